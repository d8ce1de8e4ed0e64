"""Pins for the CPU oracle: each test checks it against something other than
itself -- the pages' stated rules and worked examples (tests/golden), closed
forms, invariants, brute force on tiny inputs, Python's own sort, and an
independent Philox implementation."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from oracle import oracle as O
from spec_verification_gb300 import workloads as W
from tests.helpers import chi2_pvalue, python_order, rows, sample_case, verify_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F = W


@pytest.fixture(scope="module", autouse=True)
def _built():
    O.build()


# ----------------------------------------------------------------------------- Philox

_TRITON_PHILOX = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl

@triton.jit
def k(out_ptr, seed, c_ptr, N: tl.constexpr):
    offs = tl.arange(0, N)
    c0 = tl.load(c_ptr + offs * 4 + 0)
    c1 = tl.load(c_ptr + offs * 4 + 1)
    c2 = tl.load(c_ptr + offs * 4 + 2)
    c3 = tl.load(c_ptr + offs * 4 + 3)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out_ptr + offs * 4 + 0, a)
    tl.store(out_ptr + offs * 4 + 1, b)
    tl.store(out_ptr + offs * 4 + 2, c)
    tl.store(out_ptr + offs * 4 + 3, d)

cases = json.loads(sys.stdin.read())
res = []
for seed, ctrs in cases:
    c = torch.tensor(np.array(ctrs, dtype=np.uint32).view(np.int32).reshape(-1))
    out = torch.zeros_like(c)
    k[(1,)](out, seed, c, N=len(ctrs))
    res.append(out.numpy().view(np.uint32).reshape(-1, 4).tolist())
print(json.dumps(res))
"""


def test_philox_matches_independent_implementation():
    """Philox-4x32-10 (Salmon et al., SC'11) against Triton's implementation,
    run on the CPU by Triton's interpreter: two codes written independently."""
    pytest.importorskip("triton")
    rng = np.random.default_rng(11)
    cases = []
    for seed in [0, 1, 12345, (7 << 32) | 99, 0xFFFFFFFFFFFFFFFF, int(rng.integers(0, 2**63))]:
        ctrs = rng.integers(0, 2**32, size=(8, 4), dtype=np.uint64).astype(np.uint32)
        ctrs[0] = 0
        ctrs[1] = 0xFFFFFFFF
        cases.append([seed, ctrs.tolist()])
    env = dict(os.environ, TRITON_INTERPRET="1")
    p = subprocess.run([sys.executable, "-c", _TRITON_PHILOX], input=json.dumps(cases),
                       capture_output=True, text=True, env=env, timeout=600)
    if p.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + p.stderr[-300:])
    ref = json.loads(p.stdout.strip().splitlines()[-1])
    for (seed, ctrs), want in zip(cases, ref):
        for c, w in zip(ctrs, want):
            got = O.philox(c, seed & 0xFFFFFFFF, seed >> 32)
            assert got.tolist() == w, (seed, c)


def test_philox_words_uniform_and_uncorrelated():
    rng = np.random.default_rng(3)
    words = []
    for n in range(4000):
        words.extend(O.philox([n, 5, 7, 1], 0xDEADBEEF, 0x12345678).tolist())
    w = np.array(words, np.uint64)
    counts = np.bincount((w >> 28).astype(np.int64), minlength=16)
    assert chi2_pvalue(counts, np.full(16, 1 / 16)) > 1e-4
    u = (w.astype(np.float64) + 0.5) / 2**32
    corr = np.corrcoef(u[:-1], u[1:])[0, 1]
    assert abs(corr) < 0.02
    # counters that differ in one bit give unrelated outputs
    a = O.philox([0, 0, 0, 0], 1, 2)
    b = O.philox([1, 0, 0, 0], 1, 2)
    assert sum(bin(int(x) ^ int(y)).count("1") for x, y in zip(a, b)) > 40
    del rng


def test_uniform_is_odd_multiple_of_2pow_minus24():
    for i in range(200):
        u = O.uniform(99, i, 3, 7, i % 3)
        m = u * 2**24
        assert 0.0 < u < 1.0
        assert m == int(m) and int(m) % 2 == 1
    # word i%4 of counter floor(i/4)
    ctr = O.philox([2, 3, 7, 0], 99, 0)
    for j in range(4):
        assert O.uniform(99, 8 + j, 3, 7, 0) == ((int(ctr[j]) >> 9) * 2 + 1) / 2**24


# ----------------------------------------------------------------------------- prelude

def _processed(w, r=0, pos=0, extra=()):
    return O.prelude(w, r, pos, extra)


def test_prelude_identity_and_bf16_exact():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((1, 500)).astype(np.float32) * 3
    for dtype in ("f32", "bf16"):
        w = sample_case(x, flags=F.GREEDY, dtype=dtype)
        got, st = _processed(w)
        want = x[0] if dtype == "f32" else W.bf16_bits_to_f32(W.f32_to_bf16_bits(x))[0]
        assert st == 0
        np.testing.assert_array_equal(got, want)


def test_prelude_mask_bit_layout():
    rng = np.random.default_rng(1)
    V = 100
    x = rng.standard_normal((1, V)).astype(np.float32)
    allowed = rng.random(V) < 0.4
    # build words by hand: element i -> bit i%32 of word i//32
    words = np.zeros((1, 4), np.uint32)
    for i in np.nonzero(allowed)[0]:
        words[0, i // 32] |= np.uint32(1 << (i % 32))
    w = sample_case(x, flags=F.GREEDY | F.MASK, bitmask=words)
    got, _ = _processed(w)
    np.testing.assert_array_equal(got[allowed], x[0][allowed])
    assert np.all(np.isneginf(got[~allowed]))


def test_temperature_power_of_two_is_exact_and_order_preserving():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((1, 4096)) * 4).astype(np.float32)
    for k in (-2, -1, 0, 1, 3):
        T = np.float32(2.0 ** k)
        w = sample_case(x, flags=0, temperature=T)
        got, _ = _processed(w)
        np.testing.assert_array_equal(got, x[0] / T)   # exact: power-of-two scaling
    for T in (0.37, 0.7, 1.3, 2.9):
        w = sample_case(x, flags=0, temperature=T)
        got, _ = _processed(w)
        o = np.argsort(x[0], kind="stable")
        assert np.all(np.diff(got[o]) >= 0)            # weakly monotone (the page: T keeps order)


def test_penalties_special_cases():
    rng = np.random.default_rng(3)
    V = 64
    x = (rng.standard_normal((1, V)) * 2).astype(np.float32)
    hist = np.array([[3, 5, 5, 7, 7, 7, -1, 200]], np.int32)   # -1 padding, 200 >= V
    cnt = np.zeros(V, int)
    for t in (3, 5, 5, 7, 7, 7):
        cnt[t] += 1
    # neutral parameters -> identity
    w = sample_case(x, flags=F.GREEDY | F.PENALTY, history=hist, rep=1.0, freq=0.0, pres=0.0)
    got, st = _processed(w)
    np.testing.assert_array_equal(got, x[0])
    assert st == 4  # out-of-range history id reported
    # rep = 2 (exact halving / doubling), only where count > 0
    w = sample_case(x, flags=F.GREEDY | F.PENALTY, history=hist, rep=2.0, freq=0.0, pres=0.0)
    got, _ = _processed(w)
    for i in range(V):
        if cnt[i] == 0:
            assert got[i] == x[0, i]
        else:
            assert got[i] == (x[0, i] / 2 if x[0, i] > 0 else x[0, i] * 2)
    # frequency penalty subtracts freq per occurrence (0.25 and small ints: exact)
    xi = np.round(x * 4) / 4
    w = sample_case(xi, flags=F.GREEDY | F.PENALTY, history=hist, rep=1.0, freq=0.25, pres=0.0)
    got, _ = _processed(w)
    np.testing.assert_array_equal(got, xi[0] - 0.25 * cnt)
    # presence penalty subtracts once for present tokens
    w = sample_case(xi, flags=F.GREEDY | F.PENALTY, history=hist, rep=1.0, freq=0.0, pres=0.5)
    got, _ = _processed(w)
    np.testing.assert_array_equal(got, xi[0] - 0.5 * (cnt > 0))
    # repetition penalty > 1 never raises a present token
    w = sample_case(x, flags=F.GREEDY | F.PENALTY, history=hist, rep=1.3, freq=0.2, pres=0.3)
    got, _ = _processed(w)
    assert np.all(got[cnt > 0] < x[0][cnt > 0])


def test_bias_entries_accumulate_in_order_and_report_bad_ids():
    x = np.zeros((1, 16), np.float32)
    w = sample_case(x, flags=F.GREEDY | F.BIAS, bias_tokens=[[2, 5, 2, 99, -1]],
                    bias_values=[[0.5, -1.25, 0.25, 3.0, 7.0]])
    got, st = _processed(w)
    want = np.zeros(16, np.float32)
    want[2], want[5] = 0.75, -1.25
    np.testing.assert_array_equal(got, want)
    assert st == 8


def test_nan_becomes_neg_inf_with_status():
    x = np.array([[1.0, np.nan, 3.0, -2.0]], np.float32)
    w = sample_case(x, flags=F.GREEDY)
    got, st = _processed(w)
    assert np.isneginf(got[1]) and st == 1
    out = O.sample(w)
    assert out["tokens"][0] == 2 and out["row_status"][0] == 1


# ----------------------------------------------------------------------------- order / top-128

@pytest.mark.parametrize("V", [5, 127, 128, 129, 300])
def test_candidates_are_brute_force_order(V):
    rng = np.random.default_rng(V)
    x = np.round(rng.standard_normal((3, V)) * 3, 1).astype(np.float32)   # many ties
    x[1, ::7] = -np.inf
    x[2, 3] = -0.0
    x[2, 4] = 0.0
    w = sample_case(x, flags=F.GREEDY)
    out = O.sample(w)
    for r in range(3):
        order = python_order(x[r])
        k = min(128, V)
        assert out["cand_ids"][r, :k].tolist() == order[:k]
        assert np.all(out["cand_ids"][r, k:] == -1)
        # repeated-argmax selection, independent of any sort
        rem = list(range(V))
        sel = []
        for _ in range(k):
            best = max(rem, key=lambda i: (x[r, i], -i))
            sel.append(best)
            rem.remove(best)
        assert sel == order[:k]


def test_two_stage_decomposition_identity():
    """Every element of a row's top-128 is in its own tile's top-128 (the
    property the two-stage tile-aware top-k rests on)."""
    rng = np.random.default_rng(5)
    for trial in range(20):
        V = int(rng.integers(200, 3000))
        tile = int(rng.choice([64, 128, 256, 1000]))
        x = np.round(rng.standard_normal(V) * 2, 2).astype(np.float32)
        glob = python_order(x)[:128]
        union = set()
        for t0 in range(0, V, tile):
            sub = x[t0:t0 + tile]
            union |= {t0 + i for i in python_order(sub)[:128]}
        assert set(glob) <= union


def test_greedy_is_argmax_and_topk1_equals_greedy():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((8, 1000)) * 2).astype(np.float32)
    x[3, 10] = x[3, 20] = x[3].max() + 1   # tie -> lower index
    g = O.sample(sample_case(x, flags=F.GREEDY))
    assert g["tokens"].tolist() == [int(np.argmax(r)) for r in x]
    for seed in range(5):
        s = O.sample(sample_case(x, flags=F.TOPK, top_k=1, temperature=0.8,
                                 seeds=np.arange(8) + 100 * seed))
        assert s["tokens"].tolist() == g["tokens"].tolist()
        assert np.all(s["num_kept"] == 1)


def test_temperature_does_not_change_candidate_order():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((4, 2000)) * 2).astype(np.float32)
    base = O.sample(sample_case(x, flags=0, temperature=1.0))["cand_ids"]
    for T in (0.25, 0.5, 2.0, 8.0):
        assert np.array_equal(O.sample(sample_case(x, flags=0, temperature=T))["cand_ids"], base)


# ----------------------------------------------------------------------------- truncation

def _softmax64(l):
    m = np.max(l)
    e = np.exp(l.astype(np.float64) - m)
    return e / e.sum()


def test_golden_truncation_examples():
    for fx in json.load(open(os.path.join(GOLDEN, "truncation_examples.json"))):
        p = np.array(fx["probs"], np.float64)
        x = np.log(p).astype(np.float32)[None]
        rule = fx["rule"]
        flags, kw = 0, {}
        if "top_k" in rule:
            flags |= F.TOPK
            kw["top_k"] = rule["top_k"]
        if "top_p" in rule:
            flags |= F.TOPP
            kw["top_p"] = rule["top_p"]
        if "min_p" in rule:
            flags |= F.MINP
            kw["min_p"] = rule["min_p"]
        for exact in (False, True):
            out = O.sample(sample_case(x, flags=flags, **kw), exact=exact)
            n = int(out["num_kept"][0])
            assert sorted(out["cand_ids"][0, :n].tolist()) == fx["expected_kept_ids"], fx["name"]
            if "expected_kept_probs" in fx:
                np.testing.assert_allclose(out["cand_probs"][0, :n], fx["expected_kept_probs"],
                                           rtol=0, atol=1e-6)


def test_min_p_logit_space_equals_softmax_form():
    rng = np.random.default_rng(8)
    for trial in range(30):
        V = int(rng.integers(20, 400))
        x = (rng.standard_normal((1, V)) * rng.uniform(0.5, 3)).astype(np.float32)
        mp = float(rng.uniform(0.01, 0.9))
        out = O.sample(sample_case(x, flags=F.MINP, min_p=mp), exact=True)
        l, _ = _processed(sample_case(x, flags=F.MINP, min_p=mp))
        p = _softmax64(l)
        thr = np.float64(np.float32(mp)) * p.max()
        if np.min(np.abs(p - thr)) < 1e-12:
            continue
        assert out["num_kept"][0] == int(np.sum(p >= thr))


def test_top_p_is_smallest_prefix_reaching_p():
    rng = np.random.default_rng(9)
    for trial in range(30):
        V = int(rng.integers(10, 300))
        x = (rng.standard_normal((1, V)) * 2).astype(np.float32)
        tp = float(np.float32(rng.uniform(0.05, 0.99)))
        out = O.sample(sample_case(x, flags=F.TOPP, top_p=tp), exact=True)
        p = np.sort(_softmax64(x[0]))[::-1]
        # brute force over prefix lengths: smallest n with mass >= p
        n = next(n for n in range(1, V + 1) if p[:n].sum() >= tp or n == V)
        if abs(p[:n - 1].sum() - tp) < 1e-9 or abs(p[:n].sum() - tp) < 1e-9:
            continue
        assert out["num_kept"][0] == n
        np.testing.assert_allclose(out["cand_probs"][0, :min(n, 128)], (p[:n] / p[:n].sum())[:128],
                                   rtol=0, atol=1e-6)


def test_top_k_top_p_intersection_bruteforce():
    rng = np.random.default_rng(10)
    for trial in range(40):
        V = int(rng.integers(5, 120))
        x = (rng.standard_normal((1, V)) * 2).astype(np.float32)
        k = int(rng.integers(1, V + 1))
        tp = float(np.float32(rng.uniform(0.1, 0.99)))
        out = O.sample(sample_case(x, flags=F.TOPK | F.TOPP, top_k=k, top_p=tp))
        p = _softmax64(x[0])
        order = python_order(x[0])
        Sk = set(order[:k])
        cum, Sp = 0.0, set()
        for i in order:
            if cum >= tp:
                break
            Sp.add(i)
            cum += p[i]
        n = int(out["num_kept"][0])
        assert set(out["cand_ids"][0, :n].tolist()) == (Sk & Sp)


def test_bounded_equals_exact_when_vocab_fits():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((16, 100)) * 2).astype(np.float32)
    kw = dict(flags=F.TOPP | F.MINP, top_p=0.9, min_p=0.02, temperature=0.8)
    a = O.sample(sample_case(x, **kw))
    b = O.sample(sample_case(x, **kw), exact=True)
    for k in ("tokens", "cand_ids", "num_kept"):
        assert np.array_equal(a[k], b[k])
    np.testing.assert_allclose(a["cand_probs"], b["cand_probs"], atol=1e-7)
    assert np.all(b["mass_outside"] < 1e-12)


def test_all_masked_row():
    x = np.ones((1, 40), np.float32)
    w = sample_case(x, flags=F.MASK, bitmask=np.zeros((1, 2), np.uint32))
    out = O.sample(w)
    assert out["tokens"][0] == -1 and out["row_status"][0] == 2


def test_bad_params_rows():
    x = np.ones((4, 40), np.float32)
    w = sample_case(x, flags=F.TOPP, top_p=[0.5, 0.0, 1.5, 0.9], temperature=[1, 1, 1, -1])
    out = O.sample(w)
    assert out["row_status"].tolist() == [0, 16, 16, 16]
    assert out["tokens"].tolist()[1:] == [-1, -1, -1]


# ----------------------------------------------------------------------------- sampling statistics

def test_gumbel_sampling_follows_kept_distribution():
    """Gumbel-max (SonicSampler 3.1) samples the renormalised kept distribution."""
    rng = np.random.default_rng(13)
    V, B = 24, 40000
    x1 = (rng.standard_normal(V) * 1.2).astype(np.float32)
    x = np.repeat(x1[None], B, 0)
    w = sample_case(x, flags=F.TOPK | F.TOPP, top_k=12, top_p=0.9, temperature=0.9,
                    seeds=np.arange(B, dtype=np.uint64) * 7919 + 3)
    out = O.sample(w)
    n = int(out["num_kept"][0])
    assert np.all(out["num_kept"] == n)
    ids = out["cand_ids"][0, :n]
    probs = out["cand_probs"][0, :n].astype(np.float64)
    counts = np.array([(out["tokens"] == i).sum() for i in ids])
    assert counts.sum() == B
    assert chi2_pvalue(counts, probs / probs.sum()) > 1e-4


def _verify_stat_case(V, B, p_logits, q, gamma, flags, seed, **kw):
    rng = np.random.default_rng(seed)
    tgt = np.repeat(p_logits[None], B * (gamma + 1), 0)
    qq = np.repeat(q[None].astype(np.float32), B * gamma, 0)
    cdf = np.cumsum(q.astype(np.float64))
    d = np.minimum(np.searchsorted(cdf, rng.random(B * gamma) * cdf[-1], side="right"), V - 1)
    return verify_case(tgt, qq, d.astype(np.int32), np.full(B, gamma), flags=flags,
                       seeds=np.arange(B, dtype=np.uint64) * 104729 + seed, **kw)


@pytest.mark.parametrize("trunc", [False, True])
def test_verify_output_distributed_as_p(trunc):
    """Rejection sampling returns tokens distributed exactly as p (dl-note,
    Rejection Sampler); the acceptance rate is sum_x min(p, q)."""
    rng = np.random.default_rng(21 + trunc)
    V, B = 20, 40000
    pl = (rng.standard_normal(V) * 1.5).astype(np.float32)
    q = _softmax64((rng.standard_normal(V) * 1.5).astype(np.float32))
    flags = (F.TOPK | F.TOPP) if trunc else 0
    w = _verify_stat_case(V, B, pl, q, 1, flags, 5, top_k=10, top_p=0.95)
    out = O.verify(w)
    # p: kept distribution (truncated) or full softmax
    if trunc:
        s = O.sample(sample_case(pl[None], flags=flags, top_k=10, top_p=0.95))
        n = int(s["num_kept"][0])
        p = np.zeros(V)
        p[s["cand_ids"][0, :n]] = s["cand_probs"][0, :n]
    else:
        p = _softmax64(pl)
    first = out["tokens"][:, 0]
    counts = np.bincount(first, minlength=V)
    assert chi2_pvalue(counts, p) > 1e-4
    q32 = q.astype(np.float32).astype(np.float64)
    acc = out["num_accepted"].mean()
    want = np.minimum(p, q32).sum()
    assert abs(acc - want) < 4 * np.sqrt(want * (1 - want) / B) + 1e-3


def _one_hot(d, V):
    q = np.zeros((len(d), V), np.float32)
    q[np.arange(len(d)), d] = 1.0
    return q


@pytest.mark.parametrize("trunc", [False, True])
def test_verify_one_hot_drafts_distributed_as_p(trunc):
    """Drafts without probabilities (dl-note, Rejection Sampler, the case
    without draft probabilities): q is one-hot on the draft d, so d is kept
    with probability p(d) and a rejection draws from p without d.  Whatever
    distribution the drafts come from, the output is distributed as p and the
    acceptance rate is E[p(d)]."""
    rng = np.random.default_rng(41 + trunc)
    V, B = 20, 40000
    pl = (rng.standard_normal(V) * 1.5).astype(np.float32)
    flags = (F.TOPK | F.TOPP) if trunc else 0
    d = rng.integers(0, V, B).astype(np.int32)           # drafts from an unrelated proposal
    tgt = np.repeat(pl[None], 2 * B, 0)
    w = verify_case(tgt, _one_hot(d, V), d, np.ones(B), flags=flags, top_k=10, top_p=0.95,
                    seeds=np.arange(B, dtype=np.uint64) * 7727 + 11)
    out = O.verify(w)
    if trunc:
        s = O.sample(sample_case(pl[None], flags=flags, top_k=10, top_p=0.95))
        n = int(s["num_kept"][0])
        p = np.zeros(V)
        p[s["cand_ids"][0, :n]] = s["cand_probs"][0, :n]
    else:
        p = _softmax64(pl)
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    assert chi2_pvalue(counts, p) > 1e-4
    acc = out["num_accepted"].mean()
    want = p[d].mean()
    assert abs(acc - want) < 4 * np.sqrt(want * (1 - want) / B) + 1e-3
    # a rejection never returns the rejected draft
    rej = out["num_accepted"] == 0
    assert not np.any(out["tokens"][rej, 0] == d[rej])


def test_bounded_p_rejects_drafts_outside_the_candidates():
    """SS_BOUNDED_P: p is the softmax over the 128 candidates.  With 300 equal
    logits the candidates are tokens 0..127 (ties go to the lower index); a
    draft 200 with q = uniform is always kept under the full-vocabulary p
    (u q(d) <= p(d) = q(d)) and never under the bounded p (p(d) = 0)."""
    V, B = 300, 64
    tgt = np.zeros((2 * B, V), np.float32)
    q = np.full((B, V), 1.0 / V, np.float32)
    d = np.full(B, 200, np.int32)
    flags = np.where(np.arange(B) % 2 == 1, F.BOUNDED_P, 0).astype(np.uint32)
    w = verify_case(tgt, q, d, np.ones(B), flags=0, seeds=np.arange(B, dtype=np.uint64) + 1)
    w.rows["flags"][:] = flags
    out = O.verify(w)
    assert np.all(out["num_accepted"][0::2] == 1)
    assert np.all(out["num_accepted"][1::2] == 0)
    assert np.all(out["tokens"][1::2, 0] < 128)        # resampled among the candidates


def test_bounded_p_is_the_full_p_when_v_is_at_most_128():
    """With V <= 128 the candidates are the whole vocabulary, so the flag
    changes nothing."""
    rng = np.random.default_rng(43)
    V, B = 96, 3000
    pl = (rng.standard_normal(V) * 2).astype(np.float32)
    q = _softmax64((rng.standard_normal(V) * 2).astype(np.float32))
    w = _verify_stat_case(V, B, pl, q, 2, 0, 17)
    a = O.verify(w)
    w.rows["flags"][:] = F.BOUNDED_P
    b = O.verify(w)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    np.testing.assert_array_equal(a["num_accepted"], b["num_accepted"])


def test_exact_sampling_reaches_beyond_the_candidates():
    """SS_EXACT: an untruncated row samples by the Gumbel-max over the whole
    vocabulary, so the token follows the full softmax (Gumbel-max theorem):
    with 400 equal logits every token has probability 1/400, while the
    bounded sampler only ever returns one of the 128 candidates (0..127)."""
    V, B = 400, 40000
    x = np.zeros((B, V), np.float32)
    seeds = np.arange(B, dtype=np.uint64) * 6151 + 7
    a = O.sample(sample_case(x, flags=0, seeds=seeds))
    wb = sample_case(x, flags=F.EXACT, seeds=seeds)
    wb.meta["exact_sampling"] = True
    b = O.sample(wb)
    assert a["tokens"].max() < 128
    counts = np.bincount(b["tokens"], minlength=V)
    assert chi2_pvalue(counts, np.full(V, 1.0 / V)) > 1e-4
    assert np.all(b["row_status"] == 0)
    # truncating rows ignore the flag
    wc = sample_case(x[:2000], flags=F.EXACT | F.TOPK, top_k=50, seeds=seeds[:2000])
    wc.meta["exact_sampling"] = True
    c = O.sample(wc)
    assert c["tokens"].max() < 50
    # without exact sampling enabled: the candidates' sample and a status bit
    d = O.sample(sample_case(x[:2000], flags=F.EXACT, seeds=seeds[:2000]))
    np.testing.assert_array_equal(d["tokens"], a["tokens"][:2000])
    assert np.all(d["row_status"] == 1 << 8)


def test_exact_sampling_equals_bounded_when_v_is_at_most_128():
    rng = np.random.default_rng(44)
    V, B = 100, 2000
    x = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    seeds = np.arange(B, dtype=np.uint64) + 3
    a = O.sample(sample_case(x, flags=0, seeds=seeds))
    wb = sample_case(x, flags=F.EXACT, seeds=seeds)
    wb.meta["exact_sampling"] = True
    b = O.sample(wb)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])


def test_golden_rejection_closed_forms():
    fx = json.load(open(os.path.join(GOLDEN, "rejection_examples.json")))[0]
    p = np.array(fx["p"])
    q = np.array(fx["q"])
    V, B = p.size, 60000
    w = _verify_stat_case(V, B, np.log(p).astype(np.float32), q, 1, 0, 9)
    out = O.verify(w)
    acc = out["num_accepted"] == 1
    assert abs(acc.mean() - fx["expected_accept_rate"]) < 0.01
    d = w.draft_ids
    joint = np.array([np.mean(acc & (d == x)) for x in range(V)])
    np.testing.assert_allclose(joint, fx["expected_accept_joint"], atol=0.01)
    assert abs((~acc).mean() - fx["expected_reject_rate"]) < 0.01
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    assert chi2_pvalue(counts, p) > 1e-4


def test_verify_greedy_rows_and_bonus():
    rng = np.random.default_rng(30)
    V = 50
    tgt = (rng.standard_normal((3 * 4, V)) * 2).astype(np.float32)
    am = tgt.argmax(1)
    # row 0: all drafts = argmax -> bonus; row 1: second draft wrong; row 2: gamma 0
    gam = [3, 3, 0]
    cu = [0, 3, 6]
    pos0 = [0, 4, 8]
    d = np.array([am[0], am[1], am[2], am[4], (am[5] + 1) % V, am[6]], np.int32)
    tgt = tgt[:3 + 1 + 3 + 1 + 1]
    q = np.full((6, V), 1.0 / V, np.float32)
    w = verify_case(tgt, q, d, gam, flags=F.GREEDY)
    out = O.verify(w)
    assert out["num_accepted"].tolist() == [3, 1, 0]
    assert out["tokens"][0].tolist() == [am[0], am[1], am[2], am[3]]
    assert out["tokens"][1].tolist() == [am[4], am[5], -1, -1]
    assert out["tokens"][2].tolist() == [am[8], -1, -1, -1]
    del cu, pos0


def test_verify_zero_target_prob_rejects_and_zero_q_accepts():
    V = 8
    pl = np.log(np.array([0.5, 0.3, 0.2, 0, 0, 0, 0, 0]) + 1e-300).astype(np.float32)
    pl[3:] = -np.inf
    q = np.array([[0.0, 0.5, 0.0, 0.5, 0, 0, 0, 0]] * 2, np.float32)
    # row 0 draft 3 (p = 0): always rejected; row 1 draft 0 with q(d) = 0 and p(d) > 0: accepted
    w = verify_case(np.stack([pl, pl, pl, pl]), q, [3, 0], [1, 1])
    out = O.verify(w)
    assert out["num_accepted"].tolist() == [0, 1]
    assert out["tokens"][0, 0] in (0, 2)   # residual max(0, p - q) has mass on 0 and 2 only


def test_mass_outside_top128_report():
    c = W.topk_stress_workload(3, 4, 8192)
    out = O.sample(c, exact=True)
    m = out["mass_outside"]
    assert m[0] < 0.5 and m[1] < 0.5          # boosted rows: most mass inside
    assert m[2] > 0.9 and m[3] > 0.9          # near-flat rows: nearly all mass outside


def test_oracle_calls_are_independent_across_threads():
    """The all-cores CPU baseline calls the oracle from several threads at
    once: each call must give what it gives alone."""
    import concurrent.futures as cf
    w = W.mixed_workload(45, 12, 20000, "f32")
    subs = [W.subset(w, [r]) for r in range(w.B)]
    serial = [O.verify(s) for s in subs]
    with cf.ThreadPoolExecutor(max_workers=6) as ex:
        par = list(ex.map(O.verify, subs))
    for a, b in zip(serial, par):
        for k in ("tokens", "num_accepted", "row_status", "cand_ids", "cand_probs", "num_kept"):
            assert np.array_equal(a[k], b[k]), k


def test_packed16_staging_report():
    """The 16-bit-key report's full-precision side is the oracle's candidate
    set; its packed side loses exactly the two things a 16-bit key beside a
    tile-local index drops: mantissa bits below bf16 and the global token
    order among equal keys in different tiles."""
    from tests import key16_report as R
    w = W.topk_stress_workload(3, 4, 40000)
    out = O.sample(w)
    for r in range(w.B):
        assert R.full_key_set(R.position_logits(w, r)) == set(out["cand_ids"][r].tolist())
    # distinct bf16 values: the 16-bit keys are the full keys, so both sets agree
    bits = np.random.default_rng(0).permutation(np.arange(0x3F80, 0x3F80 + 2 * R.TILE)).astype(np.uint16)
    x = W.bf16_bits_to_f32(bits)
    assert R.packed16_set(x) == R.full_key_set(x)
    # precision: 1 + 2^-10 rounds into 1's 16-bit key, so the lower token wins
    x = np.full(R.TILE, -10.0, np.float32)
    x[:R.K - 1] = 5.0
    x[200], x[300] = 1.0, 1.0 + 2.0 ** -10
    assert 300 in R.full_key_set(x) and 200 in R.packed16_set(x)
    assert R.full_key_set(x) - R.packed16_set(x) == {300}
    # equal values in two tiles: the tile-local index decides, not the token
    x = np.full(2 * R.TILE, -10.0, np.float32)
    x[100:100 + R.K - 1] = 5.0
    x[5], x[R.TILE + 3] = 1.0, 1.0
    assert R.full_key_set(x) - R.packed16_set(x) == {5}
    assert R.packed16_set(x) - R.full_key_set(x) == {R.TILE + 3}


def test_config1_reference_behaviour():
    c = W.config1()
    out = O.sample(c)
    x = c.logits
    assert out["tokens"][0] == int(np.argmax(x[0])) and out["tokens"][1] == int(np.argmax(x[1]))
    assert np.all(out["num_kept"][2:] <= 50)
    assert np.all(out["row_status"] == 0)


# ----------------------------------------------------------------------------- temperature as division

def _nearest_f32(num):
    """The fp32 value nearest to the rational `num` (ties to the even
    significand), found from the exact rational by bracketing, independent of
    any floating-point division."""
    from fractions import Fraction
    limit = Fraction(2 ** 128) - Fraction(2 ** 103)   # FLT_MAX + half an ulp: rounds to infinity
    if abs(num) >= limit:
        return np.float32(np.inf) if num > 0 else np.float32(-np.inf)
    f = np.float32(float(num))          # within an ulp or two of the answer
    cands = [f]
    for _ in range(3):
        cands.append(np.nextafter(cands[-1], np.float32(np.inf)))
    g = f
    for _ in range(3):
        g = np.nextafter(g, np.float32(-np.inf))
        cands.append(g)
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - num),
                                     int(np.array(c, np.float32).view(np.uint32)) & 1))
    return best


def test_temperature_is_one_correctly_rounded_division():
    """dl-note, Temperature: the processed logit is z / T.  Each processed
    value must be the fp32 number nearest the exact quotient (IEEE division,
    round to nearest even), checked with exact rational arithmetic; the
    reciprocal form z * RN(1/T) is a different function and is caught."""
    from fractions import Fraction
    rng = np.random.default_rng(71)
    x = np.concatenate([rng.standard_normal(600) * 4, rng.standard_normal(100) * 1e-3,
                        [0.0, -0.0, 1e-38, -3e38, 7.0, -np.inf]]).astype(np.float32)[None]
    differs = 0
    for T in (0.37, 0.7, 1.3, 2.9, 0.5123):
        T32 = np.float32(T)
        got, _ = _processed(sample_case(x, flags=0, temperature=T32))
        with np.errstate(over="ignore"):
            recip = (x[0] * np.float32(np.float32(1.0) / T32)).astype(np.float32)
        for i, v in enumerate(x[0]):
            if not np.isfinite(v):
                assert got[i] == v
                continue
            want = _nearest_f32(Fraction(float(v)) / Fraction(float(T32)))
            assert got[i] == want, (T, i, v, got[i], want)
        differs += int(np.sum(recip != got))
    assert differs > 0


# ----------------------------------------------------------------------------- margins (parity diagnostics)

def _g32(seed, i, position, row, purpose):
    """Gumbel noise -ln(-ln u) from the pinned uniform, in fp32 steps."""
    u = np.float32(O.uniform(seed, i, position, row, purpose))
    return np.float32(-np.log(np.float32(-np.log(u))))


def test_margin_gumbel_is_relative_gap_of_the_two_best_scores():
    """The Gumbel-argmax margin is (s_1 - s_2) / |s_1| for the two best
    perturbed scores s = l + g: build rows whose two best scores are a chosen
    gap apart and check the reported margin and the winner."""
    seed = 12345
    g = [_g32(seed, i, 0, 0, 0) for i in range(3)]
    for gap in (3e-6, 2e-4, 0.5):
        l = np.zeros((1, 3), np.float32)
        l[0, 0] = np.float32(2.0) - g[0]
        l[0, 1] = np.float32(2.0 + gap) - g[1]
        l[0, 2] = np.float32(-30.0)
        w = sample_case(l, flags=0, seeds=[seed])
        out = O.sample(w)
        s = np.array([np.float32(l[0, i] + g[i]) for i in range(3)], np.float64)
        order = np.argsort(-s, kind="stable")
        want = (s[order[0]] - s[order[1]]) / abs(s[order[0]])
        assert int(out["tokens"][0]) == int(order[0])
        np.testing.assert_allclose(out["margin_gumbel"][0], want, rtol=1e-3)
        assert 0.5 * gap / 2.0 < out["margin_gumbel"][0] < 2.0 * gap / 2.0
    # one kept token (top-k = 1) and greedy rows decide nothing by noise
    x = np.array([[1.0, 0.5, 0.25]], np.float32)
    assert np.isinf(O.sample(sample_case(x, flags=F.TOPK, top_k=1))["margin_gumbel"][0])
    assert np.isinf(O.sample(sample_case(x, flags=F.GREEDY))["margin_gumbel"][0])


def test_margin_topp_is_distance_of_cumulative_mass_to_top_p():
    """The top-p margin is the smallest |mass before t - top_p| over the
    candidates (and the full mass): a top_p placed 1e-7 above and below the
    mass of the first two tokens gives that distance and keeps 3 or 2."""
    l = np.log(np.array([0.5, 0.3, 0.2])).astype(np.float32)[None]
    p = _softmax64(l[0])
    c2 = p[0] + p[1]
    for delta, keep in ((1e-7, 3), (-1e-7, 2)):
        tp = np.float32(c2 + delta)
        out = O.sample(sample_case(l, flags=F.TOPP, top_p=tp))
        cums = [0.0, p[0], c2, 1.0]
        want = min(abs(c - float(tp)) for c in cums)
        np.testing.assert_allclose(out["margin_topp"][0], want, rtol=1e-6)
        assert 3e-8 < out["margin_topp"][0] < 2e-7
        assert int(out["num_kept"][0]) == keep
    assert np.isinf(O.sample(sample_case(l, flags=0))["margin_topp"][0])


def test_margin_minp_is_distance_to_log_min_p():
    """The min-p margin is the smallest |(l_t - l_0) - ln(min_p)| over finite
    candidates (logit-space rule)."""
    l = np.array([[0.0, -1.0, -2.3, -np.inf]], np.float32)
    for mp, keep in ((0.1003, 2), (0.1002, 3)):
        mp32 = np.float32(mp)
        out = O.sample(sample_case(l, flags=F.MINP, min_p=mp32))
        thr = np.log(np.float64(mp32))
        want = min(abs(float(v) - thr) for v in l[0] if np.isfinite(v))
        np.testing.assert_allclose(out["margin_minp"][0], want, rtol=1e-9)
        assert int(out["num_kept"][0]) == keep


def test_margin_accept_is_relative_distance_of_u_q_to_p():
    """Verification margin |fp32(u q(d)) - p(d)| / p(d), with u the pinned
    acceptance uniform; q(d) is set so that u q(d) lands a chosen relative
    distance from p(d), on both sides of the accept rule."""
    V = 4
    l = np.array([0.7, 0.1, -0.4, -1.0], np.float32)
    p = _softmax64(l)
    seed, d = 777, 1
    u = np.float32(O.uniform(seed, 0, 0, 0, 1))
    for rel, acc in ((3e-4, 0), (-3e-4, 1)):
        qd = np.float32(p[d] * (1 + rel) / float(u))
        q = np.full((1, V), (1 - float(qd)) / (V - 1), np.float32)
        q[0, d] = qd
        w = verify_case(np.stack([l, l]), q, [d], [1], seeds=[seed])
        out = O.verify(w)
        prod = float(np.float32(u * qd))
        want = abs(prod - p[d]) / p[d]
        np.testing.assert_allclose(out["margin_accept"][0], want, rtol=1e-6)
        assert 1e-4 < out["margin_accept"][0] < 1e-3
        assert int(out["num_accepted"][0]) == acc
        np.testing.assert_allclose(out["p_draft"][0], p[d], rtol=1e-12)


def test_margin_resid_is_relative_gap_of_residual_scores():
    """After a rejection the residual token is the argmax of ln r_i + g_i
    (purpose 2) over r_i = max(0, p_i - q_i) > 0; the margin is the relative
    gap of its two best scores."""
    V = 4
    l = np.array([1.0, 0.9, -3.0, -3.0], np.float32)
    p = _softmax64(l)
    seed = 4242
    q = np.array([[0.0, 0.0, 0.5, 0.5]], np.float32)  # draft 2: p(2) small, u q(2) > p(2) -> reject
    w = verify_case(np.stack([l, l]), q, [2], [1], seeds=[seed])
    u = np.float32(O.uniform(seed, 0, 0, 0, 1))
    assert float(np.float32(u * np.float32(0.5))) > p[2]
    out = O.verify(w)
    assert int(out["num_accepted"][0]) == 0
    r = np.maximum(0.0, p - q[0].astype(np.float64))
    s = {i: np.float32(np.log(np.float32(r[i])) + _g32(seed, i, 0, 0, 2)) for i in range(V) if r[i] > 0}
    best = sorted(s.items(), key=lambda kv: (-float(kv[1]), kv[0]))
    assert int(out["tokens"][0, 0]) == best[0][0]
    want = (float(best[0][1]) - float(best[1][1])) / abs(float(best[0][1]))
    np.testing.assert_allclose(out["margin_resid"][0], want, rtol=1e-3)


# ----------------------------------------------------------------------------- empty residual

def test_empty_residual_draws_from_p_with_status():
    """q >= p everywhere (a bf16-rounded q can sum above 1): max(0, p - q) has
    no mass, so a rejection draws from p itself and reports the empty
    residual.  Acceptance is min(1, p(d)/q(d)) = 0.8 for q = 1.25 p, and the
    rejected rows' tokens are distributed as p."""
    rng = np.random.default_rng(91)
    V, B = 6, 30000
    l = (rng.standard_normal(V) * 1.2).astype(np.float32)
    p = _softmax64(l)
    q = (1.25 * p).astype(np.float32)
    assert np.all(q.astype(np.float64) > p)
    w = _verify_stat_case(V, B, l, q, 1, 0, 13)
    out = O.verify(w)
    rej = out["num_accepted"] == 0
    st = out["row_status"]
    assert np.all((st[rej] & (1 << 7)) != 0) and np.all((st[~rej] & (1 << 7)) == 0)
    acc = 1.0 - rej.mean()
    assert abs(acc - 0.8) < 4 * np.sqrt(0.16 / B)
    counts = np.bincount(out["tokens"][rej, 0], minlength=V)
    assert chi2_pvalue(counts, p) > 1e-4


# ----------------------------------------------------------------------------- outside-128 mass, closed form

def test_mass_outside_closed_forms():
    """1 - (full-softmax mass of the 128 candidates), against closed forms:
    128 tokens at logit 0 and V - 128 at ln(eps) leave (V-128) eps / (128 +
    (V-128) eps) outside; 300 equal logits leave 172/300."""
    V = 1000
    a = np.float32(np.log(1e-3))
    x = np.full((1, V), a, np.float32)
    x[0, 300:428] = 0.0
    out = O.sample(sample_case(x, flags=0), exact=True)
    e = np.exp(np.float64(a))
    want = (V - 128) * e / (128 + (V - 128) * e)
    np.testing.assert_allclose(out["mass_outside"][0], want, rtol=1e-9)
    assert sorted(out["cand_ids"][0].tolist()) == list(range(300, 428))
    out = O.sample(sample_case(np.zeros((1, 300), np.float32), flags=0), exact=True)
    np.testing.assert_allclose(out["mass_outside"][0], 172 / 300, rtol=1e-12)
