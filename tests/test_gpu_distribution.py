"""Distribution tests of the GPU path at tiny V: tokens drawn through
ss_sample and ss_verify over tens of thousands of seeds follow the
distribution the pages fix (chi-square against the oracle's candidate
probabilities, which the CPU tests pin against closed forms).

- Sampling draws from the kept, renormalised softmax (SonicSampler,
  section 3.3; dl-note "Decoding and sampling": temperature, top-k, top-p).
- Speculative verification returns tokens distributed as the target p,
  whatever the draft distribution q, provided the drafts are drawn from q
  (dl-note, "Rejection Sampler": accept when u * q(d) <= p(d), else draw
  from norm(max(0, p - q))); a one-hot q (drafts without probabilities) is
  the special case q = delta_d.

Each row of a call is the same problem with its own seed, so one call gives
N independent draws."""
import numpy as np
import pytest

from oracle import oracle as O
from spec_verification_gb300 import workloads as W
from tests.helpers import chi2_pvalue, sample_case, verify_case

pytestmark = pytest.mark.gpu

P_MIN = 1e-4  # chi-square p-value below which a histogram is rejected


def _run(w):
    from spec_verification_gb300.runner import DeviceRun
    d = DeviceRun(w)
    d()
    return d.results()


def _kept_probs(x, V, **rowkw):
    """The oracle's kept distribution (its candidate probabilities) for one
    sampling row with logits x and the given row parameters."""
    w1 = sample_case(x[None, :], **rowkw)
    o = O.sample(w1)
    p = np.zeros(V)
    ids, probs = o["cand_ids"][0], o["cand_probs"][0]
    ok = ids >= 0
    p[ids[ok]] = probs[ok]
    return p


@pytest.mark.parametrize("case", ["untruncated", "topk_topp"])
def test_sampled_tokens_follow_the_kept_softmax(case):
    V, N = 48, 40000
    rng = np.random.default_rng(101)
    x = rng.normal(0.0, 1.5, V).astype(np.float32)
    kw = dict(flags=0, temperature=0.8)
    if case == "topk_topp":
        kw = dict(flags=W.TOPK | W.TOPP, temperature=0.8, top_k=12, top_p=0.85)
    p = _kept_probs(x, V, **kw)
    assert abs(p.sum() - 1.0) < 1e-5
    if case == "topk_topp":
        assert 1 < np.count_nonzero(p) <= 12
    w = sample_case(np.tile(x, (N, 1)), seeds=np.arange(1, N + 1, dtype=np.uint64), **kw)
    g = _run(w)
    assert np.all(g["row_status"] == 0)
    counts = np.bincount(g["tokens"], minlength=V).astype(np.float64)
    assert counts[p == 0].sum() == 0          # nothing outside the kept set
    assert chi2_pvalue(counts, p) > P_MIN


def _verify_draws(x_t, q, draft_ids, seeds, **rowkw):
    """One drafted position per row (gamma = 1): target rows (position 0,
    then the bonus position) and the draft row q; returns the GPU output."""
    N, V = draft_ids.size, x_t.size
    target = np.empty((2 * N, V), np.float32)
    target[0::2] = x_t
    target[1::2] = x_t
    qs = np.zeros((N, V), np.float32) if q is None else np.tile(q, (N, 1))
    w = verify_case(target, qs, draft_ids, np.ones(N, np.int32), seeds=seeds, **rowkw)
    if q is None:
        w = W.with_one_hot_drafts(w)
    return _run(w)


@pytest.mark.parametrize("case", ["untruncated", "topk"])
def test_verified_tokens_follow_the_target(case):
    V, N = 32, 50000
    rng = np.random.default_rng(202)
    x_t = rng.normal(0.0, 1.2, V).astype(np.float32)
    zq = rng.normal(0.0, 1.2, V)
    q = np.exp(zq - zq.max())
    q = (q / q.sum()).astype(np.float32)
    kw = dict(flags=0, temperature=1.0)
    if case == "topk":
        kw = dict(flags=W.TOPK, temperature=1.0, top_k=8)
    p = _kept_probs(x_t, V, **kw)
    # drafts drawn from q (as a float64 distribution of the stored fp32 q)
    qd = q.astype(np.float64) / q.astype(np.float64).sum()
    drafts = rng.choice(V, size=N, p=qd).astype(np.int32)
    g = _verify_draws(x_t, q, drafts, np.arange(1, N + 1, dtype=np.uint64), **kw)
    assert np.all(g["row_status"] == 0)
    first = g["tokens"][:, 0]
    counts = np.bincount(first, minlength=V).astype(np.float64)
    assert counts[p == 0].sum() == 0
    assert chi2_pvalue(counts, p) > P_MIN
    # acceptance rate: sum_i min(p_i, q_i), within 5 binomial standard deviations
    acc = np.minimum(p, qd).sum()
    n_acc = int((g["num_accepted"] == 1).sum())
    assert abs(n_acc - N * acc) < 5 * np.sqrt(N * acc * (1 - acc)) + 1
    # an accepted draft is returned as itself
    assert np.all(first[g["num_accepted"] == 1] == drafts[g["num_accepted"] == 1])


def test_one_hot_drafts_give_the_target():
    """q = delta_d: accept with probability p(d), otherwise draw from p
    without d; overall the token follows p for any fixed draft."""
    V, N = 32, 50000
    rng = np.random.default_rng(303)
    x_t = rng.normal(0.0, 1.0, V).astype(np.float32)
    p = _kept_probs(x_t, V, flags=0, temperature=1.0)
    d = int(np.argsort(-p)[3])                # a mid-ranked draft
    drafts = np.full(N, d, np.int32)
    g = _verify_draws(x_t, None, drafts, np.arange(1, N + 1, dtype=np.uint64), flags=0, temperature=1.0)
    assert np.all(g["row_status"] == 0)
    counts = np.bincount(g["tokens"][:, 0], minlength=V).astype(np.float64)
    assert chi2_pvalue(counts, p) > P_MIN
    n_acc = int((g["num_accepted"] == 1).sum())
    assert abs(n_acc - N * p[d]) < 5 * np.sqrt(N * p[d] * (1 - p[d])) + 1
