"""Parity of the CUDA path (through the C ABI) with the CPU oracle on seeded
inputs that span several vocabulary tiles and a ragged last tile, plus the
edge cases of the method.  Comparison rules: tests/parity.py."""
import numpy as np
import pytest

from oracle import oracle as O
from spec_verification_gb300 import workloads as W
from tests import parity
from tests.helpers import gpu_rows_as, sample_case, subset, verify_case

pytestmark = pytest.mark.gpu
F = W


@pytest.fixture(scope="module", autouse=True)
def _env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from spec_verification_gb300 import build
    build.build()
    O.build()


def run_gpu(w, tile=0, **kw):
    from spec_verification_gb300.runner import DeviceRun
    d = DeviceRun(w, tile=tile, **kw)
    d()
    return d.results(), d


def check(w, tile=0, **kw):
    gpu, d = run_gpu(w, tile=tile, **kw)
    if w.is_verify:
        ora = O.verify(w, tokens_stride=gpu["tokens"].shape[1])
        rep = parity.compare_verify(w, gpu, ora)
    else:
        ora = O.sample(w)
        rep = parity.compare_sample(w, gpu, ora)
    assert rep.ok(), rep
    assert rep.ambiguous <= max(1, rep.checked // 200), rep
    return gpu, ora, d


# ------------------------------------------------------------------ sampling

@pytest.mark.parametrize("tile", [8192, 16384])
def test_config1_full(tile):
    check(W.config1(), tile=tile)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("tile", [8192, 16384])
def test_heterogeneous_sample_ragged(dtype, tile):
    # V = 40000: 5 tiles of 8192 (last 7232) or 3 of 16384 (last 7232); all processors
    w = W.sample_workload(21, 16, 40000, dtype)
    check(w, tile=tile)


def test_heterogeneous_sample_no_processors():
    w = W.sample_workload(22, 16, 50000, "bf16", processors=False)
    check(w)


@pytest.mark.parametrize("tile", [8192, 16384])
def test_topk_stress_small(tile):
    check(W.topk_stress_workload(23, 12, 70000), tile=tile)


def test_small_vocab_and_tiny_tiles():
    rng = np.random.default_rng(24)
    for V in (1, 2, 100, 127, 128, 129, 8192, 8193, 8320):
        x = (rng.standard_normal((6, V)) * 2).astype(np.float32)
        flags = np.array([F.GREEDY, 0, F.TOPK | F.TOPP, F.MINP, F.TOPP, F.TOPK], np.uint32)
        w = sample_case(x, flags=flags, top_k=[0, 0, 7, 0, 0, 3], top_p=[1, 1, 0.8, 1, 0.5, 1],
                        min_p=[0, 0, 0, 0.1, 0, 0], temperature=[1, 0.7, 1.3, 1, 0.9, 2])
        check(w)


def test_ties_and_constant_rows():
    V = 20000
    x = np.zeros((6, V), np.float32)
    x[1] = np.round(np.random.default_rng(1).standard_normal(V), 0)     # heavy ties
    x[2, ::3] = 1.0
    x[3] = -np.inf
    x[3, 5000] = 2.0
    x[4] = np.float32(-0.0)
    x[4, ::2] = 0.0
    x[5] = np.repeat(np.arange(V // 100, dtype=np.float32), 100)        # sorted runs
    for fl in (F.GREEDY, F.TOPP):
        w = sample_case(x, flags=fl, top_p=0.9)
        check(w)


def test_nan_inf_and_masked_rows():
    rng = np.random.default_rng(2)
    V = 30000
    x = rng.standard_normal((7, V)).astype(np.float32)
    x[0, 17] = np.nan
    x[1, :] = np.nan                       # every element NaN
    x[2, 99] = np.inf                      # +inf -> point mass
    x[3, ::5] = np.nan
    mask = W.bool_to_mask_bits(rng.random((7, V)) < 0.5)
    mask[4] = 0                            # all masked
    mask[5] = 0
    mask[5, 3] = 1 << 7                    # exactly one allowed token
    mask[6] = 0
    mask[6, ::97] = 0xFFFFFFFF             # sparse grammar: a few words allowed
    for fl in (F.MASK, F.MASK | F.GREEDY, F.MASK | F.TOPP | F.MINP):
        w = sample_case(x, flags=fl, bitmask=mask, top_p=0.7, min_p=0.05)
        check(w)


def _allowed(mask_row, tok):
    return (int(mask_row[tok >> 5]) >> (tok & 31)) & 1


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_late_stage_nan_inf_and_masked_extremes(dtype):
    # 96 rows x 13 stages is more stages than stage-1 CTAs, so segments run
    # over several stages and the stages after a segment's first are filtered
    # on raw (unmasked, untempered) maxima: values hidden by the mask, NaN and
    # inf planted past the first stage, all-negative rows and an infinite 1/T
    rng = np.random.default_rng(12)
    B, V = 96, 100003
    x = rng.normal(0.0, 1.5, (B, V)).astype(np.float32)
    mask = W.bool_to_mask_bits(rng.random((B, V)) < 0.6)
    late = np.arange(40000, V)

    def pick(r, allowed, n):
        c = [t for t in rng.permutation(late)[:4 * n + 64] if _allowed(mask[r], int(t)) == allowed]
        return np.asarray(c[:n], np.int64)

    for r in range(0, 4):                  # NaN where the mask hides it: no NaN status
        x[r, pick(r, 0, 50)] = np.nan
    for r in range(4, 6):                  # one visible NaN in a late stage
        x[r, pick(r, 1, 1)] = np.nan
    for r in range(6, 8):                  # visible +inf in a late stage: a point mass
        x[r, pick(r, 1, 1)] = np.inf
    for r in range(8, 10):                 # huge values and +inf hidden by the mask
        x[r, pick(r, 0, 20)] = 1e30
        x[r, pick(r, 0, 3)] = np.inf
    x[10:12] -= 40.0                       # every value negative
    x[12] = -np.abs(x[12]) - 0.5           # 1/T = +inf: one positive value left
    tpos = int(pick(12, 1, 1)[0])
    x[12, tpos] = 2.0
    x[13, 90000:98000] += 8.0              # the row's top values all in one late stage
    temp = np.ones(B, np.float32)
    temp[12] = np.float32(1e-40)           # subnormal, RN(1/T) = +inf
    fl = F.MASK | F.TOPK | F.TOPP | F.MINP
    w = sample_case(x, flags=fl, dtype=dtype, bitmask=mask, top_k=64, top_p=0.9, min_p=0.02,
                    temperature=temp)
    gpu, ora, _ = check(w)
    assert gpu["tokens"][12] == tpos


def test_bad_params_and_ids():
    rng = np.random.default_rng(3)
    V = 9000
    x = rng.standard_normal((6, V)).astype(np.float32)
    hist = rng.integers(0, V, (6, 40)).astype(np.int32)
    hist[1, 3] = V + 5                      # out-of-range history id
    hist[2, :10] = -1                       # padding
    btok = rng.integers(0, V, (6, 4)).astype(np.int32)
    btok[3, 1] = V                          # out-of-range bias id
    btok[4, 2] = btok[4, 0]                 # duplicate bias id (accumulates)
    bval = rng.uniform(-3, 3, (6, 4)).astype(np.float32)
    w = sample_case(x, flags=F.PENALTY | F.BIAS | F.TOPP, history=hist, bias_tokens=btok, bias_values=bval,
                    top_p=[0.9, 0.9, 0.9, 0.9, 0.9, 1.5], rep=1.2, freq=0.1, pres=0.2,
                    temperature=[1, 1, 1, 1, 1, 1])
    w.rows["temperature"][0] = -1.0         # invalid
    check(w)


def test_long_history_uses_count_tables():
    # more history / bias tokens than a segment's hash table lists (512): the
    # per-stage count tables of stage 1 handle these rows
    w = W.sample_workload(29, 8, 60000, "f32", H=1500, NB=24)
    assert int(w.rows["hist_len"].max()) > 512
    check(w)


def test_ascending_rows_overflow_into_exact_fallback():
    # logits rising along the row: every stage lifts a crowd of elements over
    # the running cut, the append buffer overflows and the stage is replaced
    # by its exact top-128
    # (48 rows x 16 tiles: more tiles than stage-1 CTAs, so segments span
    # several tiles and the later ones overflow)
    rng = np.random.default_rng(31)
    B, V = 48, 131072
    x = (np.linspace(-6.0, 6.0, V, dtype=np.float32)[None, :]
         + rng.standard_normal((B, V)).astype(np.float32) * np.float32(1e-3))
    w = sample_case(x, flags=F.TOPP, top_p=0.9, temperature=[1.0] * B)
    _, _, d = check(w)
    assert d.diag()[0] > 0


def test_starting_cut_fallback_on_listed_maxima():
    # every thread's largest element of the first fp32 tile is a history
    # token with a large presence penalty (thread t holds tokens 4t .. 4t + 3
    # of each 1024-token block, so tokens 4t + 3 give each of the 256 threads
    # one): the starting cut from the thread maxima is met by no unlisted
    # element, so the first stage is replaced by its exact top-128
    V = 20000
    x = np.full((2, V), -5.0, np.float32)
    x[:, 9000] = -4.0
    hot = np.arange(256) * 4 + 3
    x[:, hot] = 10.0
    hist = np.tile(hot.astype(np.int32), (2, 1))
    w = sample_case(x, flags=F.PENALTY, history=hist, rep=1.0, freq=0.0, pres=100.0,
                    temperature=[1.0, 0.7])
    _, _, d = check(w)
    assert d.diag()[0] > 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_listed_tokens_above_the_cut_in_later_stages(dtype):
    # 48 rows x 16 tiles: segments of 3 stages, so most listed tokens are met
    # by the streaming loop of a later stage.  400 history tokens and 16
    # bias tokens per row carry the largest raw logits of the row but large
    # penalties / negative bias (their processed values fall far below the
    # top-128), and 8 more bias tokens are lifted into it: each hit on a
    # listed token must be recognised (the thread's filter bit, then the
    # table) and left to its exact value, or it would enter a list twice.
    rng = np.random.default_rng(33)
    B, V = 48, 131072
    x = rng.standard_normal((B, V)).astype(np.float32)
    hist = np.stack([rng.choice(V, 400, replace=False) for _ in range(B)]).astype(np.int32)
    neg = np.stack([rng.choice(np.setdiff1d(np.arange(V), h), 24, replace=False) for h in hist]).astype(np.int32)
    rows = np.arange(B)[:, None]
    x[rows, hist] = 8.0
    x[rows, neg[:, :16]] = 7.0
    x[rows, neg[:, 16:]] = 0.0
    bval = np.concatenate([np.full((B, 16), -50.0, np.float32), np.full((B, 8), 20.0, np.float32)], axis=1)
    w = sample_case(x, flags=F.PENALTY | F.BIAS | F.TOPK, dtype=dtype, history=hist, bias_tokens=neg,
                    bias_values=bval, rep=1.0, freq=0.0, pres=100.0, top_k=[16] * B,
                    temperature=[1.0, 0.8] * (B // 2))
    gpu, ora, _ = check(w)
    # the lifted bias tokens lead every row, no penalised or lowered one is a candidate
    for r in range(B):
        assert set(gpu["cand_ids"][r][:8].tolist()) == set(neg[r, 16:].tolist())
        assert not (set(gpu["cand_ids"][r].tolist()) & (set(hist[r].tolist()) | set(neg[r, :16].tolist())))


def test_deterministic_repeat():
    w = W.sample_workload(25, 8, 60000, "bf16")
    from spec_verification_gb300.runner import DeviceRun
    d = DeviceRun(w)
    d()
    a = d.results()
    d()
    b = d.results()
    for k in a:
        assert np.array_equal(a[k], b[k]), k


# ------------------------------------------------------------------ verification

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_untruncated(dtype):
    # config-4 style: no truncation, T = 1, 25% greedy; residual passes over V
    w = W.verify_workload(31, 12, 30000, np.full(12, 3), dtype, dtype, noise=3.0)
    gpu, ora, d = check(w)
    stochastic = (w.rows["flags"] & F.GREEDY) == 0
    assert np.any(ora["num_accepted"][stochastic] < 3)   # rejections -> residual passes over V
    assert d.diag()[2] > 0


def test_verify_mixed_processors():
    w = W.mixed_workload(32, 24, 50000, "f32")
    check(w)


@pytest.mark.parametrize("tile", [8192, 16384])
def test_verify_truncated_bf16(tile):
    w = W.verify_workload(33, 10, 40000, [1, 2, 3, 4, 0, 5, 6, 7, 2, 1], "bf16", "bf16",
                          processors=True, truncation=True)
    check(w, tile=tile)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_one_hot_drafts(dtype):
    # drafts without probabilities: the library gets draft_probs = NULL and the
    # oracle the equivalent one-hot q; truncated, untruncated (residual passes
    # over V with q one-hot) and greedy rows, processors on
    w = W.verify_workload(34, 16, 40000, [1, 2, 3, 4, 0, 5, 6, 7, 2, 1, 3, 3, 2, 4, 1, 0], dtype, dtype,
                          processors=True, truncation=True, noise=2.0)
    d = w.draft_ids
    q = np.zeros((d.size, w.V), np.float32)
    q[np.arange(d.size), d] = 1.0
    w.draft_probs = W.f32_to_bf16_bits(q) if dtype == "bf16" else q
    # half of the stochastic rows without truncation, so that rejections there
    # take the pass over the vocabulary
    untr = (np.arange(w.B) % 2 == 0) & ((w.rows["flags"] & F.GREEDY) == 0)
    w.rows["flags"][untr] &= ~np.uint32(F.TOPK | F.TOPP | F.MINP)
    gpu, ora, dev = check(w, one_hot_drafts=True)
    assert np.any(ora["num_accepted"] < np.diff(w.cu_draft))   # some rejections
    assert dev.diag()[2] > 0                                    # residual passes with q one-hot


def test_verify_bounded_p_rows():
    # untruncated stochastic rows, half of them flagged SS_BOUNDED_P (candidate
    # softmax, no pass over the vocabulary)
    w = W.verify_workload(35, 12, 30000, np.full(12, 3), "bf16", "bf16", noise=3.0)
    stoch = (w.rows["flags"] & F.GREEDY) == 0
    w.rows["flags"][stoch & (np.arange(w.B) % 2 == 1)] |= np.uint32(F.BOUNDED_P)
    gpu, ora, dev = check(w)
    assert np.any(ora["num_accepted"][stoch] < 3)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_exact_sampling(dtype):
    # SS_EXACT on untruncated stochastic rows (sample positions): the
    # Gumbel-max over the whole vocabulary, with processors on (listed tokens
    # through the count tables), ragged last tile, greedy and truncated rows
    # beside them
    w = W.sample_workload(seed=36, B=40, V=50003, dtype=dtype, name="exact")
    stoch = (w.rows["flags"] & F.GREEDY) == 0
    untr = stoch & (np.arange(w.B) % 3 != 0)
    w.rows["flags"][untr] &= ~np.uint32(F.TOPK | F.TOPP | F.MINP)
    w.rows["flags"][stoch] |= np.uint32(F.EXACT)
    w.meta["exact_sampling"] = True
    gpu, ora, _ = check(w)
    # some exact samples fall outside the 128 candidates
    outside = [r for r in np.where(untr)[0] if gpu["tokens"][r] not in set(gpu["cand_ids"][r])]
    assert len(outside) >= 1


def test_exact_sampling_verify_bonus():
    # the bonus token of a verify row flagged SS_EXACT
    w = W.verify_workload(37, 16, 30000, [0, 1, 0, 2, 0, 0, 1, 0, 3, 0, 0, 1, 0, 0, 2, 0], "bf16", "bf16",
                          processors=True, noise=0.2)
    stoch = (w.rows["flags"] & F.GREEDY) == 0
    w.rows["flags"][stoch] &= ~np.uint32(F.TOPK | F.TOPP | F.MINP)
    w.rows["flags"][stoch] |= np.uint32(F.EXACT)
    w.meta["exact_sampling"] = True
    check(w)


def test_exact_flag_without_exact_plan():
    # SS_EXACT on a plan without exact sampling: candidates' sample, status bit
    w = W.sample_workload(seed=38, B=24, V=30000, dtype="bf16", name="notexact")
    stoch = (w.rows["flags"] & F.GREEDY) == 0
    w.rows["flags"][stoch] &= ~np.uint32(F.TOPK | F.TOPP | F.MINP)
    w.rows["flags"][stoch] |= np.uint32(F.EXACT)
    gpu, ora, _ = check(w)
    assert np.all((gpu["row_status"][stoch] & (1 << 8)) != 0)


def test_verify_edge_cases():
    rng = np.random.default_rng(34)
    V = 9000
    gam = np.array([2, 2, 1, 0, 3])
    npos = gam.sum() + len(gam)
    tgt = rng.standard_normal((npos, V)).astype(np.float32) * 2
    q = np.abs(rng.standard_normal((gam.sum(), V))).astype(np.float32)
    q /= q.sum(1, keepdims=True)
    d = rng.integers(0, V, gam.sum()).astype(np.int32)
    d[0] = -3                      # out-of-range draft id
    d[3] = int(np.argmax(tgt[3]))  # row 1, draft 1
    q[4, :] = 0.0                  # row 2: q(d) = 0 -> accepted when p(d) > 0
    tgt[5:7, :] = -np.inf          # row 2 positions: no finite logits at all
    w = verify_case(tgt, q, d, gam, flags=[0, F.GREEDY, F.TOPP, 0, F.TOPK], top_p=0.8, top_k=5)
    check(w)


def test_verify_beyond_max_positions():
    """cu_draft[B] + B is device data and may exceed the plan's max_positions:
    the rows whose positions all fit are verified as usual, the others report
    SS_ST_CAPACITY with no tokens, and the workspace counters stay clean for
    the next call on the same workspace."""
    from spec_verification_gb300 import native
    from spec_verification_gb300.runner import DeviceRun
    # positions: row 0 0-2, row 1 3-4, row 2 5-8, row 3 9-11, row 4 12, row 5 13-14
    w = W.verify_workload(44, 6, 20000, [2, 1, 3, 2, 0, 1], dtype="f32", q_dtype="f32", truncation=True)
    cap = 10  # row 3 straddles the bound: its position 9 is evaluated, 10 and 11 are not
    d = DeviceRun(w, max_positions=cap)
    d()
    gpu = d.results()
    fit = [0, 1, 2]
    sub = subset(w, fit)
    g = gpu_rows_as(gpu, w, fit)
    rep = parity.compare_verify(sub, g, O.verify(sub, tokens_stride=gpu["tokens"].shape[1]))
    assert rep.ok(), rep
    for r in (3, 4, 5):
        assert gpu["row_status"][r] == native.ST_CAPACITY
        assert gpu["num_accepted"][r] == 0 and np.all(gpu["tokens"][r] == -1)
    # the same plan and workspace for a batch that fits, whose row 3 is the
    # straddling row above: a counter left behind would break its walk
    w2 = subset(w, [0, 1, 4, 3])
    w2.meta.pop("row_ids")  # a batch of its own: random streams keyed by its own rows
    d2 = DeviceRun(w2, max_positions=cap)
    d2.plan, d2.workspace = d.plan, d.workspace
    for _ in range(2):
        d2()
        gpu2 = d2.results()
        rep = parity.compare_verify(w2, gpu2, O.verify(w2, tokens_stride=gpu2["tokens"].shape[1]))
        assert rep.ok(), rep
        assert not np.any(gpu2["row_status"] & native.ST_CAPACITY)


# ------------------------------------------------------------------ full-size workloads (every row)

def _oracle_chunks(w, gpu, n_chunks=16):
    """The oracle on every row of w, in row chunks run on host threads (each
    a workload of its own; ctypes releases the GIL), compared chunk by chunk
    with the GPU's rows.  Returns the merged report."""
    import concurrent.futures as cf
    chunks = [c for c in np.array_split(np.arange(w.B), n_chunks) if c.size]

    def one(rs):
        sub = subset(w, rs)
        g = gpu_rows_as(gpu, w, rs)
        if w.is_verify:
            return parity.compare_verify(sub, g, O.verify(sub, tokens_stride=gpu["tokens"].shape[1]))
        return parity.compare_sample(sub, g, O.sample(sub))

    O.lib()
    with cf.ThreadPoolExecutor(max_workers=min(16, len(chunks))) as ex:
        reps = list(ex.map(one, chunks))
    rep = parity.Report()
    for r in reps:
        rep.checked += r.checked
        rep.ambiguous += r.ambiguous
        rep.errors += r.errors
    return rep


def _full(w, tile=0):
    gpu, d = run_gpu(w, tile=tile)
    rep = _oracle_chunks(w, gpu)
    assert rep.ok(), rep
    assert rep.ambiguous <= max(1, rep.checked // 200), rep
    return rep, d


def test_config2_full():
    _full(W.config2())


def test_config3_full():
    _full(W.config3())


def test_config4_full():
    _full(W.config4())


def test_config5_full():
    rep, d = _full(W.config5())
    assert d.diag()[3] == 0


def test_config4_one_hot_full():
    # drafts without probabilities reject often: more queued residual entries
    # than one round of 2048-token pieces covers, so the pass over the
    # vocabulary takes longer pieces (streamed 2048 tokens at a time)
    from spec_verification_gb300.runner import DeviceRun
    w = W.with_one_hot_drafts(W.config4())
    d = DeviceRun(w, candidates=True)
    d()
    rep = _oracle_chunks(w, d.results())
    assert rep.ok(), rep
    assert rep.ambiguous <= max(1, rep.checked // 200), rep
    # more entries than the 608 pass CTAs cover in one round of 64 pieces each
    assert d.diag()[2] > 608 // 64, d.diag()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_low_noise_residual(dtype):
    """Untruncated stochastic rows whose target is the draft plus N(0, 0.02)
    noise: p and q nearly cancel, so the residual max(0, p - q) is a field of
    small differences, the numerically fragile case of the pass over the
    vocabulary (dl-note, Rejection Sampler).  Such drafts are rarely
    rejected, so each row's seed is picked (from the pinned acceptance
    uniform and the oracle's p(d)) to reject its first draft."""
    w = W.verify_workload(36, 24, 131072, np.full(24, 4), dtype, "f32", noise=0.02)
    w.rows["flags"][:] &= ~np.uint32(F.GREEDY)     # every row stochastic, untruncated
    q = np.asarray(w.draft_probs, np.float32)
    offs = w.position_offsets()
    # a first draft d with p(d) >= q(d) is always accepted: move it to the
    # next most likely token under q until p(d) < q(d) (p at a row's first
    # position does not depend on the drafts)
    tries = np.zeros(w.B, np.int64)
    for _ in range(64):
        ora = O.verify(w)
        todo = []
        for r in range(w.B):
            j0 = int(w.cu_draft[r])
            qd = float(np.float32(q[j0, int(w.draft_ids[j0])]))
            if float(ora["p_draft"][int(offs[r])]) * (1 + 1e-3) >= qd:
                todo.append(r)
        if not todo:
            break
        for r in todo:
            j0 = int(w.cu_draft[r])
            w.draft_ids[j0] = int(np.argsort(-q[j0], kind="stable")[tries[r]])
            tries[r] += 1
    else:
        pytest.fail("no first draft with p(d) < q(d)")
    for r in range(w.B):
        j0 = int(w.cu_draft[r])
        qd = np.float32(q[j0, int(w.draft_ids[j0])])
        pd = float(ora["p_draft"][int(offs[r])])
        for seed in range(1, 200000):
            u = np.float32(O.uniform(seed, 0, int(w.rows["position"][r]), r, 1))
            if float(np.float32(u * qd)) > pd * (1 + 1e-4):
                w.seeds[r] = np.uint64(seed)
                break
        else:
            pytest.fail(f"no rejecting seed for row {r}")
    gpu, d = run_gpu(w)
    rep = _oracle_chunks(w, gpu, n_chunks=8)
    assert rep.ok(), rep
    assert rep.ambiguous <= max(1, rep.checked // 50), rep
    assert np.all(gpu["num_accepted"] == 0)
    assert d.diag()[2] >= w.B                        # every row drew from the residual over V


def test_copy_wait_limit_gives_up_cleanly():
    """A stage-1 wait limit of one poll that does not suspend, on rows whose
    parameters are invalid (temperature -1): stage 1 then does no work per
    stage but wait for its copies, so its waits give up while the copies are
    still in flight.  The CTAs let the copies land, their rows report
    SS_ST_COPY_TIMEOUT, diagnostic counter 3 counts them, and the next call on
    the same plan and workspace, with valid rows and the default limit, is
    exact."""
    import torch
    from spec_verification_gb300 import native
    from spec_verification_gb300.runner import DeviceRun, pack_rows
    w = W.topk_stress_workload(37, 512, 32768)
    bad = {k: v.copy() for k, v in w.rows.items()}
    bad["temperature"][:] = -1.0
    d = DeviceRun(w)
    good = d.d["rows"].clone()
    d.d["rows"].copy_(torch.from_numpy(pack_rows(bad, w.B).view(np.uint8).reshape(-1)))
    d.plan.set_wait_limit(1, 1)
    d()
    g = d.results()
    diag = d.diag().copy()
    timed_out = (g["row_status"] & native.ST_COPY_TIMEOUT) != 0
    assert diag[3] > 0 and timed_out.any(), (diag, g["row_status"])
    assert np.all(g["row_status"] & native.ST_BAD_PARAM)
    d.d["rows"].copy_(good)
    d.plan.set_wait_limit(0, 0)
    d()
    g2 = d.results()
    assert not np.any(g2["row_status"] & native.ST_COPY_TIMEOUT)
    assert d.diag()[3] == diag[3]
    rep = _oracle_chunks(w, g2)
    assert rep.ok(), rep


# ------------------------------------------------------------------ graphs

def test_graph_replay_matches_eager():
    import torch
    from spec_verification_gb300.runner import DeviceRun
    w = W.mixed_workload(41, 16, 40000, "f32")
    d = DeviceRun(w)
    d()
    eager = d.results()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        d()
    d.tokens.fill_(7)
    g.replay()
    a = d.results()
    g.replay()
    b = d.results()
    for k in eager:
        assert np.array_equal(eager[k], a[k]), k
        assert np.array_equal(a[k], b[k]), k
    # new device data through the same graph: other seeds -> the oracle's answer for them
    w2 = W.mixed_workload(41, 16, 40000, "f32")
    w2.seeds = w2.seeds + np.uint64(12345)
    d.d["seeds"].copy_(torch.from_numpy(w2.seeds.view(np.int64)))
    g.replay()
    got = d.results()
    ora = O.verify(w2, tokens_stride=got["tokens"].shape[1])
    rep = parity.compare_verify(w2, got, ora)
    assert rep.ok(), rep


def test_cut_points_on_the_boundary():
    """Top-p and min-p cut points exactly on (or next to) their limits: equal
    logits make the mass before the fifth candidate exactly half of the total
    (top_p = 0.5), and min_p = exp(l_t - l_0) at a candidate.  The stage-2
    epilogue decides such cut points in fp64 (dl-note, Top-p and Min-p)."""
    V = 4096
    x = np.full((6, V), -30.0, np.float32)
    x[:, :10] = 2.0                      # ten equal logits: prefix before t is t / 10 of Z
    x[3:, 10:20] = 2.0 - np.log(4.0, dtype=np.float32)   # weights exactly 1/4 of the top ones
    w = sample_case(x, flags=[F.TOPP, F.TOPP, F.MINP, F.MINP, F.TOPP | F.MINP, F.TOPP],
                    top_p=[0.5, 0.3, 0.0, 0.25, 0.5, 0.7], min_p=[0.0, 0.0, 0.5, 0.25, 0.25, 0.0],
                    temperature=1.0)
    gpu, ora, _ = check(w)
    assert np.array_equal(gpu["num_kept"], ora["num_kept"])
