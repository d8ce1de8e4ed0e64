"""Long calls with history or bias lists launch two stage-1 forms, the lean
one (no per-stage count tables, no normaliser partials) and the full one;
every CTA checks the rows and exactly one form does the work.  These calls
are long enough (at least 10 stages per stage-1 CTA) to take that path,
once with rows the lean form can serve and once with rows that need the
full form; every row is compared with the oracle."""
import numpy as np
import pytest

from oracle import oracle as O
from spec_verification_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


def _check(w, need_full):
    from spec_verification_gb300.runner import DeviceRun
    d = DeviceRun(w)
    assert d.uses_aux
    assert w.n_positions * d.plan.num_tiles >= 10 * d.plan.stage1_ctas   # the two-form path
    d()
    d()
    g = d.results()
    if w.is_verify:
        rep = parity.compare_verify(w, g, O.verify(w, tokens_stride=g["tokens"].shape[1]))
    else:
        rep = parity.compare_sample(w, g, O.sample(w))
    assert rep.ok(), rep
    assert rep.ambiguous <= max(1, rep.checked // 200), rep
    if need_full and w.is_verify:
        assert d.diag()[2] > 0          # residual passes: the normaliser of the full form was used


def test_lean_form_serves_truncated_verification_with_processors():
    # every stochastic row truncates: no normaliser, short listed-token lists
    w = W.verify_workload(61, 64, 131072, np.full(64, 4), "bf16", "bf16", processors=True, truncation=True)
    _check(w, need_full=False)


def test_full_form_serves_untruncated_verification_with_processors():
    # untruncated stochastic rows with penalties and bias: normaliser and
    # per-stage count tables
    w = W.verify_workload(62, 64, 131072, np.full(64, 4), "bf16", "bf16", processors=True, noise=3.0)
    w.rows["flags"][:] &= ~np.uint32(W.TOPK | W.TOPP | W.MINP)
    assert np.any((w.rows["flags"] & W.GREEDY) == 0)
    _check(w, need_full=True)


def test_full_form_serves_long_histories():
    # histories of 600 tokens: more listed tokens than the hash table holds
    w = W.sample_workload(63, 200, 131072, "bf16", H=600)
    _check(w, need_full=True)


def _launches(w, mode=None, **kw):
    from spec_verification_gb300.runner import DeviceRun
    d = DeviceRun(w, **kw)
    if mode is not None:
        d.plan.set_fusion(mode)
    d()
    return d.plan.last_launches(), d


def test_launch_counts_follow_the_call_shape():
    # short call without lists: stage 1, stage 2
    n, _ = _launches(W.config1())
    assert n == 2
    # long sampling call without lists (at least two stages per stage-1
    # CTA): stage 2 runs inside stage 1 by default, as its own launch on request
    w = W.topk_stress_workload(64, 256, 32768)
    n, d = _launches(w)
    assert n == 1
    rep = parity.compare_sample(w, d.results(), O.sample(w))
    assert rep.ok(), rep
    n, _ = _launches(w, mode=2)
    assert n == 2
    # long verification call without lists: stage 1 (fused stage 2), residual pass
    v = W.verify_workload(65, 32, 65536, np.full(32, 4), "bf16", "bf16", noise=3.0)
    n, d = _launches(v)
    assert n == 2
    g = d.results()
    rep = parity.compare_verify(v, g, O.verify(v, tokens_stride=g["tokens"].shape[1]))
    assert rep.ok(), rep
    # long call with lists: lean and full stage-1 forms, stage 2, residual pass
    n, _ = _launches(W.verify_workload(61, 64, 131072, np.full(64, 4), "bf16", "bf16", processors=True,
                                       truncation=True))
    assert n == 4
