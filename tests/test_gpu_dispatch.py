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
