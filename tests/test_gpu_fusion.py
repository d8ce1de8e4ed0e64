"""Stage 2 inside the stage-1 launch (the fused form, SonicSampler 3.2's
workload-aware launch for small batches) against stage 2 as its own launch:
on the same inputs both give bit-identical outputs, both match the oracle,
and the workspace counters the fused hand-over uses (per-position segment
counts, the residual queue) come back clean for the next call."""
import numpy as np
import pytest

from oracle import oracle as O
from spec_verification_gb300 import workloads as W
from tests import parity
from tests.helpers import gpu_rows_as, subset

pytestmark = pytest.mark.gpu

FUSED, SEPARATE = 1, 2


def _cases():
    yield "c1", W.config1()
    yield "sample_processors_bf16", W.sample_workload(51, 24, 70000, "bf16")
    yield "verify_processors", W.verify_workload(52, 12, 30000, [0, 1, 2, 3, 4, 5, 6, 7, 3, 2, 1, 0], "f32", "f32",
                                                 processors=True)
    yield "verify_untruncated_residual", W.verify_workload(53, 10, 50000, [3] * 10, "bf16", "bf16", noise=3.0)
    yield "verify_one_hot", W.with_one_hot_drafts(W.verify_workload(54, 8, 20000, [2] * 8, "f32", "f32"))
    yield "topk_stress", W.topk_stress_workload(55, 64, 65536)


def _run(w, mode, calls=2, **kw):
    from spec_verification_gb300.runner import DeviceRun
    d = DeviceRun(w, **kw)
    d.plan.set_fusion(mode)
    outs = []
    for _ in range(calls):
        d()
        outs.append(d.results())
    return outs, d


@pytest.mark.parametrize("name,w", list(_cases()), ids=[c[0] for c in _cases()])
def test_fused_equals_separate_and_oracle(name, w):
    fused, df = _run(w, FUSED)
    sep, _ = _run(w, SEPARATE)
    for k in fused[0]:
        assert np.array_equal(fused[0][k], sep[0][k]), (name, k)
        assert np.array_equal(fused[1][k], fused[0][k]), (name, k)   # a second call on the same workspace
    if w.is_verify:
        rep = parity.compare_verify(w, fused[0], O.verify(w, tokens_stride=fused[0]["tokens"].shape[1]))
    else:
        rep = parity.compare_sample(w, fused[0], O.sample(w))
    assert rep.ok(), rep
    assert rep.ambiguous <= max(1, rep.checked // 200), rep
    # no position had more lists than the call's shared memory, no copy timed
    # out; a per-position count or residual queue left behind would have
    # changed the second call
    assert df.diag()[1] == 0 and df.diag()[3] == 0


def test_fused_capacity_rows():
    """Rows past the plan's max_positions are reported by the fused launch
    as by the separate one (SS_ST_CAPACITY, no tokens)."""
    from spec_verification_gb300 import native
    w = W.verify_workload(44, 6, 20000, [2, 1, 3, 2, 0, 1], dtype="f32", q_dtype="f32", truncation=True)
    fused, _ = _run(w, FUSED, max_positions=10)
    sep, _ = _run(w, SEPARATE, max_positions=10)
    for k in fused[0]:
        assert np.array_equal(fused[0][k], sep[0][k]), k
    for r in (3, 4, 5):
        assert fused[0]["row_status"][r] == native.ST_CAPACITY
    fit = [0, 1, 2]
    sub = subset(w, fit)
    g = gpu_rows_as(fused[0], w, fit)
    rep = parity.compare_verify(sub, g, O.verify(sub, tokens_stride=fused[0]["tokens"].shape[1]))
    assert rep.ok(), rep


def test_fused_copy_timeout_reports_and_recovers():
    """The wait-limit give-up under the fused form: a CTA that gives up still
    hands its positions over (empty lists with SS_ST_COPY_TIMEOUT), every row
    is written, and the next call with the default limit is exact."""
    import torch
    from spec_verification_gb300 import native
    from spec_verification_gb300.runner import DeviceRun, pack_rows
    w = W.topk_stress_workload(56, 256, 32768)
    bad = {k: v.copy() for k, v in w.rows.items()}
    bad["temperature"][:] = -1.0
    d = DeviceRun(w)
    d.plan.set_fusion(FUSED)
    good = d.d["rows"].clone()
    d.d["rows"].copy_(torch.from_numpy(pack_rows(bad, w.B).view(np.uint8).reshape(-1)))
    d.plan.set_wait_limit(1, 1)
    d()
    g = d.results()
    assert np.all(g["row_status"] & native.ST_BAD_PARAM)
    assert d.diag()[3] > 0 and np.any(g["row_status"] & native.ST_COPY_TIMEOUT)
    d.d["rows"].copy_(good)
    d.plan.set_wait_limit(0, 0)
    d()
    g2 = d.results()
    assert not np.any(g2["row_status"] & native.ST_COPY_TIMEOUT)
    rep = parity.compare_sample(w, g2, O.sample(w))
    assert rep.ok(), rep
