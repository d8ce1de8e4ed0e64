"""Canary bands around every buffer the kernels write: the workspace (staging
lists, per-segment metadata, residual queue, counters) and each output
(tokens, row status, accept counts, candidate ids / probabilities / counts)
sit inside larger allocations whose 4 KB bands before and after hold a fixed
byte pattern; after two calls on each workload the bands must be unchanged.
This stands in for a bounds checker (none runs on this GPU): a kernel write
past either end of a buffer it owns lands in a band.  The workloads cover
ragged tiles, ragged draft counts, every processor, exact sampling, drafts
without probabilities, the residual pass and the largest tile."""
import numpy as np
import pytest

from spec_verification_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096


def _cases():
    yield "c1", W.config1(), {}
    yield "sample_ragged_processors", W.sample_workload(41, 24, 40000, "bf16"), {}
    yield "sample_tile16k", W.sample_workload(42, 8, 70001, "f32"), {"tile": 16384}
    yield "verify_ragged", W.verify_workload(43, 12, 30000, [0, 1, 2, 3, 4, 5, 6, 7, 3, 2, 1, 0], "f32", "f32",
                                             processors=True), {}
    yield "verify_untruncated_residual", W.verify_workload(44, 8, 50000, [3] * 8, "bf16", "bf16", noise=3.0), {}
    yield "verify_one_hot", W.with_one_hot_drafts(W.verify_workload(45, 8, 20000, [2] * 8, "f32", "f32")), {}
    yield "exact_sampling", W.with_exact_sampling(W.sample_workload(46, 16, 33000, "f32")), {}
    yield "topk_stress", W.topk_stress_workload(47, 64, 65536), {}


@pytest.mark.parametrize("name,w,kw", list(_cases()), ids=[c[0] for c in _cases()])
def test_writes_stay_inside_their_buffers(name, w, kw):
    from spec_verification_gb300.runner import DeviceRun
    d = DeviceRun(w, guard_bytes=GUARD, **kw)
    d()
    d()
    g = d.results()
    assert d.guards_intact() == [], (name, d.guards_intact())
    # every row was processed (a token or a reported status)
    assert g["row_status"].shape == (w.B,)
    toks = g["tokens"] if g["tokens"].ndim == 1 else g["tokens"][:, 0]
    assert np.all((toks >= 0) | (g["row_status"] != 0))
    assert np.all(toks < w.V)
