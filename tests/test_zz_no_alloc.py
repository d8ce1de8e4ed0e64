"""ss_sample_noalloc (static device scratch, no workspace argument) against
ss_sample with a caller workspace: same inputs, same plan, two calls in a row
through the C ABI.  Both run the same kernels on the same data, so every
output must match; the probabilities are compared within 1e-6 absolute."""
import numpy as np
import pytest

from spec_verification_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from spec_verification_gb300 import build
    build.build()


def _noalloc_call(run):
    import torch
    from spec_verification_gb300 import native
    run.tokens.fill_(-7)
    run.row_status.fill_(0)
    run.cand_ids.fill_(-7)
    run.cand_probs.fill_(-1.0)
    run.num_kept.fill_(-7)
    d = run.d
    native.ss_sample_noalloc(run.plan, d["logits"], d["rows"], d["seeds"], tokens=run.tokens,
                             row_status=run.row_status, history=d["history"], bitmask=d.get("bitmask"),
                             bias=d["bias"], hist_stride=run.hist_stride, bias_stride=run.bias_stride,
                             cand_ids=run.cand_ids, cand_probs=run.cand_probs, num_kept=run.num_kept,
                             B=run.w.B)
    torch.cuda.synchronize()
    return run.results()


@pytest.mark.parametrize("dtype,V", [("bf16", 50000), ("f32", 20011)])
def test_noalloc_matches_workspace_call_twice(dtype, V):
    from spec_verification_gb300.runner import DeviceRun
    w = W.sample_workload(seed=91 if dtype == "bf16" else 92, B=24, V=V, dtype=dtype, name="noalloc")
    run = DeviceRun(w)
    run()
    ref = run.results()
    assert (ref["tokens"] >= 0).all()
    for _ in range(2):
        got = _noalloc_call(run)
        np.testing.assert_array_equal(got["tokens"], ref["tokens"])
        np.testing.assert_array_equal(got["row_status"], ref["row_status"])
        np.testing.assert_array_equal(got["cand_ids"], ref["cand_ids"])
        np.testing.assert_array_equal(got["num_kept"], ref["num_kept"])
        np.testing.assert_allclose(got["cand_probs"], ref["cand_probs"], rtol=0, atol=1e-6)


def test_noalloc_rejects_plan_beyond_static_scratch():
    import torch
    from spec_verification_gb300 import native
    plan = native.Plan(131072, 2048, logits_dtype="bf16")
    assert plan.workspace_bytes > (16 << 20)
    dev = torch.device("cuda:0")
    logits = torch.zeros((1, 131072), dtype=torch.int16, device=dev)
    rows = torch.zeros(44, dtype=torch.uint8, device=dev)
    seeds = torch.zeros(1, dtype=torch.int64, device=dev)
    tokens = torch.zeros(1, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(native.SSError, match="static scratch"):
        native.ss_sample_noalloc(plan, logits, rows, seeds, tokens=tokens, row_status=status, B=1)
