"""Small hand-built inputs shared by the tests (no method arithmetic here)."""
from __future__ import annotations

import numpy as np

from spec_verification_gb300 import workloads as W
from spec_verification_gb300.workloads import subset  # noqa: F401


def rows(B: int, **kw) -> dict:
    r = {k: np.zeros(B, dtype=W._ROW_DTYPES[k]) for k in W.ROW_FIELDS}
    r["temperature"][:] = 1.0
    r["top_p"][:] = 1.0
    r["rep"][:] = 1.0
    for k, v in kw.items():
        r[k][:] = v
    return r


def sample_case(logits: np.ndarray, flags=0, dtype="f32", seeds=None, history=None,
                bitmask=None, bias_tokens=None, bias_values=None, name="case", **rowkw):
    """A single-step Workload from explicit arrays (logits fp32 [B, V])."""
    logits = np.atleast_2d(np.asarray(logits, np.float32))
    B, V = logits.shape
    rw = rows(B, flags=flags, **rowkw)
    hist = np.full((B, 1), -1, np.int32) if history is None else np.atleast_2d(np.asarray(history, np.int32))
    if history is not None and "hist_len" not in rowkw:
        rw["hist_len"][:] = hist.shape[1]
    btok = np.full((B, 1), -1, np.int32) if bias_tokens is None else np.atleast_2d(np.asarray(bias_tokens, np.int32))
    bval = np.zeros(btok.shape, np.float32) if bias_values is None else np.atleast_2d(np.asarray(bias_values, np.float32))
    if bias_tokens is not None and "n_bias" not in rowkw:
        rw["n_bias"][:] = btok.shape[1]
    if seeds is None:
        seeds = np.arange(1, B + 1, dtype=np.uint64)
    data = W.f32_to_bf16_bits(logits) if dtype == "bf16" else logits
    return W.Workload(name, B, V, dtype, data, rw, hist, bitmask, btok, bval,
                      np.asarray(seeds, np.uint64))


def verify_case(target: np.ndarray, q: np.ndarray, draft_ids, gammas, flags=0, seeds=None,
                q_dtype="f32", dtype="f32", name="vcase", **rowkw):
    """A verify Workload from explicit arrays: target [B_pos, V] fp32, q [sum gamma, V]."""
    target = np.asarray(target, np.float32)
    gammas = np.asarray(gammas, np.int32)
    B = gammas.size
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(gammas)
    assert target.shape[0] == cu[-1] + B
    rw = rows(B, flags=flags, **rowkw)
    if seeds is None:
        seeds = np.arange(1, B + 1, dtype=np.uint64)
    qa = W.f32_to_bf16_bits(q) if q_dtype == "bf16" else np.asarray(q, np.float32)
    data = W.f32_to_bf16_bits(target) if dtype == "bf16" else target
    return W.Workload(name, B, target.shape[1], dtype, data, rw, np.full((B, 1), -1, np.int32),
                      None, np.full((B, 1), -1, np.int32), np.zeros((B, 1), np.float32),
                      np.asarray(seeds, np.uint64), cu_draft=cu,
                      draft_ids=np.asarray(draft_ids, np.int32), draft_probs=qa, q_dtype=q_dtype)


def python_order(x: np.ndarray) -> list:
    """Token ids by (value descending, id ascending) with Python's own sort."""
    return [i for _, i in sorted(((-float(v), i) for i, v in enumerate(x)))]


def chi2_pvalue(counts: np.ndarray, probs: np.ndarray) -> float:
    from scipy import stats
    n = counts.sum()
    exp = probs * n
    keep = exp > 0
    # pool tiny expected cells
    return float(stats.chisquare(counts[keep], exp[keep] * counts[keep].sum() / exp[keep].sum()).pvalue)


def gpu_rows_as(out: dict, w, rows) -> dict:
    """GPU outputs of a full batch restricted to `rows` (positions follow)."""
    rows = np.asarray(rows, np.int64)
    o = {"tokens": out["tokens"][rows], "row_status": out["row_status"][rows]}
    if "num_accepted" in out:
        o["num_accepted"] = out["num_accepted"][rows]
    if w.is_verify:
        offs = w.position_offsets()
        gam = w.gammas()
        pos = np.concatenate([np.arange(offs[r], offs[r] + gam[r] + 1) for r in rows])
    else:
        pos = rows
    for k in ("cand_ids", "cand_probs", "num_kept"):
        if k in out:
            o[k] = out[k][pos]
    return o
