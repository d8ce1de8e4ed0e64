"""Python front end of the CPU oracle (test infrastructure only).

Only tests/, ``__graft_entry__.smoke()`` and the cpu-baseline / reference legs
of bench.py may import this module.  The product path never does.

The oracle itself is plain single-threaded C++ (``sso.cpp``); this file only
compiles it and marshals numpy arrays into its structs with ctypes.  See the
header of ``sso.cpp`` for the definitions it follows and the readings it takes
where the pages are silent.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "sso.cpp"
BUILD_DIR = HERE / "_build"
LIB = BUILD_DIR / "liboracle.so"
K = 128

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> Path:
    """Compile the oracle with g++ (fp32 steps with one rounding each: no FMA
    contraction, no fast-math)."""
    BUILD_DIR.mkdir(exist_ok=True)
    if LIB.exists() and not force and LIB.stat().st_mtime >= SRC.stat().st_mtime:
        return LIB
    tmp = LIB.with_suffix(f".{os.getpid()}.tmp.so")
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
           "-fno-math-errno", "-fPIC", "-shared", str(SRC), "-o", str(tmp)]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


class Row(C.Structure):
    _fields_ = [("flags", C.c_uint32), ("temperature", C.c_float), ("top_p", C.c_float),
                ("min_p", C.c_float), ("rep", C.c_float), ("freq", C.c_float),
                ("pres", C.c_float), ("top_k", C.c_int32), ("hist_len", C.c_int32),
                ("n_bias", C.c_int32), ("position", C.c_uint32)]


class Problem(C.Structure):
    _fields_ = [("B", C.c_int32), ("V", C.c_int32), ("logits_bf16", C.c_int32),
                ("ld_logits", C.c_int64), ("logits", C.c_void_p), ("rows", C.c_void_p),
                ("history", C.c_void_p), ("hist_stride", C.c_int32),
                ("bitmask", C.c_void_p), ("bias_tokens", C.c_void_p),
                ("bias_values", C.c_void_p), ("bias_stride", C.c_int32),
                ("seeds", C.c_void_p), ("cu_draft", C.c_void_p), ("draft_ids", C.c_void_p),
                ("q_bf16", C.c_int32), ("ld_q", C.c_int64), ("draft_probs", C.c_void_p),
                ("row_ids", C.c_void_p), ("exact_on", C.c_int32)]


class Outputs(C.Structure):
    _fields_ = [("tokens", C.c_void_p), ("tokens_stride", C.c_int32),
                ("num_accepted", C.c_void_p), ("row_status", C.c_void_p),
                ("cand_ids", C.c_void_p), ("cand_probs", C.c_void_p), ("num_kept", C.c_void_p),
                ("margin_topp", C.c_void_p), ("margin_minp", C.c_void_p),
                ("margin_gumbel", C.c_void_p), ("margin_accept", C.c_void_p),
                ("margin_resid", C.c_void_p), ("mass_outside", C.c_void_p),
                ("p_draft", C.c_void_p), ("lse", C.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(str(LIB))
            L.sso_sample.argtypes = [C.POINTER(Problem), C.c_int, C.POINTER(Outputs)]
            L.sso_verify.argtypes = [C.POINTER(Problem), C.c_int, C.POINTER(Outputs)]
            L.sso_philox.argtypes = [C.c_void_p, C.c_uint32, C.c_uint32, C.c_void_p]
            L.sso_uniform.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint32]
            L.sso_uniform.restype = C.c_float
            L.sso_prelude.argtypes = [C.POINTER(Problem), C.c_int, C.c_int64, C.c_void_p,
                                      C.c_int, C.c_void_p, C.c_void_p]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _rows_array(rows: dict, B: int):
    arr = (Row * B)()
    for r in range(B):
        for f, _ in Row._fields_:
            setattr(arr[r], f, rows[f][r].item())
    return arr


def _problem(w, keep: list, rows_override=None):
    """Build the C problem struct from a workload-like object (duck-typed)."""
    logits = np.ascontiguousarray(w.logits)
    hist = np.ascontiguousarray(w.history, dtype=np.int32)
    btok = np.ascontiguousarray(w.bias_tokens, dtype=np.int32)
    bval = np.ascontiguousarray(w.bias_values, dtype=np.float32)
    seeds = np.ascontiguousarray(w.seeds, dtype=np.uint64)
    mask = None if w.bitmask is None else np.ascontiguousarray(w.bitmask, dtype=np.uint32)
    rows = _rows_array(rows_override if rows_override is not None else w.rows, w.B)
    keep += [logits, hist, btok, bval, seeds, mask, rows]
    P = Problem()
    P.B, P.V = w.B, w.V
    P.logits_bf16 = 1 if w.dtype == "bf16" else 0
    P.ld_logits = logits.shape[1]
    P.logits = _ptr(logits)
    P.rows = C.addressof(rows)
    P.history, P.hist_stride = _ptr(hist), hist.shape[1]
    P.bitmask = _ptr(mask)
    P.bias_tokens, P.bias_values, P.bias_stride = _ptr(btok), _ptr(bval), btok.shape[1]
    P.seeds = _ptr(seeds)
    if getattr(w, "cu_draft", None) is not None:
        cu = np.ascontiguousarray(w.cu_draft, dtype=np.int32)
        dids = np.ascontiguousarray(w.draft_ids, dtype=np.int32)
        q = np.ascontiguousarray(w.draft_probs)
        keep += [cu, dids, q]
        P.cu_draft, P.draft_ids = _ptr(cu), _ptr(dids)
        P.q_bf16 = 1 if w.q_dtype == "bf16" else 0
        P.ld_q = q.shape[1] if q.ndim == 2 and q.shape[0] else w.V
        P.draft_probs = _ptr(q)
    P.exact_on = 1 if (getattr(w, "meta", None) or {}).get("exact_sampling") else 0
    rid = getattr(w, "meta", {}).get("row_ids") if hasattr(w, "meta") else None
    if rid is not None:
        rid = np.ascontiguousarray(np.asarray(rid, np.int32))
        keep.append(rid)
        P.row_ids = _ptr(rid)
    return P


def _outputs(n_rows: int, n_pos: int, tokens_stride: int, keep: list):
    out = {
        "tokens": np.full((n_rows, tokens_stride), -1, np.int32),
        "num_accepted": np.zeros(n_rows, np.int32),
        "row_status": np.zeros(n_rows, np.uint32),
        "cand_ids": np.full((n_pos, K), -1, np.int32),
        "cand_probs": np.zeros((n_pos, K), np.float32),
        "num_kept": np.zeros(n_pos, np.int32),
    }
    for k in ("margin_topp", "margin_minp", "margin_gumbel", "margin_accept",
              "margin_resid", "mass_outside", "p_draft", "lse"):
        out[k] = np.full(n_pos, np.inf, np.float64)
    keep.append(out)
    O = Outputs()
    O.tokens_stride = tokens_stride
    for f, _ in Outputs._fields_:
        if f != "tokens_stride":
            setattr(O, f, out[f].ctypes.data)
    return O, out


def sample(w, exact: bool = False, rows=None) -> dict:
    """Oracle ss_sample on a workload: one position per row."""
    keep: list = []
    P = _problem(w, keep, rows)
    O, out = _outputs(w.B, w.B, 1, keep)
    lib().sso_sample(C.byref(P), 1 if exact else 0, C.byref(O))
    out["tokens"] = out["tokens"][:, 0]
    return out


def verify(w, exact: bool = False, rows=None, tokens_stride: int | None = None) -> dict:
    """Oracle ss_verify on a workload (cu_draft present)."""
    keep: list = []
    P = _problem(w, keep, rows)
    g = np.diff(np.asarray(w.cu_draft))
    ts = tokens_stride if tokens_stride is not None else int(g.max(initial=0)) + 1
    O, out = _outputs(w.B, int(w.cu_draft[-1]) + w.B, ts, keep)
    lib().sso_verify(C.byref(P), 1 if exact else 0, C.byref(O))
    return out


def prelude(w, r: int, pos: int, extra=()) -> tuple[np.ndarray, int]:
    """Processed logits of row r at target position pos, where pos is the
    absolute position (the logits row, not the index within row r) and extra
    holds the tokens appended to the row's history (a verify position's
    earlier drafts)."""
    keep: list = []
    P = _problem(w, keep)
    ex = np.ascontiguousarray(np.asarray(extra, np.int32))
    out = np.empty(w.V, np.float32)
    st = np.zeros(1, np.uint32)
    lib().sso_prelude(C.byref(P), r, pos, ex.ctypes.data if ex.size else None, int(ex.size),
                      out.ctypes.data, st.ctypes.data)
    return out, int(st[0])


def philox(ctr, k0: int, k1: int) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, np.uint32))
    o = np.zeros(4, np.uint32)
    lib().sso_philox(c.ctypes.data, k0 & 0xFFFFFFFF, k1 & 0xFFFFFFFF, o.ctypes.data)
    return o


def uniform(seed: int, i: int, position: int, row: int, purpose: int) -> float:
    return float(lib().sso_uniform(seed, i, position, row, purpose))
