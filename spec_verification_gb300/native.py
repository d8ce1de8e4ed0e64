"""ctypes binding of libss.so: the same entry points as include/ss.h, with
argument marshalling only (torch tensors -> device pointers, host structs).
Every step of the sampling path runs in the library's CUDA kernels; if the
library is missing this module raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes as C
from pathlib import Path

import numpy as np

PKG = Path(__file__).resolve().parent
LIB_PATH = PKG / "_build" / "libss.so"

SS_F32, SS_BF16 = 0, 1
STATUS = {0: "SS_OK", -1: "SS_ERR_ARG", -2: "SS_ERR_ALIGN", -3: "SS_ERR_UNSUPPORTED",
          -4: "SS_ERR_WORKSPACE", -5: "SS_ERR_CUDA"}
K = 128
# row_status bit of a row with invalid parameters (SS_ST_BAD_PARAM)
ST_BAD_PARAM = 1 << 4
# row_status bit of a verification row past the plan's max_positions (SS_ST_CAPACITY)
ST_CAPACITY = 1 << 9
# row_status bit of a row whose stage-1 copy did not land within the wait limit
ST_COPY_TIMEOUT = 1 << 10

# numpy layouts of the device-side structs (all 4-byte fields, no padding)
ROW_DTYPE = np.dtype([("flags", "<u4"), ("temperature", "<f4"), ("top_p", "<f4"), ("min_p", "<f4"),
                      ("rep", "<f4"), ("freq", "<f4"), ("pres", "<f4"), ("top_k", "<i4"),
                      ("hist_len", "<i4"), ("n_bias", "<i4"), ("position", "<u4")])
BIAS_DTYPE = np.dtype([("token", "<i4"), ("value", "<f4")])
assert ROW_DTYPE.itemsize == 44 and BIAS_DTYPE.itemsize == 8


class SSError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class Batch(C.Structure):
    _fields_ = [("B", C.c_int32), ("ld_logits", C.c_int64), ("ld_q", C.c_int64),
                ("rows", C.c_void_p), ("cu_draft", C.c_void_p), ("hist_stride", C.c_int32),
                ("bias_stride", C.c_int32), ("history", C.c_void_p), ("bitmask", C.c_void_p),
                ("bias", C.c_void_p), ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
                ("stream", C.c_void_p), ("plan", C.c_void_p), ("events", C.c_void_p)]


class Out(C.Structure):
    _fields_ = [("tokens", C.c_void_p), ("tokens_stride", C.c_int32), ("num_accepted", C.c_void_p),
                ("cand_ids", C.c_void_p), ("cand_probs", C.c_void_p), ("num_kept", C.c_void_p),
                ("row_status", C.c_void_p)]


EXPORTS = ["ss_plan_create", "ss_plan_destroy", "ss_workspace_bytes", "ss_plan_tile",
           "ss_plan_num_tiles", "ss_plan_stage1_ctas", "ss_sample", "ss_verify", "ss_status_str", "ss_last_error",
           "ss_workspace_diag_offset", "ss_sample_noalloc", "ss_plan_enable_exact", "ss_plan_set_wait_limit",
           "ss_plan_set_fusion", "ss_plan_last_launches"]

_lib = None


def library() -> C.CDLL:
    """Load libss.so (built by spec_verification_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not LIB_PATH.exists():
        raise ImportError(f"{LIB_PATH} is missing: run `python -m spec_verification_gb300.build` "
                          "(the CUDA library is required; there is no fallback)")
    L = C.CDLL(str(LIB_PATH))
    L.ss_plan_create.argtypes = [C.POINTER(C.c_void_p), C.c_int32, C.c_int32, C.c_int32, C.c_int,
                                 C.c_int, C.c_int32, C.c_int32]
    L.ss_plan_create.restype = C.c_int
    L.ss_plan_destroy.argtypes = [C.c_void_p]
    L.ss_workspace_bytes.argtypes = [C.c_void_p]
    L.ss_workspace_bytes.restype = C.c_size_t
    L.ss_workspace_diag_offset.argtypes = [C.c_void_p]
    L.ss_workspace_diag_offset.restype = C.c_size_t
    L.ss_plan_tile.argtypes = [C.c_void_p]
    L.ss_plan_tile.restype = C.c_int32
    L.ss_plan_num_tiles.argtypes = [C.c_void_p]
    L.ss_plan_num_tiles.restype = C.c_int32
    L.ss_plan_stage1_ctas.argtypes = [C.c_void_p]
    L.ss_plan_stage1_ctas.restype = C.c_int32
    L.ss_plan_enable_exact.argtypes = [C.c_void_p, C.c_int]
    L.ss_plan_enable_exact.restype = C.c_int
    L.ss_plan_set_wait_limit.argtypes = [C.c_void_p, C.c_uint32, C.c_uint32]
    L.ss_plan_set_wait_limit.restype = C.c_int
    L.ss_plan_set_fusion.argtypes = [C.c_void_p, C.c_int32]
    L.ss_plan_set_fusion.restype = C.c_int
    L.ss_plan_last_launches.argtypes = [C.c_void_p]
    L.ss_plan_last_launches.restype = C.c_int32
    L.ss_sample.argtypes = [C.c_void_p, C.POINTER(Batch), C.c_void_p, C.c_void_p, C.c_void_p,
                            C.c_void_p, C.POINTER(Out)]
    L.ss_sample.restype = C.c_int
    L.ss_sample_noalloc.argtypes = L.ss_sample.argtypes
    L.ss_sample_noalloc.restype = C.c_int
    L.ss_verify.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(Batch), C.c_void_p,
                            C.POINTER(Out)]
    L.ss_verify.restype = C.c_int
    L.ss_status_str.argtypes = [C.c_int]
    L.ss_status_str.restype = C.c_char_p
    L.ss_last_error.restype = C.c_char_p
    _lib = L
    return L


def _check(code: int):
    if code != 0:
        raise SSError(code, library().ss_last_error().decode())


class Plan:
    """ss_plan_create / ss_plan_destroy."""

    def __init__(self, V: int, max_rows: int, max_positions: int | None = None,
                 logits_dtype: str = "f32", q_dtype: str = "f32", tile: int = 0, device: int = 0):
        L = library()
        self._p = C.c_void_p()
        dt = {"f32": SS_F32, "bf16": SS_BF16}
        mp = max_positions if max_positions is not None else max_rows
        _check(L.ss_plan_create(C.byref(self._p), V, max_rows, mp, dt[logits_dtype], dt[q_dtype],
                                tile, device))
        self.V, self.max_rows, self.max_positions = V, max_rows, mp
        self.logits_dtype, self.q_dtype = logits_dtype, q_dtype
        self.tile = L.ss_plan_tile(self._p)
        self.num_tiles = L.ss_plan_num_tiles(self._p)
        self.stage1_ctas = L.ss_plan_stage1_ctas(self._p)
        self.workspace_bytes = L.ss_workspace_bytes(self._p)
        self.diag_offset = L.ss_workspace_diag_offset(self._p)

    def enable_exact(self, on: bool = True):
        """Run the exact-sampling variant of stage 1 (rows flagged SS_EXACT)."""
        _check(library().ss_plan_enable_exact(self._p, 1 if on else 0))

    def set_fusion(self, mode: int):
        """Where stage 2 runs: 1 inside the stage-1 launch whenever it fits,
        2 as its own launch, 0 (the default) by the call's shape."""
        _check(library().ss_plan_set_fusion(self._p, mode))

    def last_launches(self) -> int:
        """Kernels the most recent successful call with this plan launched."""
        return int(library().ss_plan_last_launches(self._p))

    def set_wait_limit(self, polls: int, suspend_ns: int = 0):
        """Polls of a stage-1 copy wait before the copy counts as lost (0:
        default) and the suspend-time hint of each poll (0: the hardware's)."""
        _check(library().ss_plan_set_wait_limit(self._p, polls, suspend_ns))

    @property
    def handle(self):
        return self._p.value

    def __del__(self):
        try:
            if self._p:
                library().ss_plan_destroy(self._p)
                self._p = C.c_void_p()
        except Exception:
            pass


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_ptr(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _events(events):
    """4 torch.cuda.Event (timing enabled) -> C array of cudaEvent_t."""
    if events is None:
        return None
    assert len(events) == 4
    assert all(e.cuda_event for e in events), "record each event once first (torch creates them lazily)"
    return (C.c_void_p * 4)(*[e.cuda_event for e in events])


def ss_sample(plan: Plan, logits, rows, seeds, *, workspace, tokens, row_status, history=None,
              bitmask=None, bias=None, hist_stride=1, bias_stride=1, cand_ids=None, cand_probs=None,
              num_kept=None, B=None, stream=None, events=None):
    """ss_sample on torch device tensors; rows = uint8 tensor of B * 44 bytes
    (ROW_DTYPE), bias = uint8 tensor of B * bias_stride * 8 bytes (BIAS_DTYPE)."""
    b = Batch()
    b.B = B if B is not None else seeds.shape[0]
    b.ld_logits = logits.stride(0)
    b.ld_q = 0
    b.rows = _ptr(rows)
    b.hist_stride, b.bias_stride = hist_stride, bias_stride
    b.workspace, b.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    b.stream = _stream_ptr(stream)
    b.plan = plan.handle
    ev = _events(events)
    b.events = C.cast(ev, C.c_void_p) if ev is not None else None
    o = Out()
    o.tokens, o.tokens_stride, o.row_status = _ptr(tokens), 1, _ptr(row_status)
    o.cand_ids, o.cand_probs, o.num_kept = _ptr(cand_ids), _ptr(cand_probs), _ptr(num_kept)
    _check(library().ss_sample(_ptr(logits), C.byref(b), _ptr(history), _ptr(bitmask), _ptr(bias),
                               _ptr(seeds), C.byref(o)))


def ss_sample_noalloc(plan: Plan, logits, rows, seeds, *, tokens, row_status, history=None,
                      bitmask=None, bias=None, hist_stride=1, bias_stride=1, cand_ids=None,
                      cand_probs=None, num_kept=None, B=None, stream=None, events=None):
    """ss_sample_noalloc: ss_sample with the library's static device scratch
    (no workspace argument)."""
    b = Batch()
    b.B = B if B is not None else seeds.shape[0]
    b.ld_logits = logits.stride(0)
    b.ld_q = 0
    b.rows = _ptr(rows)
    b.hist_stride, b.bias_stride = hist_stride, bias_stride
    b.workspace, b.workspace_bytes = None, 0
    b.stream = _stream_ptr(stream)
    b.plan = plan.handle
    ev = _events(events)
    b.events = C.cast(ev, C.c_void_p) if ev is not None else None
    o = Out()
    o.tokens, o.tokens_stride, o.row_status = _ptr(tokens), 1, _ptr(row_status)
    o.cand_ids, o.cand_probs, o.num_kept = _ptr(cand_ids), _ptr(cand_probs), _ptr(num_kept)
    _check(library().ss_sample_noalloc(_ptr(logits), C.byref(b), _ptr(history), _ptr(bitmask),
                                       _ptr(bias), _ptr(seeds), C.byref(o)))


def ss_verify(plan: Plan, target_logits, draft_probs, draft_ids, rows, cu_draft, seeds, *, workspace,
              tokens, num_accepted, row_status, history=None, bitmask=None, bias=None, hist_stride=1,
              bias_stride=1, cand_ids=None, cand_probs=None, num_kept=None, B=None, stream=None,
              events=None):
    """ss_verify on torch device tensors (see ss_sample for the struct layouts)."""
    b = Batch()
    b.B = B if B is not None else seeds.shape[0]
    b.ld_logits = target_logits.stride(0)
    # draft_probs None: drafts without probabilities (q one-hot on the draft token)
    b.ld_q = plan.V if draft_probs is None or draft_probs.dim() != 2 else draft_probs.stride(0)
    b.rows = _ptr(rows)
    b.cu_draft = _ptr(cu_draft)
    b.hist_stride, b.bias_stride = hist_stride, bias_stride
    b.history, b.bitmask, b.bias = _ptr(history), _ptr(bitmask), _ptr(bias)
    b.workspace, b.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    b.stream = _stream_ptr(stream)
    b.plan = plan.handle
    ev = _events(events)
    b.events = C.cast(ev, C.c_void_p) if ev is not None else None
    o = Out()
    o.tokens, o.tokens_stride = _ptr(tokens), tokens.shape[1]
    o.num_accepted, o.row_status = _ptr(num_accepted), _ptr(row_status)
    o.cand_ids, o.cand_probs, o.num_kept = _ptr(cand_ids), _ptr(cand_probs), _ptr(num_kept)
    _check(library().ss_verify(_ptr(target_logits), _ptr(draft_probs), _ptr(draft_ids), C.byref(b),
                               _ptr(seeds), C.byref(o)))
