"""Device-resident batch for one ss_sample / ss_verify call.

Uploads a workload (numpy arrays in the input format) into torch CUDA
tensors laid out as include/ss.h expects, allocates the outputs and the
workspace once, and issues the call through the ctypes binding.  Torch is
only used for device memory, host pinned memory and streams.
"""
from __future__ import annotations

import numpy as np

from . import native
from . import workloads as W
from .workloads import Workload


def pack_rows(rows: dict, B: int) -> np.ndarray:
    a = np.zeros(B, native.ROW_DTYPE)
    for f in native.ROW_DTYPE.names:
        a[f] = rows[f][:B]
    return a


def pack_bias(tokens: np.ndarray, values: np.ndarray) -> np.ndarray:
    a = np.zeros(tokens.shape, native.BIAS_DTYPE)
    a["token"] = tokens
    a["value"] = values
    return a


def _padded_rows(a: np.ndarray, esz: int) -> np.ndarray:
    """Rows padded to a 16-byte multiple (the ABI's row alignment); padding
    holds NaN bit patterns, which the kernels must never read as tokens."""
    if a.ndim != 2:
        return a
    per = 16 // esz
    ld = -(-a.shape[1] // per) * per
    if ld == a.shape[1]:
        return a
    out = np.empty((a.shape[0], ld), a.dtype)
    out[:, :a.shape[1]] = a
    out[:, a.shape[1]:] = np.float32(np.nan) if a.dtype == np.float32 else np.uint16(0x7FC0)
    return out


def _as_torch_bits(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    elif a.dtype == np.uint64:
        a = a.view(np.int64)
    elif a.dtype.names is not None:
        a = a.view(np.uint8).reshape(-1)
    return torch.from_numpy(a)


class DeviceRun:
    """Inputs, outputs and workspace of one call, resident on one GPU."""

    def __init__(self, w: Workload, device: str = "cuda:0", tile: int = 0, max_positions: int | None = None,
                 candidates: bool = True, tokens_stride: int | None = None, pinned_host: bool = False,
                 one_hot_drafts: bool = False, guard_bytes: int = 0):
        import torch
        self.w = w
        # guard_bytes > 0: every output buffer and the workspace sit inside a
        # larger allocation whose bands of guard_bytes before and after hold
        # GUARD; guards_intact() reports the buffers whose bands changed
        self.guard_bytes = guard_bytes
        self._guarded = {}
        # the history and bias lists go to the library only when a row uses
        # them (SS_PENALTY / SS_BIAS): a call without them runs the stage-1
        # form that has no listed-token paths
        self.uses_aux = bool(np.any(np.asarray(w.rows["flags"])[:w.B] & np.uint32(W.PENALTY | W.BIAS)))
        self.dev = torch.device(device)
        self.verify = w.is_verify
        # drafts without probabilities: nothing of q is uploaded; the library gets NULL
        self.one_hot_drafts = self.verify and (one_hot_drafts or bool(w.meta.get("one_hot_drafts")))
        npos = w.n_positions
        self.plan = native.Plan(w.V, w.B, max_positions or npos, w.dtype,
                                w.q_dtype if self.verify else "f32", tile, self.dev.index or 0)
        if (w.meta or {}).get("exact_sampling"):
            self.plan.enable_exact(True)
        host = {
            "logits": _as_torch_bits(_padded_rows(w.logits, 2 if w.dtype == "bf16" else 4)),
            "rows": _as_torch_bits(pack_rows(w.rows, w.B)),
            "seeds": _as_torch_bits(w.seeds),
            "history": _as_torch_bits(w.history.astype(np.int32)),
            "bias": _as_torch_bits(pack_bias(w.bias_tokens, w.bias_values)),
        }
        if w.bitmask is not None:
            host["bitmask"] = _as_torch_bits(w.bitmask)
        if self.verify:
            host["cu_draft"] = _as_torch_bits(w.cu_draft.astype(np.int32))
            host["draft_ids"] = _as_torch_bits(w.draft_ids.astype(np.int32))
            if not self.one_hot_drafts:
                host["draft_probs"] = _as_torch_bits(_padded_rows(w.draft_probs, 2 if w.q_dtype == "bf16" else 4))
        if pinned_host:
            host = {k: v.pin_memory() for k, v in host.items()}
        self.host = host
        self.d = {k: v.to(self.dev) for k, v in host.items()}
        self.ld_logits = int(self.host["logits"].shape[1])
        self.ld_q = int(self.host["draft_probs"].shape[1]) if "draft_probs" in self.host else 0
        self.hist_stride = int(w.history.shape[1])
        self.bias_stride = int(w.bias_tokens.shape[1])
        i32 = torch.int32
        if self.verify:
            ts = tokens_stride if tokens_stride is not None else w.max_gamma + 1
            self.tokens = self._buffer("tokens", (w.B, ts), i32, -1)
            self.num_accepted = self._buffer("num_accepted", (w.B,), i32, 0)
        else:
            self.tokens = self._buffer("tokens", (w.B,), i32, -1)
            self.num_accepted = None
        self.row_status = self._buffer("row_status", (w.B,), i32, 0)
        self.cand_ids = self.cand_probs = self.num_kept = None
        if candidates:
            self.cand_ids = self._buffer("cand_ids", (npos, native.K), i32, -1)
            self.cand_probs = self._buffer("cand_probs", (npos, native.K), torch.float32, 0)
            self.num_kept = self._buffer("num_kept", (npos,), i32, 0)
        self.workspace = self._buffer("workspace", (self.plan.workspace_bytes,), torch.uint8, 0)

    GUARD = 0xA5

    def _buffer(self, name, shape, dtype, fill):
        """A device tensor of `shape`, filled with `fill`, inside guard bands
        when guard_bytes > 0."""
        import torch
        if not self.guard_bytes:
            return torch.full(shape, fill, dtype=dtype, device=self.dev)
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        g = self.guard_bytes
        raw = torch.full((n + 2 * g,), self.GUARD, dtype=torch.uint8, device=self.dev)
        t = raw[g:g + n].view(dtype).view(shape)
        t.fill_(fill)
        self._guarded[name] = (raw, n)
        return t

    def guards_intact(self) -> list:
        """Names of the buffers whose guard bands no longer hold GUARD."""
        bad = []
        for name, (raw, n) in self._guarded.items():
            g = self.guard_bytes
            h = raw.cpu().numpy()
            if np.any(h[:g] != self.GUARD) or np.any(h[g + n:] != self.GUARD):
                bad.append(name)
        return bad

    def upload(self, non_blocking: bool = True):
        """Host -> device copy of every input (pinned host buffers)."""
        for k, v in self.host.items():
            self.d[k].copy_(v, non_blocking=non_blocking)

    def upload_split(self, main, copy_streams, events, after=None):
        """Host -> device copy of every input with the streamed tensors
        (logits, draft probabilities) cut into row ranges, one per copy
        stream, so that several copies run at once; the small inputs go on
        `main`, which then waits for every copy stream.  events: one started
        event plus one per copy stream (torch.cuda.Event, reused per call).
        The copy streams start after `after` (an event: the last work that
        read these device buffers) when given, else after everything queued
        on `main` so far."""
        import torch
        if after is None:
            events[0].record(main)
            after = events[0]
        for st in copy_streams:
            st.wait_event(after)
        for k, v in self.host.items():
            if k in ("logits", "draft_probs") and v.dim() == 2 and v.shape[0] >= len(copy_streams):
                n = v.shape[0]
                for i, st in enumerate(copy_streams):
                    r0, r1 = n * i // len(copy_streams), n * (i + 1) // len(copy_streams)
                    with torch.cuda.stream(st):
                        self.d[k][r0:r1].copy_(v[r0:r1], non_blocking=True)
            else:
                with torch.cuda.stream(main):
                    self.d[k].copy_(v, non_blocking=True)
        for i, st in enumerate(copy_streams):
            events[i + 1].record(st)
            main.wait_event(events[i + 1])

    def input_bytes(self) -> int:
        return sum(v.numel() * v.element_size() for v in self.host.values())

    def output_bytes(self) -> int:
        n = self.tokens.numel() * 4 + self.row_status.numel() * 4
        if self.num_accepted is not None:
            n += self.num_accepted.numel() * 4
        return n

    def __call__(self, stream=None, logits=None, draft_probs=None, events=None):
        d = self.d
        lg = logits if logits is not None else d["logits"]
        if self.verify:
            q = None if self.one_hot_drafts else (draft_probs if draft_probs is not None else d["draft_probs"])
            native.ss_verify(self.plan, lg, q, d["draft_ids"], d["rows"], d["cu_draft"], d["seeds"],
                             workspace=self.workspace, tokens=self.tokens, num_accepted=self.num_accepted,
                             row_status=self.row_status, history=d["history"] if self.uses_aux else None,
                             bitmask=d.get("bitmask"), bias=d["bias"] if self.uses_aux else None, hist_stride=self.hist_stride, bias_stride=self.bias_stride,
                             cand_ids=self.cand_ids, cand_probs=self.cand_probs, num_kept=self.num_kept,
                             B=self.w.B, stream=stream, events=events)
        else:
            native.ss_sample(self.plan, lg, d["rows"], d["seeds"], workspace=self.workspace,
                             tokens=self.tokens, row_status=self.row_status,
                             history=d["history"] if self.uses_aux else None,
                             bitmask=d.get("bitmask"), bias=d["bias"] if self.uses_aux else None, hist_stride=self.hist_stride,
                             bias_stride=self.bias_stride, cand_ids=self.cand_ids,
                             cand_probs=self.cand_probs, num_kept=self.num_kept, B=self.w.B, stream=stream,
                             events=events)

    def results(self) -> dict:
        import torch
        torch.cuda.synchronize(self.dev)
        out = {"tokens": self.tokens.cpu().numpy(),
               "row_status": self.row_status.cpu().numpy().view(np.uint32)}
        if self.num_accepted is not None:
            out["num_accepted"] = self.num_accepted.cpu().numpy()
        if self.cand_ids is not None:
            out["cand_ids"] = self.cand_ids.cpu().numpy()
            out["cand_probs"] = self.cand_probs.cpu().numpy()
            out["num_kept"] = self.num_kept.cpu().numpy()
        return out

    def diag(self) -> np.ndarray:
        o = self.plan.diag_offset
        return self.workspace[o:o + 32].cpu().numpy().view(np.uint32)
