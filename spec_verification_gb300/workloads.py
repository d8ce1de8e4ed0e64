"""Seeded synthetic inputs for the fused sampling / speculative-verification path.

This module only *builds inputs*: logits, grammar bitmasks, token histories,
sparse biases, per-row sampling parameters, Philox seeds and (for verification)
draft tokens with their draft-model probabilities.  It contains none of the
sampling method's arithmetic (no prelude, no selection, no truncation, no
sampling, no verification), so that the CPU oracle and the CUDA path can both
consume the same bytes without sharing any of the computation they are checked
on.

The pages measure on logits of trained LLMs, which are not available here; the
generators below stand in for them.  The structure follows the SonicSampler
page (low-entropy next-token distributions, vocabularies of 2^17..2^18 tokens,
section 1) in five standard workloads:

  c1  single-step, B=4, V=32000 fp32 N(0,2) plus five spike tokens +8..+12
  c2  single-step heterogeneous, B=64, V=131072 bf16, all processors
  c3  single-step top-k stress, B=256, V=262144 fp32, half near-flat rows
  c4  verification, B=32, gamma=4, V=131072 bf16 target and bf16 draft probs
  c5  mixed serving batch, B=512, V=151936 fp32, 60% single-step / 40% verify

Random streams come from numpy's PCG64 seeded with the config number (plus a
per-purpose stream id), so every array is reproducible within one numpy
version.  bf16 values are the round-to-nearest-even rounding of fp32 values
and are stored as their uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# Per-row flag bits (the "compact bit-level indicators" of the SonicSampler
# page, section 1).  The values are part of the input format.
GREEDY = 1 << 0
MASK = 1 << 1
PENALTY = 1 << 2
BIAS = 1 << 3
TOPK = 1 << 4
TOPP = 1 << 5
MINP = 1 << 6
BOUNDED_P = 1 << 7   # verify against the candidate softmax even without truncation
EXACT = 1 << 8       # untruncated rows sample over the whole vocabulary

ROW_FIELDS = ("flags", "temperature", "top_p", "min_p", "rep", "freq", "pres",
              "top_k", "hist_len", "n_bias", "position")
_ROW_DTYPES = {"flags": np.uint32, "temperature": np.float32, "top_p": np.float32,
               "min_p": np.float32, "rep": np.float32, "freq": np.float32,
               "pres": np.float32, "top_k": np.int32, "hist_len": np.int32,
               "n_bias": np.int32, "position": np.uint32}


@dataclass
class Workload:
    """One batch of inputs for a sample call (gamma == None) or a verify call."""
    name: str
    B: int
    V: int
    dtype: str                      # "f32" or "bf16" (target / sample logits)
    logits: np.ndarray              # [B_pos, V] float32, or uint16 bf16 bits
    rows: dict                      # ROW_FIELDS -> np.ndarray[B]
    history: np.ndarray             # [B, hist_stride] int32 (entries < 0 are padding)
    bitmask: Optional[np.ndarray]   # [B_pos, ceil(V/32)] uint32, bit=1 allowed; or None
    bias_tokens: np.ndarray         # [B, bias_stride] int32
    bias_values: np.ndarray         # [B, bias_stride] float32
    seeds: np.ndarray               # [B] uint64
    # verification only
    cu_draft: Optional[np.ndarray] = None     # [B+1] int32 prefix sums of gamma_r
    draft_ids: Optional[np.ndarray] = None    # [sum gamma] int32
    draft_probs: Optional[np.ndarray] = None  # [sum gamma, V] float32 or uint16 bf16 bits
    q_dtype: str = "f32"
    meta: dict = field(default_factory=dict)

    @property
    def is_verify(self) -> bool:
        return self.cu_draft is not None

    @property
    def n_positions(self) -> int:
        return int(self.logits.shape[0])

    @property
    def max_gamma(self) -> int:
        if self.cu_draft is None:
            return 0
        return int(np.max(np.diff(self.cu_draft))) if self.B else 0

    def gammas(self) -> np.ndarray:
        if self.cu_draft is None:
            return np.zeros(self.B, np.int32)
        return np.diff(self.cu_draft).astype(np.int32)

    def position_offsets(self) -> np.ndarray:
        """[B+1] first target position of each row (cu_draft[r] + r)."""
        if self.cu_draft is None:
            return np.arange(self.B + 1, dtype=np.int64)
        return self.cu_draft.astype(np.int64) + np.arange(self.B + 1)

    def logit_bytes(self) -> int:
        return self.logits.nbytes

    def counted_bytes(self, tile: int) -> int:
        """Bytes the throughput metric counts per call: logits + bitmask +
        draft probs (read once) + staging write and read (128 entries of 8
        bytes per vocab tile)."""
        z = -(-self.V // tile)
        n = self.logits.nbytes
        if self.bitmask is not None:
            n += self.bitmask.nbytes
        if self.draft_probs is not None and not self.meta.get("one_hot_drafts"):
            n += self.draft_probs.nbytes
        n += 2 * self.n_positions * z * 128 * 8
        return n


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16, returned as uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(x)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    r = r.astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


class _Streams:
    """Independent PCG64 streams per purpose, all derived from one seed."""

    def __init__(self, seed: int):
        self.seed = int(seed)

    def __call__(self, purpose: int) -> np.random.Generator:
        return np.random.Generator(np.random.PCG64([self.seed, int(purpose)]))


def _splitmix64(x: int) -> int:
    """SplitMix64 output for state x (Steele, Lea and Flood, OOPSLA 2014)."""
    m = (1 << 64) - 1
    z = (x + 0x9E3779B97F4A7C15) & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def row_seeds(cfg_seed: int, B: int) -> np.ndarray:
    return np.array([_splitmix64((cfg_seed << 32) ^ r) for r in range(B)], dtype=np.uint64)


def _zipf_boost(rng: np.random.Generator, V: int, n: int = 256, amp: float = 16.0,
                s: float = 1.1):
    toks = rng.choice(V, size=min(n, V), replace=False).astype(np.int64)
    ranks = np.arange(1, toks.size + 1, dtype=np.float64)
    return toks, (amp * ranks ** (-s)).astype(np.float32)


def low_entropy_logits(rng: np.random.Generator, V: int, sigma: float = 1.5,
                       boost: bool = True):
    """N(0, sigma) logits plus a Zipf(s=1.1) boost of 16 r^-1.1 on 256
    distinct random tokens ranked r = 1..256.  Returns (logits, boosted ids)."""
    x = rng.standard_normal(V, dtype=np.float32) * np.float32(sigma)
    toks = np.zeros(0, np.int64)
    if boost:
        toks, amp = _zipf_boost(rng, V)
        x[toks] += amp
    return x, toks


def _bitmask(rng: np.random.Generator, n_rows: int, V: int, p_allowed: float) -> np.ndarray:
    W = -(-V // 32)
    bits = rng.random((n_rows, W * 32), dtype=np.float32) < p_allowed
    bits[:, V:] = False
    return bool_to_mask_bits(bits)


def bool_to_mask_bits(bits: np.ndarray) -> np.ndarray:
    """[n, W*32] bool -> [n, W] uint32 with element i at bit i%32 of word i//32."""
    n = bits.shape[0]
    pad = (-bits.shape[1]) % 32
    if pad:
        bits = np.concatenate([bits, np.zeros((n, pad), bool)], axis=1)
    by = np.packbits(bits, axis=-1, bitorder="little")
    return np.ascontiguousarray(by).view("<u4").astype(np.uint32).reshape(n, -1)


def mask_bits_to_bool(mask: np.ndarray, V: int) -> np.ndarray:
    """[n, W] uint32 -> [n, V] bool (bit i%32 of word i//32)."""
    by = np.ascontiguousarray(mask.astype("<u4")).view(np.uint8).reshape(mask.shape[0], -1)
    b = np.unpackbits(by, axis=-1, bitorder="little")
    return b[:, :V].astype(bool)


def _empty_rows(B: int) -> dict:
    return {k: np.zeros(B, dtype=_ROW_DTYPES[k]) for k in ROW_FIELDS}


def _heterogeneous_rows(rng: np.random.Generator, B: int, hist_len: int, n_bias: int,
                        processors: bool = True, greedy_frac: float = 0.25) -> dict:
    """Per-row parameters with the config-2 distributions."""
    rows = _empty_rows(B)
    greedy = rng.random(B) < greedy_frac
    topk = rng.choice(np.array([0, 20, 128], np.int32), size=B)
    rows["temperature"][:] = rng.uniform(0.5, 1.5, B).astype(np.float32)
    rows["top_p"][:] = rng.uniform(0.8, 1.0, B).astype(np.float32)
    minp_on = rng.random(B) < 0.5
    rows["min_p"][:] = np.where(minp_on, np.float32(0.05), np.float32(0.0))
    rows["top_k"][:] = topk
    flags = np.zeros(B, np.uint32)
    flags |= np.where(greedy, GREEDY, 0).astype(np.uint32)
    flags |= np.where(topk > 0, TOPK, 0).astype(np.uint32)
    flags |= TOPP
    flags |= np.where(minp_on, MINP, 0).astype(np.uint32)
    if processors:
        flags |= MASK | PENALTY | BIAS
        rows["rep"][:] = 1.1
        rows["freq"][:] = 0.2
        rows["pres"][:] = 0.3
        rows["hist_len"][:] = hist_len
        rows["n_bias"][:] = n_bias
    else:
        rows["rep"][:] = 1.0
    rows["flags"][:] = flags
    return rows


def _history_and_bias(rng: np.random.Generator, V: int, boosted: list, H: int, NB: int):
    B = len(boosted)
    hist = np.empty((B, H), np.int32)
    btok = np.full((B, max(NB, 1)), -1, np.int32)
    bval = np.zeros((B, max(NB, 1)), np.float32)
    for r in range(B):
        from_boost = rng.random(H) < 0.5
        uni = rng.integers(0, V, H)
        bsel = boosted[r][rng.integers(0, len(boosted[r]), H)] if len(boosted[r]) else uni
        hist[r] = np.where(from_boost, bsel, uni).astype(np.int32)
        if NB:
            half = NB // 2
            a = rng.choice(boosted[r], size=half, replace=False) if len(boosted[r]) >= half \
                else rng.choice(V, size=half, replace=False)
            cand = rng.choice(V, size=min(V, NB + 2 * half + 8), replace=False)
            b = cand[~np.isin(cand, a)][:NB - half]
            ids = np.concatenate([a, b]).astype(np.int32)
            rng.shuffle(ids)
            btok[r, :NB] = ids
            bval[r, :NB] = rng.uniform(-5.0, 5.0, NB).astype(np.float32)
    return hist, btok, bval


def _to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    return np.ascontiguousarray(x, dtype=np.float32)


# --------------------------------------------------------------------------- configs

def config1(seed: int = 1) -> Workload:
    """B=4, V=32000 fp32 N(0,2) with five spike tokens +8..+12 per row; rows
    0-1 greedy, rows 2-3 T=0.7 top-k=50 top-p=0.9; no processors; seed 1."""
    B, V = 4, 32000
    st = _Streams(seed)
    g = st(0)
    x = g.standard_normal((B, V), dtype=np.float32) * np.float32(2.0)
    for r in range(B):
        toks = g.choice(V, size=5, replace=False)
        x[r, toks] += np.array([8, 9, 10, 11, 12], np.float32)
    rows = _empty_rows(B)
    rows["flags"][:] = [GREEDY, GREEDY, TOPK | TOPP, TOPK | TOPP]
    rows["temperature"][:] = [1.0, 1.0, 0.7, 0.7]
    rows["top_k"][:] = [0, 0, 50, 50]
    rows["top_p"][:] = [1.0, 1.0, 0.9, 0.9]
    rows["rep"][:] = 1.0
    return Workload("c1", B, V, "f32", x, rows, np.full((B, 1), -1, np.int32), None,
                    np.full((B, 1), -1, np.int32), np.zeros((B, 1), np.float32),
                    np.full(B, 1, np.uint64), meta={"config": 1})


def sample_workload(seed: int, B: int, V: int, dtype: str = "bf16", H: int = 256,
                    NB: int = 16, processors: bool = True, greedy_frac: float = 0.25,
                    p_allowed: float = 0.3, name: str = "sample") -> Workload:
    """Single-step heterogeneous batch with the config-2 distributions."""
    st = _Streams(seed)
    g = st(0)
    x = np.empty((B, V), np.float32)
    boosted = []
    for r in range(B):
        x[r], toks = low_entropy_logits(g, V)
        boosted.append(toks)
    rows = _heterogeneous_rows(st(1), B, H, NB, processors, greedy_frac)
    hist, btok, bval = _history_and_bias(st(2), V, boosted, max(H, 1), NB)
    if not processors:
        hist[:] = -1
    mask = _bitmask(st(3), B, V, p_allowed) if processors else None
    return Workload(name, B, V, dtype, _to_dtype(x, dtype), rows, hist, mask, btok, bval,
                    row_seeds(seed, B), meta={"seed": seed})


def config2(seed: int = 2) -> Workload:
    return sample_workload(seed, 64, 131072, "bf16", name="c2")


def topk_stress_workload(seed: int, B: int, V: int, name: str = "topk_stress") -> Workload:
    """Rows 0..B/2-1 Zipf-boosted N(0,1.5); rows B/2.. near-flat N(0,0.3);
    all stochastic, top-k=128, top-p=0.95, T=1, no processors, fp32."""
    st = _Streams(seed)
    g = st(0)
    x = np.empty((B, V), np.float32)
    for r in range(B):
        if r < B // 2:
            x[r], _ = low_entropy_logits(g, V)
        else:
            x[r] = g.standard_normal(V, dtype=np.float32) * np.float32(0.3)
    rows = _empty_rows(B)
    rows["flags"][:] = TOPK | TOPP
    rows["temperature"][:] = 1.0
    rows["top_k"][:] = 128
    rows["top_p"][:] = 0.95
    rows["rep"][:] = 1.0
    return Workload(name, B, V, "f32", x, rows, np.full((B, 1), -1, np.int32), None,
                    np.full((B, 1), -1, np.int32), np.zeros((B, 1), np.float32),
                    row_seeds(seed, B), meta={"seed": seed})


def config3(seed: int = 3) -> Workload:
    return topk_stress_workload(seed, 256, 262144, name="c3")


def _softmax_f64(z: np.ndarray) -> np.ndarray:
    # Draft-model probabilities (an input of the verify call, not a step of it).
    m = np.max(z)
    e = np.exp(z.astype(np.float64) - m)
    return e / e.sum()


def _inverse_cdf(rng: np.random.Generator, q: np.ndarray) -> int:
    c = np.cumsum(q.astype(np.float64))
    u = rng.random() * c[-1]
    return int(min(np.searchsorted(c, u, side="right"), q.size - 1))


def verify_workload(seed: int, B: int, V: int, gammas, dtype: str = "bf16",
                    q_dtype: str = "bf16", processors: bool = False,
                    greedy_frac: float = 0.25, truncation: bool = False,
                    noise: float = 0.5, H: int = 256, NB: int = 16,
                    p_allowed: float = 0.3, name: str = "verify") -> Workload:
    """Verification batch: per row, draft logits z_j from the low-entropy
    generator, q_j = softmax(z_j) (masked like the target when processors are
    on), target logits z_j + N(0, noise) for j < gamma_r and a fresh draw at the
    bonus position; draft ids drawn from q_j by inverse CDF in fp64."""
    st = _Streams(seed)
    g, gd, gn = st(0), st(4), st(5)
    gammas = np.asarray(gammas, np.int32)
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(gammas)
    npos = int(cu[-1]) + B
    tgt = np.empty((npos, V), np.float32)
    qs = np.empty((int(cu[-1]), V), np.float32)
    dids = np.empty(int(cu[-1]), np.int32)
    boosted = []
    if processors:
        mask = _bitmask(st(3), npos, V, p_allowed)
        allowed = mask_bits_to_bool(mask, V)
    else:
        mask, allowed = None, None
    p = 0
    for r in range(B):
        toks_r = []
        for j in range(int(gammas[r])):
            z, toks = low_entropy_logits(g, V)
            toks_r.append(toks)
            zq = z.copy()
            if allowed is not None:
                zq[~allowed[p + j]] = -np.inf
            q = _softmax_f64(zq)
            qs[cu[r] + j] = q.astype(np.float32)
            dids[cu[r] + j] = _inverse_cdf(gd, q)
            tgt[p + j] = z + gn.standard_normal(V, dtype=np.float32) * np.float32(noise)
        z, toks = low_entropy_logits(g, V)
        toks_r.append(toks)
        tgt[p + int(gammas[r])] = z
        boosted.append(np.unique(np.concatenate(toks_r)))
        p += int(gammas[r]) + 1
    if processors or truncation:
        rows = _heterogeneous_rows(st(1), B, H, NB, processors, greedy_frac)
    else:
        rows = _empty_rows(B)
        greedy = st(1).random(B) < greedy_frac
        rows["flags"][:] = np.where(greedy, GREEDY, 0).astype(np.uint32)
        rows["temperature"][:] = 1.0
        rows["top_p"][:] = 1.0
        rows["rep"][:] = 1.0
    hist, btok, bval = _history_and_bias(st(2), V, boosted, max(H, 1), NB)
    if not processors:
        hist[:] = -1
        btok[:] = -1
    if q_dtype == "bf16":
        qarr = f32_to_bf16_bits(qs)
    else:
        qarr = qs
    return Workload(name, B, V, dtype, _to_dtype(tgt, dtype), rows, hist, mask, btok, bval,
                    row_seeds(seed, B), cu_draft=cu, draft_ids=dids, draft_probs=qarr,
                    q_dtype=q_dtype, meta={"seed": seed})


def config4(seed: int = 4) -> Workload:
    return verify_workload(seed, 32, 131072, np.full(32, 4), "bf16", "bf16", name="c4")


def mixed_gammas(seed: int, B: int, p_single: float = 0.6, gmax: int = 7) -> np.ndarray:
    r = _Streams(seed)(6)
    single = r.random(B) < p_single
    g = r.integers(1, gmax + 1, B)
    return np.where(single, 0, g).astype(np.int32)


def mixed_workload(seed: int, B: int, V: int, dtype: str = "f32", gmax: int = 7,
                   name: str = "mixed") -> Workload:
    """60% single-step rows (gamma=0) and 40% verify rows with gamma in 1..gmax,
    all processors on with the config-2 distributions, one verify call."""
    return verify_workload(seed, B, V, mixed_gammas(seed, B, gmax=gmax), dtype, "f32",
                           processors=True, name=name)


def config5(seed: int = 5) -> Workload:
    return mixed_workload(seed, 512, 151936, "f32", name="c5")


def subset(w, rows) -> Workload:
    """The rows `rows` of a workload as a workload of their own.  Their
    original batch row indices are kept in meta["row_ids"] (random streams
    are keyed by batch row)."""
    rows = np.asarray(rows, np.int64)
    rw = {k: v[rows] for k, v in w.rows.items()}
    meta = dict(w.meta)
    meta["row_ids"] = rows.astype(np.int32)
    if not w.is_verify:
        return Workload(w.name + "_sub", len(rows), w.V, w.dtype, w.logits[rows], rw, w.history[rows],
                        None if w.bitmask is None else w.bitmask[rows], w.bias_tokens[rows],
                        w.bias_values[rows], w.seeds[rows], meta=meta)
    offs = w.position_offsets()
    gam = w.gammas()
    pos = np.concatenate([np.arange(offs[r], offs[r] + gam[r] + 1) for r in rows])
    qr = np.concatenate([np.arange(w.cu_draft[r], w.cu_draft[r + 1]) for r in rows] + [np.zeros(0, np.int64)])
    cu = np.zeros(len(rows) + 1, np.int32)
    cu[1:] = np.cumsum(gam[rows])
    return Workload(w.name + "_sub", len(rows), w.V, w.dtype, w.logits[pos], rw, w.history[rows],
                    None if w.bitmask is None else w.bitmask[pos], w.bias_tokens[rows], w.bias_values[rows],
                    w.seeds[rows], cu_draft=cu, draft_ids=w.draft_ids[qr], draft_probs=w.draft_probs[qr],
                    q_dtype=w.q_dtype, meta=meta)


def with_one_hot_drafts(w: Workload) -> Workload:
    """The same verify batch with drafts that carry no probabilities: the
    library is called with draft_probs = NULL (meta["one_hot_drafts"]), and
    draft_probs holds the equivalent one-hot q rows for the oracle."""
    d = np.asarray(w.draft_ids, np.int64)
    q = np.zeros((d.size, w.V), np.float32)
    q[np.arange(d.size), d] = 1.0
    w.draft_probs = f32_to_bf16_bits(q) if w.q_dtype == "bf16" else q
    w.meta = dict(w.meta, one_hot_drafts=True)
    w.name = w.name + "_onehot"
    return w


def with_bounded_p(w: Workload) -> Workload:
    """The same verify batch with every stochastic row flagged BOUNDED_P."""
    stoch = (w.rows["flags"] & GREEDY) == 0
    w.rows["flags"][stoch] |= np.uint32(BOUNDED_P)
    w.name = w.name + "_bounded"
    return w


def with_exact_sampling(w: Workload) -> Workload:
    """The same batch with every stochastic row untruncated and flagged EXACT
    (sampled over the whole vocabulary; the plan runs exact sampling)."""
    stoch = (w.rows["flags"] & GREEDY) == 0
    w.rows["flags"][stoch] &= ~np.uint32(TOPK | TOPP | MINP)
    w.rows["flags"][stoch] |= np.uint32(EXACT)
    w.meta = dict(w.meta, exact_sampling=True)
    w.name = w.name + "_exact"
    return w


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}
