"""How often packed 32-bit staging entries (a 16-bit key beside a 16-bit
tile-local index, the SonicSampler pages' staging format, section 3.2) would
select a different top-128 set than full 32-bit keys, on the oracle's
processed logits of the standard workloads.

The 16-bit key is the upper half of the order-preserving 32-bit key (sign,
exponent and 7 mantissa bits: bf16 precision).  Each 8192-token tile keeps
its top 128 by (16-bit key desc, tile-local index asc); the tile lists merge
by the same packed order.  The full-precision set is the oracle's own
candidate order: (32-bit key desc, token asc).

    python -m tests.key16_report
"""
import numpy as np

from oracle import oracle
from spec_verification_gb300 import workloads as W

K, TILE = 128, 8192


def key32(x: np.ndarray) -> np.ndarray:
    """Order-preserving key of fp32 values: the sign bit set for x >= 0,
    every bit flipped for x < 0."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return np.where((b >> 31) == 1, (~b) & 0xFFFFFFFF, b | 0x80000000)


def full_key_set(x: np.ndarray) -> set:
    k = key32(x).astype(np.int64)
    return set(np.lexsort((np.arange(x.size), -k))[:K].tolist())


def packed16_set(x: np.ndarray) -> set:
    k16 = (key32(x) >> 16).astype(np.int64)
    entries = []
    for t0 in range(0, x.size, TILE):
        kk = k16[t0:t0 + TILE]
        for i in np.lexsort((np.arange(kk.size), -kk))[:K]:
            entries.append((-int(kk[i]), int(i), t0 + int(i)))
    entries.sort()
    return {g for _, _, g in entries[:K]}


def position_logits(w, p: int) -> np.ndarray:
    """Processed logits of absolute position p (a verify position's earlier
    drafts join its row's history)."""
    offs = w.position_offsets()
    r = int(np.searchsorted(offs, p, side="right") - 1)
    j = int(p - offs[r])
    extra = w.draft_ids[w.cu_draft[r]:w.cu_draft[r] + j] if w.cu_draft is not None else ()
    return oracle.prelude(w, r, int(p), extra)[0]


def study(w, n: int, seed: int = 0) -> dict:
    rng = np.random.default_rng(seed)
    pos = rng.choice(w.n_positions, size=min(n, w.n_positions), replace=False)
    swapped, moved = [], []
    for p in pos:
        x = position_logits(w, int(p))
        a, b = full_key_set(x), packed16_set(x)
        xf = x.astype(np.float64)
        pr = np.exp(xf - xf.max())
        pr /= pr.sum()
        swapped.append(len(a - b))
        moved.append(abs(pr[list(a - b)].sum() - pr[list(b - a)].sum()))
    swapped = np.array(swapped)
    return {"positions": len(pos), "differ": int((swapped > 0).sum()),
            "swapped_mean": float(swapped.mean()), "swapped_max": int(swapped.max()),
            "mass_median": float(np.median(moved)), "mass_max": float(np.max(moved))}


if __name__ == "__main__":
    for name, make, n in [("c2", W.config2, 64), ("c3", W.config3, 128), ("c5", W.config5, 200)]:
        s = study(make(), n)
        print(f"{name}: {s['differ']} of {s['positions']} positions select another set; "
              f"tokens swapped mean {s['swapped_mean']:.2f} max {s['swapped_max']}; "
              f"full-softmax mass moved median {s['mass_median']:.2e} max {s['mass_max']:.2e}")
