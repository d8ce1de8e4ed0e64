// Stage 1 of the two-stage top-k (SonicSampler 3.2, Fig. 1 top): the logits
// prelude (grammar mask, penalties, bias, temperature) fused with a local
// top-128, every logit streamed from HBM once.
//
// Work split.  Each target position's row is cut into Z_v stages of B_N
// tokens; the npos * Z_v stages, position-major, are divided into contiguous
// ranges, one per CTA: G = min(grid, npos * Z_v) nearly equal ranges, or,
// when the grid holds two or more CTAs per position, ranges that split each
// position evenly and never cross a position boundary.  The
// part of a CTA's range inside one row is a segment, so a row has 1..Z_v
// segments; each segment leaves its exact top-128 (packed key << 32 | ~token)
// in the staging buffer and stage 2 merges a row's segments (seg_start /
// seg_cta give both kernels the same split).  This generalises the pages'
// one-list-per-tile: a list per run of tiles keeps the property stage 2 needs
// (every element of the row's top-128 is in its own list's top-128) while the
// selection work falls from once per tile to once per segment.
//
// Per CTA:
//  - a ring of shared-memory slots is filled several stages ahead by bulk
//    copies (cp.async.bulk completing on one mbarrier per slot): the stage's
//    logits and, when the rows allow it, its grammar-mask words;
//  - per segment, a candidate buffer and a cut with two invariants:
//    (a) every element seen in the segment whose packed value is >= cut is
//        in the buffer;
//    (b) at least min(128, elements seen) buffer entries are >= cut.
//    The segment's first stage takes the cut from the per-thread maxima (the
//    16th largest of each warp's 32 maxima, minimum over the 8 warps, so 128
//    maxima lie at or above it); afterwards a thread whose 32 elements all
//    fall below the cut does only the prelude and a NaN-propagating running
//    maximum, and the rare elements at or above it are appended.  When the
//    buffer passes kRaiseAt entries one histogram pass raises the cut to the
//    lower edge of the bin holding its 128th entry (dropping what lies
//    below), or, if that frees too little, it is cut back to its exact
//    top-128;
//  - history / draft / bias tokens need their count and bias entries, so they
//    are kept out of that path: per segment they are listed in a hash table
//    (which a rare append consults when the appending thread's 32-bit filter
//    of the listed tokens among its elements does not rule its token out)
//    and their exact values, read straight from HBM, are the segment's first
//    candidates; very long histories (and
//    verify positions that need the full-vocabulary normaliser) use a
//    per-stage count table instead, appending those tokens as their stage
//    streams through;
//  - what the fast path cannot certify (the buffer overflows within a stage,
//    or the first stage's cut admits fewer than 128 elements: few finite
//    values, NaN, penalised maxima) is rolled back and replaced by an exact
//    radix select of the stage's top-128, after which the cut is raised to
//    the stage's 128th value.  Both invariants survive every step.
//  - the segment's status (NaN seen; history / bias ids beyond the
//    vocabulary) and, for untruncated stochastic verify positions,
//    (max, sum exp(x - max)) over the segment go beside the list.
#pragma once

#include <type_traits>

#include "ss_common.cuh"
#include "ss_stage2.cuh"

namespace ss {

namespace {

constexpr uint32_t kDrainSpin = 1u << 22;  // polls of the final drain of copies in flight
// Loops of the cold paths (selection, hashing, raises) are kept rolled
// (#pragma unroll 1): each kernel instance is then about 207 KB of code
// instead of 275 KB, and measured 3-5 % faster.
constexpr int kMaxSlots = 4;         // ring slots at most
constexpr int kCap = 1024;           // candidate buffer entries
constexpr int kRaiseAt = 384;        // buffer fill that triggers a cut raise
constexpr int kCompactAt = 512;      // fill after a raise that triggers an exact compaction (<= kCap - kK)
constexpr int kHashBits = 10;
constexpr int kHash = 1 << kHashBits;  // hash slots for a segment's history / bias tokens
constexpr int kHashMax = 512;        // tokens a segment may list in the hash table
constexpr int kBiasPre = 64;         // bias entries prefetched per segment
constexpr int kPre = kNT;            // history / draft ids prefetched per segment
constexpr int kPT = 32;              // elements per thread per chunk
constexpr int kChunk = kPT * kNT;    // elements per chunk (a stage is 1 or 2 chunks)
constexpr float kLog2e = 1.4426950408889634f;

static_assert(kCompactAt <= kCap - kK, "a stage fallback appends 128 entries after the rollback");

// One segment's row bookkeeping, copied with cp.async one segment ahead.
struct __align__(16) RowBuf {
  ss_bias_entry bias[kBiasPre];  // bias[r][e]      (e < min(bias_stride, kBiasPre))
  int hist[kPre];                // history[r][h]   (h < min(hist_stride, kPre))
  int draft[kPre];               // drafts of the row before this position (< min(j, kPre))
  ss_row_params rp;
  int pos, r, j, c0, c1;         // position, row, draft index, cu_draft[r], cu_draft[r + 1]
  int pad[3];
};

struct __align__(16) S1Smem {
  SelectSmem sel;
  unsigned long long mbar[kMaxSlots];
  unsigned long long slots[kNT / 32];
  unsigned long long cut;
  double red[kNT / 32];
  float tw[kNT / 32];
  float lm[kNT / 32];
  int cnt[3];  // appends of stage k go to cnt[k % 3]
  int dead, nan_flag, nf, out_cnt;
  int s2_go;  // fused form: this CTA completed the position's last segment
  uint32_t rowbad;  // SS_ST_BAD_HIST / SS_ST_BAD_BIAS of the segment's row
  int pad2[2];
  unsigned long long gmax;  // the segment's Gumbel-max so far (exact sampling)
};

struct Layout {
  size_t ring, mask, cand, tmp, out, hkey, hval, ftok, finfo, sm, rb, total;
};

__host__ __device__ inline size_t up128(size_t x) { return (x + 127) & ~(size_t)127; }

__host__ __device__ inline Layout layout(int BN, int esz, int nslot) {
  Layout L;
  size_t o = 0;
  L.ring = o;  o = up128(o + (size_t)nslot * BN * esz);
  L.mask = o;  o = up128(o + (size_t)nslot * (BN / 8));
  L.cand = o;  o = up128(o + (size_t)kCap * 8);
  L.tmp = o;   o = up128(o + ((size_t)kCap * 8 > (size_t)BN * 2 ? (size_t)kCap * 8 : (size_t)BN * 2));
  L.out = o;   o = up128(o + (size_t)kK * 8);
  L.hkey = o;  o = up128(o + (size_t)kHash * 4);
  L.hval = o;  o = up128(o + (size_t)kHash * 4);
  L.ftok = o;  o = up128(o + (size_t)kHashMax * 4);
  L.finfo = o; o = up128(o + (size_t)kHashMax * 4);
  L.sm = o;    o = up128(o + sizeof(S1Smem));
  L.rb = o;    o = up128(o + 2 * sizeof(RowBuf));
  L.total = o;
  return L;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long* m) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(m)) : "memory");
}

__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, unsigned long long* m) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(m))
               : "memory");
}

// Waits for the phase of parity `parity` of mbarrier m to complete, polling
// at most `limit` times; false if it did not.  hint_ns == 0: each poll may
// suspend the thread in hardware until the phase completes or the hardware's
// time limit passes.  hint_ns > 0: each poll tests once, without suspending,
// and then sleeps about hint_ns nanoseconds.
__device__ __forceinline__ bool mbar_wait(unsigned long long* m, uint32_t parity, uint32_t limit, uint32_t hint_ns) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t ok;
    if (hint_ns == 0u) {
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(ok)
          : "r"(smem_u32(m)), "r"(parity)
          : "memory");
    } else {
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(ok)
          : "r"(smem_u32(m)), "r"(parity)
          : "memory");
      if (!ok) __nanosleep(hint_ns);
    }
    if (ok) return true;
  }
  return false;
}

// The ring's wait limits, from the plan.
struct WaitCfg {
  uint32_t spin_limit, spin_hint_ns;
};

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// max that returns NaN if either operand is NaN
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

template <bool BF16>
__device__ __forceinline__ float raw_at(const unsigned char* ring, int i) {
  if constexpr (BF16) return __uint_as_float((uint32_t) reinterpret_cast<const uint16_t*>(ring)[i] << 16);
  else return reinterpret_cast<const float*>(ring)[i];
}

template <bool BF16>
__device__ __forceinline__ float vec_elem(const uint4& v, int jj) {
  if constexpr (BF16) {
    const uint32_t w = (jj >> 1) == 0 ? v.x : (jj >> 1) == 1 ? v.y : (jj >> 1) == 2 ? v.z : v.w;
    return (jj & 1) ? bf16_hi(w) : bf16_lo(w);
  } else {
    const uint32_t w = jj == 0 ? v.x : jj == 1 ? v.y : jj == 2 ? v.z : v.w;
    return __uint_as_float(w);
  }
}

// Stage element li of chunk ch for vector v, lane element jj: vectors of a
// chunk are kNT apart so that each load is one coalesced 16-byte access.
template <int VEC>
__device__ __forceinline__ int elem_index(int ch, int v, int jj) {
  constexpr int NV = kPT / VEC;
  return ((ch * NV + v) * kNT + (int)threadIdx.x) * VEC + jj;
}

// Everything the out-of-line paths need to recompute a stage element's
// processed value, by value (nothing of the hot loop's state is addressed).
// A row's temperature step: x / T, one IEEE fp32 division (rounded to
// nearest) for stochastic rows; greedy rows keep x.
struct Temp {
  float T;
  bool stoch;
};
__device__ __forceinline__ Temp temp_of(const RowCtx& rc) { return Temp{rc.T, rc.stoch}; }
__device__ __forceinline__ float temper(float x, Temp tp) { return tp.stoch ? __fdiv_rn(x, tp.T) : x; }

// The largest raw value x0 (or less) whose processed value lies below the
// packed cut: every x <= x0 has fl(x / T) < cut's value, since rounding x / T
// (T > 0) is monotone in x.  NaN (no raw value is skipped) when the cut
// admits everything or the search does not settle.
__device__ __noinline__ float raw_threshold(unsigned long long cut, Temp tp) {
  const uint32_t ck = pk_key(cut);
  if (ck <= kKeyNegInf) return __int_as_float(0x7FC00000);
  const float cf = key2f(ck);  // processed values below cf key below ck
  if (!tp.stoch) return nextafterf(cf, -INFINITY);
  float x = __fmul_rn(cf, tp.T);
#pragma unroll 1
  for (int i = 0; i < 8; ++i) {
    if (__fdiv_rn(x, tp.T) < cf) return x;
    x = nextafterf(x, -INFINITY);
  }
  return __int_as_float(0x7FC00000);
}

// x / T for the normaliser partials only, which tolerate an ulp: the
// quotient q = RN(x * r) with r = RN(1 / T), corrected once by the residual
// x - q * T (Markstein's division step, IBM J. Res. Dev. 34(1), 1990).
__device__ __forceinline__ float quot_lse(float x, float T, float r) {
  const float q = __fmul_rn(x, r);
  return __fmaf_rn(__fmaf_rn(-q, T, x), r, q);
}

struct StageCtx {
  const unsigned char* ring;
  const uint32_t* msl;           // the stage's mask words (shared or global), or null
  const ss_bias_entry* bl;       // the row's bias list (shared copy when it fits)
  const int* hkey;
  const uint32_t* hval;
  const uint16_t* aux;
  RowCtx rc;
  int t0, nt;
  bool hashed, staged;
};

__device__ __forceinline__ uint32_t hash_of(int tok) { return ((uint32_t)tok * 0x9E3779B1u) >> (32 - kHashBits); }

// Slot of token tok in the segment's hash table, or -1.
__device__ __forceinline__ int hash_find(const int* hkey, int tok) {
  uint32_t h = hash_of(tok);
#pragma unroll 1
  for (int probe = 0; probe < kHash; ++probe) {
    const int k = hkey[h];
    if (k == tok) return (int)h;
    if (k == -1) return -1;
    h = (h + 1) & (kHash - 1);
  }
  return -1;
}

// History count (bits 0..30) and bias flag (bit 31) of stage element li.
__device__ __forceinline__ uint32_t flag_info(const StageCtx& s, int li) {
  if (s.hashed) {
    const int h = hash_find(s.hkey, s.t0 + li);
    return h >= 0 ? s.hval[h] : 0u;
  }
  if (s.staged) {
    const uint32_t a = s.aux[li];
    return (a & 0x7FFFu) | ((a & 0x8000u) << 16);
  }
  return 0u;
}

// Processed value of stage element li with history count / bias flag `info`
// (the prelude's fp32 steps in order: mask, penalties, bias, temperature).
template <bool BF16>
__device__ __forceinline__ float value_with(const StageCtx& s, int li, uint32_t info) {
  float v = raw_at<BF16>(s.ring, li);
  if (s.msl && ((s.msl[li >> 5] >> (li & 31)) & 1u) == 0u) v = -INFINITY;
  if (info) v = apply_penalty_bias(v, info & 0x7FFFFFFFu, (info >> 31) != 0u, s.t0 + li, s.rc, s.bl);
  return apply_temperature(v, s.rc);
}

// Exact top-`need` of the stage, appended to cand[cbase + *acnt]: MSB-first
// radix select on the 32-bit keys, then the lowest tokens among elements equal
// to the boundary key.  Thread t owns the contiguous elements [t*E, t*E + E)
// so that token order is (thread, element).  Sets sm.nan_flag on NaN.
template <bool BF16>
__device__ __noinline__ void stage_exact(const StageCtx& s, S1Smem& sm, int* acnt, int cbase, unsigned long long* cand,
                                         int need, int E) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int base = tid * E;
  // hash mode: the listed tokens are candidates already and take no part
  auto key_of = [&](int li, uint32_t& key) -> bool {
    if (li >= s.nt) return false;
    if (s.hashed && hash_find(s.hkey, s.t0 + li) >= 0) return false;
    const float v = value_with<BF16>(s, li, s.staged ? flag_info(s, li) : 0u);
    key = (v != v) ? kKeyNegInf : f2key(v);
    return true;
  };
  bool nan_seen = false;
  for (int k = 0; k < E; ++k) {
    const int li = base + k;
    if (li >= s.nt || (s.hashed && hash_find(s.hkey, s.t0 + li) >= 0)) continue;
    const float v = value_with<BF16>(s, li, s.staged ? flag_info(s, li) : 0u);
    nan_seen |= (v != v);
  }
  if (nan_seen) sm.nan_flag = 1;
  uint32_t prefix = 0u, pmask = 0u;
  int rem = need;
#pragma unroll 1
  for (int d = 0; d < 4; ++d) {
    const int shift = 24 - 8 * d;
    sm.sel.hist[tid & 255] = 0u;
    __syncthreads();
    for (int k = 0; k < E; ++k) {
      uint32_t key = 0u;
      const bool in = key_of(base + k, key);
      const bool match = in && ((key & pmask) == prefix);
      const uint32_t bin = match ? ((key >> shift) & 255u) : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, bin);
      if (match && lane == __ffs(peers) - 1) atomicAdd(&sm.sel.hist[bin], (uint32_t)__popc(peers));
    }
    __syncthreads();
    boundary_bin(sm.sel, rem);
    rem -= sm.sel.above;
    prefix |= (uint32_t)min(max(sm.sel.bstar, 0), 255) << shift;
    pmask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t kstar = prefix;
  int ties = 0;
  for (int k = 0; k < E; ++k) {
    uint32_t key;
    const int li = base + k;
    if (!key_of(li, key)) continue;
    if (key > kstar) {
      const int q = cbase + atomicAdd(acnt, 1);
      if (q < kCap) cand[q] = pack(key, (uint32_t)(s.t0 + li));
    } else if (key == kstar) {
      ++ties;
    }
  }
  int total;
  const int incl = block_inclusive_scan(ties, sm.sel.scan, &total);
  int rank = incl - ties;
  for (int k = 0; k < E && rank < rem; ++k) {
    uint32_t key;
    const int li = base + k;
    if (key_of(li, key) && key == kstar) {
      const int q = cbase + atomicAdd(acnt, 1);
      if (q < kCap) cand[q] = pack(kstar, (uint32_t)(s.t0 + li));
      ++rank;
    }
  }
  __syncthreads();
}

// Exact top-`need` of cand[0..n) (distinct values) to emit(); lo / hi are the
// smallest and largest entries, found here.  All threads call.
template <class Emit>
__device__ __forceinline__ void select_top(unsigned long long* cand, unsigned long long* tmp, int n, int need,
                                           S1Smem& sm, Emit emit) {
  unsigned long long mn = ~0ull, mx = 0ull;
#pragma unroll 1
  for (int i = threadIdx.x; i < n; i += kNT) {
    const unsigned long long c = cand[i];
    mn = c < mn ? c : mn;
    mx = c > mx ? c : mx;
  }
  const unsigned long long lo = block_min_u64(mn, sm.slots);
  const unsigned long long hi = block_max_u64(mx, sm.slots);
  block_select(cand, tmp, n, need, lo, hi, sm.sel, emit);
}

// Cut the buffer back to its exact top-128; returns the new cut (the 128th).
__device__ __noinline__ unsigned long long compact(unsigned long long* cand, unsigned long long* tmp,
                                                   unsigned long long* outb, int n, S1Smem& sm) {
  if (threadIdx.x == 0) sm.out_cnt = 0;
  __syncthreads();
  select_top(cand, tmp, n, kK, sm, [&](unsigned long long c) {
    const int q = atomicAdd(&sm.out_cnt, 1);
    if (q < kK) outb[q] = c;
  });
  const int t = threadIdx.x;
  const unsigned long long c = t < kK ? outb[t] : ~0ull;
  if (t < kK) cand[t] = c;
  return block_min_u64(c, sm.slots);
}

// Raise the cut with one 256-bin histogram of the buffer over [cut, max]: the
// new cut is the lower edge of the bin holding the 128th largest entry, so at
// least 128 entries stay at or above it, and the entries below it leave the
// buffer.  Returns the new cut (never below `cut`) and the new count.  Entries below `cut` (left by a stage fallback) count in bin 0.
struct Raised {
  unsigned long long cut;
  int n;
};
__device__ __noinline__ Raised raise_cut(unsigned long long* cand, unsigned long long* tmp, int n,
                                         unsigned long long cut, S1Smem& sm) {
  const int tid = threadIdx.x;
  if (tid < 256) sm.sel.hist[tid] = 0u;
  if (tid == 0) sm.out_cnt = 0;
  unsigned long long mx = 0ull;
#pragma unroll 1
  for (int i = tid; i < n; i += kNT) mx = cand[i] > mx ? cand[i] : mx;
  mx = block_max_u64(mx, sm.slots);
  const int shift = mx > cut ? max(0, 64 - __clzll((long long)(mx - cut)) - 8) : 0;
  if (mx > cut)
#pragma unroll 1
    for (int i = tid; i < n; i += kNT) atomicAdd(&sm.sel.hist[bin_of(cand[i], cut, shift)], 1u);
  __syncthreads();
  boundary_bin(sm.sel, kK);
  const int bstar = mx > cut ? sm.sel.bstar : 0;
  if (bstar <= 0) {  // no progress: keep everything
    __syncthreads();
    return Raised{cut, n};
  }
  const unsigned long long nc = cut + ((unsigned long long)bstar << shift);
#pragma unroll 1
  for (int i = tid; i < n; i += kNT) {
    const unsigned long long c = cand[i];
    if (c >= nc) tmp[atomicAdd(&sm.out_cnt, 1)] = c;
  }
  __syncthreads();
  // the count is returned, read before the final barrier: a caller that read
  // sm.out_cnt after it could race with thread 0 resetting it for the next
  // selection (compact, the segment end), and a warp that saw the reset count
  // would take other branches (and barriers) than the rest of the block
  const int m = sm.out_cnt;
#pragma unroll 1
  for (int i = tid; i < m; i += kNT) cand[i] = tmp[i];
  __syncthreads();
  return Raised{nc, m};
}

// Load chunk ch of the stage with the mask applied (masked elements -inf) but
// not the temperature: raw values, which the cut tests compare with the cut's
// raw threshold; returns their NaN-propagating maximum.  MASK: msl holds the stage's mask words (shared or
// global memory).  FULL: the stage has B_N tokens (otherwise elements past
// the last token read as -inf and are never appended).
template <bool BF16, bool MASK, bool FULL>
__device__ __forceinline__ float load_chunk(const unsigned char* ring, const uint32_t* msl, int ch, int nt,
                                            float (&x)[kPT]) {
  constexpr int VEC = BF16 ? 8 : 4;
  constexpr int NV = kPT / VEC;
  float m = -INFINITY;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int e0 = elem_index<VEC>(ch, v, 0);
    const uint4 raw = *reinterpret_cast<const uint4*>(ring + (size_t)e0 * (BF16 ? 2 : 4));
    uint32_t bits = 0xFFFFFFFFu;
    if constexpr (MASK) bits = (FULL || e0 < nt) ? msl[e0 >> 5] >> (e0 & 31) : 0u;
#pragma unroll
    for (int jj = 0; jj < VEC; ++jj) {
      float val = vec_elem<BF16>(raw, jj);
      if constexpr (MASK) {
        if (((bits >> jj) & 1u) == 0u) val = -INFINITY;
      }
      if (!FULL && e0 + jj >= nt) val = -INFINITY;
      x[v * VEC + jj] = val;
    }
  }
  // NaN-propagating maximum as a tree (depth 4, not a chain of 16)
  float t8[kPT / 2];
#pragma unroll
  for (int e = 0; e < kPT / 2; ++e) t8[e] = fmax_nan(x[2 * e], x[2 * e + 1]);
#pragma unroll
  for (int w = kPT / 4; w >= 1; w >>= 1)
#pragma unroll
    for (int e = 0; e < w; ++e) t8[e] = fmax_nan(t8[e], t8[e + w]);
  m = t8[0];
  return m;
}

template <bool BF16>
__device__ __forceinline__ float load_chunk_sel(bool mask, bool full, const unsigned char* ring, const uint32_t* msl,
                                                int ch, int nt, float (&x)[kPT]) {
  if (mask)
    return full ? load_chunk<BF16, true, true>(ring, msl, ch, nt, x)
                : load_chunk<BF16, true, false>(ring, msl, ch, nt, x);
  return full ? load_chunk<BF16, false, true>(ring, msl, ch, nt, x)
              : load_chunk<BF16, false, false>(ring, msl, ch, nt, x);
}

// Vector v of chunk ch of a full stage with the mask applied (raw values,
// as load_chunk gives them).
template <bool BF16, bool MASK>
__device__ __forceinline__ void load_vec(const unsigned char* ring, const uint32_t* msl, int ch, int v,
                                         float* y) {
  constexpr int VEC = BF16 ? 8 : 4;
  const int e0 = elem_index<VEC>(ch, v, 0);
  const uint4 raw = *reinterpret_cast<const uint4*>(ring + (size_t)e0 * (BF16 ? 2 : 4));
  uint32_t bits = 0xFFFFFFFFu;
  if constexpr (MASK) bits = msl[e0 >> 5] >> (e0 & 31);
#pragma unroll
  for (int jj = 0; jj < VEC; ++jj) {
    float val = vec_elem<BF16>(raw, jj);
    if constexpr (MASK) {
      if (((bits >> jj) & 1u) == 0u) val = -INFINITY;
    }
    y[jj] = val;
  }
}

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// NaN-propagating maxima of the RAW values of chunk ch (no mask, no
// temperature), per vector in vm and overall.  A chunk whose raw maximum m
// is at most the raw threshold of the cut (raw_threshold) holds no processed
// value at or above the cut (masked values are -inf).
template <bool BF16>
__device__ __forceinline__ float raw_chunk_max(const unsigned char* ring, int ch, float (&vm)[kPT / (BF16 ? 8 : 4)]) {
  constexpr int VEC = BF16 ? 8 : 4;
  constexpr int NV = kPT / VEC;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int e0 = elem_index<VEC>(ch, v, 0);
    const uint4 raw = *reinterpret_cast<const uint4*>(ring + (size_t)e0 * (BF16 ? 2 : 4));
    if constexpr (BF16) {
      const uint32_t c = bf16x2_max_nan(bf16x2_max_nan(raw.x, raw.y), bf16x2_max_nan(raw.z, raw.w));
      vm[v] = fmax_nan(bf16_lo(c), bf16_hi(c));
    } else {
      vm[v] = fmax_nan(fmax_nan(__uint_as_float(raw.x), __uint_as_float(raw.y)),
                       fmax_nan(__uint_as_float(raw.z), __uint_as_float(raw.w)));
    }
  }
  float t[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) t[v] = vm[v];
#pragma unroll
  for (int w = NV / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int e = 0; e < w; ++e) t[e] = fmax_nan(t[e], t[e + w]);
  return t[0];
}

// The value the stream computes for stage element li (mask and temperature:
// the same fp32 steps as load_chunk, so the same bits).
template <bool BF16>
__device__ __forceinline__ float stream_value(const unsigned char* ring, const uint32_t* msl, Temp tp, int li) {
  float v = raw_at<BF16>(ring, li);
  if (msl && ((msl[li >> 5] >> (li & 31)) & 1u) == 0u) v = -INFINITY;
  return temper(v, tp);
}

// 2^x by the hardware approximation (PTX ex2.approx, relative error about
// 2^-22): the normaliser partials feed only the full-vocabulary acceptance
// test, whose stated tolerance is 1e-5 relative.  ex2(-inf) = +0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Exact sampling: this thread's Gumbel-max of l_i + g_i over chunk ch, the
// processed values recomputed from the slot (the same fp32 steps as
// load_chunk) so that the streaming loop keeps its registers.  One Philox
// block per 4 consecutive tokens: counter (i / 4, position, row, 0), word
// i % 4.  Tokens the count table lists (aux != 0) join with their exact values
// elsewhere; NaN and -inf values take no part.
template <bool BF16>
__device__ __noinline__ void chunk_gmax(const unsigned char* ring, const uint32_t* msl, Temp tp, int ch, int nt,
                                        bool full, const uint16_t* aux, int t0, uint32_t gpos, uint32_t row,
                                        const uint64_t* seeds, unsigned long long* gmax) {
  constexpr int VEC = BF16 ? 8 : 4;
  const uint64_t seed = __ldg(seeds + row);
  unsigned long long best = 0ull;
  constexpr int NV = kPT / VEC;
  for (int v = 0; v < NV; ++v) {
    const int e0 = elem_index<VEC>(ch, v, 0);
#pragma unroll
    for (int hb = 0; hb < VEC / 4; ++hb) {
      const int b0 = e0 + 4 * hb;
      if (!full && b0 >= nt) break;
      uint32_t c0 = (uint32_t)(t0 + b0) >> 2, c1 = gpos, c2 = row, c3 = 0u;
      philox10(c0, c1, c2, c3, (uint32_t)seed, (uint32_t)(seed >> 32));
      const uint32_t wd[4] = {c0, c1, c2, c3};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int li = b0 + k;
        if (!full && li >= nt) break;
        if (aux && aux[li] != 0u) continue;
        const float xv = stream_value<BF16>(ring, msl, tp, li);
        if (xv > -INFINITY) {
          const float sc = __fadd_rn(xv, gumbel_of(word_to_uniform(wd[k])));
          const unsigned long long pk = pack(f2key(sc), (uint32_t)(t0 + li));
          best = pk > best ? pk : best;
        }
      }
    }
  }
  if (best) atomicMax(gmax, best);
}

// Running (max, sum exp(x - max)) of one thread; -inf (and NaN) terms add nothing.
__device__ __forceinline__ void lse_add(float& M, float& S, float v) {
  if (!(v > -INFINITY)) return;
  const float Mn = fmaxf(M, v);
  S = S * exp2f((M - Mn) * kLog2e) + exp2f((v - Mn) * kLog2e);
  M = Mn;
}

// ------------------------------------------------------------------ rows with penalties or bias
// These paths run once per segment (or per stage of a long-history row);
// the AUX = false variants hold none of them.  (Kept out of line they made
// the AUX = true variant 3 % slower, so they are inlined.)

// One segment's history / draft / bias lists.
struct AuxRow {
  const int32_t* hrow;       // the row's history (null: penalties off)
  const int32_t* drafts;     // the row's drafts before this position (cu_draft[r])
  const ss_bias_entry* brow; // the row's bias entries (null: bias off)
  const RowBuf* cb;          // their prefetched heads (shared memory)
  int hist_len, jn, n_bias;  // list lengths (0 when the processor is off)
};

__device__ __forceinline__ int aux_hist(const AuxRow& a, int h) { return h < kPre ? a.cb->hist[h] : __ldg(a.hrow + h); }
__device__ __forceinline__ int aux_draft(const AuxRow& a, int s) { return s < kPre ? a.cb->draft[s] : __ldg(a.drafts + s); }
__device__ __forceinline__ int aux_bias_tok(const AuxRow& a, int e) {
  return e < kBiasPre ? a.cb->bias[e].token : a.brow[e].token;
}

// A thread's listed tokens (hash mode): their logits and mask words, loaded
// at set-up and used once the first stage has been scanned; and the thread's
// filter of the listed tokens among the elements it streams (own_bit).
struct Listed {
  float raw[kHashMax / kNT];
  uint32_t mw[kHashMax / kNT];
  uint32_t own;
};

// The streaming loop gives stage element li (li = ((ch * NV + v) * kNT + tid)
// * VEC + jj, stages starting at multiples of B_N) to thread (li / VEC) % kNT.
// Of the tokens a thread streams in a segment, token tok maps to bit
// own_bit(tok) of a 32-bit filter: a hit whose bit is clear in the thread's
// filter is no listed token, so the table is consulted only when it is set
// (about one hit in 30 when a segment lists 512 tokens).  B_N / (kNT * VEC)
// is a multiple of 32 / VEC, so the bit of an element is the same whether
// counted from the token or from the stage.
template <bool BF16>
__device__ __forceinline__ int own_owner(int tok) {
  constexpr int VEC = BF16 ? 8 : 4;
  return (tok / VEC) % kNT;
}
template <bool BF16>
__device__ __forceinline__ uint32_t own_bit(int i) {
  constexpr int VEC = BF16 ? 8 : 4;
  return 1u << (((i / (kNT * VEC)) * VEC + i % VEC) & 31);
}

// Segment set-up of a row with penalties or bias.  History / bias ids beyond
// the vocabulary are reported in *rowbad.  In hash mode the segment's history,
// draft and bias tokens inside [seg_lo, seg_hi) are listed in the hash table
// (hkey / hval: count, bias flag in bit 31), then compacted to ftok / finfo
// (*nf entries), their logits (row_logits) and mask words (mask_row, or none)
// are loaded, and each thread's filter (own_bit) is built in omask (kNT
// words of scratch).  All threads call; the barriers are uniform; the first
// one also publishes the caller's counter resets.
template <bool BF16>
__device__ __forceinline__ Listed seg_aux_setup(AuxRow a, bool hashed, int V, int seg_lo, int seg_hi, int* hkey,
                                             uint32_t* hval, int* ftok, uint32_t* finfo, int* nf,
                                             uint32_t* rowbad, const void* row_logits,
                                             const uint32_t* mask_row, uint32_t* omask) {
  const int tid = threadIdx.x;
  Listed ls;
#pragma unroll
  for (int k = 0; k < kHashMax / kNT; ++k) {
    ls.raw[k] = 0.0f;
    ls.mw[k] = 0xFFFFFFFFu;
  }
  ls.own = 0u;
  if (hashed) {
    for (int q = tid; q < kHash; q += kNT) {
      hkey[q] = -1;
      hval[q] = 0u;
    }
    omask[tid] = 0u;
  }
  __syncthreads();
  // history / bias ids beyond the vocabulary are ignored and reported
  for (int h = tid; h < a.hist_len; h += kNT)
    if (aux_hist(a, h) >= V) atomicOr(rowbad, (uint32_t)SS_ST_BAD_HIST);
  for (int e = tid; e < a.n_bias; e += kNT)
    if (aux_bias_tok(a, e) >= V) atomicOr(rowbad, (uint32_t)SS_ST_BAD_BIAS);
  if (!hashed) return ls;
  auto insert = [&](int tok, uint32_t add, uint32_t orv) {
    if (tok < seg_lo || tok >= seg_hi) return;  // also drops padding (< 0) and ids >= V
    uint32_t h = hash_of(tok);
#pragma unroll 1
    for (int probe = 0; probe < kHash; ++probe) {
      const int old = atomicCAS(&hkey[h], -1, tok);
      if (old == -1 || old == tok) {
        if (add) atomicAdd(&hval[h], add);
        if (orv) atomicOr(&hval[h], orv);
        return;
      }
      h = (h + 1) & (kHash - 1);
    }
  };
  for (int h = tid; h < a.hist_len; h += kNT) insert(aux_hist(a, h), 1u, 0u);
  for (int s = tid; s < a.jn; s += kNT) insert(aux_draft(a, s), 1u, 0u);
  for (int e = tid; e < a.n_bias; e += kNT) insert(aux_bias_tok(a, e), 0u, 0x80000000u);
  __syncthreads();
  for (int q = tid; q < kHash; q += kNT) {
    const int tok = hkey[q];
    if (tok >= 0) {
      const int i = atomicAdd(nf, 1);
      ftok[i] = tok;
      finfo[i] = hval[q];
      atomicOr(&omask[own_owner<BF16>(tok)], own_bit<BF16>(tok));
    }
  }
  __syncthreads();
  ls.own = omask[tid];
  const int nfl = *nf;
#pragma unroll
  for (int k = 0; k < kHashMax / kNT; ++k) {
    const int i = tid + k * kNT;
    if (i < nfl) {
      const int tok = ftok[i];
      ls.raw[k] = BF16 ? __uint_as_float((uint32_t)__ldg(static_cast<const unsigned short*>(row_logits) + tok) << 16)
                       : __ldg(static_cast<const float*>(row_logits) + tok);
      if (mask_row) ls.mw[k] = __ldg(mask_row + (tok >> 5));
    }
  }
  return ls;
}

// The listed tokens' exact processed values (hash mode) as the segment's
// first candidates cand[0 .. nf).  Returns whether one was NaN.
__device__ __forceinline__ bool listed_candidates(Listed ls, int nf, const int* ftok, const uint32_t* finfo, RowCtx rc,
                                               const ss_bias_entry* bl, unsigned long long* cand) {
  bool nan = false;
#pragma unroll
  for (int k = 0; k < kHashMax / kNT; ++k) {
    const int i = (int)threadIdx.x + k * kNT;
    if (i < nf) {
      const int tok = ftok[i];
      const uint32_t info = finfo[i];
      float v = ls.raw[k];
      if (((ls.mw[k] >> (tok & 31)) & 1u) == 0u) v = -INFINITY;
      v = apply_penalty_bias(v, info & 0x7FFFFFFFu, (info >> 31) != 0u, tok, rc, bl);
      v = apply_temperature(v, rc);
      nan |= v != v;
      cand[i] = pack(v != v ? kKeyNegInf : f2key(v), (uint32_t)tok);
    }
  }
  return nan;
}

// Per-stage count table of a long-history row (or a normaliser position
// with processors): aux[li] = history count of stage element li, bit 15 =
// a bias entry names it.  All threads call; two uniform barriers.
__device__ __forceinline__ void count_table(AuxRow a, uint16_t* aux, int BN, int t0, int nt) {
  const int tid = threadIdx.x;
  uint4* a4 = reinterpret_cast<uint4*>(aux);
  for (int w = tid; w < BN / 8; w += kNT) a4[w] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  uint32_t* a32 = reinterpret_cast<uint32_t*>(aux);
  auto count = [&](int id) {
    if (id >= t0 && id < t0 + nt) atomicAdd(a32 + ((id - t0) >> 1), 1u << (16 * ((id - t0) & 1)));
  };
  for (int h = tid; h < a.hist_len; h += kNT) count(aux_hist(a, h));
  for (int s = tid; s < a.jn; s += kNT) count(aux_draft(a, s));
  for (int e = tid; e < a.n_bias; e += kNT) {
    const int id = aux_bias_tok(a, e);
    if (id >= t0 && id < t0 + nt) atomicOr(a32 + ((id - t0) >> 1), 0x8000u << (16 * ((id - t0) & 1)));
  }
  __syncthreads();
}

// What the count-table pass of one stage returns to the streaming loop.
struct Flagged {
  float M, S;  // the thread's normaliser partials, updated
  bool nan;
};

// The count table's tokens of this stage with their exact processed values:
// added to the normaliser partials (lse_on), to the segment's Gumbel-max
// (gmax_on: Philox purpose 0 at position gpos, row r), and appended to the
// candidates when at or above the cut.
template <bool BF16>
__device__ __forceinline__ Flagged staged_tokens(const uint16_t* aux, StageCtx sc, int BN, float M, float S, bool lse_on,
                                              bool gmax_on, uint64_t seed, uint32_t gpos, uint32_t r,
                                              unsigned long long* gmax, unsigned long long cutp, int* acnt, int n,
                                              unsigned long long* cand) {
  Flagged f{M, S, false};
  const uint4* a4 = reinterpret_cast<const uint4*>(aux);
  for (int w = (int)threadIdx.x; w < BN / 8; w += kNT) {
    const uint4 a = a4[w];
    if ((a.x | a.y | a.z | a.w) == 0u) continue;
#pragma unroll 1
    for (int q = 0; q < 8; ++q) {
      const uint32_t wq = q < 2 ? a.x : (q < 4 ? a.y : (q < 6 ? a.z : a.w));
      const uint32_t h = (wq >> (16 * (q & 1))) & 0xFFFFu;
      const int li = w * 8 + q;
      if (h == 0u || li >= sc.nt) continue;
      const float v = value_with<BF16>(sc, li, (h & 0x7FFFu) | ((h & 0x8000u) << 16));
      const bool isn = v != v;
      f.nan |= isn;
      if (lse_on) lse_add(f.M, f.S, v);
      if (gmax_on && v > -INFINITY) {
        const float g = gumbel_of(philox_uniform(seed, (uint32_t)(sc.t0 + li), gpos, r, 0u));
        atomicMax(gmax, pack(f2key(__fadd_rn(v, g)), (uint32_t)(sc.t0 + li)));
      }
      const unsigned long long pk = pack(isn ? kKeyNegInf : f2key(v), (uint32_t)(sc.t0 + li));
      if (pk >= cutp) {
        const int qq = n + atomicAdd(acnt, 1);
        if (qq < kCap) cand[qq] = pk;
      }
    }
  }
  return f;
}

}  // namespace

// The fused form: a segment's list and metadata are written; the CTA that
// completes a position's last segment (an atomic count of the position's
// written segments, released by a fence) runs the position's stage 2 at
// once, in the candidate and scratch buffers, which are free between
// segments (s2mem: P.seg_cap lists twice and the stage-2 state).  All
// threads call; the barriers are uniform.
template <bool FUSED>
__device__ __forceinline__ void segment_done(const Params& P, int pos, const Split& sp, S1Smem& sm,
                                             unsigned char* s2mem) {
  if constexpr (FUSED) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int Z = P.Z;
      const int nseg = seg_cta(sp, (long long)pos * Z + Z - 1, Z) - seg_cta(sp, (long long)pos * Z, Z) + 1;
      const uint32_t old = atomicAdd(P.ws.pos_arrive + pos, 1u);
      sm.s2_go = old == (uint32_t)(nseg - 1) ? 1 : 0;
    }
    __syncthreads();
    if (sm.s2_go) {
      __threadfence();
      const int cap = P.seg_cap * kK;
      unsigned long long* c2 = reinterpret_cast<unsigned long long*>(s2mem);
      S2Smem& s2 = *reinterpret_cast<S2Smem*>(c2 + 2 * cap);
      stage2_position<kNT>(P, P.cu_draft != nullptr ? 1 : 0, pos, sp, c2, c2 + cap, s2);
      if (threadIdx.x == 0) P.ws.pos_arrive[pos] = 0u;
    }
  }
}

// Whether any row of the call needs the count-table or normaliser paths of
// stage 1, which the lean form lacks: an untruncated stochastic row with
// drafts (its draft positions need the full-vocabulary normaliser), or a row
// with penalties or bias whose listed tokens at some position (history,
// drafts before the position, bias entries) may exceed the hash table.  The
// kernel's own per-position tests imply these (j < gamma, jn <= gamma).  All
// threads call; every CTA reaches the same answer.
__device__ __forceinline__ bool call_needs_full(const Params& P) {
  const bool verify = P.cu_draft != nullptr;
  int need = 0;
  for (int r = threadIdx.x; r < P.B; r += kNT) {
    const RowCtx rc = make_row(P.rows[r], P.hist_stride, P.bias_stride);
    if (!rc.valid) continue;
    const int gamma = verify ? __ldg(P.cu_draft + r + 1) - __ldg(P.cu_draft + r) : 0;
    const bool pen_on = (rc.flags & SS_PENALTY) && P.history != nullptr;
    const bool bias_on = (rc.flags & SS_BIAS) && P.bias != nullptr;
    if (verify && gamma > 0 && rc.stoch && !rc.trunc) need = 1;
    const int nflag_max = (pen_on ? rc.hist_len + gamma : 0) + (bias_on ? rc.n_bias : 0);
    if ((pen_on || bias_on) && nflag_max > kHashMax) need = 1;
  }
  return __syncthreads_or(need) != 0;
}

// Compile-time variants, chosen per call on the host (the fewer paths a
// variant holds, the better its streaming loop compiles: measured, the
// variant without the listed-token paths is 17 % faster on rows that use
// none of them).  AUX: rows may have penalties or bias (the call passes a
// history or a bias list).  LSE: the call verifies drafts, so untruncated
// stochastic positions need the normaliser partials.  FUSED: stage 2 runs
// inside this kernel (segment_done), for batches with few positions.
// STAGED = false (the lean form, with LSE = false): no per-stage count
// tables; the host launches it beside the full form for calls with history
// or bias lists, and P.dispatch makes exactly one of the two run
// (call_needs_full).
// EXACT: the variant that also keeps each exact-sampling segment's
// Gumbel-max; without it none of that code is in the streaming loop.
template <bool BF16, bool EXACT, bool AUX, bool LSE, bool FUSED, bool STAGED = true>
__global__ void __launch_bounds__(kNT, 2) stage1_kernel(const Params P) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int VEC = BF16 ? 8 : 4;
  constexpr int NV = kPT / VEC;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int BN = P.BN, NS = P.nslot;
  const Layout L = layout(BN, ESZ, NS);
  unsigned char* ring0 = smem_raw + L.ring;
  uint32_t* mask0 = reinterpret_cast<uint32_t*>(smem_raw + L.mask);
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(smem_raw + L.cand);
  unsigned long long* tmp = reinterpret_cast<unsigned long long*>(smem_raw + L.tmp);
  uint16_t* aux = reinterpret_cast<uint16_t*>(smem_raw + L.tmp);  // per-stage count table (shares tmp)
  unsigned long long* outb = reinterpret_cast<unsigned long long*>(smem_raw + L.out);
  int* hkey = reinterpret_cast<int*>(smem_raw + L.hkey);
  uint32_t* hval = reinterpret_cast<uint32_t*>(smem_raw + L.hval);
  int* ftok = reinterpret_cast<int*>(smem_raw + L.ftok);
  uint32_t* finfo = reinterpret_cast<uint32_t*>(smem_raw + L.finfo);
  S1Smem& sm = *reinterpret_cast<S1Smem*>(smem_raw + L.sm);
  RowBuf* rb = reinterpret_cast<RowBuf*>(smem_raw + L.rb);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V, Z = P.Z;
  // two forms launched for this call: the lean one (dispatch 1) checks the
  // rows and publishes the answer for the full one (dispatch 2), which runs
  // after it in stream order; exactly one of them does the work
  if (P.dispatch == 1) {
    const bool full = call_needs_full(P);
    if (blockIdx.x == 0 && tid == 0) P.ws.resid_count[2] = full ? 1u : 0u;
    if (full) return;
  } else if (P.dispatch == 2) {
    if (__ldcg(P.ws.resid_count + 2) == 0u) return;
  }
  const int npos = num_positions(P);
  const Split sp = make_split(P, npos);
  // fused form: verification rows past the plan's positions are reported here
  if constexpr (FUSED) stage2_capacity_rows<kNT>(P, P.cu_draft != nullptr ? 1 : 0, blockIdx.x, gridDim.x);
  if (sp.T <= 0) return;
  if ((int)blockIdx.x >= sp.G) return;
  const long long g0 = seg_start(sp, blockIdx.x, Z), g1 = seg_start(sp, blockIdx.x + 1, Z);
  const bool mask_tma = P.mask_tma != 0 && P.bitmask != nullptr;
  const int nch = BN / kChunk;

  // thread 0: bulk copies of the next stage of the range (logits, then the
  // mask words) into a slot.  Stages are issued in order, so the position
  // and tile of the next one advance by one tile per call.
  int iss_pos = (int)(g0 / Z), iss_tile = (int)(g0 - (long long)iss_pos * Z);
  auto issue = [&](int slot) {
    const int pos = iss_pos;
    const int t0 = iss_tile * BN;
    if (++iss_tile == Z) {
      iss_tile = 0;
      ++iss_pos;
    }
    const int nt = min(BN, V - t0);
    const uint32_t bytes = (uint32_t)((nt * ESZ + 15) & ~15);
    const uint32_t mbytes = mask_tma ? (uint32_t)((((nt + 31) >> 5) * 4 + 15) & ~15) : 0u;
    unsigned long long* mb = &sm.mbar[slot];
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(mb)), "r"(bytes + mbytes)
                 : "memory");
    bulk_copy(ring0 + (size_t)slot * BN * ESZ,
              static_cast<const unsigned char*>(P.logits) + ((size_t)pos * P.ld + t0) * ESZ, bytes, mb);
    if (mask_tma) bulk_copy(mask0 + (size_t)slot * (BN / 32), P.bitmask + (size_t)pos * P.mask_words + (t0 >> 5), mbytes, mb);
  };
  // warp 0: a position's row bookkeeping into nb (cp.async; c1 too when c1src is set)
  auto prefetch = [&](int pos, int r, int c0, int c1, const int32_t* c1src, RowBuf& nb) {
    const int j = P.cu_draft ? pos - c0 - r : 0;
    if (lane == 0) {
      nb.pos = pos;
      nb.r = r;
      nb.j = j;
      nb.c0 = c0;
      if (c1src) cp_async4(&nb.c1, c1src);
      else nb.c1 = c1;
    }
    if (lane < (int)(sizeof(ss_row_params) / 4))
      cp_async4(reinterpret_cast<uint32_t*>(&nb.rp) + lane, reinterpret_cast<const uint32_t*>(P.rows + r) + lane);
    if (P.history != nullptr)
      for (int q = lane; q < min(P.hist_stride, kPre); q += 32)
        cp_async4(&nb.hist[q], P.history + (size_t)r * P.hist_stride + q);
    if (P.cu_draft != nullptr)
      for (int q = lane; q < min(j, kPre); q += 32) cp_async4(&nb.draft[q], P.draft_ids + c0 + q);
    if (P.bias != nullptr)
      for (int q = lane; q < min(P.bias_stride, kBiasPre); q += 32) {  // 4-byte copies: 4-byte aligned entries
        const ss_bias_entry* be = P.bias + (size_t)r * P.bias_stride + q;
        cp_async4(&nb.bias[q].token, &be->token);
        cp_async4(&nb.bias[q].value, &be->value);
      }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // staging list of position pos for this CTA's segment: list index
  // blockIdx.x - (the CTA holding the position's first stage), which is 0 for
  // every position of the range but the first (they start inside it)
  const int pos_first = (int)(g0 / Z);
  const int first_off = (int)blockIdx.x - seg_cta(sp, (long long)pos_first * Z, Z);
  auto slot_of = [&](int pos) -> size_t {
    return (size_t)pos * Z + (size_t)(pos == pos_first ? first_off : 0);
  };

  if (tid == 0) {
    sm.dead = 0;
    for (int s = 0; s < NS; ++s) mbar_init(&sm.mbar[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int s = 0; s < NS && g0 + s < g1; ++s) issue(s);
  }
  if (warp == 0) {
    const int pos = (int)(g0 / Z);
    int r = pos, c0 = 0, c1 = 0;
    if (P.cu_draft) {
      r = warp_find_row(P.cu_draft, P.B, pos, lane);
      c0 = __ldg(P.cu_draft + r);
      c1 = __ldg(P.cu_draft + r + 1);
    }
    prefetch(pos, r, c0, c1, nullptr, rb[0]);
  }
  cp_async_wait_all();
  __syncthreads();

  WaitCfg R;
  R.spin_limit = P.spin_limit;
  R.spin_hint_ns = P.spin_hint_ns;
  long long g = g0;
  int kst = 0;           // stages consumed by this CTA
  int slot = 0;          // kst % NS
  uint32_t phase = 0u;   // (kst / NS) & 1
  int c3 = 0;            // kst % 3: this stage's append counter
  int buf = 0;
  bool dead = false;
  while (g < g1 && !dead) {
    const RowBuf& cb = rb[buf];
    const int pos = cb.pos, r = cb.r, j = cb.j;
    const int gamma = P.cu_draft ? cb.c1 - cb.c0 : 0;
    const long long gs = (long long)pos * Z;
    const long long ge = min(g1, gs + Z);
    const size_t lslot = slot_of(pos);
    const RowCtx rc = make_row(cb.rp, P.hist_stride, P.bias_stride);
    const Temp tp = temp_of(rc);
    // the next segment's bookkeeping (the next position; rows own consecutive positions)
    if (warp == 0 && ge < g1) {
      const int pn = pos + 1;
      if (P.cu_draft && pn >= cb.c1 + r + 1) prefetch(pn, r + 1, cb.c1, 0, P.cu_draft + r + 2, rb[buf ^ 1]);
      else if (P.cu_draft) prefetch(pn, r, cb.c0, cb.c1, nullptr, rb[buf ^ 1]);
      else prefetch(pn, pn, 0, 0, nullptr, rb[buf ^ 1]);
    }

    const int seg_lo = (int)(g - gs) * BN, seg_hi = min(V, (int)(ge - gs) * BN);
    const bool mask_on = (rc.flags & SS_MASK) && P.bitmask != nullptr;
    const bool pen_on = (rc.flags & SS_PENALTY) && P.history != nullptr;
    const bool bias_on = (rc.flags & SS_BIAS) && P.bias != nullptr;
    const int jn = P.cu_draft ? min(j, gamma) : 0;
    const bool lse_on = LSE && P.cu_draft != nullptr && j < gamma && rc.stoch && !rc.trunc;
    // exact sampling (a sample or bonus position of an SS_EXACT row): the
    // segment's Gumbel-max of l_i + g_i over every token (Philox purpose 0)
    const bool gmax_on = EXACT && rc.valid && rc.exact && (P.cu_draft == nullptr || j == gamma);
    const bool aux_on = AUX && rc.valid && (pen_on || bias_on);
    const int nflag = (pen_on ? rc.hist_len + jn : 0) + (bias_on ? rc.n_bias : 0);
    const bool hashed = aux_on && !lse_on && !gmax_on && nflag <= kHashMax;
    const bool staged = STAGED && aux_on && !hashed;
    const ss_bias_entry* brow = bias_on ? P.bias + (size_t)r * P.bias_stride : nullptr;
    const ss_bias_entry* bl = (bias_on && rc.n_bias <= kBiasPre) ? cb.bias : brow;

    // ---- segment set-up: counters; for rows with penalties or bias the id
    // checks and (hash mode) the listed tokens, out of line
    if (tid == 0) {
      sm.cnt[0] = sm.cnt[1] = sm.cnt[2] = 0;
      sm.nan_flag = 0;
      sm.nf = 0;
      sm.gmax = 0ull;
      sm.rowbad = 0u;
    }
    AuxRow ar;
    ar.hrow = pen_on ? P.history + (size_t)r * P.hist_stride : nullptr;
    ar.drafts = P.cu_draft ? P.draft_ids + cb.c0 : nullptr;
    ar.brow = brow;
    ar.cb = &cb;
    ar.hist_len = pen_on ? rc.hist_len : 0;
    ar.jn = pen_on ? jn : 0;
    ar.n_bias = bias_on ? rc.n_bias : 0;
    Listed ls{};
    if (aux_on)
      ls = seg_aux_setup<BF16>(ar, hashed, V, seg_lo, seg_hi, hkey, hval, ftok, finfo, &sm.nf, &sm.rowbad,
                               static_cast<const unsigned char*>(P.logits) + (size_t)pos * P.ld * ESZ,
                               mask_on ? P.bitmask + (size_t)pos * P.mask_words : nullptr,
                               reinterpret_cast<uint32_t*>(tmp));  // tmp: free until the first stage's barrier
    else
      __syncthreads();
    const int nf = hashed ? sm.nf : 0;

    unsigned long long cutp = 0ull;  // packed cut (0: everything)
    // the raw threshold of the cut x0cut: raw values <= x0 lie below it (NaN:
    // none is known to; the cut 0 admits everything)
    float x0 = __int_as_float(0x7FC00000);
    unsigned long long x0cut = 0ull;
    const float rTl = tp.stoch ? __frcp_rn(tp.T) : 1.0f;  // for the normaliser's quotients
    int n = nf;                      // buffer entries (uniform; read between barriers)
    float lM = -INFINITY, lS = 0.0f; // this thread's running (max, sum exp) for the normaliser
    bool first = true;

    for (; g < ge; ++g, ++kst, first = false) {
      const unsigned char* ring = ring0 + (size_t)slot * BN * ESZ;
      const int t0 = (int)(g - gs) * BN;
      const int nt = min(BN, V - t0);
      const bool full = nt == BN;
      const uint32_t* msl = nullptr;
      if (mask_on) msl = mask_tma ? mask0 + (size_t)slot * (BN / 32) : P.bitmask + (size_t)pos * P.mask_words + (t0 >> 5);
      int* acnt = &sm.cnt[c3];
      // the next stage's counter was last read after the barrier two stages back
      if (tid == 0) sm.cnt[c3 == 2 ? 0 : c3 + 1] = 0;
      // a copy that never lands is noticed by all threads after the stage barrier
      if (!mbar_wait(&sm.mbar[slot], phase, R.spin_limit, R.spin_hint_ns)) sm.dead = 1;

      if (rc.valid) {
        // per-stage count table (long histories, normaliser positions)
        if (staged) count_table(ar, aux, BN, t0, nt);
        auto append = [&](unsigned long long pk) {
          const int q = n + atomicAdd(acnt, 1);
          if (q < kCap) cand[q] = pk;
        };

        // pass 0 (a segment's first stage only): the cut from the per-thread
        // maxima; pass 1: the stream (prelude, running maximum, rare appends)
        bool nan_seen = false;
        // the first stage's cut: the 16th largest of each warp's 32 thread
        // maxima (bitonic sort across lanes), minimum over the warps, so at
        // least 8 * 16 elements are >= it
        auto certify = [&](float mt) -> unsigned long long {
          float v = mt;
#pragma unroll
          for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
            for (int d = kk >> 1; d > 0; d >>= 1) {
              const float o = __shfl_xor_sync(0xffffffffu, v, d);
              const bool keep_max = (((lane & d) == 0) == ((lane & kk) == 0));
              v = keep_max ? fmaxf(v, o) : fminf(v, o);
            }
          }
          if (lane == 15) sm.tw[warp] = v;
          __syncthreads();
          float tau = sm.tw[0];
#pragma unroll
          for (int w = 1; w < kNT / 32; ++w) tau = fminf(tau, sm.tw[w]);
          return pack(f2key(tau), 0xFFFFFFFFu);  // every element >= tau
        };
        // a one-chunk first stage takes the cut from the chunk it holds;
        // otherwise pass 0 scans the stage for the maxima first
        const bool merged = first && nch == 1;
        const bool lazy = !first && full && !lse_on && !gmax_on;
        for (int pass = (first && !merged) ? 0 : 1; pass < 2; ++pass) {
          if (pass == 1 && cutp != x0cut) {
            x0 = raw_threshold(cutp, tp);
            x0cut = cutp;
          }
          float mt = -INFINITY;
          for (int ch = 0; ch < nch; ++ch) {
            if (lazy) {
              // a full stage after the segment's first: the raw maxima decide,
              // and only the vectors that may hold a hit are processed
              float vm[NV];
              const float m = raw_chunk_max<BF16>(ring, ch, vm);
              if (!(m <= x0)) {
                uint32_t vb = 0u;
#pragma unroll
                for (int v = 0; v < NV; ++v) vb |= (vm[v] <= x0 ? 0u : 1u) << v;
                while (vb) {
                  const int v = __ffs((int)vb) - 1;
                  vb &= vb - 1u;
                  float y[VEC];
                  if (mask_on) load_vec<BF16, true>(ring, msl, ch, v, y);
                  else load_vec<BF16, false>(ring, msl, ch, v, y);
                  uint32_t bits = 0u;
#pragma unroll
                  for (int jj = 0; jj < VEC; ++jj) bits |= (y[jj] <= x0 ? 0u : 1u) << jj;
                  const int e0 = elem_index<VEC>(ch, v, 0);
                  while (bits) {
                    const int jj = __ffs((int)bits) - 1;
                    bits &= bits - 1u;
                    float xr = y[0];
#pragma unroll
                    for (int k = 1; k < VEC; ++k) xr = jj == k ? y[k] : xr;
                    const float xv = temper(xr, tp);
                    const int li = e0 + jj;
                    const bool isn = xv != xv;
                    nan_seen |= isn;
                    const unsigned long long pk = pack(isn ? kKeyNegInf : f2key(xv), (uint32_t)(t0 + li));
                    bool fl = false;
                    if (hashed) fl = (ls.own & own_bit<BF16>(li)) && hash_find(hkey, t0 + li) >= 0;
                    else if (staged) fl = aux[li] != 0u;
                    if (pk >= cutp && !fl) append(pk);
                  }
                }
              }
              continue;
            }
            float x[kPT];
            const float m = load_chunk_sel<BF16>(mask_on, full, ring, msl, ch, nt, x);
            if (pass == 0) {
#pragma unroll
              for (int e = 0; e < kPT; ++e) mt = fmaxf(mt, x[e]);
              continue;
            }
            if (merged) {
              float mc = m;
              if (mc != mc) {  // NaN among them: the maximum of the rest
                mc = -INFINITY;
#pragma unroll
                for (int e = 0; e < kPT; ++e) mc = fmaxf(mc, x[e]);
              }
              cutp = certify(temper(mc, tp));  // the largest processed value (temper is monotone)
              x0 = raw_threshold(cutp, tp);
              x0cut = cutp;
            }
            if (!(m <= x0)) {
              // elements at or above the cut (or NaN): re-derived from the slot
              uint32_t bits = 0u;
#pragma unroll
              for (int e = 0; e < kPT; ++e) bits |= (x[e] <= x0 ? 0u : 1u) << e;
              while (bits) {
                const int e = __ffs((int)bits) - 1;
                bits &= bits - 1u;
                const int li = ((ch * NV + e / VEC) * kNT + tid) * VEC + e % VEC;
                if (!full && li >= nt) continue;
                const float xv = stream_value<BF16>(ring, msl, tp, li);
                const bool isn = xv != xv;
                nan_seen |= isn;
                const unsigned long long pk = pack(isn ? kKeyNegInf : f2key(xv), (uint32_t)(t0 + li));
                bool fl = false;
                if (hashed) fl = (ls.own & own_bit<BF16>(li)) && hash_find(hkey, t0 + li) >= 0;
                else if (staged) fl = aux[li] != 0u;
                if (pk >= cutp && !fl) append(pk);
              }
            }
            if (lse_on) {
              // the processed values (x / T, to an ulp) and their maximum
              // without NaN; listed tokens (count-table rows) are added with
              // their exact values elsewhere
#pragma unroll
              for (int e = 0; e < kPT; ++e) x[e] = quot_lse(x[e], tp.T, rTl);
              if (staged) {
#pragma unroll
                for (int e = 0; e < kPT; ++e) {
                  const int li = elem_index<VEC>(ch, e / VEC, e % VEC);
                  if ((full || li < nt) && aux[li] != 0u) x[e] = -INFINITY;
                }
              }
              float t[kPT / 2];
#pragma unroll
              for (int e = 0; e < kPT / 2; ++e) t[e] = fmaxf(x[2 * e], x[2 * e + 1]);
#pragma unroll
              for (int w = kPT / 4; w >= 1; w >>= 1)
#pragma unroll
                for (int e = 0; e < w; ++e) t[e] = fmaxf(t[e], t[e + w]);
              const float mc = t[0];
              if (mc > -INFINITY) {
                const float Mn = fmaxf(lM, mc);
                const float off = Mn * kLog2e;
                // four independent sums; fmaxf(NaN, -inf) = -inf drops NaN terms
                float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int e = 0; e < kPT; ++e)
                  s4[e & 3] += ex2_approx(__fmaf_rn(fmaxf(x[e], -INFINITY), kLog2e, -off));
                lS = lS * ex2_approx((lM - Mn) * kLog2e) + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
                lM = Mn;
              }
            }
          }
          if (pass == 0) cutp = certify(temper(mt, tp));  // the largest processed value
        }
        // the listed tokens' exact values (hash mode), from the loads issued at set-up
        if (first && hashed) nan_seen |= listed_candidates(ls, nf, ftok, finfo, rc, bl, cand);

        // ---- the count table's tokens of this stage, with their exact values
        if (staged) {
          StageCtx sc;
          sc.ring = ring;
          sc.msl = msl;
          sc.bl = bl;
          sc.hkey = nullptr;
          sc.hval = nullptr;
          sc.aux = aux;
          sc.rc = rc;
          sc.t0 = t0;
          sc.nt = nt;
          sc.hashed = false;
          sc.staged = true;
          const Flagged f = staged_tokens<BF16>(aux, sc, BN, lM, lS, lse_on, gmax_on, __ldg(P.seeds + r),
                                                rc.position + (uint32_t)j, (uint32_t)r, &sm.gmax, cutp, acnt, n, cand);
          lM = f.M;
          lS = f.S;
          nan_seen |= f.nan;
        }
        if (nan_seen) sm.nan_flag = 1;
      }
      __syncthreads();
      if (sm.dead) {
        dead = true;
        break;
      }
      // read between this barrier and the next stage's appends, which use another counter
      int n_end = n + *acnt;

      // ---- fallback: the buffer overflowed, or the first stage's cut certified too few
      const int need_s = min(kK, nt);
      if (rc.valid && (n_end > kCap || (first && n_end - n < need_s))) {
        __syncthreads();  // every thread has read the counter
        if (tid == 0) {
          *acnt = 0;  // roll this stage's appends back
          atomicAdd(P.ws.diag + 0, 1u);
        }
        __syncthreads();
        StageCtx sc;
        sc.ring = ring;
        sc.msl = msl;
        sc.bl = bl;
        sc.hkey = hkey;
        sc.hval = hval;
        sc.aux = aux;
        sc.rc = rc;
        sc.t0 = t0;
        sc.nt = nt;
        sc.hashed = hashed;
        sc.staged = staged;
        stage_exact<BF16>(sc, sm, acnt, n, cand, need_s, BN / kNT);
        const int added = min(*acnt, need_s);  // need_s unless the keys disagreed between passes
        unsigned long long mn = ~0ull;
        for (int i = n + tid; i < n + added; i += kNT) mn = cand[i] < mn ? cand[i] : mn;
        mn = block_min_u64(mn, sm.slots);
        const unsigned long long base_cut = first ? 0ull : cutp;
        // a stage of >= 128 tokens: nothing outside its top-128 is >= its 128th value
        cutp = (nt >= kK && added == need_s && mn > base_cut) ? mn : base_cut;
        n_end = n + added;
      }
      // exact sampling: the stage's Gumbel-max, read from the slot before it is
      // refilled (and from the stage's count table, still in place)
      if (gmax_on) {
        for (int ch = 0; ch < nch; ++ch)
          chunk_gmax<BF16>(ring, msl, tp, ch, nt, full, staged ? aux : nullptr, t0, rc.position + (uint32_t)j,
                           (uint32_t)r, P.seeds, &sm.gmax);
        __syncthreads();  // every read of the slot is done before its refill
      }
      // refill this slot with the stage NS ahead (every read of it is done)
      if (tid == 0 && g + NS < g1) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(slot);
      }
      // ---- keep room in the buffer: one histogram pass raises the cut; the
      // exact top-128 only if that left too many (a crowd of equal values)
      if (rc.valid && n_end > kRaiseAt) {
        const Raised rz = raise_cut(cand, tmp, n_end, cutp, sm);
        cutp = rz.cut;
        n_end = rz.n;
        if (n_end > kCompactAt) {
          if (tid == 0) atomicAdd(P.ws.diag + 4, 1u);
          cutp = compact(cand, tmp, outb, n_end, sm);
          n_end = kK;
        }
      }
      n = n_end;
      if (++slot == NS) {
        slot = 0;
        phase ^= 1u;
      }
      c3 = c3 == 2 ? 0 : c3 + 1;
    }
    if (dead) break;

    // ---- segment end: the exact top-128 of the buffer goes to staging
    unsigned long long* stg = P.ws.staging + lslot * kK;
    if (rc.valid) {
      const int need = min(kK, seg_hi - seg_lo);
      if (tid == 0) sm.out_cnt = 0;
      __syncthreads();
      select_top(cand, tmp, n, need, sm, [&](unsigned long long c) {
        const int q = atomicAdd(&sm.out_cnt, 1);
        if (q < kK) stg[q] = c;
      });
      for (int q = min(sm.out_cnt, need) + tid; q < kK; q += kNT) stg[q] = 0ull;
      if (tid == 0) P.ws.tile_status[lslot] = (sm.nan_flag ? SS_ST_NAN : 0u) | sm.rowbad;
      if (lse_on) {
        float Mb = lM;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) Mb = fmaxf(Mb, __shfl_xor_sync(0xffffffffu, Mb, d));
        if (lane == 0) sm.lm[warp] = Mb;
        __syncthreads();
        Mb = sm.lm[0];
#pragma unroll
        for (int w = 1; w < kNT / 32; ++w) Mb = fmaxf(Mb, sm.lm[w]);
        const double part = (lM > -INFINITY) ? (double)lS * (double)exp2f((lM - Mb) * kLog2e) : 0.0;
        const double S = block_sum_d(part, sm.red);
        if (tid == 0) P.ws.tile_lse[lslot] = make_float2(Mb, (float)S);
      }
      if (gmax_on && tid == 0) P.ws.tile_gmax[lslot] = sm.gmax;  // updates end before select_top's barriers
    } else {  // invalid row parameters: stage 2 reports the row
      for (int q = tid; q < kK; q += kNT) stg[q] = 0ull;
      if (tid == 0) P.ws.tile_status[lslot] = 0u;
    }
    segment_done<FUSED>(P, pos, sp, sm, smem_raw + L.cand);
    cp_async_wait_all();  // the next segment's bookkeeping
    __syncthreads();
    buf ^= 1;
  }

  if (dead) {
    // A bulk copy did not complete within the wait limit: count it, leave
    // empty lists with SS_ST_COPY_TIMEOUT for this and the remaining
    // positions of the range, and let the copies still in flight (the stages
    // kst .. kst + NS - 1 of the range) land, with the long drain limit,
    // before the CTA exits.
    if (tid == 0) atomicAdd(P.ws.diag + 3, 1u);
    const int p_first = (int)(g / Z), p_last = (int)((g1 - 1) / Z);
    for (int p = p_first; p <= p_last; ++p) {
      const size_t ls = slot_of(p);
      for (int q = tid; q < kK; q += kNT) P.ws.staging[ls * kK + q] = 0ull;
      if (tid == 0) {
        P.ws.tile_status[ls] = (uint32_t)SS_ST_COPY_TIMEOUT;
        P.ws.tile_lse[ls] = make_float2(-INFINITY, 0.0f);
        P.ws.tile_gmax[ls] = 0ull;
      }
      segment_done<FUSED>(P, p, sp, sm, smem_raw + L.cand);
    }
    if (tid == 0)
      for (int s = 0; s < NS && g + s < g1; ++s)
        mbar_wait(&sm.mbar[(kst + s) % NS], (uint32_t)(((kst + s) / NS) & 1), kDrainSpin, 0u);
    cp_async_wait_all();
    __syncthreads();
  }
}


}  // namespace ss
