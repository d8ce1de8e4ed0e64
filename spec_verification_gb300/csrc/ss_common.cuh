// Internal declarations shared by the CUDA translation units of libss.so:
// kernel parameter block, workspace layout and small device helpers
// (order-preserving keys, Philox, row parameters, block reductions).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ss.h"

namespace ss {

constexpr int kK = 128;         // bounded candidate count (SonicSampler 1, 3.3)
constexpr int kNT = 256;        // threads per CTA in every kernel
constexpr int kCap1 = 2048;     // stage-1 survivor capacity (entries)
constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // key of -inf
constexpr int kPending = -2;    // residual token still to be drawn by the V pass

// Per-target-position result written by stage 2, read by the row walk and
// the residual pass.
struct PosResult {
  double lse;        // full-vocabulary log-sum-exp (untruncated verify positions)
  int32_t token;     // sampled / bonus / resampled token, -1 none, kPending
  int32_t accept;    // 1 if the draft at this position was accepted
  uint32_t status;   // SS_ST_* bits of this position
  int32_t pad;
};

// One queued residual pass over the vocabulary (an untruncated stochastic
// row rejected at draft index j).
struct ResidEntry {
  unsigned long long best;   // max over tiles of (key(score) << 32 | ~token)
  uint32_t arrivals;         // tiles done
  int32_t row, j, pos;
};

struct Workspace {
  unsigned long long* staging;   // [P * Z * 128] packed candidates, one list per segment
  float2* tile_lse;              // [P * Z] per segment (max, sum exp(x - max)) when requested
  unsigned long long* tile_gmax; // [P * Z] per segment Gumbel-max (key(l + g) << 32 | ~token) when requested
  uint32_t* tile_status;         // [P * Z] per segment SS_ST_* bits
  PosResult* pos;                // [P]
  uint32_t* row_count;           // [R] positions of the row done (stage-2 arrivals)
  uint32_t* resid_count;         // [3] queued residual passes, residual CTAs done (the last resets both),
                                 //     and whether the call needs the full stage-1 form (written by the lean form)
  uint32_t* pos_arrive;          // [P] fused form: segments of the position whose lists are written
  ResidEntry* resid;             // [R]
  uint32_t* diag;                // [8] diagnostic counters
};

// Everything one call's kernels read: plain pointers and sizes.
struct Params {
  const void* logits;
  int64_t ld;
  int V, Z, BN;
  int logits_bf16;
  const ss_row_params* rows;
  int B;
  const int32_t* cu_draft;  // null: single-step sampling (one position per row)
  const int32_t* history;
  int hist_stride;
  const uint32_t* bitmask;
  int mask_words;           // ceil(V / 32)
  const ss_bias_entry* bias;
  int bias_stride;
  const int32_t* draft_ids;
  const void* q;
  int64_t ld_q;
  int q_bf16;
  const uint64_t* seeds;
  int max_positions;
  int grid1;                // CTAs of the stage-1 launch (fixes the segment split)
  int nslot;                // stage-1 ring slots
  int seg_cap;              // segment lists per position that stage 2's shared memory holds
  int exact_on;             // the plan runs the exact-sampling variant of stage 1
  int mask_tma;             // bitmask rows can be bulk-copied (16-byte aligned rows)
  int dispatch;             // stage 1: 0 runs; 1 runs only if no row needs the full form, 2 only if one does
  uint32_t spin_limit;      // polls of a stage-1 ring wait before it gives up (the copy timeout)
  uint32_t spin_hint_ns;    // suspend-time hint of each poll in ns (0: the hardware's limit)
  Workspace ws;
  ss_out out;
};

// ------------------------------------------------------------------ keys
// Order-preserving map of a non-NaN float to uint32 (-0 and +0 share a key);
// a packed candidate is key << 32 | ~token, so larger packed values come first
// in the order (processed logit descending, token ascending).  Key 0 is never
// produced by a float and marks an empty staging slot.
__device__ __forceinline__ uint32_t f2key(float x) {
  const uint32_t b = __float_as_uint(x);
  return (x >= 0.0f) ? (b | 0x80000000u) : ~b;
}
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ unsigned long long pack(uint32_t key, uint32_t tok) {
  return ((unsigned long long)key << 32) | (uint32_t)(~tok);
}
__device__ __forceinline__ uint32_t pk_key(unsigned long long c) { return (uint32_t)(c >> 32); }
__device__ __forceinline__ int32_t pk_tok(unsigned long long c) { return (int32_t)(~(uint32_t)c); }

// ------------------------------------------------------------------ Philox-4x32-10
// Salmon, Moraes, Dror, Shaw, SC'11: ten rounds of two 32x32->64 multiplies
// of counter words 0 and 2, XOR of the high halves with words 1 and 3 and the
// round key, with the key advanced by the two Weyl constants each round.
__device__ __forceinline__ void philox10(uint32_t& c0, uint32_t& c1, uint32_t& c2, uint32_t& c3,
                                         uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    const uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

__device__ __forceinline__ float word_to_uniform(uint32_t w) {
  return (float)((w >> 9) * 2u + 1u) * 0x1p-24f;  // odd multiple of 2^-24 in (0, 1)
}

__device__ __forceinline__ float philox_uniform(uint64_t seed, uint32_t i, uint32_t position,
                                                uint32_t row, uint32_t purpose) {
  uint32_t c0 = i >> 2, c1 = position, c2 = row, c3 = purpose;
  philox10(c0, c1, c2, c3, (uint32_t)seed, (uint32_t)(seed >> 32));
  const uint32_t w = (i & 3u) == 0u ? c0 : (i & 3u) == 1u ? c1 : (i & 3u) == 2u ? c2 : c3;
  return word_to_uniform(w);
}

// Gumbel(0, 1) noise in fp32: -ln(-ln u).
__device__ __forceinline__ float gumbel_of(float u) { return -logf(-logf(u)); }

// ------------------------------------------------------------------ row parameters
struct RowCtx {
  uint32_t flags;
  float T, rep, freq, pres, top_p, min_p;  // T: the temperature of stochastic rows (greedy: 1)
  int top_k, hist_len, n_bias;
  uint32_t position;
  bool valid, stoch, trunc;
  bool exact;  // SS_EXACT on an untruncated stochastic row: sample over the whole vocabulary
};

__device__ __forceinline__ bool finitef(float x) { return fabsf(x) <= 3.402823466e38f; }

__device__ __forceinline__ RowCtx make_row(const ss_row_params& p, int hist_stride, int bias_stride) {
  RowCtx c;
  c.flags = p.flags;
  c.rep = p.rep;
  c.freq = p.freq;
  c.pres = p.pres;
  c.top_p = p.top_p;
  c.min_p = p.min_p;
  c.top_k = p.top_k;
  c.position = p.position;
  c.hist_len = min(max(p.hist_len, 0), hist_stride);
  c.n_bias = min(max(p.n_bias, 0), bias_stride);
  c.stoch = (p.flags & SS_GREEDY) == 0u;
  bool ok = p.hist_len >= 0 && p.hist_len <= hist_stride && p.n_bias >= 0 && p.n_bias <= bias_stride;
  if (p.flags & SS_PENALTY) ok = ok && finitef(p.rep) && p.rep > 0.0f && finitef(p.freq) && finitef(p.pres);
  if (c.stoch) {
    ok = ok && finitef(p.temperature) && p.temperature > 0.0f;
    if (p.flags & SS_TOPP) ok = ok && p.top_p > 0.0f && p.top_p <= 1.0f;
    if (p.flags & SS_MINP) ok = ok && p.min_p >= 0.0f && p.min_p <= 1.0f;
    if (p.flags & SS_TOPK) ok = ok && p.top_k >= 0;
  }
  c.valid = ok;
  c.T = c.stoch ? p.temperature : 1.0f;
  // truncating rows (and SS_BOUNDED_P rows) verify against the kept candidate
  // distribution; the others against the softmax over the whole vocabulary
  const bool cuts = ((p.flags & SS_TOPK) && p.top_k > 0) || ((p.flags & SS_TOPP) && p.top_p < 1.0f) ||
                   ((p.flags & SS_MINP) && p.min_p > 0.0f);
  c.trunc = c.stoch && (cuts || (p.flags & SS_BOUNDED_P));
  c.exact = c.stoch && !cuts && (p.flags & SS_EXACT);
  return c;
}

// Temperature (dl-note, Temperature: z / T): one IEEE fp32 division, rounded
// to nearest, for stochastic rows; greedy rows keep the logit.
__device__ __forceinline__ float apply_temperature(float x, const RowCtx& rc) {
  return rc.stoch ? __fdiv_rn(x, rc.T) : x;
}

// Penalties and bias for one element whose history count is c (> 0 only for
// tokens in the history) and whose bias flag says a bias entry names it.
// fp32, one rounding per operation, in the order of the prelude.
__device__ __forceinline__ float apply_penalty_bias(float x, uint32_t c, bool has_bias, int tok,
                                                    const RowCtx& rc, const ss_bias_entry* brow) {
  if ((rc.flags & SS_PENALTY) && c > 0u) {
    x = (x > 0.0f) ? __fdiv_rn(x, rc.rep) : __fmul_rn(x, rc.rep);
    x = __fsub_rn(x, __fmul_rn(rc.freq, (float)c));
    x = __fsub_rn(x, rc.pres);
  }
  if ((rc.flags & SS_BIAS) && has_bias) {
    for (int e = 0; e < rc.n_bias; ++e) {
      const ss_bias_entry be = brow[e];
      if (be.token == tok) x = __fadd_rn(x, be.value);
    }
  }
  return x;
}

// Out-of-line form for the unrolled hot loops: only the few tokens that are
// in the history or the bias list take it, and keeping it out of line keeps
// those loops small enough for the instruction cache.
static __device__ __noinline__ float penalize_token(float x, uint32_t a, int tok, uint32_t flags, float rep, float freq,
                                             float pres, int n_bias, const ss_bias_entry* brow) {
  RowCtx rc;
  rc.flags = flags;
  rc.rep = rep;
  rc.freq = freq;
  rc.pres = pres;
  rc.n_bias = n_bias;
  return apply_penalty_bias(x, a & 0x7FFFu, (a & 0x8000u) != 0u, tok, rc, brow);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float load_scalar(const void* base, int bf16, int64_t off) {
  if (bf16) {
    const uint16_t h = __ldg(static_cast<const unsigned short*>(base) + off);
    return __uint_as_float((uint32_t)h << 16);
  }
  return __ldg(static_cast<const float*>(base) + off);
}

// Target position -> row: largest r with cu_draft[r] + r <= pos.
__device__ __forceinline__ int find_row(const int32_t* cu, int B, int pos) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) + mid <= pos) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The same by one warp: 32-way search rounds over the row offsets (every
// lane calls and gets r).
__device__ __forceinline__ int warp_find_row(const int32_t* cu, int B, int pos, int lane) {
  int lo = 0, hi = B - 1;  // r in [lo, hi]; offset(lo) <= pos throughout
  while (hi > lo) {
    const int span = hi - lo + 1;
    const int step = (span + 31) / 32;
    const int idx = lo + lane * step;
    const bool ok = idx <= hi && __ldg(cu + idx) + idx <= pos;
    const uint32_t b = __ballot_sync(0xffffffffu, ok);
    const int k = 31 - __clz((int)b);  // the last probe at or below pos (probe 0 always is)
    lo = lo + k * step;
    hi = min(hi, lo + step - 1);
  }
  return lo;
}

__device__ __forceinline__ int num_positions(const Params& P) {
  const int n = P.cu_draft ? (__ldg(P.cu_draft + P.B) + P.B) : P.B;
  return min(n, P.max_positions);
}

// Segment split shared by stage 1 and stage 2: the T = npos * Z stages
// (position-major) are cut into G contiguous ranges, CTA c of stage 1 owning
// stages [seg_start(c), seg_start(c + 1)), at least one each.
//  - aligned (when the stage-1 grid holds two or more CTAs per position):
//    each position is cut into kk ranges of Lr stages (the last may be
//    shorter), so that no range crosses a position boundary and every CTA has
//    exactly one segment;
//  - even (otherwise): G = min(grid1, T) ranges of T / G stages.
struct Split {
  long long T;
  int G, kk, Lr;
  bool aligned;
};
__device__ __forceinline__ Split make_split(const Params& P, int npos) {
  Split s;
  s.T = (long long)npos * P.Z;
  const int k = npos > 0 ? P.grid1 / npos : 0;
  s.aligned = k >= 2;
  if (s.aligned) {
    s.Lr = (P.Z + k - 1) / k;
    s.kk = (P.Z + s.Lr - 1) / s.Lr;
    s.G = npos * s.kk;
  } else {
    s.kk = s.Lr = 0;
    s.G = (int)(s.T < (long long)P.grid1 ? s.T : (long long)P.grid1);
  }
  return s;
}
__device__ __forceinline__ long long seg_start(const Split& s, long long c, int Z) {
  if (s.aligned) return (c / s.kk) * Z + (c % s.kk) * s.Lr;
  return c * s.T / s.G;
}
// The CTA whose range holds stage g: the largest c with seg_start(c) <= g.
__device__ __forceinline__ int seg_cta(const Split& s, long long g, int Z) {
  if (s.aligned) return (int)((g / Z) * s.kk + (g % Z) / s.Lr);
  return (int)(((g + 1) * s.G - 1) / s.T);
}

// ------------------------------------------------------------------ block helpers
// Inclusive prefix sum over the kNT threads of the block (int).  All threads
// must call; `scratch` holds kNT/32 ints.
__device__ __forceinline__ int block_inclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  int add = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kNT / 32; ++w) {
    const int s = scratch[w];
    if (w < warp) add += s;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return v + add;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Sum over the block in fp64; every thread gets the total.  `scratch` holds kNT/32 doubles.
__device__ __forceinline__ double block_sum_d(double v, double* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_d(v);
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int w = 0; w < kNT / 32; ++w) t += scratch[w];
  __syncthreads();
  return t;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, d);
    v = o > v ? o : v;
  }
  return v;
}
__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, d);
    v = o < v ? o : v;
  }
  return v;
}

// Block-wide max / min of a 64-bit value through per-warp slots (no 64-bit
// shared-memory atomics, which serialise under contention).  All NT threads
// of the block call; `slots` holds NT/32 values; every thread gets the result.
template <int NT = kNT>
__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* slots) {
  v = warp_max_u64(v);
  if ((threadIdx.x & 31) == 0) slots[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long r = slots[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) r = slots[w] > r ? slots[w] : r;
  __syncthreads();
  return r;
}
template <int NT = kNT>
__device__ __forceinline__ unsigned long long block_min_u64(unsigned long long v, unsigned long long* slots) {
  v = warp_min_u64(v);
  if ((threadIdx.x & 31) == 0) slots[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long r = slots[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) r = slots[w] < r ? slots[w] : r;
  __syncthreads();
  return r;
}

// Shared-memory state of the histogram select.
struct SelectSmem {
  uint32_t hist[256];
  int scan[kNT / 32];
  int bstar, above, nb, pad;
  int tcnt[2];
};

// Find the histogram bin b* holding the need-th largest element:
// above(b*) < need <= above(b*) + hist[b*], above(b) = sum of bins > b.
// Warp 0 scans the 256 bins (8 per lane, from the top); all threads call and
// read S.bstar / S.above after the call.
__device__ __forceinline__ void boundary_bin(SelectSmem& S, int need) {
  const int t = threadIdx.x;
  if (t < 32) {
    int v[8];
    int sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      v[q] = (int)S.hist[255 - (t * 8 + q)];  // lane t holds bins 255-8t .. 248-8t
      sum += v[q];
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (t >= d) incl += o;
    }
    int above = incl - sum;  // count in bins above this lane's first bin
    if (t == 0) {
      S.bstar = 0;
      S.above = 0;
      S.nb = 0;
    }
    __syncwarp();
    if (above < need && need <= incl) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (above < need && need <= above + v[q]) {
          S.bstar = 255 - (t * 8 + q);
          S.above = above;
          S.nb = v[q];
        }
        above += v[q];
      }
    }
  }
  __syncthreads();
}

// Histogram bin of a packed value (clamped to [0, 255]).
__device__ __forceinline__ uint32_t bin_of(unsigned long long c, unsigned long long lo, int shift) {
  const unsigned long long d = c > lo ? c - lo : 0ull;
  const unsigned long long b = d >> shift;
  return (uint32_t)(b < 255ull ? b : 255ull);
}

// Exact selection of the `need` largest of cand[0..n) (distinct packed
// values, all within [lo, hi]) by repeated 256-bin histograms over the
// remaining value range; a boundary bin of at most 32 values is ranked by one
// warp.  Selected values go to emit(c) (unordered).  tmp has room for n
// values.  All threads call with uniform arguments.
template <int NT = kNT, class Emit>
__device__ void block_select(unsigned long long* cand, unsigned long long* tmp, int n, int need,
                             unsigned long long lo, unsigned long long hi, SelectSmem& S, Emit emit) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int q = tid; q < 256; q += NT) S.hist[q] = 0u;
  if (tid == 0) {
    S.tcnt[0] = 0;
    S.tcnt[1] = 0;
  }
  __syncthreads();
#pragma unroll 1
  for (int iter = 0; iter < 16; ++iter) {
    if (need <= 0) break;
    if (n <= need) {
#pragma unroll 1
      for (int i = tid; i < n; i += NT) emit(cand[i]);
      break;
    }
    if (n <= 32) {
      if (warp == 0) {
        const unsigned long long c = lane < n ? cand[lane] : 0ull;  // empty lanes rank last
        int rank = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const unsigned long long o = __shfl_sync(0xffffffffu, c, k);
          rank += (o > c) ? 1 : 0;
        }
        if (lane < n && rank < need) emit(c);
      }
      break;
    }
    const unsigned long long span = hi - lo;
    int shift = 0;
    if (span != 0ull) shift = max(0, 64 - __clzll((long long)span) - 8);
#pragma unroll 1
    for (int i = tid; i < n; i += NT) atomicAdd(&S.hist[bin_of(cand[i], lo, shift)], 1u);
    __syncthreads();
    boundary_bin(S, need);
    const uint32_t bs = (uint32_t)min(max(S.bstar, 0), 255);
    const int ab = S.above;
    const int nb = S.nb;
    int* tc = &S.tcnt[iter & 1];
#pragma unroll 1
    for (int i = tid; i < n; i += NT) {
      const unsigned long long c = cand[i];
      const uint32_t b = bin_of(c, lo, shift);
      if (b > bs) {
        emit(c);
      } else if (b == bs) {
        const int s = atomicAdd(tc, 1);
        if (s < n) tmp[s] = c;
      }
    }
    // ready for the next round: histogram cleared, the other counter reset
    for (int q = tid; q < 256; q += NT) S.hist[q] = 0u;
    if (tid == 0) S.tcnt[(iter + 1) & 1] = 0;
    __syncthreads();
    need -= ab;
    n = nb;
    lo = lo + ((unsigned long long)bs << shift);
    const unsigned long long nhi = lo + ((shift >= 64) ? ~0ull : ((1ull << shift) - 1ull));
    hi = nhi < hi ? nhi : hi;
    unsigned long long* t = cand;
    cand = tmp;
    tmp = t;
  }
  __syncthreads();
}

}  // namespace ss
