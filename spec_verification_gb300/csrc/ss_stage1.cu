// Stage 1 of the two-stage tile-aware top-k (SonicSampler 3.2, Fig. 1 top):
// one work item per (target position, vocabulary tile of B_N tokens).  Each
// item streams its tile once, applies the logits prelude (grammar mask,
// penalties, bias, temperature) and writes only the tile's 128 best packed
// candidates (key << 32 | ~token) to the staging buffer, plus a status word
// and, for untruncated verify positions, (tile max, sum of exp(x - max)).
//
// Selection is exact under the order (processed logit descending, token
// ascending).  GB300 design:
//  - persistent CTAs of 256 threads; a two-slot shared-memory ring is filled
//    by 1-D bulk copies (cp.async.bulk, completion counted on an mbarrier), so
//    the next tile streams in from HBM while the current one is processed;
//  - each thread holds E = B_N / 256 processed logits in registers;
//  - a threshold tau with at least 128 tile elements at or above it comes
//    from the per-thread maxima (the 16th largest maximum of each warp,
//    minimum over the 8 warps), so typically ~2-3% of the tile survives into
//    shared memory, where a 256-bin histogram select finishes exactly;
//  - tiles with few finite values, NaN among few finite values, or very many
//    survivors take an out-of-line radix select over the resident tile.
#include <type_traits>

#include "ss_common.cuh"

namespace ss {

namespace {

constexpr int kSpinLimit = 1 << 22;  // bounded mbarrier wait (about a second)
constexpr int kRowCache = 2048;     // rows whose position offsets stage 1 keeps in shared memory
constexpr int kSide = 1024;         // penalised tokens per tile held in the side table (power of 2)
constexpr int kBiasPre = 64;        // bias entries prefetched per item

struct __align__(16) S1Smem {
  SelectSmem sel;
  unsigned long long mbar[2];
  int cnt, nan_flag, out_cnt, nside;
  float side[kSide];  // processed-before-temperature values of the tile's history / bias tokens
  float tw[kNT / 32];
  float wmax[kNT / 32];
  double red[kNT / 32];
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(unsigned long long* m) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(m)) : "memory");
}

// One bulk copy global -> shared whose bytes complete on the slot's mbarrier.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, unsigned long long* m) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(m)), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(m))
               : "memory");
}

__device__ __forceinline__ bool mbar_wait(unsigned long long* m, uint32_t parity) {
  for (int i = 0; i < kSpinLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(m)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
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

struct TileCtx {
  int t0, nt, need, pos, r, j;
  bool mask_on, aux_on;
  bool side;  // aux entries are side-table indices + 1 (else count | bias flag)
  const ss_bias_entry* brow;
};

// Processed logit of tile element li (the same fp32 steps as the fast path).
// Penalties and bias commute with the mask (a masked token ends at -inf either
// way), so a history / bias token's value may be taken from the side table
// before the mask is applied.
template <bool BF16>
__device__ __forceinline__ float proc_elem(const Params& P, const RowCtx& rc, const TileCtx& tc,
                                           const unsigned char* ring, const uint16_t* aux, const float* side,
                                           int li) {
  float v = raw_at<BF16>(ring, li);
  const int tok = tc.t0 + li;
  if (tc.aux_on) {
    const uint32_t a = aux[li];
    if (a != 0u) {
      if (tc.side) v = side[a - 1];
      else v = apply_penalty_bias(v, a & 0x7FFFu, (a & 0x8000u) != 0u, tok, rc, tc.brow);
    }
  }
  if (tc.mask_on) {
    const uint32_t w = __ldg(P.bitmask + (size_t)tc.pos * P.mask_words + (tok >> 5));
    if (((w >> (tok & 31)) & 1u) == 0u) v = -INFINITY;
  }
  v = __fmul_rn(v, rc.rT);
  return v;
}

// Exact tile top-`need` for the cases the fast path leaves out (few finite
// values, NaN among them, or more survivors than fit in shared memory):
// MSB-first radix select on the 32-bit keys of the resident tile, then the
// lowest tokens among elements equal to the boundary key.  Thread t owns the
// contiguous elements [t*E, t*E + E), so token order is (thread, element).
template <bool BF16, int E>
__device__ __noinline__ void generic_select(const Params& P, const RowCtx& rc, const TileCtx& tc,
                                            const unsigned char* ring, const uint16_t* aux, S1Smem& sm,
                                            unsigned long long* stg) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int base = tid * E;
  auto key_of = [&](int li) -> uint32_t {
    if (li >= tc.nt) return 0u;  // not a token of this tile
    const float v = proc_elem<BF16>(P, rc, tc, ring, aux, sm.side, li);
    return (v != v) ? kKeyNegInf : f2key(v);
  };
  bool nan_seen = false;
  for (int k = 0; k < E; ++k) {
    const int li = base + k;
    if (li < tc.nt) {
      const float v = proc_elem<BF16>(P, rc, tc, ring, aux, sm.side, li);
      nan_seen |= (v != v);
    }
  }
  if (nan_seen) sm.nan_flag = 1;
  uint32_t prefix = 0u, pmask = 0u;
  int rem = tc.need;
  for (int d = 0; d < 4; ++d) {
    const int shift = 24 - 8 * d;
    sm.sel.hist[tid & 255] = 0u;
    __syncthreads();
    for (int k = 0; k < E; ++k) {
      const int li = base + k;
      const uint32_t key = key_of(li);
      const bool match = li < tc.nt && ((key & pmask) == prefix);
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
    const int li = base + k;
    if (li >= tc.nt) continue;
    const uint32_t key = key_of(li);
    if (key > kstar) {
      const int s = atomicAdd(&sm.out_cnt, 1);
      if (s < kK) stg[s] = pack(key, (uint32_t)(tc.t0 + li));
    } else if (key == kstar) {
      ++ties;
    }
  }
  int total;
  const int incl = block_inclusive_scan(ties, sm.sel.scan, &total);
  int rank = incl - ties;
  for (int k = 0; k < E && rank < rem; ++k) {
    const int li = base + k;
    if (li >= tc.nt) continue;
    if (key_of(li) == kstar) {
      const int s = atomicAdd(&sm.out_cnt, 1);
      if (s < kK) stg[s] = pack(kstar, (uint32_t)(tc.t0 + li));
      ++rank;
    }
  }
}

}  // namespace

// One work item's bookkeeping besides its tile, copied into shared memory with
// cp.async one item ahead (no registers held while the copies are in flight).
template <int MW>
struct __align__(16) NextBuf {
  ss_bias_entry bias[kBiasPre];  // bias[r][t]        (t < min(bias_stride, kBiasPre))
  int hist[kNT];            // history[r][t]          (t < hist_stride)
  int draft[kNT];           // drafts of the row      (t < min(j, gamma))
  uint32_t mask[MW];        // the tile's bitmask words
  ss_row_params rp;
  int pos, r, j, gamma;     // the item's target position, row, draft index, row draft count
};

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <bool BF16, int NCH>
__global__ void __launch_bounds__(kNT, 2) stage1_kernel(const Params P) {
  constexpr int VEC = BF16 ? 8 : 4;
  constexpr int E = NCH * VEC;
  constexpr int BN = kNT * E;
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int MW = BN / 32;
  using Bits = typename std::conditional<(E > 32), unsigned long long, uint32_t>::type;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // [ring slot 0 | ring slot 1 | aux (uint16 per token; the select's scratch
  //  afterwards) | survivors | S1Smem | NextBuf x 2 | row offsets]
  unsigned char* ring0 = smem_raw;
  uint16_t* aux = reinterpret_cast<uint16_t*>(smem_raw + 2 * BN * ESZ);
  unsigned long long* tmp = reinterpret_cast<unsigned long long*>(aux);
  unsigned long long* surv = reinterpret_cast<unsigned long long*>(smem_raw + 2 * BN * ESZ + BN * 2);
  S1Smem& sm = *reinterpret_cast<S1Smem*>(smem_raw + 2 * BN * ESZ + BN * 2 + kCap1 * 8);
  NextBuf<MW>* nbuf = reinterpret_cast<NextBuf<MW>*>(smem_raw + 2 * BN * ESZ + BN * 2 + kCap1 * 8 + sizeof(S1Smem));
  int* offs = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(nbuf) + 2 * sizeof(NextBuf<MW>));
  static_assert(BN * 2 >= kCap1 * 8, "aux region must hold the select scratch");
  static_assert(sizeof(S1Smem) % 16 == 0 && sizeof(NextBuf<MW>) % 16 == 0, "16-byte regions");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V, Z = P.Z;
  if (blockIdx.x == 0 && tid == 0) *P.ws.resid_count = 0u;  // residual queue of this call
  const int npos = num_positions(P);
  const long long total = (long long)npos * Z;
  // first target position of each row (cu_draft[r] + r), cached for the row lookups
  const bool cached = P.cu_draft != nullptr && P.B + 1 <= kRowCache;
  if (cached)
    for (int q = tid; q <= P.B; q += kNT) offs[q] = __ldg(P.cu_draft + q) + q;

  auto issue = [&](long long it, int slot) {  // thread 0 only
    const int pos = (int)(it / Z);
    const int t0 = (int)(it - (long long)pos * Z) * BN;
    const int nt = min(BN, V - t0);
    const uint32_t bytes = (uint32_t)((nt * ESZ + 15) & ~15);
    const unsigned char* src = static_cast<const unsigned char*>(P.logits) + ((size_t)pos * P.ld + t0) * ESZ;
    bulk_load(ring0 + slot * BN * ESZ, src, bytes, &sm.mbar[slot]);
  };
  // row of a work item (every thread, from the cached offsets)
  auto locate = [&](long long it, int& pos, int& r, int& j, int& gamma) {
    pos = (int)(it / Z);
    r = pos;
    j = 0;
    gamma = 0;
    if (P.cu_draft) {
      int lo = 0, hi = P.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const int o = cached ? offs[mid] : (__ldg(P.cu_draft + mid) + mid);
        if (o <= pos) lo = mid; else hi = mid - 1;
      }
      r = lo;
      const int c0 = cached ? offs[lo] - lo : __ldg(P.cu_draft + lo);
      const int c1 = cached ? offs[lo + 1] - lo - 1 : __ldg(P.cu_draft + lo + 1);
      j = pos - c0 - r;
      gamma = c1 - c0;
    }
  };
  // warp 0: locate an item's row and copy its bookkeeping into nb with
  // cp.async (the other warps never wait on these loads)
  auto prefetch = [&](long long it, NextBuf<MW>& nb) {
    int pos, r, j, gamma;
    locate(it, pos, r, j, gamma);
    if (lane == 0) {
      nb.pos = pos;
      nb.r = r;
      nb.j = j;
      nb.gamma = gamma;
    }
    const int t0 = (int)(it - (long long)pos * Z) * BN;
    const int nt = min(BN, V - t0);
    if (lane < (int)(sizeof(ss_row_params) / 4))
      cp_async4(reinterpret_cast<uint32_t*>(&nb.rp) + lane, reinterpret_cast<const uint32_t*>(P.rows + r) + lane);
    if (P.history != nullptr)
      for (int q = lane; q < min(P.hist_stride, kNT); q += 32)
        cp_async4(&nb.hist[q], P.history + (size_t)r * P.hist_stride + q);
    if (P.cu_draft != nullptr) {
      const int base = cached ? offs[r] - r : __ldg(P.cu_draft + r);
      for (int q = lane; q < min(min(j, gamma), kNT); q += 32) cp_async4(&nb.draft[q], P.draft_ids + base + q);
    }
    if (P.bias != nullptr)
      for (int q = lane; q < min(P.bias_stride, kBiasPre); q += 32) {  // 4-byte copies: 4-byte aligned entries
        const ss_bias_entry* be = P.bias + (size_t)r * P.bias_stride + q;
        cp_async4(&nb.bias[q].token, &be->token);
        cp_async4(&nb.bias[q].value, &be->value);
      }
    if (P.bitmask != nullptr)
      for (int w = lane; w < MW && w * 32 < nt; w += 32)
        cp_async4(&nb.mask[w], P.bitmask + (size_t)pos * P.mask_words + (t0 >> 5) + w);
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  if (tid == 0) {
    mbar_init(&sm.mbar[0]);
    mbar_init(&sm.mbar[1]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sm.cnt = 0;
    sm.nan_flag = 0;
    sm.out_cnt = 0;
    sm.nside = 0;
    if ((long long)blockIdx.x < total) issue(blockIdx.x, 0);
  }
  __syncthreads();  // offsets cached, barriers initialised
  if (warp == 0 && (long long)blockIdx.x < total) prefetch(blockIdx.x, nbuf[0]);
  cp_async_wait_all();
  __syncthreads();

  int k = 0;
  for (long long item = blockIdx.x; item < total; item += gridDim.x, ++k) {
    const int slot = k & 1;
    const unsigned char* ring = ring0 + slot * BN * ESZ;
    const NextBuf<MW>& cb = nbuf[slot];
    const long long nx = item + gridDim.x;
    // prefetch the next item: its tile into the other ring slot and its
    // bookkeeping into the other buffer (both freed by the previous item's
    // final barrier)
    if (nx < total && warp == 0) {
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(nx, slot ^ 1);
      }
      prefetch(nx, nbuf[slot ^ 1]);
    }
    const int pos = cb.pos, r = cb.r, j = cb.j, gamma = cb.gamma;

    const int tile = (int)(item - (long long)pos * Z);
    TileCtx tc;
    tc.pos = pos;
    tc.t0 = tile * BN;
    tc.nt = min(BN, V - tc.t0);
    tc.need = min(kK, tc.nt);
    tc.r = r;
    tc.j = j;
    const RowCtx rc = make_row(cb.rp, P.hist_stride, P.bias_stride);
    tc.mask_on = (rc.flags & SS_MASK) && P.bitmask != nullptr;
    const bool pen_on = (rc.flags & SS_PENALTY) && P.history != nullptr;
    const bool bias_on = (rc.flags & SS_BIAS) && P.bias != nullptr;
    tc.aux_on = pen_on || bias_on;
    tc.brow = bias_on ? P.bias + (size_t)r * P.bias_stride : nullptr;
    unsigned long long* stg = P.ws.staging + (size_t)item * kK;
    const int t0 = tc.t0, nt = tc.nt;
    const bool full = (nt == BN);

    // the tile's bytes
    const bool landed = mbar_wait(&sm.mbar[slot], (uint32_t)((k >> 1) & 1));
    if (!__syncthreads_and(landed)) {
      // a bulk copy did not complete: record it and stop this CTA
      if (tid == 0) {
        atomicAdd(P.ws.diag + 3, 1u);
        if (nx < total) mbar_wait(&sm.mbar[slot ^ 1], (uint32_t)(((k + 1) >> 1) & 1));
      }
      cp_async_wait_all();
      break;
    }

    // tile-local history counts and bias flags
    tc.side = tc.aux_on && (pen_on ? rc.hist_len + min(j, gamma) : 0) + (bias_on ? rc.n_bias : 0) <= kSide;
    if (tc.aux_on && rc.valid) {
      uint4* a4 = reinterpret_cast<uint4*>(aux);
      for (int w = tid; w < BN / 8; w += kNT) a4[w] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      uint32_t* a32 = reinterpret_cast<uint32_t*>(aux);
      auto count = [&](int id) {
        if (id >= t0 && id < t0 + nt) atomicAdd(a32 + ((id - t0) >> 1), 1u << (16 * ((id - t0) & 1)));
      };
      if (pen_on) {
        if (tid < rc.hist_len) count(cb.hist[tid]);
        const int32_t* hrow = P.history + (size_t)r * P.hist_stride;
        for (int h = tid + kNT; h < rc.hist_len; h += kNT) count(__ldg(hrow + h));
        if (P.cu_draft) {  // drafts accepted before this verify position
          if (tid < min(j, gamma)) count(cb.draft[tid]);
          const int base = __ldg(P.cu_draft + r);
          for (int q = tid + kNT; q < min(j, gamma); q += kNT) count(__ldg(P.draft_ids + base + q));
        }
      }
      if (bias_on) {
        auto flag = [&](int id) {
          if (id >= t0 && id < t0 + nt) atomicOr(a32 + ((id - t0) >> 1), 0x8000u << (16 * ((id - t0) & 1)));
        };
        if (tid < min(rc.n_bias, kBiasPre)) flag(cb.bias[tid].token);
        for (int e = kBiasPre + tid; e < rc.n_bias; e += kNT) flag(tc.brow[e].token);
      }
      __syncthreads();
      if (tc.side) {
        // penalised values of the flagged tokens, computed here (few live
        // registers) so the hot loop only looks them up; each thread handles
        // the tokens it owns in the hot loop's layout, so no barrier is needed
        for (int c = 0; c < NCH; ++c) {
          const int e0 = (c * kNT + tid) * VEC;
          if (e0 >= nt) break;
          uint32_t w[VEC / 2];
          if constexpr (BF16) {
            const uint4 a = *reinterpret_cast<const uint4*>(aux + e0);
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
            if ((a.x | a.y | a.z | a.w) == 0u) continue;
          } else {
            const uint2 a = *reinterpret_cast<const uint2*>(aux + e0);
            w[0] = a.x; w[1] = a.y;
            if ((a.x | a.y) == 0u) continue;
          }
          for (int jj = 0; jj < VEC; ++jj) {
            const uint32_t a = (w[jj >> 1] >> (16 * (jj & 1))) & 0xFFFFu;
            if (a == 0u) continue;
            const int li = e0 + jj;
            const float pv = apply_penalty_bias(raw_at<BF16>(ring, li), a & 0x7FFFu, (a & 0x8000u) != 0u, t0 + li,
                                                rc, tc.brow);
            const int q = atomicAdd(&sm.nside, 1);  // < kSide: bounded by the flagged-token count
            sm.side[q] = pv;
            aux[li] = (uint16_t)(q + 1);
          }
        }
      }
    }

    if (!rc.valid) {  // invalid row parameters: stage 2 reports the row, nothing to select
      for (int q = tid; q < kK; q += kNT) stg[q] = 0ull;
      if (tid == 0) P.ws.tile_status[item] = 0u;
    } else {
      // ---- prelude in registers, per-thread maximum -----------------------------
      float x[E];
      float m = -INFINITY;
      if (full && !tc.mask_on && !tc.aux_on) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const uint4 raw = *reinterpret_cast<const uint4*>(ring + (size_t)(c * kNT + tid) * 16);
#pragma unroll
          for (int jj = 0; jj < VEC; ++jj) {
            const float v = __fmul_rn(vec_elem<BF16>(raw, jj), rc.rT);
            x[c * VEC + jj] = v;
            m = fmaxf(m, v);
          }
        }
      } else {
        // general case: grammar mask and history / bias tokens; FULL drops the
        // ragged-tile check from full tiles
        auto hot = [&](auto full_c) {
          constexpr bool FULL = decltype(full_c)::value;
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const int e0 = (c * kNT + tid) * VEC;
            const uint4 raw = *reinterpret_cast<const uint4*>(ring + (size_t)(c * kNT + tid) * 16);
            const uint32_t mwc = (tc.mask_on && (FULL || e0 < nt)) ? cb.mask[e0 >> 5] : 0xFFFFFFFFu;
            uint32_t auxw[VEC / 2];
            bool any_aux = false;
            if (tc.aux_on && (FULL || e0 < nt)) {
              if constexpr (BF16) {
                const uint4 a = *reinterpret_cast<const uint4*>(aux + e0);
                auxw[0] = a.x; auxw[1] = a.y; auxw[2] = a.z; auxw[3] = a.w;
                any_aux = (a.x | a.y | a.z | a.w) != 0u;
              } else {
                const uint2 a = *reinterpret_cast<const uint2*>(aux + e0);
                auxw[0] = a.x; auxw[1] = a.y;
                any_aux = (a.x | a.y) != 0u;
              }
            }
#pragma unroll
            for (int jj = 0; jj < VEC; ++jj) {
              float v = vec_elem<BF16>(raw, jj);
              if (any_aux) {
                const uint32_t a = (auxw[jj >> 1] >> (16 * (jj & 1))) & 0xFFFFu;
                if (a != 0u) v = sm.side[(a - 1) & (kSide - 1)];
              }
              if (((mwc >> ((e0 + jj) & 31)) & 1u) == 0u) v = -INFINITY;
              v = __fmul_rn(v, rc.rT);
              if (!FULL && e0 + jj >= nt) v = -INFINITY;
              x[c * VEC + jj] = v;
              m = fmaxf(m, v);
            }
          }
        };
        if (full) hot(std::true_type{});
        else hot(std::false_type{});
      }

      // ---- threshold from the per-thread maxima ----------------------------------
      // Warp bitonic sort (descending) of the 32 maxima; lane 15 holds the 16th
      // largest.  tau = min over warps, so >= 8 * 16 = 128 threads have a
      // maximum >= tau, i.e. >= 128 tile elements are >= tau.
      {
        float v = m;
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
        if (lane == 0) sm.wmax[warp] = v;
      }
      if (tid == 0) {  // per-item counters (last read before the previous item's final barrier)
        sm.cnt = 0;
        sm.nan_flag = 0;
        sm.out_cnt = 0;
      }
      __syncthreads();
      float tau = sm.tw[0], tmax = sm.wmax[0];
#pragma unroll
      for (int w = 1; w < kNT / 32; ++w) {
        tau = fminf(tau, sm.tw[w]);
        tmax = fmaxf(tmax, sm.wmax[w]);
      }

      // ---- (tile max, sum exp) for untruncated stochastic verify positions -----
      if (P.cu_draft != nullptr && j < gamma && rc.stoch && !rc.trunc) {
        float sum = 0.0f;
        if (tmax > -INFINITY) {
          const float k2 = 1.4426950408889634f;
          const float off = tmax * k2;
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float v = x[e];
            if (v > -INFINITY) sum += exp2f(__fmaf_rn(v, k2, -off));
          }
        }
        const double S = block_sum_d((double)sum, sm.red);
        if (tid == 0) P.ws.tile_lse[item] = make_float2(tmax, (float)S);
      }

      // ---- survivors: x >= tau (tau = -inf: every finite value) -----------------
      // A bitmask per thread, one shared-memory reservation per warp; survivors
      // are re-derived from the resident tile (same fp32 steps; a survivor is
      // never masked).  NaN compares false and so survives; it is keyed as -inf
      // and reported.
      const bool few_finite = !(tau > -INFINITY);
      const float tcut = few_finite ? -3.402823466e38f : tau;
      Bits bits = 0;
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (!(x[e] < tcut)) bits |= (Bits)1 << e;
      const int cnt = (E > 32) ? __popcll((unsigned long long)bits) : __popc((uint32_t)bits);
      int incl = cnt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
      }
      int wbase = 0;
      if (lane == 31 && incl > 0) wbase = atomicAdd(&sm.cnt, incl);
      wbase = __shfl_sync(0xffffffffu, wbase, 31);
      int off = wbase + incl - cnt;
      while (bits) {
        const int e = (E > 32) ? (__ffsll((long long)bits) - 1) : (__ffs((int)(uint32_t)bits) - 1);
        bits &= bits - 1;
        const int li = ((e / VEC) * kNT + tid) * VEC + (e % VEC);
        float v = raw_at<BF16>(ring, li);
        if (tc.aux_on) {
          const uint32_t a = aux[li];
          if (a != 0u) v = sm.side[(a - 1) & (kSide - 1)];
        }
        v = __fmul_rn(v, rc.rT);
        const bool isn = (v != v);
        if (isn) sm.nan_flag = 1;
        if (off < kCap1) surv[off] = pack(isn ? kKeyNegInf : f2key(v), (uint32_t)(t0 + li));
        ++off;
      }
      __syncthreads();
      const int n = sm.cnt;
      const bool nan_here = sm.nan_flag != 0;
      auto emit = [&](unsigned long long cv) {
        const int q = atomicAdd(&sm.out_cnt, 1);
        if (q < kK) stg[q] = cv;
      };
      // few finite values: the fast path is exact only with enough of them and no NaN
      if (n <= kCap1 && n >= tc.need && !(few_finite && nan_here) && (tc.side || !tc.aux_on)) {
        const unsigned long long lo = nan_here ? pack(kKeyNegInf, 0xFFFFFFFFu) : pack(f2key(tcut), 0xFFFFFFFFu);
        const unsigned long long hi = pack(f2key(tmax), 0u);
        block_select(surv, tmp, n, tc.need, lo, hi, sm.sel, emit);
      } else {
        if (tid == 0) atomicAdd(P.ws.diag + 0, 1u);
        if (tid == 0) sm.out_cnt = 0;
        __syncthreads();
        generic_select<BF16, E>(P, rc, tc, ring, aux, sm, stg);
      }
      __syncthreads();
      // empty slots: a tile with fewer than 128 tokens (or any slot the select
      // left unwritten) holds the sentinel 0
      for (int q = min(sm.out_cnt, tc.need) + tid; q < kK; q += kNT) stg[q] = 0ull;
      if (tid == 0) P.ws.tile_status[item] = sm.nan_flag ? SS_ST_NAN : 0u;
    }
    if (tid == 0) sm.nside = 0;  // read by this item's hot loop only
    cp_async_wait_all();  // the next item's bookkeeping
    __syncthreads();
  }
}

// Explicit instantiations: fp32 / bf16 logits, B_N = 8192 and 16384.
template __global__ void stage1_kernel<false, 8>(const Params);
template __global__ void stage1_kernel<false, 16>(const Params);
template __global__ void stage1_kernel<true, 4>(const Params);
template __global__ void stage1_kernel<true, 8>(const Params);

const void* stage1_ptr(bool bf16, int BN) {
  if (!bf16) return BN == 8192 ? (const void*)stage1_kernel<false, 8> : (const void*)stage1_kernel<false, 16>;
  return BN == 8192 ? (const void*)stage1_kernel<true, 4> : (const void*)stage1_kernel<true, 8>;
}

void stage1_launch(bool bf16, int BN, int grid, size_t smem, cudaStream_t st, const Params& P) {
  if (!bf16) {
    if (BN == 8192) stage1_kernel<false, 8><<<grid, kNT, smem, st>>>(P);
    else stage1_kernel<false, 16><<<grid, kNT, smem, st>>>(P);
  } else {
    if (BN == 8192) stage1_kernel<true, 4><<<grid, kNT, smem, st>>>(P);
    else stage1_kernel<true, 8><<<grid, kNT, smem, st>>>(P);
  }
}

size_t stage1_smem_bytes(int BN, bool bf16, int max_rows) {
  const size_t nb = BN == 8192 ? sizeof(NextBuf<256>) : sizeof(NextBuf<512>);
  return (size_t)2 * BN * (bf16 ? 2 : 4) + (size_t)BN * 2 + (size_t)kCap1 * 8 + sizeof(S1Smem) + 2 * nb +
         (max_rows + 1 <= kRowCache ? (size_t)(max_rows + 1) * 4 : 0);
}

}  // namespace ss
