// Stage 1 of the two-stage tile-aware top-k (SonicSampler 3.2, Fig. 1 top):
// one work item per (target position, vocabulary tile of B_N tokens).  Each
// item streams its tile once with 128-bit loads, applies the logits prelude
// in registers (grammar mask, penalties, bias, temperature), and writes only
// the tile's 128 best packed candidates (key << 32 | ~token) to the staging
// buffer, plus the tile's smallest kept candidate, a status word and, for
// untruncated verify positions, (tile max, sum of exp(x - max)).
//
// Selection is exact under the order (processed logit descending, token
// ascending).  GB300 design: persistent CTAs of 256 threads; each thread
// holds E = B_N / 256 processed logits in registers; a threshold tau that
// provably has at least 128 elements at or above it is taken from the
// per-thread maxima (the 16th largest maximum of each warp, minimum over the
// 8 warps), so typically ~2-3% of the tile survives into shared memory, where
// a 256-bin histogram select finishes exactly.  Degenerate tiles (few finite
// values, very many survivors) take a radix select over the registers.
#include "ss_common.cuh"

namespace ss {

namespace {

struct S1Smem {
  SelectSmem sel;
  unsigned long long smin;
  int r, j, gamma;
  int cnt, nan_flag, out_cnt;
  float tw[kNT / 32];
  float wmax[kNT / 32];
  double red[kNT / 32];
};

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

// Index-ordered fill: emit the `rem` lowest-token elements among those with
// match(e) true.  Register element e = c * VEC + jj has tile offset
// (c * kNT + tid) * VEC + jj, so token order is (c, tid, jj).
template <int NCH, int VEC, class Match, class Emit>
__device__ void fill_lowest(int rem, S1Smem& sm, Match match, Emit emit) {
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    if (rem > 0) {  // uniform across the block
      int cnt = 0;
#pragma unroll
      for (int jj = 0; jj < VEC; ++jj) cnt += match(c * VEC + jj) ? 1 : 0;
      int total;
      const int incl = block_inclusive_scan(cnt, sm.sel.scan, &total);
      int rank = incl - cnt;
#pragma unroll
      for (int jj = 0; jj < VEC; ++jj) {
        const int e = c * VEC + jj;
        if (match(e)) {
          if (rank < rem) emit(e);
          ++rank;
        }
      }
      rem -= min(total, rem);
    }
  }
}

}  // namespace

template <bool BF16, int NCH>
__global__ void __launch_bounds__(kNT, 2) stage1_kernel(const Params P) {
  constexpr int VEC = BF16 ? 8 : 4;
  constexpr int E = NCH * VEC;
  constexpr int BN = kNT * E;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // aux: per-token history count (bits 0..14) and bias flag (bit 15), one
  // uint16 per tile token; reused as the select's scratch list afterwards.
  uint16_t* aux = reinterpret_cast<uint16_t*>(smem_raw);
  unsigned long long* tmp = reinterpret_cast<unsigned long long*>(smem_raw);
  unsigned long long* surv = reinterpret_cast<unsigned long long*>(smem_raw + (size_t)BN * 2);
  S1Smem& sm = *reinterpret_cast<S1Smem*>(smem_raw + (size_t)BN * 2 + (size_t)kCap1 * 8);
  static_assert((size_t)BN * 2 >= (size_t)kCap1 * 8, "aux region must hold the select scratch");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V, Z = P.Z;
  if (blockIdx.x == 0 && tid == 0) *P.ws.resid_count = 0u;  // residual queue of this call
  const int npos = num_positions(P);
  const long long total = (long long)npos * Z;
  const size_t esz = BF16 ? 2 : 4;

  for (long long item = blockIdx.x; item < total; item += gridDim.x) {
    const int pos = (int)(item / Z);
    const int tile = (int)(item - (long long)pos * Z);
    const int t0 = tile * BN;
    const int nt = min(BN, V - t0);

    // ---- 1. issue the tile's loads (depend only on the position) ------------
    const unsigned char* rowp = static_cast<const unsigned char*>(P.logits) + ((size_t)pos * P.ld + t0) * esz;
    uint4 raw[NCH];
    uint32_t mw[NCH];
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int e0 = (c * kNT + tid) * VEC;
      if (e0 < nt) raw[c] = __ldcs(reinterpret_cast<const uint4*>(rowp + (size_t)e0 * esz));
      else raw[c] = make_uint4(0u, 0u, 0u, 0u);
      mw[c] = 0xFFFFFFFFu;
      if (P.bitmask != nullptr && e0 < nt)
        mw[c] = __ldg(P.bitmask + (size_t)pos * P.mask_words + ((t0 + e0) >> 5));
    }
    // ---- 2. row of this position ---------------------------------------------
    if (tid == 0) {
      int r = pos, j = 0, g = 0;
      if (P.cu_draft) {
        r = find_row(P.cu_draft, P.B, pos);
        const int c0 = __ldg(P.cu_draft + r);
        j = pos - c0 - r;
        g = __ldg(P.cu_draft + r + 1) - c0;
      }
      sm.r = r;
      sm.j = j;
      sm.gamma = g;
      sm.cnt = 0;
      sm.nan_flag = 0;
      sm.out_cnt = 0;
      sm.smin = ~0ull;
    }
    __syncthreads();
    const int r = sm.r, j = sm.j, gamma = sm.gamma;
    const RowCtx rc = make_row(P.rows[r], P.hist_stride, P.bias_stride);
    const bool mask_on = (rc.flags & SS_MASK) && P.bitmask != nullptr;
    const bool pen_on = (rc.flags & SS_PENALTY) && P.history != nullptr;
    const bool bias_on = (rc.flags & SS_BIAS) && P.bias != nullptr;
    const bool aux_on = pen_on || bias_on;
    const ss_bias_entry* brow = bias_on ? P.bias + (size_t)r * P.bias_stride : nullptr;
    unsigned long long* stg = P.ws.staging + (size_t)item * kK;
    if (!rc.valid) {  // invalid row parameters: stage 2 reports the row, nothing to select
      for (int s = tid; s < kK; s += kNT) stg[s] = 0ull;
      if (tid == 0) {
        P.ws.tile_min[item] = 0ull;
        P.ws.tile_status[item] = 0u;
      }
      __syncthreads();
      continue;
    }

    // ---- 3. tile-local history counts and bias flags -------------------------
    if (aux_on) {
      uint4* a4 = reinterpret_cast<uint4*>(aux);
      for (int w = tid; w < BN / 8; w += kNT) a4[w] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      uint32_t* a32 = reinterpret_cast<uint32_t*>(aux);
      if (pen_on) {
        const int32_t* hrow = P.history + (size_t)r * P.hist_stride;
        for (int h = tid; h < rc.hist_len; h += kNT) {
          const int id = __ldg(hrow + h);
          if (id >= t0 && id < t0 + nt) atomicAdd(a32 + ((id - t0) >> 1), 1u << (16 * ((id - t0) & 1)));
        }
        if (P.cu_draft) {  // drafts accepted before this verify position
          const int base = __ldg(P.cu_draft + r);
          for (int s = tid; s < min(j, gamma); s += kNT) {
            const int id = __ldg(P.draft_ids + base + s);
            if (id >= t0 && id < t0 + nt) atomicAdd(a32 + ((id - t0) >> 1), 1u << (16 * ((id - t0) & 1)));
          }
        }
      }
      if (bias_on) {
        for (int e = tid; e < rc.n_bias; e += kNT) {
          const int id = brow[e].token;
          if (id >= t0 && id < t0 + nt) atomicOr(a32 + ((id - t0) >> 1), 0x8000u << (16 * ((id - t0) & 1)));
        }
      }
      __syncthreads();
    }

    // ---- 4. prelude in registers, per-thread maximum ---------------------------
    float x[E];
    float m = -INFINITY;
    const bool full = (nt == BN);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int e0 = (c * kNT + tid) * VEC;
      uint32_t auxw[VEC / 2];
      bool any_aux = false;
      if (aux_on && (full || e0 < nt)) {
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
        const int e = c * VEC + jj;
        float v = vec_elem<BF16>(raw[c], jj);
        const bool valid = full || (e0 + jj < nt);
        if (mask_on && ((mw[c] >> ((e0 + jj) & 31)) & 1u) == 0u) v = -INFINITY;
        if (any_aux) {
          const uint32_t a = (auxw[jj >> 1] >> (16 * (jj & 1))) & 0xFFFFu;
          if (a != 0u) v = apply_penalty_bias(v, a & 0x7FFFu, (a & 0x8000u) != 0u, t0 + e0 + jj, rc, brow);
        }
        if (rc.stoch) v = __fmul_rn(v, rc.rT);
        if (!valid) v = -INFINITY;
        x[e] = v;
        m = fmaxf(m, v);
      }
    }

    // ---- 5. threshold from the per-thread maxima --------------------------------
    // Warp bitonic sort (descending) of the 32 maxima; lane 15 holds the 16th
    // largest.  tau = min over warps, so >= 8 * 16 = 128 threads have a
    // maximum >= tau, i.e. >= 128 tile elements are >= tau.
    {
      float v = m;
#pragma unroll
      for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int d = k >> 1; d > 0; d >>= 1) {
          const float o = __shfl_xor_sync(0xffffffffu, v, d);
          const bool keep_max = (((lane & d) == 0) == ((lane & k) == 0));
          v = keep_max ? fmaxf(v, o) : fminf(v, o);
        }
      }
      if (lane == 15) sm.tw[warp] = v;
      if (lane == 0) sm.wmax[warp] = v;
    }
    __syncthreads();
    float tau = sm.tw[0], tmax = sm.wmax[0];
#pragma unroll
    for (int w = 1; w < kNT / 32; ++w) {
      tau = fminf(tau, sm.tw[w]);
      tmax = fmaxf(tmax, sm.wmax[w]);
    }

    // ---- 6. (tile max, sum exp) for untruncated stochastic verify positions ---
    const bool need_lse = P.cu_draft != nullptr && j < gamma && rc.stoch && !rc.trunc && rc.valid;
    if (need_lse) {
      float s = 0.0f;
      if (tmax > -INFINITY) {
        const float k2 = 1.4426950408889634f;
        const float off = tmax * k2;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float v = x[e];
          if (v > -INFINITY) s += exp2f(__fmaf_rn(v, k2, -off));
        }
      }
      const double S = block_sum_d((double)s, sm.red);
      if (tid == 0) P.ws.tile_lse[item] = make_float2(tmax, (float)S);
    }

    // ---- 7. exact tile top-128 -------------------------------------------------
    auto emit = [&](unsigned long long c) {
      const int s = atomicAdd(&sm.out_cnt, 1);
      if (s < kK) stg[s] = c;
      atomicMin(&sm.smin, c);
    };
    auto tok_of = [&](int e) { return t0 + ((e / VEC) * kNT + tid) * VEC + (e % VEC); };
    auto valid_e = [&](int e) { return full || (((e / VEC) * kNT + tid) * VEC + (e % VEC)) < nt; };
    const int need = min(kK, nt);
    bool generic = false;
    if (tau > -INFINITY) {
      // Path A: survivors x >= tau (NaN survives as -inf and is reported).
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float v = x[e];
        if (!(v < tau)) {
          const bool isn = (v != v);
          if (isn) sm.nan_flag = 1;
          const uint32_t key = isn ? kKeyNegInf : f2key(v);
          const int slot = atomicAdd(&sm.cnt, 1);
          if (slot < kCap1) surv[slot] = pack(key, (uint32_t)tok_of(e));
        }
      }
      __syncthreads();
      const int n = sm.cnt;
      if (n <= kCap1) {
        const unsigned long long lo = sm.nan_flag ? pack(kKeyNegInf, 0xFFFFFFFFu) : pack(f2key(tau), 0xFFFFFFFFu);
        const unsigned long long hi = pack(f2key(tmax), 0u);
        block_select(surv, tmp, n, need, lo, hi, sm.sel, emit);
      } else {
        generic = true;
      }
    } else {
      // Path B: tau = -inf (few finite values): survivors are the finite ones.
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float v = x[e];
        if (valid_e(e)) {
          if (v != v) sm.nan_flag = 1;
          if (v > -INFINITY) {
            const int slot = atomicAdd(&sm.cnt, 1);
            if (slot < kCap1) surv[slot] = pack(f2key(v), (uint32_t)tok_of(e));
          }
        }
      }
      __syncthreads();
      const int n = sm.cnt;
      if (n > kCap1) {
        generic = true;
      } else if (n >= need) {
        block_select(surv, tmp, n, need, pack(kKeyNegInf, 0xFFFFFFFFu), ~0ull, sm.sel, emit);
      } else {
        for (int i = tid; i < n; i += kNT) emit(surv[i]);
        // the rest: lowest tokens among -inf / NaN elements
        fill_lowest<NCH, VEC>(need - n, sm,
                              [&](int e) { return valid_e(e) && !(x[e] > -INFINITY); },
                              [&](int e) { emit(pack(kKeyNegInf, (uint32_t)tok_of(e))); });
        __syncthreads();
      }
    }
    if (generic) {
      // Path C: MSB-first radix select over the register keys (4 x 8 bits),
      // then the lowest tokens among elements equal to the boundary key.
      if (tid == 0) atomicAdd(P.ws.diag + 0, 1u);
      auto key_of = [&](int e) -> uint32_t {
        const float v = x[e];
        return (v != v) ? kKeyNegInf : f2key(v);
      };
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (valid_e(e) && x[e] != x[e]) sm.nan_flag = 1;
      uint32_t prefix = 0u, pmask = 0u;
      int rem = need;
      for (int d = 0; d < 4; ++d) {
        const int shift = 24 - 8 * d;
        sm.sel.hist[tid & 255] = 0u;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint32_t k = key_of(e);
          const bool match = valid_e(e) && ((k & pmask) == prefix);
          const uint32_t bin = match ? ((k >> shift) & 255u) : 256u;
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
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (valid_e(e)) {
          const uint32_t k = key_of(e);
          if (k > kstar) emit(pack(k, (uint32_t)tok_of(e)));
        }
      }
      fill_lowest<NCH, VEC>(rem, sm, [&](int e) { return valid_e(e) && key_of(e) == kstar; },
                            [&](int e) { emit(pack(kstar, (uint32_t)tok_of(e))); });
    }
    __syncthreads();
    // sentinel slots of a tile with fewer than 128 tokens
    for (int s = need + tid; s < kK; s += kNT) stg[s] = 0ull;
    if (tid == 0) {
      P.ws.tile_min[item] = (need == kK) ? sm.smin : 0ull;
      P.ws.tile_status[item] = sm.nan_flag ? SS_ST_NAN : 0u;
    }
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

size_t stage1_smem_bytes(int BN) {
  return (size_t)BN * 2 + (size_t)kCap1 * 8 + sizeof(S1Smem);
}

}  // namespace ss
