// Stage 2 (SonicSampler 3.2, Fig. 1 bottom) and the rejection-sampling
// verification (SonicSampler 3.1 "Speculative verification"; dl-note
// "Rejection Sampler").
//
// One work item per target position (persistent CTAs of 256 threads):
//  1. merge: each of the position's segments (1..Z_v runs of tiles, one per
//     stage-1 CTA) left its top-128 packed candidates in the staging buffer.
//     tau2 = the largest "smallest kept candidate" of a full list certifies
//     128 candidates, so only packed values >= tau2 enter
//     shared memory, and a histogram select picks the exact top-128, which a
//     bitonic network then sorts (processed logit descending, token ascending).
//  2. epilogue (dl-note Combination): fp64 softmax over the candidates,
//     top-k / top-p / logit-space min-p cut (shortest prefix), renormalised
//     kept probabilities; Gumbel-max token in fp32 with Philox noise keyed by
//     (seed, row, position, token), or the first candidate for greedy rows.
//  3. verification positions: accept the draft d iff p(d) > 0 and
//     fp32(u q(d)) <= p(d); on rejection draw from norm(max(0, p - q)) over
//     the kept set (truncated rows) or queue a pass over the vocabulary
//     (untruncated rows).  The last position of a row to finish walks the
//     row: accepted prefix, then the resampled or bonus token.
#include "ss_common.cuh"

namespace ss {

namespace {

struct S2Smem {
  SelectSmem sel;
  unsigned long long top[kK];
  unsigned long long slots[kNT / 32];
  int r, j, gamma, cnt, out_cnt, last;
  uint32_t status;
  int d_found;
  float d_l;
  double pd, lse, red[kNT / 32];
};

// Exclusive prefix sum of v over threads 0..kNT-1 in fp64.
__device__ __forceinline__ double block_exclusive_scan_d(double v, double* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  double add = 0.0;
  for (int w = 0; w < warp; ++w) add += scratch[w];
  __syncthreads();
  return add + incl - v;
}

// Processed logit of one token at one position (the same fp32 steps as the
// stage-1 prelude), for a draft token outside the candidate list.  All
// threads call.
__device__ float prelude_single(const Params& P, const RowCtx& rc, int pos, int r, int j, int tok,
                                S2Smem& sm) {
  float x = load_scalar(P.logits, P.logits_bf16, (int64_t)pos * P.ld + tok);
  int cnt = 0;
  if ((rc.flags & SS_PENALTY) && P.history) {
    const int32_t* hrow = P.history + (size_t)r * P.hist_stride;
    for (int h = threadIdx.x; h < rc.hist_len; h += kNT) cnt += (__ldg(hrow + h) == tok) ? 1 : 0;
    if (P.cu_draft) {
      const int base = __ldg(P.cu_draft + r);
      const int jn = min(j, __ldg(P.cu_draft + r + 1) - base);
      for (int s = threadIdx.x; s < jn; s += kNT) cnt += (__ldg(P.draft_ids + base + s) == tok) ? 1 : 0;
    }
  }
  int total;
  block_inclusive_scan(cnt, sm.sel.scan, &total);
  if ((rc.flags & SS_MASK) && P.bitmask) {
    const uint32_t w = __ldg(P.bitmask + (size_t)pos * P.mask_words + (tok >> 5));
    if (((w >> (tok & 31)) & 1u) == 0u) x = -INFINITY;
  }
  const ss_bias_entry* brow = (rc.flags & SS_BIAS) && P.bias ? P.bias + (size_t)r * P.bias_stride : nullptr;
  x = apply_penalty_bias(x, (uint32_t)total, brow != nullptr, tok, rc, brow);
  if (rc.stoch) x = __fmul_rn(x, rc.rT);
  if (x != x) x = -INFINITY;
  return x;
}

// Position results written by other CTAs of this kernel: read past L1.
__device__ __forceinline__ PosResult load_pos_result(const PosResult* p) {
  PosResult q;
  q.lse = __ldcg(&p->lse);
  q.token = __ldcg(&p->token);
  q.accept = __ldcg(&p->accept);
  q.status = __ldcg(&p->status);
  q.pad = 0;
  return q;
}

}  // namespace

__global__ void __launch_bounds__(kNT) stage2_kernel(const Params P, int verify) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int cap = P.Z * kK;
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(smem_raw);
  unsigned long long* tmp = cand + cap;
  S2Smem& sm = *reinterpret_cast<S2Smem*>(tmp + cap);
  const int tid = threadIdx.x, lane = tid & 31;
  const int npos = num_positions(P);
  const int V = P.V, Z = P.Z;

  for (int pos = blockIdx.x; pos < npos; pos += gridDim.x) {
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
      sm.out_cnt = 0;
      sm.status = 0u;
      sm.d_found = 0;
      sm.pd = 0.0;
      sm.last = 0;
    }
    __syncthreads();
    const int r = sm.r, j = sm.j, gamma = sm.gamma;
    const RowCtx rc = make_row(P.rows[r], P.hist_stride, P.bias_stride);
    const uint32_t position = rc.position + (uint32_t)j;
    // the position's segment lists (the stage-1 split of the npos * Z stages)
    const long long T = (long long)npos * Z, G = seg_grid(P, T);
    const int nseg = seg_cta((long long)pos * Z + Z - 1, T, G) - seg_cta((long long)pos * Z, T, G) + 1;
    const uint64_t seed = P.seeds[r];
    const bool is_draft = verify && j >= 0 && j < gamma;
    int32_t* cid = P.out.cand_ids ? P.out.cand_ids + (size_t)pos * kK : nullptr;
    float* cpr = P.out.cand_probs ? P.out.cand_probs + (size_t)pos * kK : nullptr;

    int32_t token = -1;      // sampled / bonus token (or resampled token on rejection)
    int accept = 0;
    double lse = 0.0;

    if (!rc.valid) {
      if (tid < kK) {
        if (cid) cid[tid] = -1;
        if (cpr) cpr[tid] = 0.0f;
      }
      if (tid == 0) {
        if (P.out.num_kept) P.out.num_kept[pos] = 0;
        atomicOr(&sm.status, (uint32_t)SS_ST_BAD_PARAM);
      }
    } else {
      // ---- row-level input checks (history / bias ids beyond the vocabulary)
      if ((rc.flags & SS_PENALTY) && P.history) {
        const int32_t* hrow = P.history + (size_t)r * P.hist_stride;
        for (int h = tid; h < rc.hist_len; h += kNT)
          if (__ldg(hrow + h) >= V) atomicOr(&sm.status, (uint32_t)SS_ST_BAD_HIST);
      }
      if ((rc.flags & SS_BIAS) && P.bias) {
        for (int e = tid; e < rc.n_bias; e += kNT)
          if (P.bias[(size_t)r * P.bias_stride + e].token >= V) atomicOr(&sm.status, (uint32_t)SS_ST_BAD_BIAS);
      }
      // ---- 1. merge the tiles' candidates
      // Load the Z_v * 128 packed candidates; a tile whose 128 slots are all
      // real certifies 128 candidates >= its smallest one, so tau2 = the
      // largest such minimum bounds the position's top-128 from below.
      const size_t tbase = (size_t)pos * Z;
      uint32_t tst = 0u;
      for (int t = tid; t < nseg; t += kNT) tst |= P.ws.tile_status[tbase + t];
      if (tst) atomicOr(&sm.status, tst);
      const unsigned long long* stg = P.ws.staging + tbase * kK;
      for (int i = tid; i < nseg * kK; i += kNT) tmp[i] = stg[i];
      __syncthreads();
      unsigned long long tm = 0ull;
      for (int t = tid >> 5; t < nseg; t += kNT / 32) {
        unsigned long long mn = ~0ull;
#pragma unroll
        for (int q = 0; q < kK / 32; ++q) {
          const unsigned long long c = tmp[t * kK + q * 32 + lane];
          mn = c < mn ? c : mn;   // an empty slot (0) makes the tile certify nothing
        }
        mn = warp_min_u64(mn);
        tm = mn > tm ? mn : tm;
      }
      const unsigned long long tau2 = block_max_u64(tm, sm.slots);
      unsigned long long lmin = ~0ull, lmax = 0ull;
      for (int i = tid; i < nseg * kK; i += kNT) {
        const unsigned long long c = tmp[i];
        if (c != 0ull && c >= tau2) {
          cand[atomicAdd(&sm.cnt, 1)] = c;
          lmin = c < lmin ? c : lmin;
          lmax = c > lmax ? c : lmax;
        }
      }
      const unsigned long long lo = block_min_u64(lmin, sm.slots);
      const unsigned long long hi = block_max_u64(lmax, sm.slots);
      const int n = sm.cnt;
      const int need = min(kK, V);
      block_select(cand, tmp, n, need, lo, hi, sm.sel,
                   [&](unsigned long long c) {
                     const int s = atomicAdd(&sm.out_cnt, 1);
                     if (s < kK) sm.top[s] = c;
                   });
      // slots the select did not fill (only if its count invariant broke) stay empty
      if (tid < kK && tid >= min(sm.out_cnt, need)) sm.top[tid] = 0ull;
      __syncthreads();
      // bitonic sort of the 128 candidates, descending
      for (int k = 2; k <= kK; k <<= 1) {
        for (int d = k >> 1; d > 0; d >>= 1) {
          if (tid < kK) {
            const int p = tid ^ d;
            if (p > tid) {
              const unsigned long long a = sm.top[tid], b = sm.top[p];
              const bool desc = (tid & k) == 0;
              if ((a < b) == desc) {
                sm.top[tid] = b;
                sm.top[p] = a;
              }
            }
          }
          __syncthreads();
        }
      }

      // ---- 2. epilogue over the candidates (thread t < 128 holds candidate t)
      const int t = tid;
      const unsigned long long c = t < kK ? sm.top[t] : 0ull;
      const bool real = t < need && c != 0ull;
      const int32_t tok = pk_tok(c);
      const float l = real ? key2f(pk_key(c)) : -INFINITY;
      const float l0 = key2f(pk_key(sm.top[0]));
      const int32_t tok0 = pk_tok(sm.top[0]);
      const bool finite = real && l > -INFINITY;
      const int n_f = __syncthreads_count(finite);
      const bool no_finite = n_f == 0;
      const bool pos_inf = !no_finite && l0 == INFINITY;
      const bool point = no_finite || pos_inf || !rc.stoch;
      int nk = 0;
      double w = 0.0, zk = 1.0;
      if (no_finite) {
        nk = 0;
      } else if (point) {
        nk = 1;
      } else {
        w = finite ? exp((double)l - (double)l0) : 0.0;
        const double Zall = block_sum_d(w, sm.red);
        int n2 = min(need, n_f);
        if ((rc.flags & SS_TOPK) && rc.top_k > 0) n2 = min(n2, rc.top_k);
        if ((rc.flags & SS_TOPP) && rc.top_p < 1.0f) {
          const double ex = block_exclusive_scan_d(t < need ? w / Zall : 0.0, sm.red);
          const int np = __syncthreads_count(t < need && ex < (double)rc.top_p);
          n2 = min(n2, np);
        }
        if ((rc.flags & SS_MINP) && rc.min_p > 0.0f) {
          const double thr = log((double)rc.min_p);
          const int nm = __syncthreads_count(t < need && ((double)l - (double)l0) >= thr);
          n2 = min(n2, nm);
        }
        nk = max(1, n2);
        zk = block_sum_d(t < nk ? w : 0.0, sm.red);
      }
      // candidate outputs
      if (t < kK) {
        if (cid) cid[t] = real ? tok : -1;
        if (cpr) {
          float pr = 0.0f;
          if (t < nk) pr = point ? (t == 0 ? 1.0f : 0.0f) : (float)(w / zk);
          cpr[t] = pr;
        }
      }
      if (tid == 0 && P.out.num_kept) P.out.num_kept[pos] = nk;
      if (no_finite) {
        if (tid == 0) atomicOr(&sm.status, (uint32_t)SS_ST_NO_FINITE);
      } else if (pos_inf && tid == 0) {
        atomicOr(&sm.status, (uint32_t)SS_ST_POS_INF);
      }

      // ---- 3. token of this position (sample / bonus)
      if (!is_draft) {
        if (no_finite) {
          token = -1;
        } else if (point) {
          token = tok0;
        } else {
          unsigned long long sc = 0ull;
          if (t < nk) {
            const float g = gumbel_of(philox_uniform(seed, (uint32_t)tok, position, (uint32_t)r, 0u));
            sc = pack(f2key(__fadd_rn(l, g)), (uint32_t)tok);
          }
          token = pk_tok(block_max_u64(sc, sm.slots));
        }
      } else {
        // ---- 4. verification of draft j
        const int32_t d = __ldg(P.draft_ids + __ldg(P.cu_draft + r) + j);
        const bool d_ok = d >= 0 && d < V;
        if (!d_ok && tid == 0) atomicOr(&sm.status, (uint32_t)SS_ST_BAD_DRAFT);
        if (no_finite) {
          accept = 0;
          token = -1;
        } else if (point) {
          accept = (d_ok && d == tok0) ? 1 : 0;
          token = tok0;
        } else {
          const int64_t qrow = (int64_t)__ldg(P.cu_draft + r) + j;
          if (rc.trunc) {
            if (t < nk && tok == d) sm.pd = w / zk;
            __syncthreads();
          } else {
            // full-vocabulary softmax: LSE from the tiles' (max, sum exp) partials
            if (tid == 0) {
              float M = -INFINITY;
              for (int tt = 0; tt < nseg; ++tt) M = fmaxf(M, P.ws.tile_lse[(size_t)pos * Z + tt].x);
              double S = 0.0;
              for (int tt = 0; tt < nseg; ++tt) {
                const float2 ms = P.ws.tile_lse[(size_t)pos * Z + tt];
                if (ms.x > -INFINITY) S += (double)ms.y * exp((double)ms.x - (double)M);
              }
              sm.lse = (double)M + log(S);
            }
            if (real && tok == d) {
              sm.d_found = 1;
              sm.d_l = l;
            }
            __syncthreads();
            lse = sm.lse;
            float ld = sm.d_l;
            if (!sm.d_found && d_ok) ld = prelude_single(P, rc, pos, r, j, d, sm);
            if (tid == 0 && d_ok) sm.pd = exp((double)ld - lse);
            __syncthreads();
          }
          const double pd = sm.pd;
          if (d_ok) {
            const float u = philox_uniform(seed, 0u, position, (uint32_t)r, 1u);
            const float prod = __fmul_rn(u, load_scalar(P.q, P.q_bf16, qrow * P.ld_q + d));
            accept = (pd > 0.0 && (double)prod <= pd) ? 1 : 0;
          }
          if (!accept) {
            if (rc.trunc) {
              // residual norm(max(0, p - q)) over the kept candidates
              double rr = 0.0;
              if (t < nk) rr = fmax(0.0, w / zk - (double)load_scalar(P.q, P.q_bf16, qrow * P.ld_q + tok));
              const int anypos = __syncthreads_or(t < nk && rr > 0.0);
              unsigned long long sc = 0ull;
              if (t < nk) {
                const float g = gumbel_of(philox_uniform(seed, (uint32_t)tok, position, (uint32_t)r, 2u));
                if (anypos) {
                  if (rr > 0.0) sc = pack(f2key(__fadd_rn(logf((float)rr), g)), (uint32_t)tok);
                } else {
                  sc = pack(f2key(__fadd_rn(l, g)), (uint32_t)tok);
                }
              }
              token = pk_tok(block_max_u64(sc, sm.slots));
              if (!anypos && tid == 0) atomicOr(&sm.status, (uint32_t)SS_ST_RESID_EMPTY);
            } else {
              token = kPending;  // drawn by the pass over the vocabulary
            }
          }
        }
      }
    }
    __syncthreads();
    const uint32_t status = sm.status;

    // ---- 5. outputs
    if (!verify) {
      if (tid == 0) {
        P.out.tokens[r] = rc.valid ? token : -1;
        P.out.row_status[r] = status;
      }
    } else {
      if (tid == 0) {
        PosResult pr;
        pr.lse = lse;
        pr.token = token;
        pr.accept = accept;
        pr.status = status;
        pr.pad = 0;
        P.ws.pos[pos] = pr;
        __threadfence();
        const uint32_t old = atomicAdd(P.ws.row_count + r, 1u);
        sm.last = (old == (uint32_t)gamma) ? 1 : 0;
      }
      __syncthreads();
      if (sm.last && tid == 0) {
        // the row's last position: walk the drafts
        __threadfence();
        const int pos0 = __ldg(P.cu_draft + r) + r;
        int32_t* tk = P.out.tokens + (size_t)r * P.out.tokens_stride;
        const int stride = P.out.tokens_stride;
        uint32_t st = 0u;
        int n_acc = 0;
        if (!rc.valid) {
          for (int s = 0; s < stride; ++s) tk[s] = -1;
          st = SS_ST_BAD_PARAM;
        } else {
          int stop = gamma;
          for (int s = 0; s < gamma; ++s) {
            const PosResult q = load_pos_result(P.ws.pos + pos0 + s);
            st |= q.status;
            if (!q.accept) {
              stop = s;
              break;
            }
          }
          const int base = __ldg(P.cu_draft + r);
          for (int s = 0; s < stop && s < stride; ++s) tk[s] = __ldg(P.draft_ids + base + s);
          const PosResult fin = load_pos_result(P.ws.pos + pos0 + stop);
          if (stop == gamma) st |= fin.status;
          int32_t ft = fin.token;
          if (ft == kPending) {
            if (stop < stride) {
              const uint32_t e = atomicAdd(P.ws.resid_count, 1u);
              P.ws.resid[e].row = r;
              P.ws.resid[e].j = stop;
              P.ws.resid[e].pos = pos0 + stop;
            }
            ft = -1;  // written by the residual pass
          }
          if (stop < stride) tk[stop] = ft;
          for (int s = stop + 1; s < stride; ++s) tk[s] = -1;
          n_acc = stop;
        }
        if (P.out.num_accepted) P.out.num_accepted[r] = n_acc;
        P.out.row_status[r] = st;
        P.ws.row_count[r] = 0u;
      }
    }
    __syncthreads();
  }
}

size_t stage2_smem_bytes(int Z) { return (size_t)Z * kK * 8 * 2 + sizeof(S2Smem); }

}  // namespace ss
