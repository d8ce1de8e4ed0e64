// Stage 2 (SonicSampler 3.2, Fig. 1 bottom) and the rejection-sampling
// verification (SonicSampler 3.1 "Speculative verification"; dl-note
// "Rejection Sampler").
//
// One work item per target position (persistent CTAs of 128 threads, one
// per candidate):
//  1. merge: each of the position's segments (1..Z_v runs of tiles, one per
//     stage-1 CTA) left its top-128 packed candidates in the staging buffer.
//     One segment is the answer already; otherwise tau2 = the largest
//     "smallest kept candidate" of a full list certifies 128 candidates, only
//     packed values >= tau2 enter shared memory, and a histogram select picks
//     the exact top-128.  The 128 are ordered (processed logit descending,
//     token ascending) by ranking: a candidate's place is the number of
//     candidates above it.
//  2. epilogue (dl-note Combination): the fp64 softmax weights
//     w_t = exp(l_t - l_0), one candidate per thread of four warps; then one
//     warp holding four consecutive candidates per lane: top-k / top-p
//     (mass before t below top_p) / min-p (l_t - l_0 >= ln min_p, i.e.
//     w_t >= min_p) cut (shortest prefix), renormalised kept probabilities;
//     Gumbel-max token in fp32 with Philox noise keyed by (seed, row,
//     position, token), or the first candidate for greedy rows.
//  3. verification positions: accept the draft d iff p(d) > 0 and
//     fp32(u q(d)) <= p(d); on rejection draw from norm(max(0, p - q)) over
//     the kept set (truncated rows) or queue a pass over the vocabulary
//     (untruncated rows).  The last position of a row to finish walks the
//     row: accepted prefix, then the resampled or bonus token.
// The position's global reads are issued together at its start (row lookup
// by a 32-way search in one warp while the other warps fetch the lists), so
// a position costs a few memory round trips and a handful of barriers.
#pragma once

#include "ss_common.cuh"

namespace ss {

namespace {

constexpr int kNT2 = 128;  // threads of a stage-2 CTA (one per candidate)

struct S2Smem {
  SelectSmem sel;
  unsigned long long top[kK];  // the selected candidates (unordered)
  unsigned long long srt[kK];  // the same, ordered
  double w[kK];                // exp(l_t - l_0) of the ordered candidates (stochastic rows)
  float w32[kK];               // the same in fp32 (stochastic sample / bonus positions)
  float g[kK];                 // their Gumbel noise: sample (purpose 0) or residual (purpose 2)
  float qv[kK];                // their draft probability q (truncated draft positions)
  float u_acc;                 // the acceptance uniform (draft positions)
  unsigned long long slots[kNT / 32];
  double lse;
  int r, j, gamma, c0, cnt, out_cnt, last, token, accept, d;
  float qd;
  uint32_t status;
};

// Merges (m2, s2) into the running (max, sum exp(x - max)) pair (m, s);
// pairs with m = -inf add nothing.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  if (!(m2 > -INFINITY)) return;
  if (!(m > -INFINITY)) {
    m = m2;
    s = s2;
    return;
  }
  const float mx = fmaxf(m, m2);
  s = s * expf(m - mx) + s2 * expf(m2 - mx);
  m = mx;
}

// Processed logit of one token at one position (the same fp32 steps as the
// stage-1 prelude), for a draft token outside the candidate list.  One warp.
__device__ float prelude_single_warp(const Params& P, const RowCtx& rc, int pos, int r, int c0, int jn, int tok,
                                     int lane) {
  float x = load_scalar(P.logits, P.logits_bf16, (int64_t)pos * P.ld + tok);
  int cnt = 0;
  if ((rc.flags & SS_PENALTY) && P.history) {
    const int32_t* hrow = P.history + (size_t)r * P.hist_stride;
    for (int h = lane; h < rc.hist_len; h += 32) cnt += (__ldg(hrow + h) == tok) ? 1 : 0;
    if (P.cu_draft)
      for (int s = lane; s < jn; s += 32) cnt += (__ldg(P.draft_ids + c0 + s) == tok) ? 1 : 0;
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, d);
  if ((rc.flags & SS_MASK) && P.bitmask) {
    const uint32_t w = __ldg(P.bitmask + (size_t)pos * P.mask_words + (tok >> 5));
    if (((w >> (tok & 31)) & 1u) == 0u) x = -INFINITY;
  }
  const ss_bias_entry* brow = (rc.flags & SS_BIAS) && P.bias ? P.bias + (size_t)r * P.bias_stride : nullptr;
  x = apply_penalty_bias(x, (uint32_t)cnt, brow != nullptr, tok, rc, brow);
  x = apply_temperature(x, rc);
  if (x != x) x = -INFINITY;
  return x;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
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


// One target position's stage 2: merge of its segment lists, epilogue,
// sample or accept test, outputs and (the last position of a row) the row
// walk.  Called by all NT >= 128 threads of a CTA (the candidate-parallel
// steps use the first 128); cand / tmp hold P.seg_cap lists each.  The
// segment lists and metadata may have been written by other CTAs of the
// same launch (the fused form): they are read through L2.
template <int NT>
__device__ __forceinline__ void stage2_position(const Params& P, int verify, int pos, const Split& sp,
                                                unsigned long long* cand, unsigned long long* tmp, S2Smem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V, Z = P.Z;
  const int need = min(kK, V);
  // ---- the position's reads: row lookup (warp 0) beside the lists (all);
  // every read of the previous position's shared state ended at its last barrier
  if (tid == 0) {
    sm.cnt = 0;
    sm.out_cnt = 0;
    sm.status = 0u;
    sm.last = 0;
    sm.token = -1;
    sm.accept = 0;
    sm.lse = 0.0;
  }
  const int nseg = seg_cta(sp, (long long)pos * Z + Z - 1, Z) - seg_cta(sp, (long long)pos * Z, Z) + 1;
  const size_t tbase = (size_t)pos * Z;
  if (warp == 0) {
    int r = pos, c0 = 0, c1 = 0;
    if (P.cu_draft) {
      r = warp_find_row(P.cu_draft, P.B, pos, lane);
      c0 = __ldg(P.cu_draft + r);
      c1 = __ldg(P.cu_draft + r + 1);
    }
    if (lane == 0) {
      const int j = P.cu_draft ? pos - c0 - r : 0;
      const int gamma = P.cu_draft ? c1 - c0 : 0;
      sm.r = r;
      sm.c0 = c0;
      sm.j = j;
      sm.gamma = gamma;
      // a draft position's token and q(d), fetched beside the lists
      int32_t d = -1;
      float qd = 0.0f;
      if (verify && j < gamma) {
        d = __ldg(P.draft_ids + c0 + j);
        if (d >= 0 && d < V) qd = P.q ? load_scalar(P.q, P.q_bf16, ((int64_t)c0 + j) * P.ld_q + d) : 1.0f;
      }
      sm.d = d;
      sm.qd = qd;
    }
  }
  uint32_t tst = 0u;
  for (int t = tid; t < nseg; t += NT) tst |= __ldcg(P.ws.tile_status + tbase + t);
  // the host sizes seg_cap so that no position has more lists; should that
  // bound ever fail, the position is reported as invalid rather than merged
  const bool fits = nseg <= P.seg_cap;
  const unsigned long long* stg = P.ws.staging + tbase * kK;
  if (fits)
    for (int i = tid; i < nseg * kK; i += NT) tmp[i] = __ldcg(stg + i);
  __syncthreads();
  if (tst) atomicOr(&sm.status, tst);
  const int r = sm.r, j = sm.j, gamma = sm.gamma, c0 = sm.c0;
  RowCtx rc = make_row(P.rows[r], P.hist_stride, P.bias_stride);
  if (!fits) {
    rc.valid = false;
    if (tid == 0) atomicAdd(P.ws.diag + 1, 1u);
  }
  const uint32_t position = rc.position + (uint32_t)j;
  const uint64_t seed = P.seeds[r];
  const bool is_draft = verify && j >= 0 && j < gamma;
  int32_t* cid = P.out.cand_ids ? P.out.cand_ids + (size_t)pos * kK : nullptr;
  float* cpr = P.out.cand_probs ? P.out.cand_probs + (size_t)pos * kK : nullptr;

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
    // ---- 1. merge the segments' candidates
    if (nseg == 1) {
      // one segment: its list is the position's top-min(128, V) already
      if (tid < kK) sm.top[tid] = tid < need ? tmp[tid] : 0ull;
    } else {
      unsigned long long tm = 0ull;
      for (int t = warp; t < nseg; t += NT / 32) {
        unsigned long long mn = ~0ull;
#pragma unroll
        for (int q = 0; q < kK / 32; ++q) {
          const unsigned long long c = tmp[t * kK + q * 32 + lane];
          mn = c < mn ? c : mn;  // an empty slot (0) makes the list certify nothing
        }
        mn = warp_min_u64(mn);
        tm = mn > tm ? mn : tm;
      }
      const unsigned long long tau2 = block_max_u64<NT>(tm, sm.slots);
      unsigned long long lmin = ~0ull, lmax = 0ull;
      for (int i = tid; i < nseg * kK; i += NT) {
        const unsigned long long c = tmp[i];
        if (c != 0ull && c >= tau2) {
          cand[atomicAdd(&sm.cnt, 1)] = c;
          lmin = c < lmin ? c : lmin;
          lmax = c > lmax ? c : lmax;
        }
      }
      const unsigned long long lo = block_min_u64<NT>(lmin, sm.slots);
      const unsigned long long hi = block_max_u64<NT>(lmax, sm.slots);
      const int n = sm.cnt;
      block_select<NT>(cand, tmp, n, need, lo, hi, sm.sel, [&](unsigned long long c) {
        const int s = atomicAdd(&sm.out_cnt, 1);
        if (s < kK) sm.top[s] = c;
      });
      // slots the select did not fill (only if its count invariant broke) stay empty
      if (tid < kK && tid >= min(sm.out_cnt, need)) sm.top[tid] = 0ull;
    }
    __syncthreads();
    // order: a candidate's place is the number of candidates above it
    // (distinct values; empty slots (0) rank below every candidate).  What a
    // candidate needs that does not depend on its place is computed first,
    // so that its latency overlaps the ordering: its softmax weight
    // w_t = exp(l_t - l_0) against the largest logit l_0 (each warp finds
    // it; fp64 for a draft position, fp32 for a sample / bonus position), its Gumbel noise (one Philox draw: the sample of a sampled / bonus
    // position, or the truncated residual's of a draft) and, for a truncated
    // draft position, its q.  Weights are unused for point masses.
    const unsigned long long v = tid < kK ? sm.top[tid] : 0ull;
    unsigned long long vmax = 0ull;
#pragma unroll
    for (int q = 0; q < kK / 32; ++q) {
      const unsigned long long c = sm.top[q * 32 + lane];
      vmax = c > vmax ? c : vmax;
    }
    vmax = warp_max_u64(vmax);
    const float lz = key2f(pk_key(vmax));
    const bool real = v != 0ull;
    double wv = 0.0;
    float wf = 0.0f, gv = 0.0f, qvv = 0.0f;
    if (real) {
      const float lt = key2f(pk_key(v));
      const int32_t tk = pk_tok(v);
      if (rc.stoch && lt > -INFINITY && lz < INFINITY) {
        // fp64 for a draft position (its accept test and residual); a
        // sample / bonus position takes fp32 and computes fp64 weights only
        // in the rare fallback below (fp64 is the GPU's slowest pipe)
        if (is_draft) wv = exp((double)lt - (double)lz);
        else wf = expf(__fsub_rn(lt, lz));
      }
      if (rc.stoch && (!is_draft || rc.trunc))
        gv = gumbel_of(philox_uniform(seed, (uint32_t)tk, position, (uint32_t)r, is_draft ? 2u : 0u));
      if (is_draft && rc.stoch && rc.trunc)
        qvv = P.q ? load_scalar(P.q, P.q_bf16, ((int64_t)c0 + j) * P.ld_q + tk) : (tk == sm.d ? 1.0f : 0.0f);
    }
    const int nz = __syncthreads_count(real);
    if (real) {
      int rank = 0;
#pragma unroll 8
      for (int u = 0; u < kK; ++u) rank += sm.top[u] > v ? 1 : 0;
      sm.srt[rank] = v;
      sm.w[rank] = wv;
      sm.w32[rank] = wf;
      sm.g[rank] = gv;
      sm.qv[rank] = qvv;
    }
    if (tid < kK && tid >= nz) {
      sm.srt[tid] = 0ull;
      sm.w[tid] = 0.0;
      sm.w32[tid] = 0.0f;
    }
    if (tid == 0 && is_draft && rc.stoch) sm.u_acc = philox_uniform(seed, 0u, position, (uint32_t)r, 1u);
    __syncthreads();

    if (warp == 0) {
      // ---- 2. epilogue: lane L holds the ordered candidates 4L .. 4L + 3
      unsigned long long cv[4];
      bool real[4], fin[4];
      int32_t tok[4];
      float l[4];
      int nfin = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = 4 * lane + k;
        cv[k] = sm.srt[t];
        real[k] = t < need && cv[k] != 0ull;
        tok[k] = pk_tok(cv[k]);
        l[k] = real[k] ? key2f(pk_key(cv[k])) : -INFINITY;
        fin[k] = real[k] && l[k] > -INFINITY;
        nfin += fin[k] ? 1 : 0;
      }
      const float l0 = key2f(pk_key(sm.srt[0]));
      const int32_t tok0 = pk_tok(sm.srt[0]);
      const int n_f = warp_sum_i(nfin);
      const bool no_finite = n_f == 0;
      const bool pos_inf = !no_finite && l0 == INFINITY;
      const bool point = no_finite || pos_inf || !rc.stoch;
      int nk = 0;
      double w[4] = {0.0, 0.0, 0.0, 0.0};
      double zk = 1.0;
      float wf[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      float izkf = 1.0f;
      bool f32 = false;  // the kept set and probabilities came from the fp32 weights
      if (no_finite) {
        nk = 0;
      } else if (point) {
        nk = 1;
      } else {
        int n2 = min(need, n_f);
        if ((rc.flags & SS_TOPK) && rc.top_k > 0) n2 = min(n2, rc.top_k);
        if (!is_draft) {
          // A sample / bonus position takes its cut points from the fp32
          // weights when they are certain: w32 is within (|l_t - l_0| 2^-24 +
          // 2 ulp) of w relative, so the sums and prefixes are within 1.5e-5
          // Z of the fp64 ones; a top-p prefix or a min-p weight closer than
          // the stated margin to its limit sends the position to the fp64
          // path below, which the oracle's fp64 decisions then match.
          float lsf = 0.0f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            wf[k] = sm.w32[4 * lane + k];
            lsf += wf[k];
          }
          const float Zf = warp_sum_f(lsf);
          int m2 = n2;
          bool unsure = false;
          if ((rc.flags & SS_TOPP) && rc.top_p < 1.0f) {
            float e[4], run = 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              e[k] = run;
              run += (4 * lane + k < need) ? wf[k] : 0.0f;
            }
            float incl = run;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
              const float o = __shfl_up_sync(0xffffffffu, incl, d);
              if (lane >= d) incl += o;
            }
            const float base = incl - run;
            const float lim = rc.top_p * Zf;
            const float tol = 2e-5f * Zf;
            int c = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if (4 * lane + k < need) {
                const float pre = base + e[k];
                c += pre < lim ? 1 : 0;
                unsure |= fabsf(pre - lim) <= tol;
              }
            }
            m2 = min(m2, warp_sum_i(c));
          }
          if ((rc.flags & SS_MINP) && rc.min_p > 0.0f) {
            int c = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if (4 * lane + k < need) {
                c += wf[k] >= rc.min_p ? 1 : 0;
                unsure |= fabsf(wf[k] - rc.min_p) <= 2e-5f * fmaxf(wf[k], rc.min_p) + 1e-37f;
              }
            }
            m2 = min(m2, warp_sum_i(c));
          }
          if (__any_sync(0xffffffffu, unsure)) {
            if (lane == 0) atomicAdd(P.ws.diag + 5, 1u);
          } else {
            nk = max(1, m2);
            float kz = 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) kz += (4 * lane + k < nk) ? wf[k] : 0.0f;
            izkf = 1.0f / warp_sum_f(kz);
            f32 = true;
          }
        }
        if (!f32) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            w[k] = is_draft ? sm.w[4 * lane + k] : (fin[k] ? exp((double)l[k] - (double)l0) : 0.0);
          double ls = 0.0;
#pragma unroll
          for (int k = 0; k < 4; ++k) ls += w[k];
          const double Zall = warp_sum_d(ls);
          if ((rc.flags & SS_TOPP) && rc.top_p < 1.0f) {
            // t is kept iff the mass before it, sum_{u<t} w_u / Z, is below top_p:
            // the exclusive prefix of w in candidate order against top_p * Z
            double e[4], run = 0.0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              e[k] = run;
              run += (4 * lane + k < need) ? w[k] : 0.0;
            }
            double incl = run;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
              const double o = __shfl_up_sync(0xffffffffu, incl, d);
              if (lane >= d) incl += o;
            }
            const double base = incl - run;
            const double lim = (double)rc.top_p * Zall;
            int c = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) c += (4 * lane + k < need && base + e[k] < lim) ? 1 : 0;
            n2 = min(n2, warp_sum_i(c));
          }
          if ((rc.flags & SS_MINP) && rc.min_p > 0.0f) {
            // l_t - l_0 >= ln(min_p)  <=>  w_t = exp(l_t - l_0) >= min_p
            int c = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) c += (4 * lane + k < need && w[k] >= (double)rc.min_p) ? 1 : 0;
            n2 = min(n2, warp_sum_i(c));
          }
          nk = max(1, n2);
          double kz = 0.0;
#pragma unroll
          for (int k = 0; k < 4; ++k) kz += (4 * lane + k < nk) ? w[k] : 0.0;
          zk = warp_sum_d(kz);
        }
      }
      const double izk = (f32 || point || no_finite) ? 1.0 : 1.0 / zk;
      // candidate outputs
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = 4 * lane + k;
        if (cid) cid[t] = real[k] ? tok[k] : -1;
        if (cpr) {
          float pr = 0.0f;
          if (t < nk) pr = point ? (t == 0 ? 1.0f : 0.0f) : (f32 ? wf[k] * izkf : (float)(w[k] * izk));
          cpr[t] = pr;
        }
      }
      uint32_t st = 0u;
      if (no_finite) st |= SS_ST_NO_FINITE;
      else if (pos_inf) st |= SS_ST_POS_INF;
      // SS_EXACT on a plan without exact sampling: sampled from the candidates
      if (rc.exact && !P.exact_on && !is_draft && !point) st |= SS_ST_NOT_EXACT;

      // ---- 3. token of this position (sample / bonus)
      int32_t token = -1;
      int accept = 0;
      double lse = 0.0;
      if (!is_draft) {
        if (no_finite) {
          token = -1;
        } else if (point) {
          token = tok0;
        } else if (rc.exact && P.exact_on) {
          // exact sampling: the Gumbel-max over the whole vocabulary, the
          // largest of the segments' maxima (stage 1)
          unsigned long long gb = 0ull;
          for (int t = lane; t < nseg; t += 32) {
            const unsigned long long v = __ldcg(P.ws.tile_gmax + tbase + t);
            gb = v > gb ? v : gb;
          }
          gb = warp_max_u64(gb);
          token = gb ? pk_tok(gb) : tok0;
        } else {
          unsigned long long sc = 0ull;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (4 * lane + k < nk) {
              const float g = sm.g[4 * lane + k];
              const unsigned long long s = pack(f2key(__fadd_rn(l[k], g)), (uint32_t)tok[k]);
              sc = s > sc ? s : sc;
            }
          }
          token = pk_tok(warp_max_u64(sc));
        }
      } else {
        // ---- 4. verification of draft j
        const int32_t d = sm.d;
        const bool d_ok = d >= 0 && d < V;
        if (!d_ok) st |= SS_ST_BAD_DRAFT;
        if (no_finite) {
          accept = 0;
          token = -1;
        } else if (point) {
          accept = (d_ok && d == tok0) ? 1 : 0;
          token = tok0;
        } else {
          double pd = 0.0;
          if (rc.trunc) {
            double mine = 0.0;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (4 * lane + k < nk && tok[k] == d) mine = w[k] * izk;
#pragma unroll
            for (int dd = 16; dd > 0; dd >>= 1) mine = fmax(mine, __shfl_xor_sync(0xffffffffu, mine, dd));
            pd = mine;
          } else {
            // full-vocabulary softmax: LSE from the segments' (max, sum exp)
            // partials, lane-parallel in fp32 (the partials are fp32 sums;
            // this acceptance test is held to 1e-5 relative)
            float M = -INFINITY, S = 0.0f;
            for (int tt = lane; tt < nseg; tt += 32) {
              const float2 ms = __ldcg(P.ws.tile_lse + tbase + tt);
              lse_merge(M, S, ms.x, ms.y);
            }
#pragma unroll
            for (int dd = 16; dd > 0; dd >>= 1) {
              const float M2 = __shfl_xor_sync(0xffffffffu, M, dd);
              const float S2 = __shfl_xor_sync(0xffffffffu, S, dd);
              lse_merge(M, S, M2, S2);
            }
            lse = (double)(M + logf(S));
            // d among the candidates: its logit; else recompute it
            bool found = false;
            float dl = 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (real[k] && tok[k] == d) {
                found = true;
                dl = l[k];
              }
            const uint32_t fb = __ballot_sync(0xffffffffu, found);
            if (fb) {
              dl = __shfl_sync(0xffffffffu, dl, __ffs((int)fb) - 1);
            } else if (d_ok) {
              dl = prelude_single_warp(P, rc, pos, r, c0, min(j, gamma), d, lane);
            }
            if (d_ok) pd = (double)expf(dl - (float)lse);
          }
          if (d_ok) {
            const float u = sm.u_acc;
            const float prod = __fmul_rn(u, sm.qd);
            accept = (pd > 0.0 && (double)prod <= pd) ? 1 : 0;
          }
          if (!accept) {
            if (rc.trunc) {
              // residual norm(max(0, p - q)) over the kept candidates
              double rr[4];
              bool pos_any = false;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                rr[k] = 0.0;
                if (4 * lane + k < nk)
                  rr[k] = fmax(0.0, w[k] * izk - (double)sm.qv[4 * lane + k]);
                pos_any |= (4 * lane + k < nk && rr[k] > 0.0);
              }
              const bool anypos = __any_sync(0xffffffffu, pos_any);
              unsigned long long sc = 0ull;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                if (4 * lane + k < nk) {
                  const float g = sm.g[4 * lane + k];
                  unsigned long long s = 0ull;
                  if (anypos) {
                    if (rr[k] > 0.0) s = pack(f2key(__fadd_rn(logf((float)rr[k]), g)), (uint32_t)tok[k]);
                  } else {
                    s = pack(f2key(__fadd_rn(l[k], g)), (uint32_t)tok[k]);
                  }
                  sc = s > sc ? s : sc;
                }
              }
              token = pk_tok(warp_max_u64(sc));
              if (!anypos) st |= SS_ST_RESID_EMPTY;
            } else {
              token = kPending;  // drawn by the pass over the vocabulary
            }
          }
        }
      }
      if (lane == 0) {
        if (P.out.num_kept) P.out.num_kept[pos] = nk;
        if (st) atomicOr(&sm.status, st);
        sm.token = token;
        sm.accept = accept;
        sm.lse = lse;
      }
    }
  }
  __syncthreads();
  const uint32_t status = sm.status;
  const int32_t token = rc.valid ? sm.token : -1;
  const int accept = rc.valid ? sm.accept : 0;
  const double lse = sm.lse;

  // ---- 5. outputs
  if (!verify) {
    if (tid == 0) {
      P.out.tokens[r] = token;
      P.out.row_status[r] = status;
    }
  } else if (warp == 0 && c0 + gamma + r < P.max_positions) {
    // (a row whose positions reach past max_positions is reported below)
    if (lane == 0) {
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
    __syncwarp();
    if (sm.last) {
      // the row's last position: walk the drafts (one warp; positions read in parallel)
      __threadfence();
      const int pos0 = c0 + r;
      int32_t* tk = P.out.tokens + (size_t)r * P.out.tokens_stride;
      const int stride = P.out.tokens_stride;
      uint32_t st = 0u;
      int n_acc = 0;
      if (!rc.valid) {
        for (int s = lane; s < stride; s += 32) tk[s] = -1;
        st = SS_ST_BAD_PARAM;
      } else {
        int stop = gamma;
        for (int s0 = 0; s0 < gamma && stop == gamma; s0 += 32) {
          const int s = s0 + lane;
          PosResult q;
          q.status = 0u;
          q.accept = 1;
          if (s < gamma) q = load_pos_result(P.ws.pos + pos0 + s);
          const uint32_t rej = __ballot_sync(0xffffffffu, s < gamma && !q.accept);
          const int first = rej ? s0 + __ffs((int)rej) - 1 : gamma;
          // statuses of the drafts up to and including the first rejection
          uint32_t sv = (s < gamma && s <= first) ? q.status : 0u;
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) sv |= __shfl_xor_sync(0xffffffffu, sv, d);
          st |= sv;
          stop = first;
        }
        for (int s = lane; s < stop && s < stride; s += 32) tk[s] = __ldg(P.draft_ids + c0 + s);
        const PosResult fin = load_pos_result(P.ws.pos + pos0 + stop);
        if (stop == gamma) st |= fin.status;
        if (lane == 0) {
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
        }
        for (int s = stop + 1 + lane; s < stride; s += 32) tk[s] = -1;
        n_acc = stop;
      }
      if (lane == 0) {
        if (P.out.num_accepted) P.out.num_accepted[r] = n_acc;
        P.out.row_status[r] = st;
        P.ws.row_count[r] = 0u;
      }
    }
  }
  __syncthreads();
}

// A verification batch with more target positions than the plan holds: the
// positions past max_positions were not evaluated, and a row reaching past
// it was neither counted nor walked, so it is reported here (CTA `cta` of
// `ncta`, NT threads each).
template <int NT>
__device__ __forceinline__ void stage2_capacity_rows(const Params& P, int verify, int cta, int ncta) {
  if (verify && __ldg(P.cu_draft + P.B) + P.B > P.max_positions) {
    for (int r = cta * NT + (int)threadIdx.x; r < P.B; r += ncta * NT) {
      if (__ldg(P.cu_draft + r + 1) + r < P.max_positions) continue;
      int32_t* tk = P.out.tokens + (size_t)r * P.out.tokens_stride;
      for (int s = 0; s < P.out.tokens_stride; ++s) tk[s] = -1;
      if (P.out.num_accepted) P.out.num_accepted[r] = 0;
      P.out.row_status[r] = SS_ST_CAPACITY;
    }
  }
}

// Shared memory of stage2_position for `lists` segment lists per position.
__host__ __device__ constexpr size_t stage2_smem_for(int lists) { return (size_t)lists * kK * 8 * 2 + sizeof(S2Smem); }

}  // namespace

}  // namespace ss
