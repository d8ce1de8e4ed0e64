// Residual resampling over the whole vocabulary for untruncated stochastic
// rows (SonicSampler 3.1 "Speculative verification": on rejection sample from
// p~(x) proportional to max{0, p(x) - q(x)}; dl-note "Rejection Sampler").
//
// The row walk of stage 2 queues (row, rejected draft index, target position)
// entries.  This kernel has a fixed launch shape (persistent CTAs) and loops
// over (entry, piece) items: each piece recomputes the processed
// logits with the stage-1 prelude, p_i = exp(l_i - LSE) with the LSE stage 2
// assembled from the tiles' (max, sum exp) partials, r_i = p_i - q_i, and the
// Gumbel-max score ln r_i + g_i (Philox purpose 2) over r_i > 0.  Pieces
// combine by a 64-bit atomicMax of (key(score) << 32 | ~token); the last piece
// of an entry writes the token.  If no r_i is positive, the last piece draws
// from p itself (Gumbel-max of l_i + g_i over the vocabulary, by B_N tiles).
#include "ss_common.cuh"

namespace ss {

namespace {

constexpr int kGroups = 2;                // groups of 4 tokens per thread in a work item (4: slower, spills)
constexpr int kSub = 4 * kGroups * kNT;  // tokens per work item

struct S3Smem {
  unsigned long long slots[kNT / 32];
  int last;
  int pad;
};

// Word w (0..3) of a Philox block, by selects (an index into a local array
// would go through local memory).  Groups start at multiples of 4 tokens, so
// token i0 + k of a group takes word k of block i0 / 4.
__device__ __forceinline__ uint32_t word_of4(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, int w) {
  return w == 0 ? c0 : (w == 1 ? c1 : (w == 2 ? c2 : c3));
}

// Processed logits of 4 consecutive tokens i0..i0+3 of one position (the
// fp32 steps of the stage-1 prelude); counts come from the tile's aux table.
__device__ __forceinline__ void prelude4(const Params& P, const RowCtx& rc, int pos, int i0, int n_valid,
                                         const uint16_t* aux, int t0, const ss_bias_entry* brow,
                                         bool aux_on, float out[4]) {
  uint32_t mw = 0xFFFFFFFFu;
  if ((rc.flags & SS_MASK) && P.bitmask) mw = __ldg(P.bitmask + (size_t)pos * P.mask_words + (i0 >> 5));
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = i0 + k;
    if (k >= n_valid) {
      out[k] = -INFINITY;
      continue;
    }
    float x = load_scalar(P.logits, P.logits_bf16, (int64_t)pos * P.ld + i);
    if ((rc.flags & SS_MASK) && P.bitmask && ((mw >> (i & 31)) & 1u) == 0u) x = -INFINITY;
    if (aux_on) {
      const uint32_t a = aux[i - t0];
      if (a != 0u) x = apply_penalty_bias(x, a & 0x7FFFu, (a & 0x8000u) != 0u, i, rc, brow);
    }
    x = apply_temperature(x, rc);
    if (x != x) x = -INFINITY;
    out[k] = x;
  }
}

// Four consecutive values i0..i0+3 of a row (fp32 or bf16 bits widened),
// n_valid of them real (the rest 0): one 16- or 8-byte load when all four
// are (rows are 16-byte aligned and i0 is a multiple of 4), else scalar.
__device__ __forceinline__ void load4(const void* base, int bf16, int64_t row_off, int i0, int n_valid, float v[4]) {
  if (n_valid >= 4) {
    if (bf16) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(base) + row_off + i0));
      v[0] = bf16_lo(u.x);
      v[1] = bf16_hi(u.x);
      v[2] = bf16_lo(u.y);
      v[3] = bf16_hi(u.y);
    } else {
      const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + row_off + i0));
      v[0] = f.x;
      v[1] = f.y;
      v[2] = f.z;
      v[3] = f.w;
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = k < n_valid ? load_scalar(base, bf16, row_off + i0 + k) : 0.0f;
}

// prelude4 on loaded logits x (mask word mw of the group's tokens).
__device__ __forceinline__ void prelude_loaded(const RowCtx& rc, int i0, int n_valid, uint32_t mw, bool masked,
                                               const uint16_t* aux, int t0, const ss_bias_entry* brow, bool aux_on,
                                               float x[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = i0 + k;
    if (k >= n_valid) {
      x[k] = -INFINITY;
      continue;
    }
    float v = x[k];
    if (masked && ((mw >> (i & 31)) & 1u) == 0u) v = -INFINITY;
    if (aux_on) {
      const uint32_t a = aux[i - t0];
      if (a != 0u) v = apply_penalty_bias(v, a & 0x7FFFu, (a & 0x8000u) != 0u, i, rc, brow);
    }
    v = apply_temperature(v, rc);
    if (v != v) v = -INFINITY;
    x[k] = v;
  }
}

// Fill the tile's aux table (history counts incl. drafts before j, bias flags).
__device__ void build_aux(const Params& P, const RowCtx& rc, int r, int j, int t0, int nt, uint16_t* aux,
                          bool pen_on, bool bias_on, const ss_bias_entry* brow) {
  const int tid = threadIdx.x;
  uint32_t* a32 = reinterpret_cast<uint32_t*>(aux);
  for (int w = tid; w < (nt + 1) / 2; w += kNT) a32[w] = 0u;
  __syncthreads();
  if (pen_on) {
    const int32_t* hrow = P.history + (size_t)r * P.hist_stride;
    for (int h = tid; h < rc.hist_len; h += kNT) {
      const int id = __ldg(hrow + h);
      if (id >= t0 && id < t0 + nt) atomicAdd(a32 + ((id - t0) >> 1), 1u << (16 * ((id - t0) & 1)));
    }
    const int base = __ldg(P.cu_draft + r);
    const int jn = min(j, __ldg(P.cu_draft + r + 1) - base);
    for (int s = tid; s < jn; s += kNT) {
      const int id = __ldg(P.draft_ids + base + s);
      if (id >= t0 && id < t0 + nt) atomicAdd(a32 + ((id - t0) >> 1), 1u << (16 * ((id - t0) & 1)));
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

}  // namespace

__global__ void __launch_bounds__(kNT, 4) residual_kernel(const Params P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint16_t* aux = reinterpret_cast<uint16_t*>(smem_raw);
  S3Smem& sm = *reinterpret_cast<S3Smem*>(smem_raw + (size_t)P.BN * 2);
  const int tid = threadIdx.x;
  const int Z = P.Z, V = P.V;
  const int count = (int)__ldcg(P.ws.resid_count);
  // items are (entry, piece): an entry's pieces run on many CTAs, so a
  // handful of rejections still spreads over the whole GPU.  A piece is a
  // multiple of kSub tokens (at most B_N, the aux table), as few as spread
  // the entries over the grid in one round: pieces of kSub when the entries
  // are few, longer ones (streamed kSub at a time, one prelude, reduction
  // and arrival per piece) when more entries would need several rounds.
  int psz = kSub;
  if (count > 0) {
    const int want = max(1, (int)gridDim.x / count);  // pieces per entry for one round
    psz = (((V + want - 1) / want) + kSub - 1) / kSub * kSub;
    psz = max(kSub, min(psz, P.BN / kSub * kSub));
  }
  const int nsub = (V + psz - 1) / psz;
  const long long total = (long long)count * nsub;
  for (long long item = blockIdx.x; item < total; item += gridDim.x) {
    const int e = (int)(item / nsub);
    const int piece = (int)(item - (long long)e * nsub);
    ResidEntry* ent = P.ws.resid + e;
    const int r = __ldcg(&ent->row), j = __ldcg(&ent->j), pos = __ldcg(&ent->pos);
    const RowCtx rc = make_row(P.rows[r], P.hist_stride, P.bias_stride);
    const uint32_t position = rc.position + (uint32_t)j;
    const uint64_t seed = P.seeds[r];
    const float lse = (float)__ldcg(&P.ws.pos[pos].lse);
    const int64_t qrow = (int64_t)__ldg(P.cu_draft + r) + j;
    const int32_t dtok = P.q ? -1 : __ldg(P.draft_ids + qrow);  // one-hot drafts: q = [i == dtok]
    const bool pen_on = (rc.flags & SS_PENALTY) && P.history != nullptr;
    const bool bias_on = (rc.flags & SS_BIAS) && P.bias != nullptr;
    const bool aux_on = pen_on || bias_on;
    const ss_bias_entry* brow = bias_on ? P.bias + (size_t)r * P.bias_stride : nullptr;
    const int t0 = piece * psz;
    const int nt = min(psz, V - t0);
    if (tid == 0) sm.last = 0;
    if (aux_on) build_aux(P, rc, r, j, t0, nt, aux, pen_on, bias_on, brow);
    else __syncthreads();

    unsigned long long best = 0ull;
    const bool masked = (rc.flags & SS_MASK) && P.bitmask;
#pragma unroll 1
    for (int s0 = t0; s0 < t0 + nt; s0 += kSub) {
      // the thread's kGroups groups of four tokens of this kSub-token part:
      // every load of every group goes out before the first value is used
      float xg[kGroups][4], qg[kGroups][4];
      uint32_t mw[kGroups];
      int ig[kGroups], nv[kGroups];
#pragma unroll
      for (int gi = 0; gi < kGroups; ++gi) {
        ig[gi] = s0 + 4 * tid + gi * 4 * kNT;
        nv[gi] = min(4, t0 + nt - ig[gi]);
        mw[gi] = 0xFFFFFFFFu;
        if (nv[gi] > 0) {
          load4(P.logits, P.logits_bf16, (int64_t)pos * P.ld, ig[gi], nv[gi], xg[gi]);
          if (P.q) load4(P.q, P.q_bf16, qrow * P.ld_q, ig[gi], nv[gi], qg[gi]);
          if (masked) mw[gi] = __ldg(P.bitmask + (size_t)pos * P.mask_words + (ig[gi] >> 5));
        }
      }
#pragma unroll
      for (int gi = 0; gi < kGroups; ++gi) {
        if (nv[gi] <= 0) continue;
        const int i0 = ig[gi];
        float* x = xg[gi];
        prelude_loaded(rc, i0, nv[gi], mw[gi], masked, aux, t0, brow, aux_on, x);
        float rr[4];
        bool any = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          rr[k] = -1.0f;
          if (x[k] > -INFINITY && k < nv[gi]) {
            // q one-hot on the draft (drafts without probabilities): r_i = p_i
            // for every other token and 0 at the draft, so ln r_i is l_i - LSE
            // with no exp or log; rr only marks the support then
            if (P.q) rr[k] = expf(x[k] - lse) - qg[gi][k];
            else rr[k] = i0 + k == dtok ? 0.0f : 1.0f;
            any |= rr[k] > 0.0f;
          }
        }
        if (any) {
          uint32_t c0 = (uint32_t)i0 >> 2, c1 = position, c2 = (uint32_t)r, c3 = 2u;
          philox10(c0, c1, c2, c3, (uint32_t)seed, (uint32_t)(seed >> 32));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (rr[k] > 0.0f) {
              const float g = gumbel_of(word_to_uniform(word_of4(c0, c1, c2, c3, k)));
              const float lr = P.q ? logf(rr[k]) : __fsub_rn(x[k], lse);
              const unsigned long long sc = pack(f2key(__fadd_rn(lr, g)), (uint32_t)(i0 + k));
              best = sc > best ? sc : best;
            }
          }
        }
      }
    }
    best = block_max_u64(best, sm.slots);
    if (tid == 0) {
      if (best) atomicMax(&ent->best, best);
      __threadfence();
      const uint32_t old = atomicAdd(&ent->arrivals, 1u);
      sm.last = (old == (uint32_t)(nsub - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (sm.last) {
      __threadfence();
      const unsigned long long fin = atomicAdd(&ent->best, 0ull);
      int32_t token;
      uint32_t extra = 0u;
      if (fin != 0ull) {
        token = pk_tok(fin);
      } else {
        // no residual mass: Gumbel-max over l_i + g_i, i.e. a draw from p
        extra = SS_ST_RESID_EMPTY;
        unsigned long long fb = 0ull;
        for (int tt = 0; tt < Z; ++tt) {
          const int u0 = tt * P.BN;
          const int un = min(P.BN, V - u0);
          if (aux_on) build_aux(P, rc, r, j, u0, un, aux, pen_on, bias_on, brow);
          for (int i0 = u0 + 4 * tid; i0 < u0 + un; i0 += 4 * kNT) {
            float x[4];
            prelude4(P, rc, pos, i0, min(4, u0 + un - i0), aux, u0, brow, aux_on, x);
            uint32_t c0 = (uint32_t)i0 >> 2, c1 = position, c2 = (uint32_t)r, c3 = 2u;
            philox10(c0, c1, c2, c3, (uint32_t)seed, (uint32_t)(seed >> 32));
            
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if (x[k] > -INFINITY && i0 + k < u0 + un) {
                const float g = gumbel_of(word_to_uniform(word_of4(c0, c1, c2, c3, k)));
                const unsigned long long sc = pack(f2key(__fadd_rn(x[k], g)), (uint32_t)(i0 + k));
                fb = sc > fb ? sc : fb;
              }
            }
          }
          __syncthreads();
        }
        fb = block_max_u64(fb, sm.slots);
        token = fb ? pk_tok(fb) : -1;
      }
      if (tid == 0) {
        if (j < P.out.tokens_stride) P.out.tokens[(size_t)r * P.out.tokens_stride + j] = token;
        if (extra) P.out.row_status[r] |= extra;
        ent->best = 0ull;
        ent->arrivals = 0u;
        atomicAdd(P.ws.diag + 2, 1u);
      }
    }
    __syncthreads();
  }
  // the queue is consumed: the last CTA to finish (every CTA has read the
  // count by then) empties it for the next call
  if (tid == 0) {
    __threadfence();
    const uint32_t done = atomicAdd(P.ws.resid_count + 1, 1u);
    if (done == gridDim.x - 1u) {
      P.ws.resid_count[0] = 0u;
      P.ws.resid_count[1] = 0u;
    }
  }
}

size_t residual_smem_bytes(int BN) { return (size_t)BN * 2 + sizeof(S3Smem) + 16; }

int residual_piece_tokens() { return kSub; }

}  // namespace ss
