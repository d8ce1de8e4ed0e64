// CPU oracle for the fused LLM sampling / speculative-verification path.
//
// TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
// cpu_baseline / reference legs of bench.py may load or run this code.  It
// shares no code, header, table or helper with the CUDA path.
//
// Plain, slow, single-threaded C++.  Every step is the plain definition from
// the pages, in the pages' order; library primitives (std::sort, exp, log)
// serve as steps.  Floating point: the logits prelude is fp32 with one IEEE
// rounding per operation (built with -ffp-contract=off, no fast-math), because
// the selection keys are a function of the fp32 processed logits; probabilities
// and truncation cut points are fp64; the Gumbel argmax is fp32 (the precision
// the kernel takes that decision in).
//
// Sources (page title, section):
//  [SS]  "SonicSampler: unified tile-aware kernels for LLM sampling and
//        speculative verification" -- 3.1 Background (logits processing,
//        truncation, Gumbel-max sampling, speculative verification), 3.2
//        execution model, Fig. 1 (stage-1 prelude order; top-k with k = 128).
//  [DN]  "Decoding and sampling" (dl-note) -- Temperature, Top-k, Top-p, Min-p,
//        "Combination" (Temperature -> Softmax -> top-k/top-p/min-p ->
//        Renormalize -> Sample; top-k with top-p keeps the intersection),
//        "Rejection Sampler" (accept rule, residual norm(max(0, p - q)),
//        exactness of the resulting distribution).
//  [PX]  Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
//        1, 2, 3", SC'11 -- Philox-4x32 with 10 rounds.
//
// Readings where the pages are silent:
//  - penalty formulas (the paper's appendix C is missing): CTRL repetition
//    penalty x/rep for x > 0 else x*rep, then x - freq*count, then x - pres,
//    applied only to tokens with count > 0;
//  - temperature divides each logit by T ([DN] Temperature: z_i / T), one
//    IEEE fp32 division rounded to nearest; greedy rows skip temperature and
//    truncation;
//  - the order is (processed logit descending, token index ascending); NaN
//    after the prelude becomes -inf and sets a status bit; -0 == +0;
//  - bounded mode: the candidate universe is the first min(128, V) tokens of
//    that order; exact mode: all V;
//  - top-p keeps the smallest prefix whose cumulative probability reaches p
//    (t is kept iff the mass strictly before it is < p); min-p is evaluated in
//    logit space, l_t - l_0 >= ln(min_p); the kept set is the shortest of the
//    active prefixes (intersection), and at least one token;
//  - verification: rows that request any truncation use the kept
//    distribution as p; untruncated rows use the full-vocabulary softmax,
//    unless flagged bounded-p (then the candidate softmax); greedy rows
//    accept iff the draft equals the argmax.  Drafts without probabilities
//    are given to the oracle as a one-hot q row (q(d) = 1);
//  - rows flagged exact (untruncated, stochastic) sample by the Gumbel-max
//    over every finite token of the vocabulary instead of the candidates.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <numeric>
#include <vector>

namespace {

// Per-row flag bits ("compact bit-level indicators", [SS] 1).
constexpr uint32_t kGreedy = 1u << 0;
constexpr uint32_t kMask = 1u << 1;
constexpr uint32_t kPenalty = 1u << 2;
constexpr uint32_t kBias = 1u << 3;
constexpr uint32_t kTopK = 1u << 4;
constexpr uint32_t kTopP = 1u << 5;
constexpr uint32_t kMinP = 1u << 6;
constexpr uint32_t kBoundedP = 1u << 7;  // verify against the candidate distribution
constexpr uint32_t kExact = 1u << 8;     // sample over the whole vocabulary

// Per-row status bits.
constexpr uint32_t kStNan = 1u << 0;         // a processed logit was NaN -> -inf
constexpr uint32_t kStNoFinite = 1u << 1;    // every candidate is -inf -> token -1
constexpr uint32_t kStBadHist = 1u << 2;     // history id >= V ignored
constexpr uint32_t kStBadBias = 1u << 3;     // bias id >= V ignored
constexpr uint32_t kStBadParam = 1u << 4;    // invalid parameters -> no tokens
constexpr uint32_t kStBadDraft = 1u << 5;    // draft id outside [0, V) -> rejected
constexpr uint32_t kStPosInf = 1u << 6;      // +inf processed logit -> point mass
constexpr uint32_t kStResidEmpty = 1u << 7;  // residual had no mass -> sampled from p
constexpr uint32_t kStNotExact = 1u << 8;    // SS_EXACT without exact sampling -> candidates

constexpr int kK = 128;  // bounded candidate count ([SS] 1, 3.3)
constexpr float kNegInf = -std::numeric_limits<float>::infinity();
constexpr double kInfD = std::numeric_limits<double>::infinity();

enum Purpose : uint32_t { kPurposeSample = 0, kPurposeAccept = 1, kPurposeResidual = 2 };

}  // namespace

extern "C" {

struct sso_row {
  uint32_t flags;
  float temperature, top_p, min_p, rep, freq, pres;
  int32_t top_k, hist_len, n_bias;
  uint32_t position;
};

struct sso_problem {
  int32_t B, V;
  int32_t logits_bf16;        // 0: fp32 logits, 1: bf16 bit patterns
  int64_t ld_logits;          // row stride (elements)
  const void* logits;         // [B_pos, ld_logits]
  const sso_row* rows;        // [B]
  const int32_t* history;     // [B, hist_stride]
  int32_t hist_stride;
  const uint32_t* bitmask;    // [B_pos, ceil(V/32)] or null
  const int32_t* bias_tokens; // [B, bias_stride]
  const float* bias_values;   // [B, bias_stride]
  int32_t bias_stride;
  const uint64_t* seeds;      // [B]
  const int32_t* cu_draft;    // [B+1] (null: single-step sampling)
  const int32_t* draft_ids;   // [cu_draft[B]]
  int32_t q_bf16;
  int64_t ld_q;
  const void* draft_probs;    // [cu_draft[B], ld_q]
  const int32_t* row_ids;     // [B] batch row index used in the Philox counter, or null (= r)
  int32_t exact_on;           // SS_EXACT rows sample over the vocabulary (else: candidates + status)
};

struct sso_outputs {
  int32_t* tokens;          // [B, tokens_stride]
  int32_t tokens_stride;
  int32_t* num_accepted;    // [B] (verify) or null
  uint32_t* row_status;     // [B]
  int32_t* cand_ids;        // [B_pos, 128] or null
  float* cand_probs;        // [B_pos, 128] or null
  int32_t* num_kept;        // [B_pos] or null
  // diagnostics per position (may be null)
  double* margin_topp;      // min |cum_before(t) - top_p|
  double* margin_minp;      // min |(l_t - l_0) - ln(min_p)|
  double* margin_gumbel;    // relative gap of the two best perturbed scores
  double* margin_accept;    // |u*q(d) - p(d)| / p(d)
  double* margin_resid;     // relative gap of the two best residual scores
  double* mass_outside;     // 1 - (top-128 mass of the full-V softmax)
  double* p_draft;          // p_j(d_j) used by the accept test
  double* lse;              // full-V log-sum-exp of the processed logits
};

}  // extern "C"

namespace {

// ------------------------------------------------------------------ Philox [PX]
// Philox-4x32-10: each round multiplies counter words 0 and 2 by the two round
// constants, takes high and low halves, XORs the high halves with the other two
// counter words and the round key, and permutes; the key advances by the Weyl
// constants between rounds.
void philox4x32_10(uint32_t ctr[4], uint32_t k0, uint32_t k1) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  for (int round = 0; round < 10; ++round) {
    const uint64_t prod0 = (uint64_t)M0 * ctr[0];
    const uint64_t prod1 = (uint64_t)M1 * ctr[2];
    const uint32_t out0 = (uint32_t)(prod1 >> 32) ^ ctr[1] ^ k0;
    const uint32_t out1 = (uint32_t)prod1;
    const uint32_t out2 = (uint32_t)(prod0 >> 32) ^ ctr[3] ^ k1;
    const uint32_t out3 = (uint32_t)prod0;
    ctr[0] = out0; ctr[1] = out1; ctr[2] = out2; ctr[3] = out3;
    k0 += W0;
    k1 += W1;
  }
}

// Uniform in (0, 1): an odd multiple of 2^-24 built from the top 23 bits of
// word (i mod 4) of Philox at counter (floor(i/4), position, row, purpose).
float uniform01(uint64_t seed, uint32_t i, uint32_t position, uint32_t row, uint32_t purpose) {
  uint32_t c[4] = {i / 4u, position, row, purpose};
  philox4x32_10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
  const uint32_t w = c[i % 4u];
  return (float)((w >> 9) * 2u + 1u) * 0x1p-24f;
}

// Gumbel(0,1) noise in fp32: -ln(-ln u).
float gumbel(uint64_t seed, uint32_t i, uint32_t position, uint32_t row, uint32_t purpose) {
  const float u = uniform01(seed, i, position, row, purpose);
  const float e = -logf(u);
  return -logf(e);
}

float load_elem(const void* base, int bf16, int64_t off) {
  if (bf16) {
    const uint16_t h = static_cast<const uint16_t*>(base)[off];
    const uint32_t b = (uint32_t)h << 16;
    float f;
    std::memcpy(&f, &b, 4);
    return f;
  }
  return static_cast<const float*>(base)[off];
}

bool row_params_valid(const sso_row& rp, const sso_problem& P) {
  if (rp.hist_len < 0 || rp.hist_len > P.hist_stride) return false;
  if (rp.n_bias < 0 || rp.n_bias > P.bias_stride) return false;
  if (rp.flags & kPenalty) {
    if (!(std::isfinite(rp.rep) && rp.rep > 0.0f)) return false;
    if (!std::isfinite(rp.freq) || !std::isfinite(rp.pres)) return false;
  }
  if (rp.flags & kGreedy) return true;
  if (!(std::isfinite(rp.temperature) && rp.temperature > 0.0f)) return false;
  if ((rp.flags & kTopP) && !(rp.top_p > 0.0f && rp.top_p <= 1.0f)) return false;
  if ((rp.flags & kMinP) && !(rp.min_p >= 0.0f && rp.min_p <= 1.0f)) return false;
  if ((rp.flags & kTopK) && rp.top_k < 0) return false;
  return true;
}

// A stochastic row that asks for top-k, top-p or min-p.
bool row_cuts(const sso_row& rp) {
  if (rp.flags & kGreedy) return false;
  if ((rp.flags & kTopK) && rp.top_k > 0) return true;
  if ((rp.flags & kTopP) && rp.top_p < 1.0f) return true;
  if ((rp.flags & kMinP) && rp.min_p > 0.0f) return true;
  return false;
}

bool row_truncates(const sso_row& rp) {
  if (rp.flags & kGreedy) return false;
  if (row_cuts(rp)) return true;
  if (rp.flags & kBoundedP) return true;  // p = the kept (here: all finite) candidates
  return false;
}

// ------------------------------------------------------------ prelude ([SS] 3.1, Fig. 1)
// Processed logits of one target position.  `extra` are token ids appended to
// the row's history (the drafts accepted before this verify position).
std::vector<float> prelude(const sso_problem& P, int r, int64_t pos, const std::vector<int32_t>& extra,
                           uint32_t* status) {
  const sso_row& rp = P.rows[r];
  const int V = P.V;
  std::vector<float> x(V);
  for (int i = 0; i < V; ++i) x[i] = load_elem(P.logits, P.logits_bf16, pos * P.ld_logits + i);

  // 1. grammar mask: bit (i mod 32) of word floor(i/32); 1 = allowed.
  if ((rp.flags & kMask) && P.bitmask) {
    const int64_t W = (V + 31) / 32;
    const uint32_t* m = P.bitmask + pos * W;
    for (int i = 0; i < V; ++i)
      if (((m[i / 32] >> (i % 32)) & 1u) == 0u) x[i] = kNegInf;
  }
  // 2. repetition, frequency and presence penalties over the token history.
  if (rp.flags & kPenalty) {
    std::vector<int32_t> count(V, 0);
    const int hl = std::min(std::max(rp.hist_len, 0), P.hist_stride);
    for (int h = 0; h < hl; ++h) {
      const int32_t t = P.history[(int64_t)r * P.hist_stride + h];
      if (t < 0) continue;  // padding
      if (t >= V) { *status |= kStBadHist; continue; }
      count[t] += 1;
    }
    for (int32_t t : extra)
      if (t >= 0 && t < V) count[t] += 1;
    for (int i = 0; i < V; ++i) {
      const int32_t c = count[i];
      if (c > 0) {
        float v = x[i];
        v = (v > 0.0f) ? (v / rp.rep) : (v * rp.rep);
        v = v - rp.freq * (float)c;
        v = v - rp.pres;
        x[i] = v;
      }
    }
  }
  // 3. sparse logit bias, entries applied in list order.
  if (rp.flags & kBias) {
    const int nb = std::min(std::max(rp.n_bias, 0), P.bias_stride);
    for (int e = 0; e < nb; ++e) {
      const int32_t t = P.bias_tokens[(int64_t)r * P.bias_stride + e];
      if (t < 0) continue;
      if (t >= V) { *status |= kStBadBias; continue; }
      x[t] = x[t] + P.bias_values[(int64_t)r * P.bias_stride + e];
    }
  }
  // 4. temperature (stochastic rows only): x / T, one fp32 division.
  if (!(rp.flags & kGreedy)) {
    const float T = rp.temperature;
    for (int i = 0; i < V; ++i) x[i] = x[i] / T;
  }
  // 5. NaN -> -inf.
  for (int i = 0; i < V; ++i)
    if (std::isnan(x[i])) { x[i] = kNegInf; *status |= kStNan; }
  return x;
}

// (processed logit descending, index ascending); float comparison, so -0 == +0.
std::vector<int32_t> order_of(const std::vector<float>& x) {
  std::vector<int32_t> idx(x.size());
  std::iota(idx.begin(), idx.end(), 0);
  std::sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) {
    if (x[a] > x[b]) return true;
    if (x[a] < x[b]) return false;
    return a < b;
  });
  return idx;
}

struct Dist {
  int universe = 0;              // candidates considered (128 bounded, V exact)
  int n = 0;                     // kept prefix length
  std::vector<double> w;         // exp(l_t - l_0) over the universe
  double z_kept = 0.0;           // sum of kept w
  bool no_finite = false, pos_inf = false;
  double margin_topp = kInfD, margin_minp = kInfD;
};

// Softmax over the candidate universe and the truncation rules ([DN] Top-k,
// Top-p, Min-p, Combination; min-p in logit space [SS] 3.1).
Dist truncate(const sso_row& rp, const std::vector<float>& x, const std::vector<int32_t>& ord,
              int universe) {
  Dist d;
  d.universe = universe;
  const float l0 = x[ord[0]];
  int n_fin = 0;
  for (int t = 0; t < universe; ++t)
    if (x[ord[t]] > kNegInf) ++n_fin;
  if (n_fin == 0) { d.no_finite = true; d.n = 0; return d; }
  if (l0 == std::numeric_limits<float>::infinity()) {
    d.pos_inf = true; d.n = 1; d.w.assign(universe, 0.0); d.w[0] = 1.0; d.z_kept = 1.0;
    return d;
  }
  if (rp.flags & kGreedy) {  // greedy: a point mass on the argmax (top-k with k = 1)
    d.n = 1; d.w.assign(universe, 0.0); d.w[0] = 1.0; d.z_kept = 1.0;
    return d;
  }
  d.w.resize(universe);
  double Z = 0.0;
  for (int t = 0; t < universe; ++t) {
    d.w[t] = std::exp((double)x[ord[t]] - (double)l0);
    Z += d.w[t];
  }
  int n = universe;
  n = std::min(n, n_fin);
  if ((rp.flags & kTopK) && rp.top_k > 0) n = std::min(n, (int)rp.top_k);
  if ((rp.flags & kTopP) && rp.top_p < 1.0f) {
    const double tp = (double)rp.top_p;
    double cum = 0.0;
    int np_ = 0;
    for (int t = 0; t < universe; ++t) {
      d.margin_topp = std::min(d.margin_topp, std::fabs(cum - tp));
      if (cum < tp) ++np_;
      cum += d.w[t] / Z;
    }
    d.margin_topp = std::min(d.margin_topp, std::fabs(cum - tp));
    n = std::min(n, np_);
  }
  if ((rp.flags & kMinP) && rp.min_p > 0.0f) {
    const double thr = std::log((double)rp.min_p);
    int nm = 0;
    for (int t = 0; t < universe; ++t) {
      const double diff = (double)x[ord[t]] - (double)l0;
      if (std::isfinite(diff)) d.margin_minp = std::min(d.margin_minp, std::fabs(diff - thr));
      if (diff >= thr) ++nm;
    }
    n = std::min(n, nm);
  }
  d.n = std::max(1, n);
  double zk = 0.0;
  for (int t = 0; t < d.n; ++t) zk += d.w[t];
  d.z_kept = zk;
  return d;
}

struct Pick { int32_t token = -1; double margin = kInfD; };

// Gumbel-max over scores s_t = base_t + g_t in fp32 ([SS] 3.1 Sampling); ties
// go to the lower token index.
Pick gumbel_argmax(const std::vector<int32_t>& ids, const std::vector<float>& base, uint64_t seed,
                   uint32_t position, uint32_t row, uint32_t purpose) {
  Pick p;
  float best = kNegInf, second = kNegInf;
  int32_t best_id = -1;
  for (size_t t = 0; t < ids.size(); ++t) {
    const float s = base[t] + gumbel(seed, (uint32_t)ids[t], position, row, purpose);
    if (best_id < 0 || s > best || (s == best && ids[t] < best_id)) {
      second = best;
      best = s;
      best_id = ids[t];
    } else if (s > second) {
      second = s;
    }
  }
  p.token = best_id;
  if (ids.size() >= 2 && std::isfinite(best) && std::isfinite(second)) {
    const double scale = std::max(std::fabs((double)best), 1e-30);
    p.margin = ((double)best - (double)second) / scale;
  }
  return p;
}

double full_lse(const std::vector<float>& x, float l0) {
  if (!(l0 > kNegInf)) return -kInfD;
  double s = 0.0;
  for (float v : x) s += std::exp((double)v - (double)l0);
  return (double)l0 + std::log(s);
}

struct PosResult {
  std::vector<float> x;
  std::vector<int32_t> ord;
  Dist d;
};

PosResult eval_position(const sso_problem& P, int r, int64_t pos, const std::vector<int32_t>& extra,
                        int exact, uint32_t* status) {
  PosResult R;
  R.x = prelude(P, r, pos, extra, status);
  R.ord = order_of(R.x);
  const int universe = exact ? P.V : std::min(kK, P.V);
  R.d = truncate(P.rows[r], R.x, R.ord, universe);
  return R;
}

void write_candidates(const sso_outputs& O, int64_t pos, const PosResult& R) {
  const int nk = std::min(kK, (int)R.ord.size());
  if (O.cand_ids)
    for (int t = 0; t < kK; ++t) O.cand_ids[pos * kK + t] = t < nk ? R.ord[t] : -1;
  if (O.cand_probs)
    for (int t = 0; t < kK; ++t)
      O.cand_probs[pos * kK + t] =
          (t < R.d.n && R.d.z_kept > 0.0) ? (float)(R.d.w[t] / R.d.z_kept) : 0.0f;
  if (O.num_kept) O.num_kept[pos] = R.d.n;
  if (O.margin_topp) O.margin_topp[pos] = R.d.margin_topp;
  if (O.margin_minp) O.margin_minp[pos] = R.d.margin_minp;
  if (O.mass_outside || O.lse) {
    const float l0 = R.x[R.ord[0]];
    const double lse = full_lse(R.x, l0);
    if (O.lse) O.lse[pos] = lse;
    if (O.mass_outside) {
      double in = 0.0;
      for (int t = 0; t < nk; ++t) in += std::exp((double)R.x[R.ord[t]] - lse);
      O.mass_outside[pos] = std::isfinite(lse) ? std::max(0.0, 1.0 - in) : 0.0;
    }
  }
}

void clear_candidates(const sso_outputs& O, int64_t pos) {
  for (int t = 0; t < kK; ++t) {
    if (O.cand_ids) O.cand_ids[pos * kK + t] = -1;
    if (O.cand_probs) O.cand_probs[pos * kK + t] = 0.0f;
  }
  if (O.num_kept) O.num_kept[pos] = 0;
}

// One sampled token from the kept distribution of a position ([DN]
// Combination; Gumbel-max [SS] 3.1).
uint32_t philox_row(const sso_problem& P, int r) { return P.row_ids ? (uint32_t)P.row_ids[r] : (uint32_t)r; }

Pick sample_position(const sso_problem& P, int r, uint32_t position, const PosResult& R,
                     uint32_t* status) {
  Pick p;
  if (R.d.no_finite) { *status |= kStNoFinite; return p; }
  if (R.d.pos_inf) { *status |= kStPosInf; p.token = R.ord[0]; return p; }
  if (P.rows[r].flags & kGreedy) { p.token = R.ord[0]; return p; }
  std::vector<int32_t> ids;
  std::vector<float> base;
  const bool exact_row = (P.rows[r].flags & kExact) && !row_cuts(P.rows[r]);
  if (exact_row && !P.exact_on) *status |= kStNotExact;
  if (exact_row && P.exact_on) {
    // exact sampling: the Gumbel-max over every finite token of the vocabulary
    for (int32_t i = 0; i < (int32_t)R.x.size(); ++i)
      if (R.x[i] > -std::numeric_limits<float>::infinity()) { ids.push_back(i); base.push_back(R.x[i]); }
  } else {
    ids.assign(R.ord.begin(), R.ord.begin() + R.d.n);
    for (int t = 0; t < R.d.n; ++t) base.push_back(R.x[R.ord[t]]);
  }
  return gumbel_argmax(ids, base, P.seeds[r], position, philox_row(P, r), kPurposeSample);
}

}  // namespace

extern "C" {

int sso_abi_version() { return 1; }

// Philox word access for tests (counter (c0..c3), key (k0,k1)).
void sso_philox(const uint32_t* ctr_in, uint32_t k0, uint32_t k1, uint32_t* out) {
  uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
  philox4x32_10(c, k0, k1);
  for (int i = 0; i < 4; ++i) out[i] = c[i];
}

float sso_uniform(uint64_t seed, uint32_t i, uint32_t position, uint32_t row, uint32_t purpose) {
  return uniform01(seed, i, position, row, purpose);
}

// Processed logits of one position (for tests).
int sso_prelude(const sso_problem* P, int r, int64_t pos, const int32_t* extra, int n_extra,
                float* out, uint32_t* status) {
  std::vector<int32_t> ex(extra, extra + n_extra);
  uint32_t st = 0;
  std::vector<float> x = prelude(*P, r, pos, ex, &st);
  std::memcpy(out, x.data(), sizeof(float) * x.size());
  if (status) *status = st;
  return 0;
}

// Single-step sampling: one position per row.  mode 0 = bounded (k = 128), 1 = exact.
int sso_sample(const sso_problem* Pp, int exact, const sso_outputs* Op) {
  const sso_problem& P = *Pp;
  const sso_outputs& O = *Op;
  for (int r = 0; r < P.B; ++r) {
    uint32_t status = 0;
    const sso_row& rp = P.rows[r];
    if (!row_params_valid(rp, P)) {
      status |= kStBadParam;
      clear_candidates(O, r);
      O.tokens[(int64_t)r * O.tokens_stride] = -1;
      O.row_status[r] = status;
      continue;
    }
    PosResult R = eval_position(P, r, r, {}, exact, &status);
    write_candidates(O, r, R);
    Pick p = sample_position(P, r, rp.position, R, &status);
    if (O.margin_gumbel) O.margin_gumbel[r] = p.margin;
    O.tokens[(int64_t)r * O.tokens_stride] = p.token;
    O.row_status[r] = status;
  }
  return 0;
}

// Speculative verification ([SS] 3.1; [DN] Rejection Sampler).  Row r has
// gamma_r = cu_draft[r+1] - cu_draft[r] drafts and gamma_r + 1 target
// positions starting at cu_draft[r] + r.
int sso_verify(const sso_problem* Pp, int exact, const sso_outputs* Op) {
  const sso_problem& P = *Pp;
  const sso_outputs& O = *Op;
  const int V = P.V;
  for (int r = 0; r < P.B; ++r) {
    uint32_t status = 0;
    const sso_row& rp = P.rows[r];
    const int gamma = P.cu_draft[r + 1] - P.cu_draft[r];
    const int64_t pos0 = (int64_t)P.cu_draft[r] + r;
    int32_t* tok = O.tokens + (int64_t)r * O.tokens_stride;
    for (int j = 0; j < O.tokens_stride; ++j) tok[j] = -1;
    if (!row_params_valid(rp, P)) {
      for (int j = 0; j <= gamma; ++j) clear_candidates(O, pos0 + j);
      O.num_accepted[r] = 0;
      O.row_status[r] = status | kStBadParam;
      continue;
    }
    const bool greedy = (rp.flags & kGreedy) != 0;
    const bool trunc = row_truncates(rp);
    std::vector<int32_t> accepted_prefix;
    bool done = false;
    int n_acc = 0;
    // Every position's candidates are reported; decisions stop at the first rejection.
    for (int j = 0; j <= gamma; ++j) {
      const int64_t pos = pos0 + j;
      const uint32_t position = rp.position + (uint32_t)j;
      std::vector<int32_t> extra;
      for (int s = 0; s < j; ++s) extra.push_back(P.draft_ids[P.cu_draft[r] + s]);
      uint32_t pst = 0;
      PosResult R = eval_position(P, r, pos, extra, exact, &pst);
      write_candidates(O, pos, R);
      if (done) continue;
      status |= pst;
      if (j == gamma) {  // bonus token: all drafts accepted
        Pick p = sample_position(P, r, position, R, &status);
        if (O.margin_gumbel) O.margin_gumbel[pos] = p.margin;
        tok[j] = p.token;
        n_acc = gamma;
        break;
      }
      const int32_t d = P.draft_ids[P.cu_draft[r] + j];
      const bool d_ok = d >= 0 && d < V;
      if (!d_ok) status |= kStBadDraft;
      if (R.d.no_finite) {  // nothing to accept or resample
        status |= kStNoFinite;
        tok[j] = -1;
        n_acc = j;
        done = true;
        continue;
      }
      if (greedy || R.d.pos_inf) {
        if (R.d.pos_inf) status |= kStPosInf;
        if (d_ok && d == R.ord[0]) { tok[j] = d; continue; }
        tok[j] = R.ord[0];
        n_acc = j;
        done = true;
        continue;
      }
      // p_j: kept distribution (truncated rows) or full-V softmax (untruncated rows).
      std::vector<double> pfull;     // untruncated: p over V
      double lse = -kInfD;
      if (!trunc) {
        lse = full_lse(R.x, R.x[R.ord[0]]);
        pfull.resize(V);
        for (int i = 0; i < V; ++i) pfull[i] = std::exp((double)R.x[i] - lse);
      }
      auto p_of = [&](int32_t i) -> double {
        if (i < 0 || i >= V) return 0.0;
        if (!trunc) return pfull[i];
        for (int t = 0; t < R.d.n; ++t)
          if (R.ord[t] == i) return R.d.w[t] / R.d.z_kept;
        return 0.0;
      };
      const int64_t qrow = (int64_t)P.cu_draft[r] + j;
      auto q_of = [&](int32_t i) -> float { return load_elem(P.draft_probs, P.q_bf16, qrow * P.ld_q + i); };
      const double pd = p_of(d);
      bool accept = false;
      if (d_ok) {
        const float u = uniform01(P.seeds[r], 0u, position, philox_row(P, r), kPurposeAccept);
        const float prod = u * q_of(d);
        accept = pd > 0.0 && (double)prod <= pd;
        if (O.margin_accept) O.margin_accept[pos] = pd > 0.0 ? std::fabs((double)prod - pd) / pd : kInfD;
      }
      if (O.p_draft) O.p_draft[pos] = pd;
      if (accept) { tok[j] = d; continue; }
      // Rejected: resample from norm(max(0, p - q)) over the support of p_j.
      std::vector<int32_t> ids;
      std::vector<double> resid;
      std::vector<float> lbase;
      if (trunc) {
        for (int t = 0; t < R.d.n; ++t) {
          const int32_t i = R.ord[t];
          ids.push_back(i);
          resid.push_back(std::max(0.0, R.d.w[t] / R.d.z_kept - (double)q_of(i)));
          lbase.push_back(R.x[i]);
        }
      } else {
        for (int i = 0; i < V; ++i) {
          ids.push_back(i);
          resid.push_back(std::max(0.0, pfull[i] - (double)q_of(i)));
          lbase.push_back(R.x[i]);
        }
      }
      double rsum = 0.0;
      for (double v : resid) rsum += v;
      Pick pk;
      if (rsum > 0.0) {
        std::vector<int32_t> ids2;
        std::vector<float> base2;
        for (size_t t = 0; t < ids.size(); ++t)
          if (resid[t] > 0.0) { ids2.push_back(ids[t]); base2.push_back(logf((float)resid[t])); }
        pk = gumbel_argmax(ids2, base2, P.seeds[r], position, philox_row(P, r), kPurposeResidual);
      } else {
        status |= kStResidEmpty;
        pk = gumbel_argmax(ids, lbase, P.seeds[r], position, philox_row(P, r), kPurposeResidual);
      }
      if (O.margin_resid) O.margin_resid[pos] = pk.margin;
      tok[j] = pk.token;
      n_acc = j;
      done = true;
    }
    O.num_accepted[r] = n_acc;
    O.row_status[r] = status;
  }
  return 0;
}

}  // extern "C"
