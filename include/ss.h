/* ss.h -- fused LLM sampling and speculative verification on one GB300 GPU.
 *
 * C ABI of libss.so.  Every entry point takes plain pointers and sizes; all
 * tensors are caller-owned device memory unless stated otherwise.  The
 * library never allocates device memory, never synchronises the device and
 * never copies to the host inside ss_sample / ss_verify: both are a fixed
 * sequence of kernel launches on the caller's stream whose launch shapes
 * depend only on the plan, so a call can be captured in a CUDA Graph and
 * replayed with new device-resident data (logits, parameters, draft offsets,
 * seeds).  Each call is also marked with NVTX ranges ("ss_sample" /
 * "ss_verify", and one per launch: stage 1, stage 2, the residual pass) for
 * profilers that record them.
 *
 * What is computed (page titles and sections of the source material):
 *  - "SonicSampler: unified tile-aware kernels for LLM sampling and
 *    speculative verification", 3.1 Background: logits processing (grammar
 *    mask, repetition / frequency / presence penalties, logit bias,
 *    temperature) is a map over the vocabulary; truncation (top-k, top-p,
 *    min-p; min-p can be evaluated without a softmax) needs a global
 *    reduction; sampling is x* = argmax_i (x_i + eps_i) (Gumbel-max, eps = 0
 *    for greedy); a draft token d is accepted when u q(d) <= p(d), u ~ U(0,1),
 *    and otherwise a token is resampled from max(0, p - q) normalised.
 *  - same page, 3.2 Workload-aware execution model and Fig. 1: a two-stage
 *    hierarchical top-k with k = 128.  Stage 1 runs one program per
 *    (row, vocabulary tile of B_N tokens) and fuses the prelude with a
 *    tile-local top-k; only k packed candidates per tile reach HBM.  Stage 2
 *    runs per row, merges the Z_v * k candidates (Z_v = ceil(V / B_N)) and
 *    applies truncation, Gumbel noise and argmax.
 *  - "Decoding and sampling" (dl-note), sections Temperature, Top-k, Top-p,
 *    Min-p and Combination (Temperature -> Softmax -> top-k/top-p/min-p ->
 *    Renormalize -> Sample; top-k with top-p keeps the intersection), and
 *    Rejection Sampler (accept / residual; the output is distributed as p).
 *
 * Semantics fixed where the pages are silent:
 *  - prelude per element, fp32 with one rounding per operation, in this
 *    order: mask (bit i%32 of word i/32, 1 = allowed, else -inf); if count
 *    c of token i in the history is > 0 and SS_PENALTY: x = x>0 ? x/rep :
 *    x*rep, then x -= freq*c, then x -= pres; if SS_BIAS: each bias entry for
 *    token i is added in list order; stochastic rows: x /= T (one IEEE
 *    division, dl-note Temperature); a NaN
 *    result becomes -inf (status SS_ST_NAN);
 *  - candidate order: processed logit descending, token id ascending (-0 and
 *    +0 are equal); candidates are the first min(128, V) tokens in that order;
 *  - probabilities are the softmax over those candidates; top-k keeps k,
 *    top-p keeps token t iff the probability mass before it is < top_p,
 *    min-p keeps t iff l_t - l_0 >= ln(min_p); the kept set is the shortest
 *    active prefix and at least one token; greedy rows take the first
 *    candidate and ignore temperature and truncation;
 *  - random numbers: Philox-4x32-10 (Salmon et al., SC'11) with key = the
 *    row's 64-bit seed and counter (i/4, position, row, purpose), word i%4;
 *    u = ((w >> 9) * 2 + 1) * 2^-24; Gumbel noise -ln(-ln u) in fp32;
 *    purpose 0 = sample / bonus token (i = token id), 1 = accept uniform
 *    (i = 0), 2 = residual resampling (i = token id); position =
 *    rows[r].position + j for draft index j;
 *  - verification p: the kept distribution for rows that request any
 *    truncation, else the full-vocabulary softmax; greedy rows accept iff
 *    the draft equals the argmax.
 */
#ifndef SS_H_
#define SS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes.  Host-detectable misuse returns a negative code before any
 * launch; SS_ERR_CUDA means a launch failed (ss_last_error() has the text). */
typedef enum {
  SS_OK = 0,
  SS_ERR_ARG = -1,          /* null pointer, size out of range, B > max_rows */
  SS_ERR_ALIGN = -2,        /* logits / draft-prob rows not 16-byte aligned */
  SS_ERR_UNSUPPORTED = -3,  /* vocabulary or tile size outside the plan's range */
  SS_ERR_WORKSPACE = -4,    /* workspace missing or smaller than ss_workspace_bytes */
  SS_ERR_CUDA = -5          /* CUDA runtime error */
} ss_status;

typedef enum { SS_F32 = 0, SS_BF16 = 1 } ss_dtype;

/* Per-row flag bits: the "compact bit-level indicators" that select
 * per-request behaviour inside one batch (SonicSampler page, section 1). */
enum {
  SS_GREEDY = 1u << 0,   /* argmax; ignore temperature and truncation */
  SS_MASK = 1u << 1,     /* apply the grammar bitmask */
  SS_PENALTY = 1u << 2,  /* repetition / frequency / presence penalties */
  SS_BIAS = 1u << 3,     /* sparse logit bias */
  SS_TOPK = 1u << 4,     /* top_k > 0 keeps the top_k most probable */
  SS_TOPP = 1u << 5,     /* top_p < 1 keeps the nucleus */
  SS_MINP = 1u << 6,     /* min_p > 0 keeps p >= min_p * p_max */
  SS_BOUNDED_P = 1u << 7, /* verify: p is the softmax over the row's 128
                             candidates even without truncation (no pass
                             over the vocabulary; a draft outside them is
                             rejected) */
  SS_EXACT = 1u << 8      /* untruncated stochastic rows: the sample (and
                             the bonus token of a verify row) is the
                             Gumbel-max over the whole vocabulary, not over
                             the 128 candidates (exact softmax sampling);
                             needs a plan with ss_plan_enable_exact */
};

/* Per-row status bits written to ss_out.row_status.  Data errors never trap. */
enum {
  SS_ST_NAN = 1u << 0,         /* a processed logit was NaN; treated as -inf */
  SS_ST_NO_FINITE = 1u << 1,   /* every candidate is -inf; token = -1 */
  SS_ST_BAD_HIST = 1u << 2,    /* a history id >= V was ignored */
  SS_ST_BAD_BIAS = 1u << 3,    /* a bias id >= V was ignored */
  SS_ST_BAD_PARAM = 1u << 4,   /* invalid parameters: no tokens (-1) */
  SS_ST_BAD_DRAFT = 1u << 5,   /* a draft id outside [0, V): rejected */
  SS_ST_POS_INF = 1u << 6,     /* +inf processed logit: point mass on it */
  SS_ST_RESID_EMPTY = 1u << 7, /* residual max(0, p - q) had no mass: sampled from p */
  SS_ST_NOT_EXACT = 1u << 8,    /* SS_EXACT on a plan without exact sampling:
                                   sampled from the 128 candidates */
  SS_ST_CAPACITY = 1u << 9,     /* verification: the row's target positions reach
                                   past the plan's max_positions; not verified,
                                   tokens -1, num_accepted 0 */
  SS_ST_COPY_TIMEOUT = 1u << 10 /* a stage-1 copy of this row's logits did not
                                   land within the wait limit: the row's result
                                   is not valid (not expected; see
                                   ss_plan_set_wait_limit) */
};

/* One row's sampling parameters (device array of B entries, 44 bytes each).
 * Valid ranges: stochastic rows need 0 < temperature < inf; top_p in (0, 1]
 * when SS_TOPP; min_p in [0, 1] when SS_MINP; top_k >= 0 when SS_TOPK;
 * rep > 0 and finite freq, pres when SS_PENALTY; 0 <= hist_len <= hist_stride;
 * 0 <= n_bias <= bias_stride.  A row outside them gets SS_ST_BAD_PARAM. */
typedef struct {
  uint32_t flags;
  float temperature, top_p, min_p;
  float rep, freq, pres;
  int32_t top_k;
  int32_t hist_len;     /* entries of the history row in use; ids < 0 are padding */
  int32_t n_bias;       /* entries of the bias row in use; ids < 0 are padding */
  uint32_t position;    /* Philox position of the row's first target position */
} ss_row_params;

/* One sparse-bias entry (device array [B, bias_stride]). */
typedef struct {
  int32_t token;
  float value;
} ss_bias_entry;

/* Opaque, immutable plan: vocabulary size, capacities, dtypes and the tile
 * size B_N, chosen once per shape on the host. */
typedef struct ss_plan ss_plan;

/* Per-call batch description (host struct; the pointers inside are device
 * pointers unless noted). */
typedef struct {
  int32_t B;                       /* rows in this call, 1 <= B <= max_rows */
  int64_t ld_logits;               /* row stride of the logits in elements (>= V) */
  int64_t ld_q;                    /* row stride of draft_probs in elements (>= V) */
  const ss_row_params* rows;       /* [B] */
  const int32_t* cu_draft;         /* verify: [B+1] prefix sums of gamma_r, cu_draft[0] = 0
                                      (non-decreasing; not checked: other values are undefined) */
  int32_t hist_stride;             /* ints per history row (>= 1) */
  int32_t bias_stride;             /* entries per bias row (>= 1) */
  /* ss_verify only (ss_sample takes these as arguments): */
  const int32_t* history;          /* [B, hist_stride] or NULL */
  const uint32_t* bitmask;         /* [B_pos, ceil(V/32)] per target position, or NULL */
  const ss_bias_entry* bias;       /* [B, bias_stride] or NULL */
  void* workspace;                 /* caller-allocated device scratch, 256-byte aligned */
  size_t workspace_bytes;          /* >= ss_workspace_bytes(plan) */
  void* stream;                    /* cudaStream_t (NULL = legacy default stream) */
  const ss_plan* plan;
  void* const* events;             /* optional: 4 cudaEvent_t (timing enabled) recorded on the
                                      stream before stage 1, after stage 1, after stage 2 and
                                      after the residual pass (ss_verify) or again after stage 2
                                      (ss_sample); NULL = none.  Captured into CUDA Graphs as
                                      event-record nodes. */
} ss_batch;

/* Outputs (device pointers, caller-owned). */
typedef struct {
  int32_t* tokens;         /* sample: [B]; verify: [B, tokens_stride], -1 padded */
  int32_t tokens_stride;   /* verify: >= max gamma + 1 (ignored by ss_sample) */
  int32_t* num_accepted;   /* verify: [B] accepted drafts; ignored by ss_sample */
  int32_t* cand_ids;       /* optional [B_pos, 128]: candidates in order, -1 padded */
  float* cand_probs;       /* optional [B_pos, 128]: kept renormalised probs, 0 beyond */
  int32_t* num_kept;       /* optional [B_pos]: kept prefix length */
  uint32_t* row_status;    /* [B]: SS_ST_* bits */
} ss_out;

/* Create a plan.  V in [1, 2^20]; max_rows >= 1; max_positions >= max_rows
 * bounds B_pos (B for sampling, cu_draft[B] + B for verification; a
 * verification call whose device-side cu_draft[B] + B exceeds it verifies
 * the rows whose positions all lie below max_positions and reports the
 * others with SS_ST_CAPACITY; candidate outputs are written for positions
 * below max_positions only);
 * tile = 0 chooses B_N automatically, else 8192 or 16384.  device is the
 * CUDA ordinal the plan is for.  Returns SS_ERR_ARG / SS_ERR_UNSUPPORTED on
 * bad sizes; *plan is NULL on failure.  The plan is host memory owned by the
 * caller (ss_plan_destroy). */
ss_status ss_plan_create(ss_plan** plan, int32_t V, int32_t max_rows, int32_t max_positions,
                         ss_dtype logits_dtype, ss_dtype q_dtype, int32_t tile, int32_t device);
void ss_plan_destroy(ss_plan* plan);

/* Device scratch a call needs: per-tile staging (B_pos * Z_v * 128 entries
 * of 8 bytes), per-tile metadata and per-row bookkeeping.  Must be zeroed
 * once before the first call with a plan (the library keeps its counters at
 * zero between calls); a workspace that held another plan's data must be
 * zeroed again. */
size_t ss_workspace_bytes(const ss_plan* plan);

/* Tile size B_N and tile count Z_v the plan uses. */
int32_t ss_plan_tile(const ss_plan* plan);
int32_t ss_plan_num_tiles(const ss_plan* plan);

/* CTAs of the stage-1 launch.  Stage 1 splits the B_pos * Z_v tiles into
 * min(this, B_pos * Z_v) contiguous runs, one per CTA; a run's part inside
 * one position is a segment, which leaves one list of 128 candidates. */
int32_t ss_plan_stage1_ctas(const ss_plan* plan);

/* Exact sampling for rows flagged SS_EXACT (an addition of this library,
 * following the pages' note that a tile-local Gumbel-max is exact and
 * decomposes over tiles): enable != 0 makes the plan run the stage-1 variant
 * that also keeps, per segment, the Gumbel-max of l_i + g_i over every token
 * (g_i the Philox purpose-0 noise of the sampler); stage 2 then takes the
 * largest of a position's segment maxima as the token.  Off by default: the
 * default variant's streaming loop carries none of this work.  On a plan
 * without it, SS_EXACT rows are sampled from their 128 candidates and report
 * SS_ST_NOT_EXACT.  Not thread-safe against calls using the plan.
 * Returns SS_ERR_ARG for a NULL plan, SS_ERR_CUDA if the kernel cannot be
 * configured. */
ss_status ss_plan_enable_exact(ss_plan* plan, int enable);

/* Single-step sampling (SonicSampler 3.1-3.2; dl-note Combination).
 * logits:  [B, ld_logits] fp32 or bf16 (plan dtype), rows 16-byte aligned.
 * params:  host batch description (B, rows, strides, workspace, stream, plan).
 * history: [B, hist_stride] int32 or NULL; with NULL, SS_PENALTY is ignored.
 * bitmask: [B, ceil(V/32)] uint32 or NULL; with NULL, SS_MASK is ignored.
 * bias:    [B, bias_stride] ss_bias_entry or NULL; with NULL, SS_BIAS is ignored.
 * seeds:   [B] uint64 Philox keys.
 * out:     host struct of device outputs: tokens [B], row_status [B], and the
 *          optional candidate outputs indexed by row.
 * Asynchronous on params->stream. */
ss_status ss_sample(const void* logits, const ss_batch* params, const int32_t* history,
                    const uint32_t* bitmask, const ss_bias_entry* bias, const uint64_t* seeds,
                    ss_out* out);

/* Speculative verification (SonicSampler 3.1; dl-note Rejection Sampler).
 * Row r has gamma_r = cu_draft[r+1] - cu_draft[r] drafts and gamma_r + 1
 * target positions starting at cu_draft[r] + r; gamma_r = 0 is a single-step
 * row whose bonus token is its sample.
 * target_logits: [cu_draft[B] + B, ld_logits] (plan dtype).
 * draft_probs:   [cu_draft[B], ld_q] draft-model probabilities q (plan q dtype),
 *                or NULL for drafts without probabilities (n-gram or
 *                prompt-lookup drafts): q is then one-hot on the draft token,
 *                so a draft is accepted iff u <= p(d) and a rejection samples
 *                from p with the draft token removed (dl-note "Decoding and
 *                sampling", Rejection Sampler, its example's no-draft-probs
 *                case).  ld_q is ignored then.
 * draft_ids:     [cu_draft[B]] int32.
 * params:        as for ss_sample, plus cu_draft and the processor inputs
 *                history / bitmask (per target position) / bias, each NULL
 *                or not as for ss_sample (a NULL history also leaves the
 *                drafts uncounted: SS_PENALTY is ignored).
 * seeds:         [B] uint64.
 * out:           tokens [B, tokens_stride] (accepted drafts, then the
 *                resampled or bonus token, then -1), num_accepted [B],
 *                row_status [B], optional candidate outputs per target position.
 * Asynchronous on params->stream. */
ss_status ss_verify(const void* target_logits, const void* draft_probs, const int32_t* draft_ids,
                    const ss_batch* params, const uint64_t* seeds, ss_out* out);

/* ss_sample_noalloc -- the source material has no counterpart to this call;
 * it is an addition of this library.  It is ss_sample for callers that cannot
 * provide the workspace: a runtime that hands nearly all free device memory
 * to its own pool (a KV cache) and exposes no allocator, or a C caller in a
 * decode loop that must not call cudaMalloc / cudaFree because both
 * synchronise the device.  It allocates nothing.
 *
 * Arguments, outputs and results are those of ss_sample; params->workspace
 * and params->workspace_bytes are ignored.  The scratch is a device array
 * of SS_NOALLOC_SCRATCH_BYTES inside libss.so, one per device per process:
 *  - the first call for a device (the plan's device) does the set-up: it
 *    looks the array's address up and clears it on params->stream;
 *  - the address is looked up once per process and device: do not use this
 *    call across a cudaDeviceReset of that device;
 *  - the diagnostic counters (ss_workspace_diag_offset) of these calls live
 *    in the library's array, which the caller never sees: they cannot be
 *    read for this call;
 *  - the whole array starts at zero (set-up clears it); the counters in it
 *    must be zero when a call starts, and each completed call leaves them
 *    at zero again; stage 2 always runs as its own launch here (the array
 *    is shared by every plan, see ss_plan_set_fusion);
 *  - plans whose ss_workspace_bytes exceeds SS_NOALLOC_SCRATCH_BYTES are
 *    rejected with SS_ERR_UNSUPPORTED (use ss_sample with a workspace);
 *  - calls on the same device that overlap in time (different streams or
 *    host threads without ordering between them) share the array and race:
 *    order them on one stream or serialise them. */
#define SS_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20) /* 16 MiB */
ss_status ss_sample_noalloc(const void* logits, const ss_batch* params, const int32_t* history,
                            const uint32_t* bitmask, const ss_bias_entry* bias, const uint64_t* seeds,
                            ss_out* out);

const char* ss_status_str(ss_status s);

/* Text of the last error on the calling host thread ("" if none). */
const char* ss_last_error(void);

/* Where stage 2 (merge, epilogue, sampling / accept test, row walk) runs.
 * Fused: inside the stage-1 launch, where the CTA that writes a position's
 * last segment list runs that position's stage 2 at once (only when a
 * position's lists fit that launch's shared memory; otherwise, and
 * unfused, stage 2 is its own launch after stage 1).  Fusing saves a launch
 * and lets a position's stage 2 overlap the streaming of other positions,
 * but it delays the rest of the fusing CTA's stage-1 range.
 *  - mode 0 (the default): fused when the call passes no history and no
 *    bias list and the positions it can have (B for ss_sample, the plan's
 *    max_positions for ss_verify) span at least two stage-1 stages per
 *    stage-1 CTA.  Calls with lists keep their lean / full stage-1 dispatch,
 *    which the fused form does not have.
 *  - mode 1: fused whenever the lists fit.
 *  - mode 2: never.
 * Plans with exact sampling enabled never fuse.  Results do not depend on
 * the mode.  Not thread-safe against calls using the plan.  SS_ERR_ARG for a
 * NULL plan or another mode. */
ss_status ss_plan_set_fusion(ss_plan* plan, int32_t mode);

/* Kernels launched by the most recent successful ss_sample / ss_verify /
 * ss_sample_noalloc call with this plan (stage-1 forms, stage 2 unless
 * fused, the residual pass of ss_verify); 0 before the first.  A host-side
 * record of the launch decisions, for accounting; not thread-safe against
 * calls using the plan. */
int32_t ss_plan_last_launches(const ss_plan* plan);

/* Wait limit of stage 1's copy ring: a thread polls a ring slot's
 * completion at most `polls` times (0 restores the default, 2^22 polls)
 * before it counts the copy as lost.  suspend_ns == 0 (the default): each
 * poll may suspend the thread in hardware until the copy lands or the
 * hardware's time limit passes (2^22 such polls of a copy that never lands
 * take about 15 s).  suspend_ns > 0: each poll tests once without suspending
 * and then sleeps about suspend_ns nanoseconds.  A CTA that gives up stops
 * waiting, writes empty candidate lists with SS_ST_COPY_TIMEOUT for its
 * remaining positions (so their rows report it), counts itself in
 * diagnostic counter 3 and lets the copies it issued land (waiting up to
 * 2^22 suspending polls for them) before it exits.  A lost copy is not
 * expected: a short limit (one poll, suspend_ns = 1) is a way to exercise
 * this path, since the copies still land, only later than the waits allow.
 * Not thread-safe against calls using the plan.  Returns SS_ERR_ARG for a
 * NULL plan. */
ss_status ss_plan_set_wait_limit(ss_plan* plan, uint32_t polls, uint32_t suspend_ns);

/* Byte offset, inside the workspace, of 8 uint32 diagnostic counters the
 * kernels increment: 0: stage-1 stages replaced by their exact top-128 (the
 * candidate buffer overflowed within the stage, or a segment's first stage
 * certified fewer than 128 elements); 1: stage-2 positions with more segment
 * lists than the call's shared memory holds (reported SS_ST_BAD_PARAM; not
 * expected); 2: residual passes over V; 3: stage-1 CTAs that gave up
 * waiting for a copy (their positions are left without candidates and
 * report SS_ST_COPY_TIMEOUT; not expected); 4: stage-1 candidate buffers cut
 * back to their exact top-128 after a histogram raise left too many; 5:
 * stage-2 sample / bonus positions whose top-p or min-p cut point lay too
 * close to its limit for the fp32 weights and was decided in fp64.  They
 * are cumulative and only cleared by the caller. */
size_t ss_workspace_diag_offset(const ss_plan* plan);

#ifdef __cplusplus
}
#endif

#endif /* SS_H_ */
