// Host side of libss.so: plans, argument checks, workspace layout and the
// fixed launch sequence of ss_sample / ss_verify (see include/ss.h).
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "ss.h"
#include "ss_common.cuh"

namespace ss {
const void* stage1_ptr(bool bf16, bool exact, bool aux, bool lse, bool fused);
void stage1_launch(bool bf16, bool exact, bool aux, bool lse, bool fused, int grid, size_t smem, cudaStream_t st,
                   const Params& P);
size_t stage1_fused_room(int BN, bool bf16, int nslot);
const void* stage1_lean_ptr(bool bf16);
int stage1_hash_tokens();
void stage1_launch_lean(bool bf16, int grid, size_t smem, cudaStream_t st, const Params& P);
ss_status sample_call(const void* logits, const ss_batch* params, const int32_t* history, const uint32_t* bitmask,
                      const ss_bias_entry* bias, const uint64_t* seeds, ss_out* out, bool allow_fusion);
__global__ void stage2_kernel(const Params P, int verify);
__global__ void residual_kernel(const Params P);
size_t stage1_smem_bytes(int BN, bool bf16, int nslot);
int stage1_max_slots();
size_t stage2_smem_bytes(int Z);
int stage2_threads();
size_t residual_smem_bytes(int BN);
int residual_piece_tokens();
}  // namespace ss

struct ss_plan {
  int V, max_rows, max_positions, BN, Z, device, sms, nslot;
  int exact;  // stage 1 runs its exact-sampling variant
  int fuse;   // stage 2 inside stage 1: 1 whenever it fits; 2 never; 0 (the default) by the call's shape
  size_t fused_room;  // shared memory the fused form has for stage 2
  uint32_t spin_limit;  // polls of a stage-1 ring wait before it gives up
  uint32_t spin_hint_ns;  // suspend-time hint of each poll (0: the hardware's)
  ss_dtype ldt, qdt;
  int grid1, grid2, grid3;
  std::vector<int> grid2_by_cap;  // stage-2 grid for a shared-memory capacity of c lists (index c)
  size_t smem1, smem2, smem3;
  const void* k1;
  size_t off_staging, off_tlse, off_tgm, off_tst, off_pos, off_rowc, off_rescnt, off_parr, off_res, off_diag, ws_bytes;
  mutable int last_launches;  // kernels the most recent call launched
};

namespace {

thread_local std::string g_err;

// Polls of a stage-1 ring wait before the copy counts as lost.  The hardware
// suspends a polling thread between polls; measured, 2^22 polls of a copy
// that never lands take about 15 s.
constexpr uint32_t kDefaultSpin = 1u << 22;

ss_status fail(ss_status s, const char* msg) {
  g_err = msg;
  return s;
}

ss_status cuda_fail(cudaError_t e, const char* where) {
  g_err = std::string(where) + ": " + cudaGetErrorString(e);
  return SS_ERR_CUDA;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u; }

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev);
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    cudaGetDevice(&cur);
    if (prev >= 0 && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

extern "C" {

const char* ss_last_error(void) { return g_err.c_str(); }

const char* ss_status_str(ss_status s) {
  switch (s) {
    case SS_OK: return "ok";
    case SS_ERR_ARG: return "invalid argument";
    case SS_ERR_ALIGN: return "misaligned row";
    case SS_ERR_UNSUPPORTED: return "unsupported size";
    case SS_ERR_WORKSPACE: return "workspace too small";
    case SS_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

ss_status ss_plan_create(ss_plan** out, int32_t V, int32_t max_rows, int32_t max_positions,
                         ss_dtype logits_dtype, ss_dtype q_dtype, int32_t tile, int32_t device) {
  if (out == nullptr) return fail(SS_ERR_ARG, "plan pointer is NULL");
  *out = nullptr;
  if (V < 1 || V > (1 << 20)) return fail(SS_ERR_UNSUPPORTED, "V must be in [1, 2^20]");
  if (max_rows < 1 || max_positions < max_rows || max_positions > (1 << 24))
    return fail(SS_ERR_ARG, "need 1 <= max_rows <= max_positions <= 2^24");
  if ((logits_dtype != SS_F32 && logits_dtype != SS_BF16) || (q_dtype != SS_F32 && q_dtype != SS_BF16))
    return fail(SS_ERR_ARG, "dtype must be SS_F32 or SS_BF16");
  if (tile != 0 && tile != 8192 && tile != 16384) return fail(SS_ERR_UNSUPPORTED, "tile must be 0, 8192 or 16384");
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (device < 0 || device >= ndev) return fail(SS_ERR_ARG, "device ordinal out of range");
  DeviceGuard guard(device);
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  int smem_optin = 0;
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);

  int smem_sm = 0;
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device);

  const bool bf16 = logits_dtype == SS_BF16;
  int BN = tile;
  if (BN == 0) {
    // 8192-token stages, larger only when the stage-2 merge of Z_v lists of
    // 128 would not fit in shared memory
    BN = 8192;
    while (BN < 16384 && (long long)ss::stage2_smem_bytes((V + BN - 1) / BN) > smem_optin) BN *= 2;
  }
  // ring slots: as many as keep two CTAs per SM, else as many as fit one
  int nslot = 0;
  for (int s = ss::stage1_max_slots(); s >= 2 && nslot == 0; --s)
    if (2 * ((long long)ss::stage1_smem_bytes(BN, bf16, s) + 1024) <= smem_sm) nslot = s;
  for (int s = ss::stage1_max_slots(); s >= 2 && nslot == 0; --s)
    if ((long long)ss::stage1_smem_bytes(BN, bf16, s) <= smem_optin) nslot = s;
  if (nslot == 0) return fail(SS_ERR_UNSUPPORTED, "stage size too large for shared memory");
  ss_plan* p = new (std::nothrow) ss_plan();
  if (!p) return fail(SS_ERR_ARG, "out of host memory");
  p->V = V;
  p->max_rows = max_rows;
  p->max_positions = max_positions;
  p->BN = BN;
  p->Z = (V + BN - 1) / BN;
  p->device = device;
  p->sms = sms;
  p->nslot = nslot;
  p->ldt = logits_dtype;
  p->qdt = q_dtype;
  p->k1 = ss::stage1_ptr(bf16, false, true, true, false);
  p->exact = 0;
  p->fuse = 0;
  p->last_launches = 0;
  p->fused_room = ss::stage1_fused_room(BN, bf16, nslot);
  p->spin_limit = kDefaultSpin;
  p->spin_hint_ns = 0u;
  p->smem1 = ss::stage1_smem_bytes(BN, bf16, nslot);
  p->smem2 = ss::stage2_smem_bytes(p->Z);
  p->smem3 = ss::residual_smem_bytes(BN);
  if ((long long)p->smem2 > smem_optin || (long long)p->smem1 > smem_optin) {
    delete p;
    return fail(SS_ERR_UNSUPPORTED, "vocabulary too large for the stage-2 shared-memory merge");
  }
  // every default-variant form of stage 1 (listed-token paths, normaliser, fused stage 2)
  for (int v = 0; v < 8 && e == cudaSuccess; ++v)
    e = cudaFuncSetAttribute(ss::stage1_ptr(bf16, false, (v & 1) != 0, (v & 2) != 0, (v & 4) != 0),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p->smem1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ss::stage1_lean_ptr(bf16), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p->smem1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ss::stage2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p->smem2);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ss::residual_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p->smem3);
  int occ1 = 0, occ2 = 0, occ3 = 0;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ1, p->k1, ss::kNT, p->smem1);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, ss::stage2_kernel, ss::stage2_threads(), p->smem2);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ3, ss::residual_kernel, ss::kNT, p->smem3);
  if (e != cudaSuccess) {
    delete p;
    return cuda_fail(e, "kernel attributes");
  }
  const long long items1 = (long long)max_positions * p->Z;
  p->grid1 = (int)std::min<long long>(items1, (long long)std::max(occ1, 1) * sms);
  p->grid2 = std::min(max_positions, std::max(occ2, 1) * sms);
  // stage 2 sized per call by the lists a position can have (ss::seg_cap_for)
  p->grid2_by_cap.assign(p->Z + 1, p->grid2);
  for (int c = 1; c < p->Z && e == cudaSuccess; ++c) {
    int o = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, ss::stage2_kernel, ss::stage2_threads(),
                                                      ss::stage2_smem_bytes(c));
    p->grid2_by_cap[c] = std::min(max_positions, std::max(o, 1) * sms);
  }
  if (e != cudaSuccess) {
    delete p;
    return cuda_fail(e, "kernel attributes");
  }
  // residual items are (entry, vocabulary piece); at most four CTAs per SM so
  // that a call with no rejection spends little on empty CTAs
  const int piece = ss::residual_piece_tokens();
  const long long items3 = (long long)max_rows * ((V + piece - 1) / piece);
  p->grid3 = (int)std::min<long long>(items3, (long long)std::min(std::max(occ3, 1), 4) * sms);

  // workspace layout (256-byte aligned regions)
  size_t off = 0;
  const size_t P = (size_t)max_positions, R = (size_t)max_rows, PZ = P * p->Z;
  p->off_staging = off; off = align_up(off + PZ * ss::kK * 8, 256);
  p->off_tlse = off;    off = align_up(off + PZ * 8, 256);
  p->off_tgm = off;     off = align_up(off + PZ * 8, 256);
  p->off_tst = off;     off = align_up(off + PZ * 4, 256);
  p->off_pos = off;     off = align_up(off + P * sizeof(ss::PosResult), 256);
  p->off_rowc = off;    off = align_up(off + R * 4, 256);
  p->off_rescnt = off;  off = align_up(off + 12, 256);
  p->off_parr = off;    off = align_up(off + P * 4, 256);
  p->off_res = off;     off = align_up(off + R * sizeof(ss::ResidEntry), 256);
  p->off_diag = off;    off = align_up(off + 8 * 4, 256);
  p->ws_bytes = off;
  *out = p;
  return SS_OK;
}

void ss_plan_destroy(ss_plan* plan) { delete plan; }

size_t ss_workspace_bytes(const ss_plan* p) { return p ? p->ws_bytes : 0; }
int32_t ss_plan_tile(const ss_plan* p) { return p ? p->BN : 0; }
int32_t ss_plan_num_tiles(const ss_plan* p) { return p ? p->Z : 0; }
int32_t ss_plan_stage1_ctas(const ss_plan* p) { return p ? p->grid1 : 0; }

ss_status ss_plan_enable_exact(ss_plan* p, int enable) {
  if (!p) return fail(SS_ERR_ARG, "plan is required");
  if (enable) {
    DeviceGuard guard(p->device);
    // same launch bounds and shared memory as the default variant, so the
    // occupancy (and with it the stage-1 split) does not change
    const cudaError_t e = cudaFuncSetAttribute(ss::stage1_ptr(p->ldt == SS_BF16, true, true, true, false),
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p->smem1);
    if (e != cudaSuccess) return cuda_fail(e, "kernel attributes");
  }
  p->exact = enable ? 1 : 0;
  return SS_OK;
}
size_t ss_workspace_diag_offset(const ss_plan* p) { return p ? p->off_diag : 0; }

int32_t ss_plan_last_launches(const ss_plan* p) { return p ? p->last_launches : 0; }

ss_status ss_plan_set_fusion(ss_plan* p, int32_t mode) {
  if (!p) return fail(SS_ERR_ARG, "plan is required");
  if (mode < 0 || mode > 2) return fail(SS_ERR_ARG, "fusion mode must be 0 (default: by the call's shape), 1 (on) or 2 (off)");
  p->fuse = mode;
  return SS_OK;
}

ss_status ss_plan_set_wait_limit(ss_plan* p, uint32_t polls, uint32_t suspend_ns) {
  if (!p) return fail(SS_ERR_ARG, "plan is required");
  p->spin_limit = polls == 0 ? kDefaultSpin : polls;
  p->spin_hint_ns = suspend_ns;
  return SS_OK;
}

}  // extern "C"

namespace {

ss_status fill_common(const ss_plan* pl, const ss_batch* b, const void* logits, const uint64_t* seeds,
                      const ss_out* out, ss::Params& P) {
  if (b->B < 1 || b->B > pl->max_rows) return fail(SS_ERR_ARG, "B must be in [1, max_rows]");
  if (!logits || !b->rows || !seeds || !out->tokens || !out->row_status)
    return fail(SS_ERR_ARG, "logits, rows, seeds, tokens and row_status are required");
  const size_t esz = pl->ldt == SS_BF16 ? 2 : 4;
  if (b->ld_logits < pl->V) return fail(SS_ERR_ARG, "ld_logits < V");
  if (!aligned16(logits) || ((size_t)b->ld_logits * esz) % 16 != 0)
    return fail(SS_ERR_ALIGN, "logit rows must start on 16-byte boundaries");
  if (b->hist_stride < 1 || b->hist_stride > 16384 || b->bias_stride < 1 || b->bias_stride > 4096)
    return fail(SS_ERR_ARG, "hist_stride must be in [1, 16384] and bias_stride in [1, 4096]");
  if (!b->workspace || b->workspace_bytes < pl->ws_bytes)
    return fail(SS_ERR_WORKSPACE, "workspace missing or smaller than ss_workspace_bytes()");
  if ((reinterpret_cast<uintptr_t>(b->workspace) & 255u) != 0u)
    return fail(SS_ERR_ALIGN, "workspace must be 256-byte aligned");
  std::memset(&P, 0, sizeof(P));
  P.logits = logits;
  P.ld = b->ld_logits;
  P.V = pl->V;
  P.Z = pl->Z;
  P.BN = pl->BN;
  P.logits_bf16 = pl->ldt == SS_BF16;
  P.rows = b->rows;
  P.B = b->B;
  P.hist_stride = b->hist_stride;
  P.bias_stride = b->bias_stride;
  P.mask_words = (pl->V + 31) / 32;
  P.seeds = seeds;
  P.max_positions = pl->max_positions;
  P.grid1 = pl->grid1;
  P.nslot = pl->nslot;
  P.spin_limit = pl->spin_limit;
  P.spin_hint_ns = pl->spin_hint_ns;
  char* w = static_cast<char*>(b->workspace);
  P.ws.staging = reinterpret_cast<unsigned long long*>(w + pl->off_staging);
  P.ws.tile_lse = reinterpret_cast<float2*>(w + pl->off_tlse);
  P.ws.tile_gmax = reinterpret_cast<unsigned long long*>(w + pl->off_tgm);
  P.ws.tile_status = reinterpret_cast<uint32_t*>(w + pl->off_tst);
  P.ws.pos = reinterpret_cast<ss::PosResult*>(w + pl->off_pos);
  P.ws.row_count = reinterpret_cast<uint32_t*>(w + pl->off_rowc);
  P.ws.resid_count = reinterpret_cast<uint32_t*>(w + pl->off_rescnt);
  P.ws.pos_arrive = reinterpret_cast<uint32_t*>(w + pl->off_parr);
  P.ws.resid = reinterpret_cast<ss::ResidEntry*>(w + pl->off_res);
  P.ws.diag = reinterpret_cast<uint32_t*>(w + pl->off_diag);
  P.out = *out;
  return SS_OK;
}

// Grammar-mask rows start on 16-byte boundaries (so stage 1 bulk-copies the
// words of each stage with its logits) when the array does and ceil(V/32) is
// a multiple of 4.
int mask_rows_copyable(const ss::Params& P) {
  return P.bitmask != nullptr && aligned16(P.bitmask) && P.mask_words % 4 == 0 ? 1 : 0;
}

// Segment lists stage 2 must hold for one position.  A position's Z_v stages
// meet at most 1 + ceil((Z_v - 1) / L) stage-1 ranges when every range has at
// least L stages.  A call has at least B positions (exactly B when sampling),
// and once B * Z_v >= grid1 the ranges are at least floor(B * Z_v / grid1)
// stages long; below that a range may be a single stage.
// Under the aligned split (two or more stage-1 CTAs per position) a position
// has kk <= grid1 / npos <= grid1 / B lists.
int seg_cap_for(const ss_plan* pl, int B) {
  const int bmin = std::max(1, std::min(B, pl->max_positions));
  const long long tmin = (long long)bmin * pl->Z;
  int cap = pl->Z;
  if (tmin >= pl->grid1) {
    const long long L = tmin / pl->grid1;
    cap = (int)std::min<long long>(pl->Z, 1 + (pl->Z - 1 + L - 1) / L);
  }
  if (pl->grid1 / bmin >= 2) cap = std::max(cap, std::min(pl->Z, pl->grid1 / bmin));
  return cap;
}

// NVTX ranges (a call, and each launch in it) for profilers that record
// them; without a tool attached each push or pop is a test of a pointer.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

ss_status launch(const ss_plan* pl, const ss::Params& P0, cudaStream_t st, bool verify, void* const* ev,
                 bool allow_fusion = true) {
  const NvtxRange call_range(verify ? "ss_verify" : "ss_sample");
  ss::Params P = P0;
  P.seg_cap = seg_cap_for(pl, P.B);
  P.exact_on = pl->exact;
  const size_t smem2 = ss::stage2_smem_bytes(P.seg_cap);
  const int grid2 = pl->grid2_by_cap[P.seg_cap];
  cudaError_t e = cudaSuccess;
  // Under stream capture a plain event record is only a fork/join marker;
  // the external flag makes it an event-record node that fires at replay.
  unsigned int rec_flags = cudaEventRecordDefault;
  if (ev) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(st, &cs);
    if (cs == cudaStreamCaptureStatusActive) rec_flags = cudaEventRecordExternal;
  }
  auto rec = [&](int i) {
    if (ev && ev[i] && e == cudaSuccess)
      e = cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev[i]), st, rec_flags);
  };
  rec(0);
  const bool aux = P.history != nullptr || P.bias != nullptr;
  const long long npos_bound = verify ? pl->max_positions : std::min(P.B, pl->max_positions);
  // the stage-1 form holding only the paths this call can take: listed-token
  // paths when it passes a history or a bias list, the normaliser when it
  // verifies drafts.  Stage 2 runs inside it (fused) when a position's lists
  // fit the fused form's shared memory and the plan asks for it, or, by
  // default, when the call has no history or bias lists (those calls use the
  // lean / full dispatch below, which the fused form does not have) and at
  // least two stages per stage-1 CTA for the positions it can have.
  // Measured (us per call, fused against separate): 4 x 32000 fp32 18.8 /
  // 18.4 and a 64-row sampling call with lists 35.6 / 34.2 (not fused by
  // default), 256 x 262144 fp32 73.3 / 74.8 (fused by default).
  const bool shape_fuse = !aux && npos_bound * pl->Z >= 2LL * pl->grid1;
  const bool fused = allow_fusion && pl->exact == 0 && smem2 <= pl->fused_room &&
                     (pl->fuse == 1 || (pl->fuse == 0 && shape_fuse));
  // A long call with history or bias lists launches the lean form
  // (listed-token paths without count tables or normaliser) and then the full
  // form: each CTA first checks the rows (call_needs_full) and exactly one of
  // the two does the work, so the calls whose rows need neither path (the
  // common case) stream through the leaner loop.  Measured: the mixed serving
  // batch (76 stages per CTA) 6 % faster; a call of 3 stages per CTA 7 %
  // slower (the second launch costs more than the leaner loop saves), hence
  // the length test (at least 10 stages per CTA for the positions a call
  // can have).
  // A sampling call whose history and bias strides together fit the hash
  // table needs neither path (no drafts, and no row can list more tokens
  // than the strides hold): the lean form alone serves it.
  const int listed_max = (P.history ? P.hist_stride : 0) + (P.bias ? P.bias_stride : 0);
  const bool lean_only = aux && !verify && pl->exact == 0 && !fused && listed_max <= ss::stage1_hash_tokens();
  const bool dual = aux && !lean_only && pl->exact == 0 && !fused && npos_bound * pl->Z >= 10LL * pl->grid1;
  P.dispatch = 0;
  nvtxRangePushA(fused ? "ss stage 1 + 2" : "ss stage 1");
  if (lean_only) {
    ss::stage1_launch_lean(pl->ldt == SS_BF16, pl->grid1, pl->smem1, st, P);
  } else {
    if (dual) {
      P.dispatch = 1;
      ss::stage1_launch_lean(pl->ldt == SS_BF16, pl->grid1, pl->smem1, st, P);
      P.dispatch = 2;
    }
    ss::stage1_launch(pl->ldt == SS_BF16, pl->exact != 0, aux, P.cu_draft != nullptr, fused, pl->grid1, pl->smem1, st,
                      P);
  }
  nvtxRangePop();
  rec(1);
  if (!fused) {
    const NvtxRange r2("ss stage 2");
    ss::stage2_kernel<<<grid2, ss::stage2_threads(), smem2, st>>>(P, verify ? 1 : 0);
  }
  rec(2);
  if (verify) {
    const NvtxRange r3("ss residual pass");
    ss::residual_kernel<<<pl->grid3, ss::kNT, pl->smem3, st>>>(P);
  }
  rec(3);
  pl->last_launches = 1 + (dual ? 1 : 0) + (fused ? 0 : 1) + (verify ? 1 : 0);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return SS_OK;
}

}  // namespace

extern "C" {

ss_status ss_sample(const void* logits, const ss_batch* params, const int32_t* history,
                    const uint32_t* bitmask, const ss_bias_entry* bias, const uint64_t* seeds,
                    ss_out* out) {
  return ss::sample_call(logits, params, history, bitmask, bias, seeds, out, true);
}

}  // extern "C"

namespace ss {

// ss_sample; allow_fusion = false keeps stage 2 as its own launch (the
// no-alloc entry point, whose shared scratch may hold another plan's data
// where this plan keeps the fused form's per-position counters).
ss_status sample_call(const void* logits, const ss_batch* params, const int32_t* history,
                      const uint32_t* bitmask, const ss_bias_entry* bias, const uint64_t* seeds, ss_out* out,
                      bool allow_fusion) {
  if (!params || !out || !params->plan) return fail(SS_ERR_ARG, "params, out and plan are required");
  const ss_plan* pl = params->plan;
  if (params->B > pl->max_positions) return fail(SS_ERR_ARG, "B exceeds max_positions");
  ss::Params P;
  ss_status s = fill_common(pl, params, logits, seeds, out, P);
  if (s != SS_OK) return s;
  P.cu_draft = nullptr;
  P.history = history;
  P.bitmask = bitmask;
  P.bias = bias;
  P.mask_tma = mask_rows_copyable(P);
  DeviceGuard guard(pl->device);
  return launch(pl, P, static_cast<cudaStream_t>(params->stream), false, params->events, allow_fusion);
}

}  // namespace ss

extern "C" {

ss_status ss_verify(const void* target_logits, const void* draft_probs, const int32_t* draft_ids,
                    const ss_batch* params, const uint64_t* seeds, ss_out* out) {
  if (!params || !out || !params->plan) return fail(SS_ERR_ARG, "params, out and plan are required");
  const ss_plan* pl = params->plan;
  ss::Params P;
  ss_status s = fill_common(pl, params, target_logits, seeds, out, P);
  if (s != SS_OK) return s;
  if (!params->cu_draft || !draft_ids || !out->num_accepted)
    return fail(SS_ERR_ARG, "cu_draft, draft_ids and num_accepted are required");
  if (out->tokens_stride < 1) return fail(SS_ERR_ARG, "tokens_stride must be >= 1");
  if (draft_probs && params->ld_q < pl->V) return fail(SS_ERR_ARG, "ld_q < V");
  P.cu_draft = params->cu_draft;
  P.history = params->history;
  P.bitmask = params->bitmask;
  P.bias = params->bias;
  P.draft_ids = draft_ids;
  P.q = draft_probs;  // NULL: one-hot drafts
  P.ld_q = draft_probs ? params->ld_q : 0;
  P.q_bf16 = pl->qdt == SS_BF16;
  P.mask_tma = mask_rows_copyable(P);
  DeviceGuard guard(pl->device);
  return launch(pl, P, static_cast<cudaStream_t>(params->stream), true, params->events);
}

}  // extern "C"

namespace ss {
// Used by the static-scratch entry point (ss_noalloc.cu).
int plan_device(const ss_plan* p) { return p->device; }
void set_last_error(const char* msg) { g_err = msg; }
}  // namespace ss
