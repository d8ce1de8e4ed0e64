// ss_sample_noalloc: the single-step sampling call with its scratch held in a
// fixed-size device array of this library instead of a caller workspace.
//
// Who needs it: callers that have no way to obtain device memory for the
// workspace.  A serving runtime that reserves nearly all free HBM for its
// KV-cache pool at start-up and gives plug-ins no allocator is one; a plain C
// caller inside a decode loop is another, because cudaMalloc / cudaFree
// synchronise the whole device and would stall every stream each step.
//
// How: the scratch is a file-scope __device__ array; the first call on a
// device (with that device current) looks up its address once with
// cudaGetSymbolAddress, clears it on the call's stream, and every call then
// hands that address to ss_sample as its workspace.  Nothing here allocates
// device memory, and the launch sequence is ss_sample's with stage 2 as its
// own launch.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "ss.h"

namespace ss {
int plan_device(const ss_plan* p);
void set_last_error(const char* msg);
ss_status sample_call(const void* logits, const ss_batch* params, const int32_t* history, const uint32_t* bitmask,
                      const ss_bias_entry* bias, const uint64_t* seeds, ss_out* out, bool allow_fusion);
}  // namespace ss

namespace {

constexpr size_t kScratchBytes = SS_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

// One copy per device per process (a __device__ variable lives in every
// device's image of the module).  Zero at set-up; the kernels return their
// counters to zero at the end of each call.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices];  // device address of g_scratch, per ordinal; null until set up

ss_status fail(ss_status s, const char* msg) {
  ss::set_last_error(msg);
  return s;
}

// Set-up for one device: address lookup (the device must be current) and a
// clear of the whole array on the caller's stream.  Refused while the stream
// is being captured, so that the one-time clear is not recorded into a graph.
ss_status setup_device(int dev, cudaStream_t st, void** out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_ptr[dev] != nullptr) {
    *out = g_scratch_ptr[dev];
    return SS_OK;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return fail(SS_ERR_CUDA, "ss_sample_noalloc: cudaStreamIsCapturing failed");
  if (cs != cudaStreamCaptureStatusNone)
    return fail(SS_ERR_ARG,
                "ss_sample_noalloc: the first call on a device sets up the static scratch and must not "
                "run under stream capture");
  int prev = -1;
  e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return fail(SS_ERR_CUDA, "ss_sample_noalloc: cudaGetDevice failed");
  if (prev != dev && (e = cudaSetDevice(dev)) != cudaSuccess)
    return fail(SS_ERR_CUDA, "ss_sample_noalloc: cudaSetDevice failed");
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_scratch);
  if (e == cudaSuccess && p == nullptr) e = cudaErrorInvalidSymbol;
  if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, kScratchBytes, st);
  if (prev != dev) cudaSetDevice(prev);
  if (e != cudaSuccess) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "ss_sample_noalloc: scratch set-up failed: %s", cudaGetErrorString(e));
    return fail(SS_ERR_CUDA, msg);
  }
  g_scratch_ptr[dev] = p;
  *out = p;
  return SS_OK;
}

}  // namespace

extern "C" ss_status ss_sample_noalloc(const void* logits, const ss_batch* params, const int32_t* history,
                                       const uint32_t* bitmask, const ss_bias_entry* bias,
                                       const uint64_t* seeds, ss_out* out) {
  if (!params || !out || !params->plan) return fail(SS_ERR_ARG, "params, out and plan are required");
  const size_t need = ss_workspace_bytes(params->plan);
  if (need > kScratchBytes) {
    char msg[200];
    std::snprintf(msg, sizeof(msg),
                  "ss_sample_noalloc: the plan needs %zu bytes of scratch but the static scratch holds "
                  "%zu; use ss_sample with a caller workspace",
                  need, kScratchBytes);
    return fail(SS_ERR_UNSUPPORTED, msg);
  }
  const int dev = ss::plan_device(params->plan);
  if (dev < 0 || dev >= kMaxDevices) return fail(SS_ERR_UNSUPPORTED, "ss_sample_noalloc: device ordinal >= 64");
  void* scratch = nullptr;
  const ss_status s = setup_device(dev, static_cast<cudaStream_t>(params->stream), &scratch);
  if (s != SS_OK) return s;
  ss_batch b = *params;
  b.workspace = scratch;
  b.workspace_bytes = kScratchBytes;
  // stage 2 as its own launch: the scratch is shared by every plan, so the
  // words where this plan keeps the fused form's per-position counters may
  // hold another plan's lists
  return ss::sample_call(logits, &b, history, bitmask, bias, seeds, out, false);
}
