// Stage-1 kernels for fp32 logits: the default variant in its four
// compile-time forms (listed-token paths on / off, normaliser on / off).
#include "ss_stage1.cuh"

namespace ss {

template __global__ void stage1_kernel<false, false, false, false>(const Params);
template __global__ void stage1_kernel<false, false, true, false>(const Params);
template __global__ void stage1_kernel<false, false, false, true>(const Params);
template __global__ void stage1_kernel<false, false, true, true>(const Params);

const void* stage1_ptr_f32(bool aux, bool lse) {
  if (aux) return lse ? (const void*)stage1_kernel<false, false, true, true> : (const void*)stage1_kernel<false, false, true, false>;
  return lse ? (const void*)stage1_kernel<false, false, false, true> : (const void*)stage1_kernel<false, false, false, false>;
}

void stage1_launch_f32(bool aux, bool lse, int grid, size_t smem, cudaStream_t st, const Params& P) {
  if (aux) {
    if (lse) stage1_kernel<false, false, true, true><<<grid, kNT, smem, st>>>(P);
    else stage1_kernel<false, false, true, false><<<grid, kNT, smem, st>>>(P);
  } else {
    if (lse) stage1_kernel<false, false, false, true><<<grid, kNT, smem, st>>>(P);
    else stage1_kernel<false, false, false, false><<<grid, kNT, smem, st>>>(P);
  }
}

// Shared memory of a plan's stage-1 CTAs, and the most ring slots a plan may use.
size_t stage1_smem_bytes(int BN, bool bf16, int nslot) { return layout(BN, bf16 ? 2 : 4, nslot).total; }

int stage1_max_slots() { return kMaxSlots; }

}  // namespace ss
