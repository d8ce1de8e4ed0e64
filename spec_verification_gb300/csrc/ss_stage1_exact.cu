// Stage-1 kernels of the exact-sampling variant (every path present), for
// fp32 and bf16 logits.
#include "ss_stage1.cuh"

namespace ss {

template __global__ void stage1_kernel<false, true, true, true, false>(const Params);
template __global__ void stage1_kernel<true, true, true, true, false>(const Params);

const void* stage1_ptr_exact(bool bf16) {
  return bf16 ? (const void*)stage1_kernel<true, true, true, true, false> : (const void*)stage1_kernel<false, true, true, true, false>;
}

void stage1_launch_exact(bool bf16, int grid, size_t smem, cudaStream_t st, const Params& P) {
  if (bf16) stage1_kernel<true, true, true, true, false><<<grid, kNT, smem, st>>>(P);
  else stage1_kernel<false, true, true, true, false><<<grid, kNT, smem, st>>>(P);
}

}  // namespace ss
