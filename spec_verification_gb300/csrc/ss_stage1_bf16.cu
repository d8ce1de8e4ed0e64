// Stage-1 kernels for bf16 logits: the default variant in its four
// compile-time forms (listed-token paths on / off, normaliser on / off).
#include "ss_stage1.cuh"

namespace ss {

template __global__ void stage1_kernel<true, false, false, false>(const Params);
template __global__ void stage1_kernel<true, false, true, false>(const Params);
template __global__ void stage1_kernel<true, false, false, true>(const Params);
template __global__ void stage1_kernel<true, false, true, true>(const Params);

const void* stage1_ptr_bf16(bool aux, bool lse) {
  if (aux) return lse ? (const void*)stage1_kernel<true, false, true, true> : (const void*)stage1_kernel<true, false, true, false>;
  return lse ? (const void*)stage1_kernel<true, false, false, true> : (const void*)stage1_kernel<true, false, false, false>;
}

void stage1_launch_bf16(bool aux, bool lse, int grid, size_t smem, cudaStream_t st, const Params& P) {
  if (aux) {
    if (lse) stage1_kernel<true, false, true, true><<<grid, kNT, smem, st>>>(P);
    else stage1_kernel<true, false, true, false><<<grid, kNT, smem, st>>>(P);
  } else {
    if (lse) stage1_kernel<true, false, false, true><<<grid, kNT, smem, st>>>(P);
    else stage1_kernel<true, false, false, false><<<grid, kNT, smem, st>>>(P);
  }
}

}  // namespace ss
