// Stage-1 kernels for bf16 logits: the default variant in its eight
// compile-time forms (listed-token paths on / off, normaliser on / off,
// stage 2 fused or not).
#include "ss_stage1.cuh"

namespace ss {

template __global__ void stage1_kernel<true, false, false, false, false>(const Params);
template __global__ void stage1_kernel<true, false, true, false, false, false>(const Params);
template __global__ void stage1_kernel<true, false, false, true, false>(const Params);
template __global__ void stage1_kernel<true, false, true, false, false>(const Params);
template __global__ void stage1_kernel<true, false, true, true, false>(const Params);
template __global__ void stage1_kernel<true, false, false, false, true>(const Params);
template __global__ void stage1_kernel<true, false, false, true, true>(const Params);
template __global__ void stage1_kernel<true, false, true, false, true>(const Params);
template __global__ void stage1_kernel<true, false, true, true, true>(const Params);

template <bool AUX, bool LSE, bool FUSED>
static const void* ptr_of() { return (const void*)stage1_kernel<true, false, AUX, LSE, FUSED>; }

template <bool AUX, bool LSE, bool FUSED>
static void launch_of(int grid, size_t smem, cudaStream_t st, const Params& P) {
  stage1_kernel<true, false, AUX, LSE, FUSED><<<grid, kNT, smem, st>>>(P);
}

const void* stage1_ptr_bf16(bool aux, bool lse, bool fused) {
  if (fused) {
    if (aux) return lse ? ptr_of<true, true, true>() : ptr_of<true, false, true>();
    return lse ? ptr_of<false, true, true>() : ptr_of<false, false, true>();
  }
  if (aux) return lse ? ptr_of<true, true, false>() : ptr_of<true, false, false>();
  return lse ? ptr_of<false, true, false>() : ptr_of<false, false, false>();
}

void stage1_launch_bf16(bool aux, bool lse, bool fused, int grid, size_t smem, cudaStream_t st, const Params& P) {
  if (fused) {
    if (aux) lse ? launch_of<true, true, true>(grid, smem, st, P) : launch_of<true, false, true>(grid, smem, st, P);
    else lse ? launch_of<false, true, true>(grid, smem, st, P) : launch_of<false, false, true>(grid, smem, st, P);
  } else {
    if (aux) lse ? launch_of<true, true, false>(grid, smem, st, P) : launch_of<true, false, false>(grid, smem, st, P);
    else lse ? launch_of<false, true, false>(grid, smem, st, P) : launch_of<false, false, false>(grid, smem, st, P);
  }
}

// The lean form: listed-token paths without count tables, no normaliser.
const void* stage1_ptr_bf16_lean() { return (const void*)stage1_kernel<true, false, true, false, false, false>; }

void stage1_launch_bf16_lean(int grid, size_t smem, cudaStream_t st, const Params& P) {
  stage1_kernel<true, false, true, false, false, false><<<grid, kNT, smem, st>>>(P);
}

}  // namespace ss
