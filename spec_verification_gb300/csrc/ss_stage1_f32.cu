// Stage-1 kernels for fp32 logits: the default variant in its eight
// compile-time forms (listed-token paths on / off, normaliser on / off,
// stage 2 fused or not).
#include "ss_stage1.cuh"

namespace ss {

template __global__ void stage1_kernel<false, false, false, false, false>(const Params);
template __global__ void stage1_kernel<false, false, true, false, false, false>(const Params);
template __global__ void stage1_kernel<false, false, false, true, false>(const Params);
template __global__ void stage1_kernel<false, false, true, false, false>(const Params);
template __global__ void stage1_kernel<false, false, true, true, false>(const Params);
template __global__ void stage1_kernel<false, false, false, false, true>(const Params);
template __global__ void stage1_kernel<false, false, false, true, true>(const Params);
template __global__ void stage1_kernel<false, false, true, false, true>(const Params);
template __global__ void stage1_kernel<false, false, true, true, true>(const Params);

template <bool AUX, bool LSE, bool FUSED>
static const void* ptr_of() { return (const void*)stage1_kernel<false, false, AUX, LSE, FUSED>; }

template <bool AUX, bool LSE, bool FUSED>
static void launch_of(int grid, size_t smem, cudaStream_t st, const Params& P) {
  stage1_kernel<false, false, AUX, LSE, FUSED><<<grid, kNT, smem, st>>>(P);
}

const void* stage1_ptr_f32(bool aux, bool lse, bool fused) {
  if (fused) {
    if (aux) return lse ? ptr_of<true, true, true>() : ptr_of<true, false, true>();
    return lse ? ptr_of<false, true, true>() : ptr_of<false, false, true>();
  }
  if (aux) return lse ? ptr_of<true, true, false>() : ptr_of<true, false, false>();
  return lse ? ptr_of<false, true, false>() : ptr_of<false, false, false>();
}

void stage1_launch_f32(bool aux, bool lse, bool fused, int grid, size_t smem, cudaStream_t st, const Params& P) {
  if (fused) {
    if (aux) lse ? launch_of<true, true, true>(grid, smem, st, P) : launch_of<true, false, true>(grid, smem, st, P);
    else lse ? launch_of<false, true, true>(grid, smem, st, P) : launch_of<false, false, true>(grid, smem, st, P);
  } else {
    if (aux) lse ? launch_of<true, true, false>(grid, smem, st, P) : launch_of<true, false, false>(grid, smem, st, P);
    else lse ? launch_of<false, true, false>(grid, smem, st, P) : launch_of<false, false, false>(grid, smem, st, P);
  }
}

// Shared memory of a plan's stage-1 CTAs, the most ring slots a plan may use,
// and the room the fused form has for stage 2 (the candidate and scratch
// buffers).
size_t stage1_smem_bytes(int BN, bool bf16, int nslot) { return layout(BN, bf16 ? 2 : 4, nslot).total; }

int stage1_max_slots() { return kMaxSlots; }

int stage1_hash_tokens() { return kHashMax; }

size_t stage1_fused_room(int BN, bool bf16, int nslot) {
  const Layout L = layout(BN, bf16 ? 2 : 4, nslot);
  return L.out - L.cand;
}

// The lean form: listed-token paths without count tables, no normaliser.
const void* stage1_ptr_f32_lean() { return (const void*)stage1_kernel<false, false, true, false, false, false>; }

void stage1_launch_f32_lean(int grid, size_t smem, cudaStream_t st, const Params& P) {
  stage1_kernel<false, false, true, false, false, false><<<grid, kNT, smem, st>>>(P);
}

}  // namespace ss
