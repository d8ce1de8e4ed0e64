// Stage 1 on the host side: which compiled variant a call launches.  The
// kernel itself is in
// ss_stage1.cuh, instantiated by ss_stage1_f32.cu, ss_stage1_bf16.cu and
// ss_stage1_exact.cu (compiled in parallel).
#include "ss_common.cuh"

namespace ss {

const void* stage1_ptr_f32(bool aux, bool lse, bool fused);
const void* stage1_ptr_bf16(bool aux, bool lse, bool fused);
const void* stage1_ptr_exact(bool bf16);
void stage1_launch_f32(bool aux, bool lse, bool fused, int grid, size_t smem, cudaStream_t st, const Params& P);
void stage1_launch_bf16(bool aux, bool lse, bool fused, int grid, size_t smem, cudaStream_t st, const Params& P);
void stage1_launch_exact(bool bf16, int grid, size_t smem, cudaStream_t st, const Params& P);
const void* stage1_ptr_f32_lean();
const void* stage1_ptr_bf16_lean();
void stage1_launch_f32_lean(int grid, size_t smem, cudaStream_t st, const Params& P);
void stage1_launch_bf16_lean(int grid, size_t smem, cudaStream_t st, const Params& P);

// aux: the call passes a history or a bias list (rows may have penalties or
// bias); lse: the call verifies drafts; fused: stage 2 runs inside stage 1.
// The exact-sampling variant holds every path and is never fused.
const void* stage1_ptr(bool bf16, bool exact, bool aux, bool lse, bool fused) {
  if (exact) return stage1_ptr_exact(bf16);
  return bf16 ? stage1_ptr_bf16(aux, lse, fused) : stage1_ptr_f32(aux, lse, fused);
}

void stage1_launch(bool bf16, bool exact, bool aux, bool lse, bool fused, int grid, size_t smem, cudaStream_t st,
                   const Params& P) {
  if (exact) stage1_launch_exact(bf16, grid, smem, st, P);
  else if (bf16) stage1_launch_bf16(aux, lse, fused, grid, smem, st, P);
  else stage1_launch_f32(aux, lse, fused, grid, smem, st, P);
}

// The lean form (listed-token paths without count tables, no normaliser),
// launched before the full form for calls with history or bias lists; their
// P.dispatch makes exactly one of the two run.
const void* stage1_lean_ptr(bool bf16) { return bf16 ? stage1_ptr_bf16_lean() : stage1_ptr_f32_lean(); }

void stage1_launch_lean(bool bf16, int grid, size_t smem, cudaStream_t st, const Params& P) {
  if (bf16) stage1_launch_bf16_lean(grid, smem, st, P);
  else stage1_launch_f32_lean(grid, smem, st, P);
}

}  // namespace ss
