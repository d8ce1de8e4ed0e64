// The stage-2 kernel: one position per CTA iteration (persistent CTAs of
// 128 threads, one per candidate); the per-position work is
// stage2_position (ss_stage2.cuh), which the fused stage-1 form also runs.
#include "ss_stage2.cuh"

namespace ss {

__global__ void __launch_bounds__(kNT2, 9) stage2_kernel(const Params P, int verify) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int cap = P.seg_cap * kK;  // the lists of one position (at most seg_cap of them)
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(smem_raw);
  unsigned long long* tmp = cand + cap;
  S2Smem& sm = *reinterpret_cast<S2Smem*>(tmp + cap);
  const int npos = num_positions(P);
  const Split sp = make_split(P, npos);
  for (int pos = blockIdx.x; pos < npos; pos += gridDim.x) stage2_position<kNT2>(P, verify, pos, sp, cand, tmp, sm);
  stage2_capacity_rows<kNT2>(P, verify, blockIdx.x, gridDim.x);
}

size_t stage2_smem_bytes(int Z) { return stage2_smem_for(Z); }

int stage2_threads() { return kNT2; }

}  // namespace ss
