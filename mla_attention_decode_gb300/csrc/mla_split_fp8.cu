// mla_split_fp8.cu -- e4m3 KV: the tcgen05 split kernel (one query token per
// work unit; two-token plans go to the instance in mla_split_fp8_t2.cu).
#include "mla_tc.cuh"

namespace mla {
cudaError_t launch_stage1_fp8(const Stage1Params& p, cudaStream_t s) {
  return p.tok == 2 ? launch_stage1_fp8_t2(p, s) : launch_split_tc<false>(p, s);
}
}  // namespace mla
