// mla_split_mxfp4.cu -- MXFP4 KV: the tcgen05 split kernel with e2m1 -> e4m3
// conversion warps.
#include "mla_tc.cuh"

namespace mla {
cudaError_t launch_stage1_mxfp4(const Stage1Params& p, cudaStream_t s) { return launch_split_tc<true>(p, s); }
}  // namespace mla
