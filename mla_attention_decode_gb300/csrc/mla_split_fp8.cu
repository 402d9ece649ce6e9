// mla_split_fp8.cu -- e4m3 KV: the tcgen05 split kernel.
#include "mla_tc.cuh"

namespace mla {
cudaError_t launch_stage1_fp8(const Stage1Params& p, cudaStream_t s) { return launch_split_tc<false>(p, s); }
}  // namespace mla
