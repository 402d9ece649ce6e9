// mla_split_fp8_t2.cu -- e4m3 KV, two query tokens per work unit: the tcgen05
// split kernel that reads each cache row once for both tokens of a sequence.
#include "mla_tc.cuh"

namespace mla {
cudaError_t launch_stage1_fp8_t2(const Stage1Params& p, cudaStream_t s) { return launch_split_tc<false, 2>(p, s); }
}  // namespace mla
