// mla_split_bf16.cu -- instantiation of the split-K decode kernel for bf16 KV.
#include "mla_stage1.cuh"

namespace mla {
cudaError_t launch_stage1_bf16(const Stage1Params& p, cudaStream_t s) { return launch_split<0>(p, s); }
}  // namespace mla
