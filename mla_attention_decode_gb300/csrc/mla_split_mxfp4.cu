// mla_split_mxfp4.cu -- instantiation of the split-K decode kernel for MXFP4 KV.
#include "mla_stage1.cuh"

namespace mla {
cudaError_t launch_stage1_mxfp4(const Stage1Params&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace mla
