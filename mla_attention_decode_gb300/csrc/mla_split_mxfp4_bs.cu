// mla_split_mxfp4_bs.cu -- MXFP4 KV with the scores from block-scaled tensor-core
// MMAs (kind::mxf8f6f4, e2m1 K tile x e4m3 query, the cache's e8m0 block scales
// as the A scale factors) read straight from the TMA-loaded tile; the converter
// warps rewrite only the 512 V features as e4m3 for the P.V.
#include "mla_tc.cuh"

namespace mla {
cudaError_t launch_stage1_mxfp4_bs(const Stage1Params& p, cudaStream_t s) {
  return launch_split_tc<true, 1, tcfp8::kPathBlockScaled>(p, s);
}
}  // namespace mla
