// mla_split_mxfp4.cu -- MXFP4 KV: the tcgen05 split kernel with e2m1 -> e4m3
// conversion warps (pages of fewer than 64 rows: mla_split_small_pages.cu;
// scores by block-scaled MMAs: mla_split_mxfp4_bs.cu).
#include "mla_tc.cuh"

namespace mla {
cudaError_t launch_stage1_mxfp4(const Stage1Params& p, cudaStream_t s) {
  if (p.paged && p.page_shift < 6) return launch_stage1_small_pages(p, true, s);
  if (p.mx_bs) return launch_stage1_mxfp4_bs(p, s);
  return launch_split_tc<true>(p, s);
}
}  // namespace mla
