// mla_split_small_pages.cu -- the tcgen05 split kernel for paged caches whose
// pages hold fewer than 64 rows (e4m3 and MXFP4, one token per sequence): a
// tile's rows lie in several pages, so the producer warp fetches them with
// per-page lookups (four-row TMA gathers for e4m3, one bulk copy per packed row
// for MXFP4).  A separate instance, so that the contiguous-cache kernels carry
// none of this code.
#include "mla_tc.cuh"

namespace mla {
cudaError_t launch_stage1_small_pages(const Stage1Params& p, bool mx, cudaStream_t s) {
  return mx ? launch_split_tc<true, 1, tcfp8::kPathSmallPages>(p, s)
            : launch_split_tc<false, 1, tcfp8::kPathSmallPages>(p, s);
}
}  // namespace mla
