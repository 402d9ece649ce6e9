// mla_split_fp8.cu -- e4m3 KV: the tcgen05 split kernel (one query token per
// work unit; two-token plans go to the instance in mla_split_fp8_t2.cu, and
// paged caches with pages of fewer than 64 rows to mla_split_small_pages.cu).
#include "mla_tc.cuh"

namespace mla {
cudaError_t launch_stage1_fp8(const Stage1Params& p, cudaStream_t s) {
  if (p.tok == 2) return launch_stage1_fp8_t2(p, s);
  if (p.paged && p.page_shift < 6) return launch_stage1_small_pages(p, false, s);
  return launch_split_tc<false>(p, s);
}
}  // namespace mla
