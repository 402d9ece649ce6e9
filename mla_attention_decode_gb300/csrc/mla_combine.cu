// mla_combine.cu -- log-sum-exp combine of split partials (sm_103a).
//
// For every sequence b that the plan split into S_b > 1 units and every head h
// (kernelindex "amd-mixed-mla" submission 593653, stage-2 kernel
// "_flash_fp8_split_s2", written here in closed form like submission 703488's
// "_reduce_splitk_parallel" kernels):
//   M = max_s lse_s,  w_s = exp(lse_s - M),
//   out[b,h,:] = sum_s w_s o_s / sum_s w_s,   lse[b,h] = M + ln(sum_s w_s),
// skipping splits whose lse is -inf.  o_s are the normalised fp32 partials the
// split kernel left in the workspace.  Launched with programmatic dependent
// launch: the CTAs may start early and block in griddepcontrol.wait until the
// split kernel has completed and its writes are visible.
#include <cuda_runtime.h>

#include "mla_internal.h"
#include "mla_ptx.cuh"

namespace mla {

// One CTA per (sequence, head); 128 threads, 4 output features each.
__global__ void __launch_bounds__(128) mla_combine_kernel(const __grid_constant__ CombineParams p) {
  pdl_wait_primary();
  const int b = blockIdx.x / kHeads, h = blockIdx.x % kHeads;
  const int first = p.ws_seq[2 * b], ns = p.ws_seq[2 * b + 1];
  if (ns <= 1) return;  // written directly by the split kernel
  const float* lse = p.ws_lse + (size_t)first * kHeads + h;
  float m = -INFINITY;
  for (int s = 0; s < ns; ++s) m = fmaxf(m, lse[(size_t)s * kHeads]);
  const int f = 4 * threadIdx.x;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (m != -INFINITY) {
    const float* o = p.ws_o + ((size_t)first * kHeads + h) * kVDim + f;
    for (int s = 0; s < ns; ++s) {
      const float l = lse[(size_t)s * kHeads];
      if (l == -INFINITY) continue;
      const float w = __expf(l - m);
      const float4 v = *reinterpret_cast<const float4*>(o + (size_t)s * kHeads * kVDim);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
      wsum += w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint16_t* out = p.out + ((size_t)b * kHeads + h) * kVDim + f;
  *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (threadIdx.x == 0 && p.lse) p.lse[b * kHeads + h] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.batch * kHeads);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_combine_kernel, p);
}

}  // namespace mla
