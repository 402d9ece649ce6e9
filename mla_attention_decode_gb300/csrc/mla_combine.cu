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

// One CTA per (sequence, head, quarter of the 512 features); 128 threads.
// Warp w takes splits w, w + 4, ... for its 128 features (lane: 4 features),
// loading each split's lse and partial together, four splits in flight at a
// time, and keeps a running log-sum-exp against its own maximum; the four
// warps' sums meet in shared memory, rescaled to the common maximum.  After
// the split table, the latency is one L2 round trip whatever the split count.
__global__ void __launch_bounds__(128) mla_combine_kernel(const __grid_constant__ CombineParams p) {
  __shared__ float4 part[4][32];
  __shared__ float wpart[4], mpart[4];
  pdl_wait_primary();
  const int b = blockIdx.x >> 6, h = (blockIdx.x >> 2) & 15, quarter = blockIdx.x & 3;
  const int first = p.ws_seq[2 * b], ns = p.ws_seq[2 * b + 1];
  if (ns <= 1) return;  // written directly by the split kernel
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* lse = p.ws_lse + (size_t)first * kHeads + h;
  const int f = 128 * quarter + 4 * lane;
  const float* o = p.ws_o + ((size_t)first * kHeads + h) * kVDim + f;
  float m = -INFINITY;  // this warp's running maximum of the split lse values
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  for (int s0 = warp; s0 < ns; s0 += 16) {
    float l[4];
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int s = s0 + 4 * i;
      l[i] = s < ns ? lse[(size_t)s * kHeads] : -INFINITY;
      v[i] = s < ns ? *reinterpret_cast<const float4*>(o + (size_t)s * kHeads * kVDim) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float mb = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
    if (mb > m) {
      // the maximum rises: what was summed so far is rescaled to it
      const float c = m == -INFINITY ? 0.f : __expf(m - mb);
      acc.x *= c;
      acc.y *= c;
      acc.z *= c;
      acc.w *= c;
      wsum *= c;
      m = mb;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (l[i] == -INFINITY) continue;  // an empty split
      const float w = __expf(l[i] - m);
      acc.x += w * v[i].x;
      acc.y += w * v[i].y;
      acc.z += w * v[i].z;
      acc.w += w * v[i].w;
      wsum += w;
    }
  }
  part[warp][lane] = acc;
  if (lane == 0) {
    wpart[warp] = wsum;
    mpart[warp] = m;
  }
  __syncthreads();
  if (warp == 0) {
    const float M = fmaxf(fmaxf(mpart[0], mpart[1]), fmaxf(mpart[2], mpart[3]));
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    float ws = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (mpart[w] == -INFINITY) continue;  // no non-empty split in this warp
      const float c = __expf(mpart[w] - M);
      const float4 y = part[w][lane];
      t.x += c * y.x;
      t.y += c * y.y;
      t.z += c * y.z;
      t.w += c * y.w;
      ws += c * wpart[w];
    }
    const float inv = ws > 0.f ? 1.f / ws : 0.f;
    uint16_t* out = p.out + ((size_t)b * kHeads + h) * kVDim + f;
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16x2(t.x * inv, t.y * inv), pack_bf16x2(t.z * inv, t.w * inv));
    if (quarter == 0 && lane == 0 && p.lse) p.lse[b * kHeads + h] = ws > 0.f ? M + logf(ws) : -INFINITY;
  }
}

// Few splits per sequence (at most 4 in the plan): one CTA per (sequence, head)
// for all 512 features (thread t: features 4t .. 4t + 3), every split's lse and
// partial in flight at once; a quarter of the CTAs of the kernel above, no
// shared memory and no cross-warp step, so that one of its CTAs fits on each
// SM beside a split CTA and waits there (measured: 1.3 us off a bs64/kv8192
// call).  More splits than 4 (a device layout the plan did not see) are still
// summed, four at a time.
__global__ void __launch_bounds__(128) mla_combine_few_kernel(const __grid_constant__ CombineParams p) {
  pdl_wait_primary();
  const int b = blockIdx.x >> 4, h = blockIdx.x & 15;
  const int first = p.ws_seq[2 * b], ns = p.ws_seq[2 * b + 1];
  if (ns <= 1) return;  // written directly by the split kernel
  const int f = 4 * threadIdx.x;
  const float* lse = p.ws_lse + (size_t)first * kHeads + h;
  const float* o = p.ws_o + ((size_t)first * kHeads + h) * kVDim + f;
  float m = -INFINITY;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  for (int s0 = 0; s0 < ns; s0 += 4) {
    float l[4];
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int s = s0 + i;
      l[i] = s < ns ? lse[(size_t)s * kHeads] : -INFINITY;
      v[i] = s < ns ? *reinterpret_cast<const float4*>(o + (size_t)s * kHeads * kVDim) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float mb = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
    if (mb > m) {
      const float c = m == -INFINITY ? 0.f : __expf(m - mb);
      acc.x *= c;
      acc.y *= c;
      acc.z *= c;
      acc.w *= c;
      wsum *= c;
      m = mb;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (l[i] == -INFINITY) continue;  // an empty split
      const float w = __expf(l[i] - m);
      acc.x += w * v[i].x;
      acc.y += w * v[i].y;
      acc.z += w * v[i].z;
      acc.w += w * v[i].w;
      wsum += w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint16_t* out = p.out + ((size_t)b * kHeads + h) * kVDim + f;
  *reinterpret_cast<uint2*>(out) =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (threadIdx.x == 0 && p.lse) p.lse[b * kHeads + h] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.batch * kHeads * (p.few_splits ? 1 : 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.few_splits ? cudaLaunchKernelEx(&cfg, mla_combine_few_kernel, p)
                      : cudaLaunchKernelEx(&cfg, mla_combine_kernel, p);
}

}  // namespace mla
