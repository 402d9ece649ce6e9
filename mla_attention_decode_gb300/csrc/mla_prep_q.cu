// mla_prep_q.cu -- the two-term e4m3 query of every sequence, prepared once per
// call for the tcgen05 split kernel (e4m3 and MXFP4 KV).
//
// The tcgen05 MMA of kind::f8f6f4 takes 8-bit operands, so the bf16 query row
// of sequence b (kernelindex "amd-mixed-mla" submission 593653, "Slow
// fallback": q[qo_indptr[b], h, :576]) is carried as x = 2^-s_h (hi + lo) with
// hi = e4m3(2^s_h x), lo = e4m3(2^s_h x - hi) and a power-of-two scale 2^s_h
// per head (amax * 2^s_h <= 448).  This kernel writes, per sequence, the
// 32 x 576 B image (rows h: hi, rows 16 + h: lo; K-major, 64-byte swizzle)
// that the split kernel copies into shared memory unchanged, and the 16 score
// factors sm_scale * log2(e) * kv_scale * 2^-s_h (kv_scale = 1 for MXFP4).
//
// It runs ahead of the split kernel (programmatic dependent launch): it waits
// for the previous kernel, then lets the split kernel start its set-up, which
// reads the prepared queries only after this grid has completed.
#include <cuda_runtime.h>

#include "mla_common.cuh"

namespace mla {

// One CTA of 128 threads per sequence: thread j handles head j/8, features
// [72 (j%8), 72 (j%8) + 72), all nine 16-byte loads in flight for the head
// maximum, then the same row again (L1 hits) for the conversion, in 53
// registers.  Measured against one CTA of 64 threads at 174 registers (a
// thread per 144 features): calls 1.4-1.9 us faster at bs32/kv1024 and
// bs64/kv8192.  The split CTAs placed on this grid's SMs still start when its
// CTAs have finished (a per-CTA trace shows them entering about 3.3 us late).
template <bool kMx>
__global__ void __launch_bounds__(128, 9) mla_prep_q_kernel(const __grid_constant__ Stage1Params p) {
  if (threadIdx.x == 0) trace_stamp(p, kTrPrepEntry);
  pdl_wait_primary();      // q and qo_indptr written by earlier work are visible
  pdl_launch_dependents();  // the split kernel may begin its set-up
  if (threadIdx.x == 0) trace_stamp(p, kTrPrepWaited);
  const int b = blockIdx.x, j = threadIdx.x;
  const int qrow = query_row(p, b);
  // bring the sequence's kv_indptr entries into L2 for the split kernel's unit
  // scan (the comparison only keeps the load; offsets are never negative)
  if (j == 0 && __ldg(p.kv_indptr + (p.q_len > 1 ? b / p.q_len : b)) < 0) p.ws_err[1] = 1;
  if (qrow < 0) return;  // the split kernel reports the bad index
  const int h = j >> 3, part = j & 7;  // 8 threads per head, 72 features each
  const float kv_scale = kMx ? 1.f : *static_cast<const float*>(p.kv_scale);
  const uint4* src = reinterpret_cast<const uint4*>(p.q + (((size_t)qrow * kHeads + h) * kQkDim + 72 * part) * 2);
  float amax = 0.f;
  {
    uint4 raw[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) raw[i] = __ldg(src + i);
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const float4 a = bf16x4_to_f4(make_uint2(raw[i].x, raw[i].y));
      const float4 c = bf16x4_to_f4(make_uint2(raw[i].z, raw[i].w));
      amax = fmaxf(amax, fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                               fmaxf(fmaxf(fabsf(c.x), fabsf(c.y)), fmaxf(fabsf(c.z), fabsf(c.w)))));
    }
  }
  amax = quad_max(amax);  // over the head's 8 threads
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  // power-of-two scale with amax * scale <= 448 (e4m3 max); 1 for an all-zero head
  float sc = 1.f;
  if (amax > 0.f) {
    sc = exp2f(floorf(log2f(448.f / amax)));
    if (amax * sc > 448.f) sc *= 0.5f;
  }
  uint8_t* dst = p.ws_q + (size_t)b * kQPrepBytes;
#pragma unroll 3
  for (int i = 0; i < 9; ++i) {
    const int f0 = 72 * part + 8 * i;  // 8 features, inside one 16-byte unit of a 64-byte block
    const uint4 r = __ldg(src + i);
    const float4 a = bf16x4_to_f4(make_uint2(r.x, r.y));
    const float4 c = bf16x4_to_f4(make_uint2(r.z, r.w));
    uint32_t hi0, lo0, hi1, lo1;
    two_term_e4m3(a.x * sc, a.y * sc, a.z * sc, a.w * sc, hi0, lo0);
    two_term_e4m3(c.x * sc, c.y * sc, c.z * sc, c.w * sc, hi1, lo1);
    const int blk = f0 >> 6, col = f0 & 63;
    *reinterpret_cast<uint2*>(dst + blk * 2048 + sw64_off(h, col)) = make_uint2(hi0, hi1);
    *reinterpret_cast<uint2*>(dst + blk * 2048 + sw64_off(16 + h, col)) = make_uint2(lo0, lo1);
  }
  if (part == 0) reinterpret_cast<float*>(dst + kQImageBytes)[h] = p.sm_scale * kLog2e * kv_scale / sc;
#if MLA_TRACE
  __syncthreads();
  if (threadIdx.x == 0) trace_stamp(p, kTrPrepDone);
#endif
}

cudaError_t launch_prep_q(const Stage1Params& p, bool mx, cudaStream_t s) {
  if (p.batch <= 0) return cudaSuccess;
  cudaError_t e = mx ? launch_overlapped(mla_prep_q_kernel<true>, dim3(p.batch), dim3(128), 0, s, p)
                     : launch_overlapped(mla_prep_q_kernel<false>, dim3(p.batch), dim3(128), 0, s, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
