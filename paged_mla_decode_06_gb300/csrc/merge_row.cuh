// merge_row.cuh -- one warp merges the base-2 partials of one (token, head)
// row into its bf16 output and natural-log LSE (rocm_aiter_mla_merge page,
// merge_mla_segments_triton): partial s sits at index base + s * stride of
// the max / expsum arrays and at that index times the row width in the
// outputs.
// Partials with expsum > 0 take part with weight l_s * 2^(m2_s - M), M the
// largest of their maxima and the sink's base-2 logit; the sink adds
// 2^(sink2 - M) to the denominator only. A row with no mass gets zeros and
// -inf. Coherent selects L2 loads (partials written by other CTAs of the
// same grid) instead of the read-only path.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace mla {

template <bool Coherent>
__device__ __forceinline__ float4 merge_load(const float4* p) {
  if constexpr (Coherent) return __ldcg(p);
  else return __ldg(p);
}

template <bool Coherent>
__device__ __forceinline__ float merge_load_f(const float* p) {
  if constexpr (Coherent) return __ldcg(p);
  else return __ldg(p);
}

// Rows of VPL * 128 values: lane i handles float4 i, i + 32, ...
template <int VPL, bool Coherent>
__device__ void merge_row(const float* segm_out, const float* segm_max, const float* segm_expsum,
                          int64_t base, int64_t stride, int live, float sink2, __nv_bfloat16* out,
                          float* lse, int lane) {
  // (unrolled so that the loads of several partials are in flight together)
  float M = -INFINITY;
#pragma unroll 4
  for (int s = 0; s < live; ++s) {
    const int64_t i = base + s * stride;
    if (merge_load_f<Coherent>(segm_expsum + i) > 0.f) M = fmaxf(M, merge_load_f<Coherent>(segm_max + i));
  }
  M = fmaxf(M, sink2);
  if (M == -INFINITY) {
#pragma unroll
    for (int v = 0; v < VPL; ++v)
      *reinterpret_cast<uint2*>(out + (v * 32 + lane) * 4) = make_uint2(0u, 0u);
    if (lane == 0) *lse = -INFINITY;
    return;
  }
  float acc[VPL][4];
#pragma unroll
  for (int v = 0; v < VPL; ++v) acc[v][0] = acc[v][1] = acc[v][2] = acc[v][3] = 0.f;
  float W = 0.f;
#pragma unroll 2
  for (int s = 0; s < live; ++s) {
    const int64_t i = base + s * stride;
    const float l = merge_load_f<Coherent>(segm_expsum + i);
    if (!(l > 0.f)) continue;
    const float w = l * exp2f(merge_load_f<Coherent>(segm_max + i) - M);
    W += w;
    const float4* src = reinterpret_cast<const float4*>(segm_out + i * (VPL * 128));
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      const float4 x = merge_load<Coherent>(src + v * 32 + lane);
      acc[v][0] += w * x.x;
      acc[v][1] += w * x.y;
      acc[v][2] += w * x.z;
      acc[v][3] += w * x.w;
    }
  }
  if (sink2 != -INFINITY) W += exp2f(sink2 - M);
  const float inv = 1.f / W;
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[v][0] * inv, acc[v][1] * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[v][2] * inv, acc[v][3] * inv);
    *reinterpret_cast<uint2*>(out + (v * 32 + lane) * 4) =
        make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
  if (lane == 0) *lse = kLn2 * (M + log2f(W));
}

}  // namespace mla
