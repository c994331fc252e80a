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

// Rows of VPL * 128 values: lane i handles float4 i, i + 32, ... . The
// (max, expsum) pairs of the first kMeta partials are loaded together and
// kept; the outputs of four partials at a time are loaded together, so that a
// row costs about two memory round trips.
constexpr int kMeta = 8;

template <int VPL, bool Coherent>
__device__ void merge_row(const float* segm_out, const float* segm_max, const float* segm_expsum,
                          int64_t base, int64_t stride, int live, float sink2, __nv_bfloat16* out,
                          float* lse, int lane) {
  float lk[kMeta], mk[kMeta];
#pragma unroll
  for (int u = 0; u < kMeta; ++u) {
    lk[u] = u < live ? merge_load_f<Coherent>(segm_expsum + base + u * stride) : 0.f;
    mk[u] = u < live ? merge_load_f<Coherent>(segm_max + base + u * stride) : -INFINITY;
  }
  // the outputs of the first four partials are loaded with no wait for their
  // weights (one memory round trip instead of two); a partial that carries
  // no mass (possibly never written: stale or NaN) is excluded by select
  float4 x0[4][VPL];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float4* src = reinterpret_cast<const float4*>(segm_out + (base + u * stride) * (VPL * 128));
#pragma unroll
    for (int v = 0; v < VPL; ++v)
      x0[u][v] = u < live ? merge_load<Coherent>(src + v * 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float M = sink2;
#pragma unroll
  for (int u = 0; u < kMeta; ++u)
    if (lk[u] > 0.f) M = fmaxf(M, mk[u]);
  for (int s = kMeta; s < live; ++s) {
    const int64_t i = base + s * stride;
    if (merge_load_f<Coherent>(segm_expsum + i) > 0.f) M = fmaxf(M, merge_load_f<Coherent>(segm_max + i));
  }
  float acc[VPL][4];
#pragma unroll
  for (int v = 0; v < VPL; ++v) acc[v][0] = acc[v][1] = acc[v][2] = acc[v][3] = 0.f;
  float W = 0.f;
  if (M == -INFINITY) {
#pragma unroll
    for (int v = 0; v < VPL; ++v)
      *reinterpret_cast<uint2*>(out + (v * 32 + lane) * 4) = make_uint2(0u, 0u);
    if (lane == 0) *lse = -INFINITY;
    return;
  }
  // weight of partial s (its (max, expsum) pair from the first kMeta kept in
  // registers, else loaded)
  auto weight = [&](int s) {
    float l = 0.f, m = 0.f;
    if (s < kMeta) {
#pragma unroll
      for (int k = 0; k < kMeta; ++k)
        if (k == s) { l = lk[k]; m = mk[k]; }
    } else if (s < live) {
      l = merge_load_f<Coherent>(segm_expsum + base + s * stride);
      m = merge_load_f<Coherent>(segm_max + base + s * stride);
    }
    return l > 0.f ? l * exp2f(m - M) : 0.f;
  };
  auto add = [&](float wu, const float4 (&xu)[VPL]) {
    W += wu;
    if (wu != 0.f) {
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        acc[v][0] += wu * xu[v].x;
        acc[v][1] += wu * xu[v].y;
        acc[v][2] += wu * xu[v].z;
        acc[v][3] += wu * xu[v].w;
      }
    }
  };
#pragma unroll
  for (int u = 0; u < 4; ++u) add(weight(u), x0[u]);
  for (int s0 = 4; s0 < live; s0 += 4) {
    float w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) w[u] = weight(s0 + u);
    float4 x[4][VPL];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4* src = reinterpret_cast<const float4*>(segm_out + (base + (s0 + u) * stride) * (VPL * 128));
#pragma unroll
      for (int v = 0; v < VPL; ++v)
        x[u][v] = w[u] != 0.f ? merge_load<Coherent>(src + v * 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) add(w[u], x[u]);
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
