// q_prep.cu -- the q pre-step of the decode: q = ql_nope || q_pe along the
// last dim (the absorbed latent query and its rope part), written as bf16 or
// quantised to e4m3 with a static per-tensor scale (code = sat(round_rn(q /
// q_scale)), magnitudes above 448 saturated). One thread per 8 output columns.
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kChunks = kHeadDim / 8;        // 72 groups of 8 columns per row
constexpr int kNopeChunks = kRank / 8;       // 64 of them come from ql_nope

__global__ void __launch_bounds__(kThreads) concat_q_kernel(const QPrepParams p) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t rows = static_cast<int64_t>(p.num_tokens) * p.num_heads;
  if (i >= rows * kChunks) return;
  const int64_t row = i / kChunks;
  const int ch = static_cast<int>(i - row * kChunks);
  const int64_t t = row / p.num_heads;
  const int64_t h = row - t * p.num_heads;
  const __nv_bfloat16* src =
      ch < kNopeChunks
          ? static_cast<const __nv_bfloat16*>(p.nope) + t * p.nope_st + h * p.nope_sh + ch * 8
          : static_cast<const __nv_bfloat16*>(p.pe) + t * p.pe_st + h * p.pe_sh + (ch - kNopeChunks) * 8;
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
  if (!p.fp8) {
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + row * kHeadDim + ch * 8) = v;
    return;
  }
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t packed[2] = {0u, 0u};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    const float2 s = make_float2(f.x / p.q_scale, f.y / p.q_scale);
    const uint32_t c = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(s, __NV_SATFINITE, __NV_E4M3));
    packed[k >> 1] |= (c & 0xFFFFu) << ((k & 1) * 16);
  }
  *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * kHeadDim + ch * 8) =
      make_uint2(packed[0], packed[1]);
}

}  // namespace

cudaError_t launch_concat_q(const QPrepParams& p, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(p.num_tokens) * p.num_heads * kChunks;
  if (n == 0) return cudaSuccess;
  concat_q_kernel<<<static_cast<unsigned>((n + kThreads - 1) / kThreads), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
