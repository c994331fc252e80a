// merge.cu -- merge split-K segment partials into the output and a
// natural-log LSE (rocm_aiter_mla_merge page, merge_mla_segments_triton).
//
// One warp per (token, head). The token's partition length and the tile size
// give the segments that exist (start < len, tiles_per_segment =
// cdiv(len, NS * tile)); of those, segments with expsum > 0 contribute.
// Under the balanced schedule the row's pieces come from the unit table
// instead, and rows whose unit was not split are left as the decode kernel
// wrote them.
// Pass 1 reads the base-2 maxima, pass 2 streams each live segment's
// normalised output coalesced (lane i reads float4 i, i + 32, ...) and
// accumulates it with weight l_s * 2^(m2_s - M). The sink logit, when given,
// adds 2^(sink * log2 e - M) to the denominator only.
#include <cfloat>

#include "common.cuh"
#include "internal.h"
#include "merge_row.cuh"

namespace mla {
namespace {

constexpr int kWarpsPerBlock = 4;

// Request of token t: the last r with qo_indptr[r] <= t.
__device__ __forceinline__ int request_of(const PartLens& pl, int t) {
  int lo = 0, hi = pl.num_reqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pl.qo_indptr[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int part_len_of(const PartLens& pl, int t) {
  switch (pl.mode) {
    case 0: return pl.lens[t];
    case 1: return pl.qo_indptr == nullptr ? pl.seq_lens[t] : pl.seq_lens[request_of(pl, t)];
    case 2: return pl.indptr[t + 1] - pl.indptr[t];
    default: return pl.constant;
  }
}

template <int VPL>  // float4 values per lane: rank / 128
__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_kernel(const MergeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t total = static_cast<int64_t>(p.num_tokens) * p.num_heads;
  if (gw >= total) return;
  const int t = static_cast<int>(gw / p.num_heads);
  const int h = static_cast<int>(gw % p.num_heads);
  const float sink2 = p.sinks != nullptr ? p.sinks[h] * kLog2e : -INFINITY;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + gw * p.rank;
  if (p.unit_tab != nullptr) {
    // balanced schedule: the rows of a (unit, row tile) split into k > 1
    // pieces own k consecutive slots of tile_rows rows; k == 1 rows were
    // written by the decode kernel itself. The unit table comes from the
    // schedule kernel, which completed before the decode began, so it is
    // read while the decode (this grid's programmatic primary) may still
    // run, and a row that was not split leaves at once; only the partials
    // wait for the decode to complete.
    int u = t, tok0 = t;
    if (!p.sparse && p.part.qo_indptr != nullptr) {
      u = request_of(p.part, t);
      tok0 = p.part.qo_indptr[u];
    }
    const int r = (t - tok0) * p.num_heads + h;
    const int tr = p.tile_rows;
    int2 e = make_int2(-1, 0);
    if (r / tr < p.tiles_max)
      e = reinterpret_cast<const int2*>(p.unit_tab)[static_cast<int64_t>(u) * p.tiles_max + r / tr];
    if (e.y <= 1) return;
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    merge_row<VPL, true>(p.segm_out, p.segm_max, p.segm_expsum, static_cast<int64_t>(e.x) * tr + r % tr,
                         tr, e.y, sink2, out, p.lse + gw, lane);
    return;
  }
  // uniform partition: an ordinary launch (the wait is a no-op)
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const int NS = p.num_segments;
  const int len = part_len_of(p.part, t);
  const int span = NS * p.tile_size;
  const int tps = len > 0 ? cdiv(len, span) : 0;
  const int seg = tps * p.tile_size;
  const int live = len > 0 ? min(NS, cdiv(len, seg)) : 0;
  merge_row<VPL, false>(p.segm_out, p.segm_max, p.segm_expsum, gw * NS, 1, live, sink2, out, p.lse + gw,
                        lane);
}

// Natural-log (out, lse) pairs of W key shards of the same rows: weights
// e^(lse_w - M), one warp per (token, head), bf16 shard outputs read 8 bytes
// per lane per step (coalesced).
template <int VPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_lse_kernel(const LseMergeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t rows = static_cast<int64_t>(p.num_tokens) * p.num_heads;
  if (gw >= rows) return;
  const int h = static_cast<int>(gw % p.num_heads);
  float M = -INFINITY;
  for (int w = 0; w < p.num_shards; ++w) M = fmaxf(M, p.shard_lse[w * rows + gw]);
  const bool has_sink = p.sinks != nullptr;
  const float sink = has_sink ? p.sinks[h] : -INFINITY;
  M = fmaxf(M, sink);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + gw * p.rank;
  if (M == -INFINITY) {
#pragma unroll
    for (int v = 0; v < VPL; ++v)
      *reinterpret_cast<uint2*>(out + (v * 32 + lane) * 4) = make_uint2(0u, 0u);
    if (lane == 0) p.lse[gw] = -INFINITY;
    return;
  }
  float acc[VPL][4];
#pragma unroll
  for (int v = 0; v < VPL; ++v) acc[v][0] = acc[v][1] = acc[v][2] = acc[v][3] = 0.f;
  float Z = 0.f;
  for (int w = 0; w < p.num_shards; ++w) {
    const float l = p.shard_lse[w * rows + gw];
    if (l == -INFINITY) continue;
    const float e = expf(l - M);
    Z += e;
    const uint2* src = reinterpret_cast<const uint2*>(
        static_cast<const __nv_bfloat16*>(p.shard_out) + (w * rows + gw) * p.rank);
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      const uint2 x = __ldg(src + v * 32 + lane);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
      acc[v][0] += e * a.x;
      acc[v][1] += e * a.y;
      acc[v][2] += e * b.x;
      acc[v][3] += e * b.y;
    }
  }
  if (has_sink) Z += expf(sink - M);
  const float inv = 1.f / Z;
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[v][0] * inv, acc[v][1] * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[v][2] * inv, acc[v][3] * inv);
    *reinterpret_cast<uint2*>(out + (v * 32 + lane) * 4) =
        make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
  if (lane == 0) p.lse[gw] = M + logf(Z);
}

}  // namespace

cudaError_t launch_merge_lse(const LseMergeParams& p, cudaStream_t stream) {
  const int64_t warps = static_cast<int64_t>(p.num_tokens) * p.num_heads;
  if (warps == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
  switch (p.rank / 128) {
    case 1: merge_lse_kernel<1><<<blocks, kWarpsPerBlock * 32, 0, stream>>>(p); break;
    case 2: merge_lse_kernel<2><<<blocks, kWarpsPerBlock * 32, 0, stream>>>(p); break;
    case 4: merge_lse_kernel<4><<<blocks, kWarpsPerBlock * 32, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
  const int64_t warps = static_cast<int64_t>(p.num_tokens) * p.num_heads;
  if (warps == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
  if (p.unit_tab != nullptr) {
    // balanced schedule: programmatic dependent launch after the decode, so
    // that the grid is in place when the decode completes
    if (p.rank != 512) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(blocks, 1, 1);
    cfg.blockDim = dim3(kWarpsPerBlock * 32, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_kernel<4>, p);
  }
  switch (p.rank / 128) {
    case 1: merge_kernel<1><<<blocks, kWarpsPerBlock * 32, 0, stream>>>(p); break;
    case 2: merge_kernel<2><<<blocks, kWarpsPerBlock * 32, 0, stream>>>(p); break;
    case 4: merge_kernel<4><<<blocks, kWarpsPerBlock * 32, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mla
