// decode_mma.cu -- split-K paged MLA decode on warp-level tensor-core MMAs.
//
// One CTA owns (row tile, segment, unit). A unit is a request (dense: all of
// its qlen x H query rows share one pass over its KV) or a token (sparse:
// its own slot list). Rows are (token, head) pairs, 16 x RG per CTA. The
// CTA walks its segment of the key list in chunks of KC keys:
//   gather   cp.async 16-byte pieces of each 576-wide row, located through
//            the block table (dense) or the slot list (sparse), into a
//            STAGES-deep shared-memory ring; keys outside the segment or
//            with slot -1 are zero-filled and never read from global memory;
//   QK^T     S[rows, KC] = Q[rows, 576] . K^T, fp32 accumulation;
//   softmax  base-2 online softmax with per-row running max m and sum l;
//            masked keys (outside the segment, past the row's causal end,
//            invalid sparse slot) score -inf;
//   P.V      O[rows, 512] += P[rows, KC] . V[KC, 512] where V is the first
//            512 columns of the same shared-memory rows.
// bf16 inputs use bf16 MMAs; e4m3 inputs are widened exactly to f16 in
// shared memory and use f16 MMAs (scores are rescaled by q_scale * kv_scale,
// values by kv_scale).
//
// Epilogue: either the segment's base-2 partials (m2, l, O / l), the format
// of the rocm_aiter_mla_merge page, or -- when the whole row is one segment
// -- the final bf16 output and natural-log LSE with the sink folded into
// the denominator (rocm_aiter_mla_sparse page, _forward_mla).
//
// Warp layout: 8 warps; warp w serves row group w % RG and column slice
// w / RG: in QK^T a slice of the chunk's keys, in P.V a slice of the 512
// value columns. Row maxima and sums are combined through shared memory.
#include <atomic>
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kQStride = kHeadDim + 8;   // 16-bit elements per smem row (1168 B, conflict-free)
constexpr int kRawStride = kHeadDim + 16;  // bytes per raw fp8 smem row

template <int RG, bool FP8>
struct Cfg {
  static constexpr int kRows = 16 * RG;
  static constexpr int kCS = kWarps / RG;            // warps sharing a row group
  static constexpr int kKC = (RG == 1) ? 64 : 32;    // keys per chunk
  static constexpr int kStages = FP8 ? (RG == 1 ? 3 : 4) : (RG == 1 ? 2 : 3);
  static constexpr int kKW = kKC / kCS;              // keys per warp in QK^T
  static constexpr int kNTS = kKW / 8;
  static constexpr int kVW = kRank / kCS;            // value columns per warp in P.V
  static constexpr int kNTV = kVW / 8;
  static constexpr int kPStride = kKC + 8;           // 16-bit elements per P row
  static constexpr int kPieces = FP8 ? kHeadDim / 16 : kHeadDim * 2 / 16;  // 16-B pieces per row
  static constexpr int kQBytes = kRows * kQStride * 2;
  static constexpr int kStageBytes = FP8 ? kKC * kRawStride : kKC * kQStride * 2;
  static constexpr int kComputeBytes = FP8 ? kKC * kQStride * 2 : 0;
  static constexpr int kPBytes = kRows * kPStride * 2;
  static constexpr int kRedBytes = RG * kCS * 16 * 4;
  static constexpr int kOkBytes = kStages * kKC * 4;
  static constexpr int kOffStage = kQBytes;
  static constexpr int kOffCompute = kOffStage + kStages * kStageBytes;
  static constexpr int kOffP = kOffCompute + kComputeBytes;
  static constexpr int kOffRed = kOffP + kPBytes;
  static constexpr int kOffOk = kOffRed + kRedBytes;
  static constexpr int kSmem = kOffOk + kOkBytes;
  static_assert(kNTS >= 1 && kKW % 8 == 0, "key slice per warp must be whole n-tiles");
  static_assert(kNTV % 2 == 0, "value slice must be an even number of n-tiles");
  static_assert(kSmem <= 232448, "shared memory budget");
};

template <int RG, bool FP8>
__global__ void __launch_bounds__(kThreads, 1) decode_mma_kernel(const DecodeParams p) {
  using C = Cfg<RG, FP8>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int rg = warp % RG;
  const int cs = warp / RG;
  const int tile = blockIdx.x;
  const int seg = blockIdx.y;
  const int unit = blockIdx.z;
  const int H = p.num_heads;
  const bool sparse = p.slots != nullptr;

  // ---------------------------------------------------------------- unit
  int qlen = 1, tok0 = unit, part_len = 0;
  int64_t list_base = 0;
  const int32_t* bt_row = nullptr;
  if (!sparse) {
    if (p.qo_indptr != nullptr) {
      tok0 = p.qo_indptr[unit];
      qlen = p.qo_indptr[unit + 1] - tok0;
    }
    part_len = p.seq_lens[unit];
    bt_row = p.block_table + static_cast<int64_t>(unit) * p.bt_stride;
  } else if (p.slot_indptr != nullptr) {
    list_base = p.slot_indptr[unit];
    part_len = p.slot_indptr[unit + 1] - p.slot_indptr[unit];
  } else {
    list_base = static_cast<int64_t>(unit) * p.topk;
    part_len = p.topk;
  }
  const int rows_total = qlen * H;
  const int row0 = tile * C::kRows;
  if (row0 >= rows_total) return;  // whole CTA: this request has fewer rows

  // Segment of the partition: tps = cdiv(len, NS * tile).
  const int span = p.num_segments * p.tile_size;
  const int tps = part_len > 0 ? cdiv(part_len, span) : 0;
  const int seg_len = tps * p.tile_size;
  const int seg_start = seg * seg_len;
  const int seg_end = min(seg_start + seg_len, part_len);
  const int n_chunks = seg_end > seg_start ? cdiv(seg_end - seg_start, C::kKC) : 0;

  uint8_t* sQ = smem;
  uint8_t* sP = smem + C::kOffP;
  float* red = reinterpret_cast<float*>(smem + C::kOffRed);
  int* key_ok = reinterpret_cast<int*>(smem + C::kOffOk);

  // Rows of this thread: r_a = rg*16 + lane/4 and r_a + 8 (within the tile).
  const int ra = rg * 16 + (lane >> 2);
  int vis[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int rho = row0 + ra + 8 * i;
    const int j = rho / H;
    vis[i] = (rho >= rows_total) ? 0 : (sparse ? INT_MAX : part_len - qlen + j + 1);
  }

  // ---------------------------------------------------------------- Q
  const uint8_t* qbytes = static_cast<const uint8_t*>(p.q);
  if constexpr (!FP8) {
    for (int i = tid; i < C::kRows * 72; i += kThreads) {
      const int r = i / 72, part = i % 72;
      const int rho = row0 + r;
      const bool ok = rho < rows_total;
      const int64_t qrow = ok ? (static_cast<int64_t>(tok0 + rho / H) * H + rho % H) : 0;
      cp_async_16(smem_u32(sQ + r * kQStride * 2 + part * 16), qbytes + qrow * kHeadDim * 2 + part * 16,
                  ok ? 16u : 0u);
    }
    cp_async_commit();
  } else {
    for (int i = tid; i < C::kRows * 36; i += kThreads) {
      const int r = i / 36, part = i % 36;
      const int rho = row0 + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (rho < rows_total) {
        const int64_t qrow = static_cast<int64_t>(tok0 + rho / H) * H + rho % H;
        v = *reinterpret_cast<const uint4*>(qbytes + qrow * kHeadDim + part * 16);
      }
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t h[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        h[2 * k] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xFFFF));
        h[2 * k + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16));
      }
      uint4* dst = reinterpret_cast<uint4*>(sQ + r * kQStride * 2 + part * 32);
      dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
      dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }

  // ---------------------------------------------------------------- KV gather
  const uint8_t* kvbytes = static_cast<const uint8_t*>(p.kv);
  const int64_t row_bytes = FP8 ? kHeadDim : kHeadDim * 2;
  const int bs = p.block_size;
  auto load_chunk = [&](int c, int stage) {
    const int c0 = seg_start + c * C::kKC;
    uint8_t* dst = smem + C::kOffStage + stage * C::kStageBytes;
    int* ok = key_ok + stage * C::kKC;
    constexpr int kRowStrideB = FP8 ? kRawStride : kQStride * 2;
    for (int i = tid; i < C::kKC * C::kPieces; i += kThreads) {
      const int k = i / C::kPieces, part = i % C::kPieces;
      const int pos = c0 + k;
      int64_t slot = -1;
      if (pos < seg_end) {
        if (!sparse) {
          const int blk = pos / bs;
          slot = static_cast<int64_t>(bt_row[blk]) * bs + (pos - blk * bs);
        } else {
          slot = p.slots[list_base + pos];
        }
      }
      const bool live = slot >= 0;
      cp_async_16(smem_u32(dst + k * kRowStrideB + part * 16),
                  live ? kvbytes + slot * row_bytes + part * 16 : kvbytes, live ? 16u : 0u);
      if (part == 0) ok[k] = live ? 1 : 0;
    }
  };

#pragma unroll
  for (int s = 0; s < C::kStages - 1; ++s) {
    if (s < n_chunks) load_chunk(s, s);
    cp_async_commit();
  }

  float o[C::kNTV][4];
#pragma unroll
  for (int n = 0; n < C::kNTV; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  const float scale2 = p.score_scale_log2;

  const uint32_t sQ_u32 = smem_u32(sQ);
  const uint32_t sP_u32 = smem_u32(sP);

  for (int c = 0; c < n_chunks; ++c) {
    cp_async_wait<C::kStages - 2>();
    __syncthreads();
    const int stage = c % C::kStages;
    {
      const int nc = c + C::kStages - 1;
      if (nc < n_chunks) load_chunk(nc, nc % C::kStages);
      cp_async_commit();
    }
    const uint8_t* kvs;
    if constexpr (FP8) {
      const uint8_t* raw = smem + C::kOffStage + stage * C::kStageBytes;
      uint8_t* comp = smem + C::kOffCompute;
      for (int i = tid; i < C::kKC * 36; i += kThreads) {
        const int k = i / 36, part = i % 36;
        const uint4 v = *reinterpret_cast<const uint4*>(raw + k * kRawStride + part * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          h[2 * e] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[e] & 0xFFFF));
          h[2 * e + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[e] >> 16));
        }
        uint4* d = reinterpret_cast<uint4*>(comp + k * kQStride * 2 + part * 32);
        d[0] = make_uint4(h[0], h[1], h[2], h[3]);
        d[1] = make_uint4(h[4], h[5], h[6], h[7]);
      }
      __syncthreads();
      kvs = comp;
    } else {
      kvs = smem + C::kOffStage + stage * C::kStageBytes;
    }
    const uint32_t kv_u32 = smem_u32(kvs);
    const int* ok = key_ok + stage * C::kKC;

    // ---- S = Q K^T for rows of group rg, keys [cs*KW, cs*KW + KW)
    float sacc[C::kNTS][4];
#pragma unroll
    for (int n = 0; n < C::kNTS; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
    const uint32_t qa = sQ_u32 + ((rg * 16 + (lane & 15)) * kQStride + (lane >> 4) * 8) * 2;
    const uint32_t kb = kv_u32 + ((cs * C::kKW + (lane & 7)) * kQStride + ((lane >> 3) & 1) * 8) * 2;
#pragma unroll 4
    for (int ks = 0; ks < kHeadDim / 16; ++ks) {
      uint32_t a[4];
      ldmatrix_x4(qa + ks * 32, a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int n = 0; n < C::kNTS; ++n) {
        uint32_t b0, b1;
        ldmatrix_x2(kb + (n * 8 * kQStride) * 2 + ks * 32, b0, b1);
        mma_16816<FP8>(sacc[n], a, b0, b1);
      }
    }

    // ---- mask, chunk max
    const int c0 = seg_start + c * C::kKC;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < C::kNTS; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kl = cs * C::kKW + n * 8 + 2 * (lane & 3) + e;
        const int pos = c0 + kl;
        const bool live = ok[kl] != 0;
        const float s0 = (live && pos < vis[0]) ? sacc[n][e] * scale2 : -INFINITY;
        const float s1 = (live && pos < vis[1]) ? sacc[n][2 + e] * scale2 : -INFINITY;
        sacc[n][e] = s0;
        sacc[n][2 + e] = s1;
        mx[0] = fmaxf(mx[0], s0);
        mx[1] = fmaxf(mx[1], s1);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
    }
    if ((lane & 3) == 0) {
      red[(rg * C::kCS + cs) * 16 + (lane >> 2)] = mx[0];
      red[(rg * C::kCS + cs) * 16 + (lane >> 2) + 8] = mx[1];
    }
    __syncthreads();
    float base[2], alpha[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float cm = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::kCS; ++w) cm = fmaxf(cm, red[(rg * C::kCS + w) * 16 + (lane >> 2) + 8 * i]);
      const float mn = fmaxf(m_run[i], cm);
      base[i] = (mn == -INFINITY) ? 0.f : mn;
      alpha[i] = fast_exp2(m_run[i] - base[i]);
      m_run[i] = mn;
    }

    // ---- P = 2^(s - m), to shared memory
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < C::kNTS; ++n) {
      const float p00 = fast_exp2(sacc[n][0] - base[0]);
      const float p01 = fast_exp2(sacc[n][1] - base[0]);
      const float p10 = fast_exp2(sacc[n][2] - base[1]);
      const float p11 = fast_exp2(sacc[n][3] - base[1]);
      psum[0] += p00 + p01;
      psum[1] += p10 + p11;
      const int col = cs * C::kKW + n * 8 + 2 * (lane & 3);
      *reinterpret_cast<uint32_t*>(sP + (ra * C::kPStride + col) * 2) = pack2<FP8>(p00, p01);
      *reinterpret_cast<uint32_t*>(sP + ((ra + 8) * C::kPStride + col) * 2) = pack2<FP8>(p10, p11);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) l_run[i] = l_run[i] * alpha[i] + psum[i];
#pragma unroll
    for (int n = 0; n < C::kNTV; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    __syncthreads();

    // ---- O += P V for value columns [cs*VW, cs*VW + VW)
    const uint32_t pa = sP_u32 + ((rg * 16 + (lane & 15)) * C::kPStride + (lane >> 4) * 8) * 2;
    const uint32_t vb = kv_u32 + (((lane & 7) + ((lane >> 3) & 1) * 8) * kQStride +
                                  cs * C::kVW + (lane >> 4) * 8) * 2;
#pragma unroll
    for (int ks = 0; ks < C::kKC / 16; ++ks) {
      uint32_t a[4];
      ldmatrix_x4(pa + ks * 32, a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int n = 0; n < C::kNTV; n += 2) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vb + (ks * 16 * kQStride + n * 8) * 2, b0, b1, b2, b3);
        mma_16816<FP8>(o[n], a, b0, b1);
        mma_16816<FP8>(o[n + 1], a, b2, b3);
      }
    }
  }
  cp_async_wait<0>();

  // ---------------------------------------------------------------- epilogue
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 1);
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 2);
  }
  __syncthreads();
  if ((lane & 3) == 0) {
    red[(rg * C::kCS + cs) * 16 + (lane >> 2)] = l_run[0];
    red[(rg * C::kCS + cs) * 16 + (lane >> 2) + 8] = l_run[1];
  }
  __syncthreads();
  float ltot[2] = {0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int w = 0; w < C::kCS; ++w) ltot[i] += red[(rg * C::kCS + w) * 16 + (lane >> 2) + 8 * i];

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int rho = row0 + ra + 8 * i;
    if (rho >= rows_total) continue;
    const int tok = tok0 + rho / H;
    const int head = rho % H;
    const int64_t th = static_cast<int64_t>(tok) * H + head;
    const float L = ltot[i];
    const float m = m_run[i];
    if (p.final_mode) {
      float mult, lse;
      if (p.sinks != nullptr) {
        const float s2 = p.sinks[head] * kLog2e;
        const float M = fmaxf(m, s2);
        const float wk = L > 0.f ? L * exp2f(m - M) : 0.f;
        const float W = wk + exp2f(s2 - M);
        mult = L > 0.f ? exp2f(m - M) / W : 0.f;
        lse = kLn2 * (M + log2f(W));
      } else if (L > 0.f) {
        mult = 1.f / L;
        lse = kLn2 * (m + log2f(L));
      } else {
        mult = 0.f;
        lse = -INFINITY;
      }
      mult *= p.kv_scale;
      __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out) + th * kRank + cs * C::kVW + 2 * (lane & 3);
#pragma unroll
      for (int n = 0; n < C::kNTV; ++n) {
        *reinterpret_cast<__nv_bfloat162*>(outp + n * 8) =
            __floats2bfloat162_rn(o[n][2 * i] * mult, o[n][2 * i + 1] * mult);
      }
      if (cs == 0 && (lane & 3) == 0) p.lse[th] = lse;
    } else {
      const float mult = L > 0.f ? p.kv_scale / L : 0.f;
      const int64_t ts = th * p.num_segments + seg;
      float* dst = p.segm_out + ts * kRank + cs * C::kVW + 2 * (lane & 3);
#pragma unroll
      for (int n = 0; n < C::kNTV; ++n) {
        *reinterpret_cast<float2*>(dst + n * 8) = make_float2(o[n][2 * i] * mult, o[n][2 * i + 1] * mult);
      }
      if (cs == 0 && (lane & 3) == 0) {
        p.segm_max[ts] = L > 0.f ? m : -INFINITY;
        p.segm_expsum[ts] = L;
      }
    }
  }
}

// Raise the dynamic shared-memory limit of a kernel once per device, so that
// later launches (including ones recorded into a CUDA graph) make no
// attribute calls.
template <typename K>
cudaError_t ensure_smem_limit(K kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <int RG, bool FP8>
cudaError_t launch_variant(const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  using C = Cfg<RG, FP8>;
  static std::atomic<uint64_t> done{0};
  cudaError_t e = ensure_smem_limit(decode_mma_kernel<RG, FP8>, C::kSmem, done);
  if (e != cudaSuccess) return e;
  decode_mma_kernel<RG, FP8><<<grid, kThreads, C::kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int decode_mma_smem_bytes(int32_t kernel, bool fp8) {
  switch (kernel) {
    case kMmaRows16: return fp8 ? Cfg<1, true>::kSmem : Cfg<1, false>::kSmem;
    case kMmaRows32: return fp8 ? Cfg<2, true>::kSmem : Cfg<2, false>::kSmem;
    case kMmaRows64: return fp8 ? Cfg<4, true>::kSmem : Cfg<4, false>::kSmem;
    default: return -1;
  }
}

cudaError_t launch_decode_mma(int32_t kernel, bool fp8, const DecodeParams& p, dim3 grid,
                              cudaStream_t stream) {
  switch (kernel) {
    case kMmaRows16: return fp8 ? launch_variant<1, true>(p, grid, stream) : launch_variant<1, false>(p, grid, stream);
    case kMmaRows32: return fp8 ? launch_variant<2, true>(p, grid, stream) : launch_variant<2, false>(p, grid, stream);
    case kMmaRows64: return fp8 ? launch_variant<4, true>(p, grid, stream) : launch_variant<4, false>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
