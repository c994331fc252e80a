// decode_tc.cu -- split-K paged MLA decode on tcgen05 tensor cores (sm_103a).
//
// A CTA pair (thread-block cluster of 2) owns one (128-row tile, segment,
// request). Rows are (token, head) pairs of the request; all of them share
// one pass over each KV page. The 576 score columns and the 512 value
// columns are split between the two CTAs so that neither re-reads the
// other's bytes:
//   CTA 0 loads cache columns [0, 256):   QK^T over dims [0, 256),   O[:, 0:256)
//   CTA 1 loads cache columns [256, 576): QK^T over dims [256, 576), O[:, 256:512)
// Per 64-key chunk (one TMA box of 64 rows x 64 columns per 128 bytes):
//   TMA warp   -- loads this CTA's boxes of the page into a 2-stage ring
//                 (block-table lookup per chunk, 128-byte swizzle);
//   MMA thread -- S_c = Q_c K_c^T (M=128, N=64, bf16, fp32 in TMEM), and after
//                 the softmax, O_c += P V_c (A = P in TMEM, B = V MN-major);
//   softmax    -- 4 warps, one row per thread: read the partial scores from
//                 TMEM, send them to the peer through distributed shared
//                 memory, add the peer's partial, mask, base-2 online
//                 softmax with a lazily updated reference max (O in TMEM is
//                 rescaled only when the max grows by more than 2^8), write P
//                 (bf16) back into TMEM over the scores.
// Both CTAs compute identical P, m and l (the same fp32 sum in either order).
// TMEM: O at columns [0, 256), S/P double buffer at [256, 384).
// Every wait is bounded; on a timeout the kernel records an error code in
// the status word, stops issuing work, drains what it issued and exits.
#include <atomic>
#include <cfloat>
#include <climits>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ops.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 softmax
constexpr int kRows = 128;
constexpr int kKeys = 64;
constexpr int kBoxQ = kRows * 128;     // 128 rows x 64 bf16 columns
constexpr int kBoxKV = kKeys * 128;    // 64 rows x 64 bf16 columns
constexpr int kMaxBoxes = 5;
constexpr int kStages = 2;
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kMaxBoxes * kBoxQ;
constexpr int kRecvBytes = kRows * kKeys * 4;
constexpr int kOffRecv = kOffKV + kStages * kMaxBoxes * kBoxKV;
constexpr int kOffBar = kOffRecv + 2 * kRecvBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;  // barriers, TMEM slot, flags, 1 KB alignment
static_assert(kSmemBytes <= 232448, "shared memory budget");

enum : int {
  kQFull = 0, kKvFull = 1, kKvEmpty = 3, kSFull = 5, kPFull = 7, kRecvFull = 9, kPeerFree = 11,
  kPvDone = 13, kOFinal = 15, kDrain = 16, kNumBars = 17
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct TcMaps {
  CUtensorMap q;   // q viewed as [T*H rows, 576] bf16, box 64 x 128
  CUtensorMap kv;  // cache viewed as [NB*BS rows, 576] bf16, box 64 x 64
};

struct Shared {
  uint8_t* base;
  uint32_t bar0;
  volatile int* abort;
  __device__ uint32_t bar(int i) const { return bar0 + 8u * i; }
};

__device__ __forceinline__ void report(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Bounded wait on a local barrier phase; `cluster` selects acquire.cluster
// (for barriers a peer CTA arrives on). Returns false on timeout or abort.
__device__ bool wait_phase(const Shared& sh, int* status, uint32_t bar, uint32_t parity,
                           bool cluster, int code) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    const bool ok = cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    if (ok) return true;
    if (*sh.abort) return false;
    if ((it & 63u) == 0) {
      const uint64_t now = global_timer_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > kTimeoutNs) {
        report(status, code);
        *sh.abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ TcMaps maps, const DecodeParams p, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t peer = crank ^ 1u;
  const int tile = blockIdx.x >> 1;
  const int seg = blockIdx.y;
  const int unit = blockIdx.z;
  const int H = p.num_heads;

  int qlen = 1, tok0 = unit;
  if (p.qo_indptr != nullptr) {
    tok0 = p.qo_indptr[unit];
    qlen = p.qo_indptr[unit + 1] - tok0;
  }
  const int part_len = p.seq_lens[unit];
  const int rows_total = qlen * H;
  const int row0 = tile * kRows;
  if (row0 >= rows_total) return;  // both CTAs of the pair take this branch together

  const int span = p.num_segments * p.tile_size;
  const int tps = part_len > 0 ? cdiv(part_len, span) : 0;
  const int seg_len = tps * p.tile_size;
  const int seg_start = seg * seg_len;
  const int seg_end = min(seg_start + seg_len, part_len);
  const int n_chunks = seg_end > seg_start ? cdiv(seg_end - seg_start, kKeys) : 0;
  const int nbox = crank == 0 ? 4 : 5;
  const int col0 = crank == 0 ? 0 : 256;

  Shared sh;
  sh.base = smem;
  sh.bar0 = smem_u32(smem + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kNumBars);
  sh.abort = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * kNumBars + 4);

  if (tid == 0) {
    *sh.abort = 0;
    mbar_init(sh.bar(kQFull), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(sh.bar(kKvFull + b), 1);
      mbar_init(sh.bar(kKvEmpty + b), 1);
      mbar_init(sh.bar(kSFull + b), 1);
      mbar_init(sh.bar(kPFull + b), 128);
      mbar_init(sh.bar(kRecvFull + b), 128);
      mbar_init(sh.bar(kPeerFree + b), 128);
      mbar_init(sh.bar(kPvDone + b), 1);
    }
    mbar_init(sh.bar(kOFinal), 1);
    mbar_init(sh.bar(kDrain), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tslot), kTmemCols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote arrive
  fence_after_sync();
  const uint32_t tbase = *tslot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.kv);
      mbar_arrive_expect_tx(sh.bar(kQFull), nbox * kBoxQ);
      const int qrow = tok0 * H + row0;
      for (int j = 0; j < nbox; ++j)
        tma_load_2d(smem_u32(smem + kOffQ + j * kBoxQ), &maps.q, col0 + 64 * j, qrow,
                    sh.bar(kQFull));
      const int32_t* bt_row = p.block_table + static_cast<int64_t>(unit) * p.bt_stride;
      const int bs = p.block_size;
      int issued = 0;
      for (int c = 0; c < n_chunks; ++c) {
        const int s = c & 1;
        if (c >= 2 && !wait_phase(sh, status, sh.bar(kKvEmpty + s), ((c - 2) >> 1) & 1, false, 11))
          break;
        const int pos = seg_start + c * kKeys;
        const int blk = pos / bs;
        const int row = bt_row[blk] * bs + (pos - blk * bs);
        mbar_arrive_expect_tx(sh.bar(kKvFull + s), nbox * kBoxKV);
        for (int j = 0; j < nbox; ++j)
          tma_load_2d(smem_u32(smem + kOffKV + (s * kMaxBoxes + j) * kBoxKV), &maps.kv,
                      col0 + 64 * j, row, sh.bar(kKvFull + s));
        issued = c + 1;
      }
      // Drain: the last two loads issued must have landed before the CTA exits.
      for (int c = max(0, issued - 2); c < issued; ++c) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(sh.bar(kKvFull + (c & 1)), (c >> 1) & 1)) {
          if (global_timer_ns() - t0 > kTimeoutNs) {
            report(status, 12);
            break;
          }
        }
      }
      {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(sh.bar(kQFull), 0)) {
          if (global_timer_ns() - t0 > kTimeoutNs) {
            report(status, 13);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = instr_desc(kRows, kKeys, 1, 1, false, false);
      const uint32_t idesc_pv = instr_desc(kRows, 256, 1, 1, false, true);
      const uint32_t q_base = smem_u32(smem + kOffQ);
      const uint32_t kv_base = smem_u32(smem + kOffKV);
      bool ok = n_chunks == 0 || wait_phase(sh, status, sh.bar(kQFull), 0, false, 21);
      auto issue_pv = [&](int cc) -> bool {
        const int b = cc & 1;
        if (!wait_phase(sh, status, sh.bar(kPFull + b), (cc >> 1) & 1, false, 22)) return false;
        fence_after_sync();
        const uint32_t v0 = kv_base + (b * kMaxBoxes) * kBoxKV;
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks) {
          const uint64_t bd = smem_desc_sw128(v0 + ks * 2048, kBoxKV, 1024);
          mma_ts(tbase + kTmemO, tbase + kTmemS + 64 * b + 8 * ks, bd, idesc_pv,
                 (cc | ks) != 0 ? 1u : 0u);
        }
        mma_commit(sh.bar(kKvEmpty + b));
        mma_commit(sh.bar(kPvDone + b));
        return true;
      };
      for (int c = 0; c < n_chunks && ok; ++c) {
        const int b = c & 1;
        if (!wait_phase(sh, status, sh.bar(kKvFull + b), (c >> 1) & 1, false, 23)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint32_t kv0 = kv_base + (b * kMaxBoxes) * kBoxKV;
        for (int j = 0; j < nbox; ++j) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = smem_desc_sw128(q_base + j * kBoxQ + k * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(kv0 + j * kBoxKV + k * 32, 16, 1024);
            mma_ss(tbase + kTmemS + 64 * b, ad, bd, idesc_qk, (j | k) != 0 ? 1u : 0u);
          }
        }
        mma_commit(sh.bar(kSFull + b));
        if (c >= 1 && !issue_pv(c - 1)) ok = false;
      }
      if (ok && n_chunks >= 1 && issue_pv(n_chunks - 1)) mma_commit(sh.bar(kOFinal));
      // Drain every MMA this thread issued before TMEM is released.
      mma_commit(sh.bar(kDrain));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(sh.bar(kDrain), 0)) {
        if (global_timer_ns() - t0 > kTimeoutNs) {
          report(status, 24);
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int q4 = warp & 3;                 // TMEM lane quarter of this warp
    const int r = q4 * 32 + lane;            // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int rho = row0 + r;
    const bool row_ok = rho < rows_total;
    const int vis = row_ok ? part_len - qlen + rho / H + 1 : 0;
    const float scale2 = p.score_scale_log2;
    const uint32_t recv_local = smem_u32(smem + kOffRecv);
    const uint32_t recv_peer = map_to_rank(recv_local, peer);
    const uint32_t bar_peer = map_to_rank(sh.bar0, peer);
    float m_ref = -INFINITY, m_true = -INFINITY, l = 0.f;
    bool ok = true;
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int b = c & 1;
      const uint32_t par = (c >> 1) & 1;
      ok = __all_sync(0xffffffffu, wait_phase(sh, status, sh.bar(kSFull + b), par, false, 31));
      if (!ok) break;
      fence_after_sync();
      uint32_t sr[64];
      tmem_ld_32x32b_x64(tbase + lane_off + kTmemS + 64 * b, sr);
      tmem_ld_wait();
      // exchange partial scores with the peer CTA
      if (c >= 2) {
        ok = __all_sync(0xffffffffu,
                        wait_phase(sh, status, sh.bar(kPeerFree + b), ((c - 2) >> 1) & 1, true, 32));
        if (!ok) break;
      }
      const uint32_t dst = recv_peer + b * kRecvBytes + r * 256;
#pragma unroll
      for (int q = 0; q < 16; ++q)
        st_cluster_v4(dst + ((q ^ (r & 15)) << 4), sr[4 * q], sr[4 * q + 1], sr[4 * q + 2],
                      sr[4 * q + 3]);
      mbar_arrive_cluster(bar_peer + 8u * (kRecvFull + b));
      ok = __all_sync(0xffffffffu, wait_phase(sh, status, sh.bar(kRecvFull + b), par, true, 33));
      if (!ok) break;
      const uint8_t* src = smem + kOffRecv + b * kRecvBytes + r * 256;
      float s[64];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(src + ((q ^ (r & 15)) << 4));
        s[4 * q + 0] = __uint_as_float(sr[4 * q + 0]) + v.x;
        s[4 * q + 1] = __uint_as_float(sr[4 * q + 1]) + v.y;
        s[4 * q + 2] = __uint_as_float(sr[4 * q + 2]) + v.z;
        s[4 * q + 3] = __uint_as_float(sr[4 * q + 3]) + v.w;
      }
      mbar_arrive_cluster(bar_peer + 8u * (kPeerFree + b));

      // mask and chunk maximum
      const int c0 = seg_start + c * kKeys;
      const int lim = min(seg_end, vis) - c0;
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        s[j] = j < lim ? s[j] * scale2 : -INFINITY;
        mx = fmaxf(mx, s[j]);
      }
      m_true = fmaxf(m_true, mx);
      float alpha = 1.f;
      bool resc = false;
      if (mx > m_ref + 8.f) {
        if (m_ref != -INFINITY) {
          alpha = fast_exp2(m_ref - mx);
          resc = true;
          l *= alpha;
        }
        m_ref = mx;
      }
      if (__any_sync(0xffffffffu, resc)) {
        // O rows of this warp are relative to the old reference: wait for
        // P.V of the previous chunk, then rescale them in TMEM.
        ok = __all_sync(0xffffffffu, wait_phase(sh, status, sh.bar(kPvDone + ((c - 1) & 1)),
                                                 ((c - 1) >> 1) & 1, false, 34));
        if (!ok) break;
        fence_after_sync();
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          uint32_t o[64];
          tmem_ld_32x32b_x64(tbase + lane_off + kTmemO + 64 * g, o);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 64; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          uint32_t o0[32], o1[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            o0[j] = o[j];
            o1[j] = o[32 + j];
          }
          tmem_st_32x32b_x32(tbase + lane_off + kTmemO + 64 * g, o0);
          tmem_st_32x32b_x32(tbase + lane_off + kTmemO + 64 * g + 32, o1);
        }
        tmem_st_wait();
      }
      // P = 2^(s - m_ref) as bf16, into TMEM over the scores
      const float base = m_ref == -INFINITY ? 0.f : m_ref;
      uint32_t pk[32];
      float ps = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float p0 = fast_exp2(s[2 * j] - base);
        const float p1 = fast_exp2(s[2 * j + 1] - base);
        ps += p0 + p1;
        pk[j] = pack_bf16(p0, p1);
      }
      l += ps;
      tmem_st_32x32b_x32(tbase + lane_off + kTmemS + 64 * b, pk);
      tmem_st_wait();
      // A partial last chunk: zero the value rows past the segment so that
      // whatever the cache holds there cannot reach O through P = 0.
      const int nvalid = seg_end - c0;
      if (nvalid < kKeys) {
        uint8_t* vbase = smem + kOffKV + (b * kMaxBoxes) * kBoxKV;
        const int pieces = (kKeys - nvalid) * 8;  // 16-byte pieces per box
        for (int i = tid - 64; i < 4 * pieces; i += 128) {
          const int box = i / pieces;
          const int rem = i - box * pieces;
          const int row = nvalid + rem / 8;
          *reinterpret_cast<uint4*>(vbase + box * kBoxKV + row * 128 + (rem & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      }
      fence_before_sync();
      mbar_arrive(sh.bar(kPFull + b));
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n_chunks > 0) {
      ok = __all_sync(0xffffffffu, wait_phase(sh, status, sh.bar(kOFinal), 0, false, 35));
      fence_after_sync();
    }
    if (ok && row_ok) {
      const int tok = tok0 + rho / H;
      const int head = rho % H;
      const int64_t th = static_cast<int64_t>(tok) * H + head;
      float mult;
      float lse = -INFINITY;
      if (p.final_mode) {
        if (p.sinks != nullptr) {
          const float s2 = p.sinks[head] * kLog2e;
          const float M = fmaxf(m_ref, s2);
          const float e = l > 0.f ? exp2f(m_ref - M) : 0.f;
          const float W = l * e + exp2f(s2 - M);
          mult = e / W;
          lse = kLn2 * (M + log2f(W));
        } else if (l > 0.f) {
          mult = 1.f / l;
          lse = kLn2 * (m_ref + log2f(l));
        } else {
          mult = 0.f;
        }
      } else {
        mult = l > 0.f ? 1.f / l : 0.f;
      }
      mult *= p.kv_scale;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        uint32_t o[64];
        if (n_chunks > 0) {
          tmem_ld_32x32b_x64(tbase + lane_off + kTmemO + 64 * g, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) o[j] = 0u;
        }
        if (p.final_mode) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + th * kRank +
                                                col0 + 64 * g);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            dst[q] = make_uint4(
                pack_bf16(__uint_as_float(o[8 * q + 0]) * mult, __uint_as_float(o[8 * q + 1]) * mult),
                pack_bf16(__uint_as_float(o[8 * q + 2]) * mult, __uint_as_float(o[8 * q + 3]) * mult),
                pack_bf16(__uint_as_float(o[8 * q + 4]) * mult, __uint_as_float(o[8 * q + 5]) * mult),
                pack_bf16(__uint_as_float(o[8 * q + 6]) * mult, __uint_as_float(o[8 * q + 7]) * mult));
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(
              p.segm_out + (th * p.num_segments + seg) * kRank + col0 + 64 * g);
#pragma unroll
          for (int q = 0; q < 16; ++q)
            dst[q] = make_float4(__uint_as_float(o[4 * q]) * mult, __uint_as_float(o[4 * q + 1]) * mult,
                                 __uint_as_float(o[4 * q + 2]) * mult, __uint_as_float(o[4 * q + 3]) * mult);
        }
      }
      if (crank == 0) {
        if (p.final_mode) {
          p.lse[th] = lse;
        } else {
          const int64_t ts = th * p.num_segments + seg;
          p.segm_max[ts] = l > 0.f ? m_true : -INFINITY;
          p.segm_expsum[ts] = l > 0.f ? l * exp2f(m_ref - m_true) : 0.f;
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  fence_before_sync();
  __syncthreads();
  cluster_sync();  // no remote access to this CTA's shared memory after here
  fence_after_sync();
  if (warp == 1) tmem_dealloc(tbase, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::atomic<bool> tried{false};
  if (!tried.load(std::memory_order_acquire)) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    tried.store(true, std::memory_order_release);
  }
  return fn;
}

cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

int decode_tc_smem_bytes() { return kSmemBytes; }

cudaError_t launch_decode_tc(const DecodeParams& p, int64_t q_rows, int64_t kv_rows, dim3 grid,
                             int* status, cudaStream_t stream) {
  TcMaps maps;
  cudaError_t e = make_map(&maps.q, p.q, static_cast<uint64_t>(q_rows), kRows);
  if (e != cudaSuccess) return e;
  e = make_map(&maps.kv, p.kv, static_cast<uint64_t>(kv_rows), kKeys);
  if (e != cudaSuccess) return e;
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_acq_rel);
  }
  decode_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(maps, p, status);
  return cudaGetLastError();
}

}  // namespace mla
