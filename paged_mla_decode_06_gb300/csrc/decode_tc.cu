// decode_tc.cu -- split-K paged MLA decode on tcgen05 tensor cores (sm_103a).
//
// A CTA pair (thread-block cluster of 2) owns one (128-row tile, segment,
// request). Rows are (token, head) pairs of the request; all of them share
// one pass over each KV page. The 576 score columns and the 512 value
// columns are split between the two CTAs so that neither loads the other's
// bytes:
//   CTA 0 loads cache columns [0, 256):   QK^T over dims [0, 256),   O[:, 0:256)
//   CTA 1 loads cache columns [256, 576): QK^T over dims [256, 576), O[:, 256:512)
// Per 64-key chunk (one 128-byte-wide TMA box per 64 bf16 / 128 e4m3 columns):
//   TMA warp   -- block-table lookup, this CTA's boxes of the page into a
//                 STAGES-deep ring (128-byte swizzle);
//   MMA thread -- S_c = Q_c K_c^T (M=128, N=64, fp32 in TMEM; kind::f16 for
//                 bf16, kind::f8f6f4 for e4m3), then O_c += P V_c with P in
//                 TMEM as the A operand and V an MN-major B operand (bf16, or
//                 f16 for e4m3 caches);
//   softmax    -- 4 warps, one row per thread: partial scores from TMEM, sent
//                 to the peer through distributed shared memory, the peer's
//                 partial added, masks, base-2 online softmax with a lazily
//                 moved reference max (O in TMEM is rescaled only when the
//                 max grows by more than 2^8), P written back into TMEM;
//   convert    -- (e4m3 only) 4 warps widen the chunk's value columns to f16
//                 in shared memory (exact), zeroing rows past the segment.
// Both CTAs compute identical P, m and l (the same fp32 sum in either order).
// TMEM: O at columns [0, 256), scores/P double buffer at [256, 384).
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

constexpr int kRows = 128;
constexpr int kKeys = 64;
constexpr int kBoxQ = kRows * 128;     // 128 rows x 128 bytes
constexpr int kBoxKV = kKeys * 128;    // 64 rows x 128 bytes
constexpr int kRecvBytes = kRows * kKeys * 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;
constexpr uint32_t kTmemQ = 384;  // bf16: q of the CTA's 256 latent dims (A operand of QK^T)
constexpr uint64_t kTimeoutNs = 2000000000ull;

enum : int {
  kQFull = 0, kKvFull = 1, kKvEmpty = 4, kSFull = 7, kPFull = 9, kRecvFull = 11,
  kPeerFree = 13, kPvDone = 15, kOFinal = 17, kDrain = 18, kV16Full = 19, kQTmem = 20,
  kSRead = 21, kNumBars = 23
};

template <bool FP8, bool SPARSE = false>
struct Cfg {
  // warp 0 loads, warp 1 issues MMAs, warps 2..5 softmax, warps 6..9 send
  // the partial scores to the peer (and, for e4m3, widen the values to f16)
  static constexpr int kThreads = 320;
  static constexpr int kBoxCols = FP8 ? 128 : 64;   // elements per 128-byte box row
  static constexpr int kNbox0 = FP8 ? 2 : 4;        // CTA 0: columns [0, 256)
  static constexpr int kNbox1 = FP8 ? 3 : 5;        // CTA 1: columns [256, 576 (+ zero fill))
  static constexpr int kMaxBoxes = kNbox1;
  // bf16 keeps q's 256 latent dims in TMEM and only CTA 1's rope box in
  // shared memory; e4m3 keeps all of q in shared memory.
  static constexpr int kQSmemBoxes = FP8 ? kNbox1 : 1;
  static constexpr int kStages = 3;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQSmemBoxes * kBoxQ;
  static constexpr int kOffV16 = kOffKV + kStages * kMaxBoxes * kBoxKV;
  static constexpr int kV16Bytes = FP8 ? 4 * kBoxKV : 0;
  // partial scores: one buffer the peer fills, one this CTA sends from
  static constexpr int kOffRecv = kOffV16 + kV16Bytes;
  static constexpr int kOffSend = kOffRecv + kRecvBytes;
  static constexpr int kOffBar = kOffSend + kRecvBytes;
  static constexpr int kSmem = kOffBar + 256 + 1024;  // barriers, TMEM slot, flag, alignment
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kStages <= 3, "barrier slots");
};

struct TcMaps {
  CUtensorMap q;   // q viewed as [T*H rows, 576], box 128 bytes x 128 rows
  CUtensorMap kv;  // cache viewed as [NB*BS rows, 576], box 128 bytes x 64 rows
};

struct Shared {
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
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kTimeoutNs) {
        report(status, code);
        *sh.abort = 1;
        return false;
      }
    }
  }
}

// Wait that ignores the abort flag (teardown drains), still bounded.
__device__ void drain_wait(int* status, uint32_t bar, uint32_t parity, int code) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kTimeoutNs) {
      report(status, code);
      return;
    }
  }
}

template <bool F16>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// The part of q that lives in shared memory: every box for e4m3; for bf16
// only CTA 1's rope box (x = 512), CTA 0 has none and just arrives.
template <bool FP8>
__device__ void load_q_smem(const TcMaps& maps, uint8_t* dst, uint32_t bar, uint32_t crank,
                            int nbox, int col0, int qrow) {
  tma_prefetch_desc(&maps.q);
  if constexpr (FP8) {
    mbar_arrive_expect_tx(bar, nbox * kBoxQ);
    for (int j = 0; j < nbox; ++j)
      tma_load_2d(smem_u32(dst + j * kBoxQ), &maps.q, col0 + 128 * j, qrow, bar);
  } else if (crank == 1) {
    mbar_arrive_expect_tx(bar, kBoxQ);
    tma_load_2d(smem_u32(dst), &maps.q, 512, qrow, bar);
  } else {
    mbar_arrive(bar);
  }
}

template <bool FP8, bool SPARSE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<FP8>::kThreads, 1)
    decode_tc_kernel(const __grid_constant__ TcMaps maps, const DecodeParams p, int* status) {
  using C = Cfg<FP8>;
  static_assert(!(FP8 && SPARSE), "the sparse variant is bf16");
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

  int qlen = 1, tok0 = unit, part_len = 0;
  int64_t list_base = 0;
  if constexpr (SPARSE) {
    if (p.slot_indptr != nullptr) {
      list_base = p.slot_indptr[unit];
      part_len = p.slot_indptr[unit + 1] - p.slot_indptr[unit];
    } else {
      list_base = static_cast<int64_t>(unit) * p.topk;
      part_len = p.topk;
    }
  } else {
    if (p.qo_indptr != nullptr) {
      tok0 = p.qo_indptr[unit];
      qlen = p.qo_indptr[unit + 1] - tok0;
    }
    part_len = p.seq_lens[unit];
  }
  const int rows_total = qlen * H;
  const int row0 = tile * kRows;
  if (row0 >= rows_total) return;  // both CTAs of the pair take this branch together

  const int span = p.num_segments * p.tile_size;
  const int tps = part_len > 0 ? cdiv(part_len, span) : 0;
  const int seg_len = tps * p.tile_size;
  const int seg_start = seg * seg_len;
  const int seg_end = min(seg_start + seg_len, part_len);
  const int n_chunks = seg_end > seg_start ? cdiv(seg_end - seg_start, kKeys) : 0;
  const int nbox = crank == 0 ? C::kNbox0 : C::kNbox1;
  const int col0 = crank == 0 ? 0 : 256;

  Shared sh;
  sh.bar0 = smem_u32(smem + C::kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 8 * kNumBars);
  sh.abort = reinterpret_cast<volatile int*>(smem + C::kOffBar + 8 * kNumBars + 4);

  if (tid == 0) {
    *sh.abort = 0;
    mbar_init(sh.bar(kQFull), 1);
    for (int s = 0; s < C::kStages; ++s) {
      // sparse: every lane of the gather warp arrives after its copies land
      mbar_init(sh.bar(kKvFull + s), SPARSE ? 32 : 1);
      // e4m3: the stage is free once QK^T (MMA commit) and the conversion
      // warps (128 arrivals) have read it; bf16: once P.V has.
      mbar_init(sh.bar(kKvEmpty + s), FP8 ? 129 : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sh.bar(kSFull + b), 1);
      mbar_init(sh.bar(kPFull + b), 128);
      // the receiver arms its own barrier with the 32 KB the peer sends;
      // one arrival per softmax warp of the peer frees the buffer
      if (b == 0) {
        mbar_init(sh.bar(kRecvFull), 1);
        mbar_init(sh.bar(kPeerFree), 4);
      }
      mbar_init(sh.bar(kPvDone + b), 1);
    }
    mbar_init(sh.bar(kOFinal), 1);
    mbar_init(sh.bar(kDrain), 1);
    mbar_init(sh.bar(kV16Full), 128);
    mbar_init(sh.bar(kQTmem), 128);
    // the sender warps have read the scores of buffer b out of TMEM
    mbar_init(sh.bar(kSRead), 128);
    mbar_init(sh.bar(kSRead + 1), 128);
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

  if (SPARSE && warp == 0) {
    // ------------------------------------------------------------ row gather (sparse)
    // Lane l copies rows 2l and 2l+1 of each chunk (this CTA's 128-byte column
    // groups, swizzled like a TMA box); rows with no valid slot are skipped.
    if (lane == 0) load_q_smem<FP8>(maps, smem + C::kOffQ, sh.bar(kQFull), crank, nbox, col0,
                                    tok0 * H + row0);
    const uint8_t* kvbytes = static_cast<const uint8_t*>(p.kv);
    int c = 0;
    for (; c < n_chunks; ++c) {
      const int st = c % C::kStages;
      if (c >= C::kStages) {
        const bool okw = __all_sync(0xffffffffu, wait_phase(sh, status, sh.bar(kKvEmpty + st),
                                                            (c / C::kStages - 1) & 1, false, 14));
        if (!okw) break;
      }
      const int c0 = seg_start + c * kKeys;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rr = 2 * lane + h;
        const int pos = c0 + rr;
        const int64_t slot = pos < seg_end ? static_cast<int64_t>(p.slots[list_base + pos]) : -1;
        if (slot >= 0) {
          const uint8_t* src = kvbytes + slot * (kHeadDim * 2) + col0 * 2;
          const uint32_t dst = smem_u32(smem + C::kOffKV + (st * C::kMaxBoxes) * kBoxKV + rr * 128);
          for (int j = 0; j < nbox; ++j)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              cp_async_16(dst + j * kBoxKV + ((k ^ (rr & 7)) << 4), src + j * 128 + k * 16, 16u);
        }
      }
      cp_async_commit();
      if (c >= 1) {
        cp_async_wait<1>();
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        mbar_arrive(sh.bar(kKvFull + (c - 1) % C::kStages));
      }
    }
    cp_async_wait<0>();
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    if (c >= 1) mbar_arrive(sh.bar(kKvFull + (c - 1) % C::kStages));
    if (lane == 0) drain_wait(status, sh.bar(kQFull), 0, 13);
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.kv);
      load_q_smem<FP8>(maps, smem + C::kOffQ, sh.bar(kQFull), crank, nbox, col0, tok0 * H + row0);
      const int32_t* bt_row = p.block_table + static_cast<int64_t>(unit) * p.bt_stride;
      const int bs = p.block_size;
      int issued = 0;
      for (int c = 0; c < n_chunks; ++c) {
        const int st = c % C::kStages;
        if (c >= C::kStages &&
            !wait_phase(sh, status, sh.bar(kKvEmpty + st), (c / C::kStages - 1) & 1, false, 11))
          break;
        const int pos = seg_start + c * kKeys;
        const int blk = pos / bs;
        const int row = bt_row[blk] * bs + (pos - blk * bs);
        mbar_arrive_expect_tx(sh.bar(kKvFull + st), nbox * kBoxKV);
        for (int j = 0; j < nbox; ++j)
          tma_load_2d(smem_u32(smem + C::kOffKV + (st * C::kMaxBoxes + j) * kBoxKV), &maps.kv,
                      col0 + C::kBoxCols * j, row, sh.bar(kKvFull + st));
        issued = c + 1;
      }
      // Drain: every load issued must have landed before the CTA exits.
      for (int c = max(0, issued - C::kStages); c < issued; ++c)
        drain_wait(status, sh.bar(kKvFull + c % C::kStages), (c / C::kStages) & 1, 12);
      drain_wait(status, sh.bar(kQFull), 0, 13);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = FP8 ? instr_desc(kRows, kKeys, 0, 0, false, false)
                                    : instr_desc(kRows, kKeys, 1, 1, false, false);
      const uint32_t idesc_pv = FP8 ? instr_desc(kRows, 256, 0, 0, false, true)
                                    : instr_desc(kRows, 256, 1, 1, false, true);
      const uint32_t q_base = smem_u32(smem + C::kOffQ);
      const uint32_t kv_base = smem_u32(smem + C::kOffKV);
      const uint32_t v16_base = smem_u32(smem + C::kOffV16);
      bool ok = n_chunks == 0 || wait_phase(sh, status, sh.bar(kQFull), 0, false, 21);
      if (!FP8 && ok && n_chunks > 0) ok = wait_phase(sh, status, sh.bar(kQTmem), 0, false, 26);
      auto issue_pv = [&](int cc) -> bool {
        const int b = cc & 1;
        if (!wait_phase(sh, status, sh.bar(kPFull + b), (cc >> 1) & 1, false, 22)) return false;
        if (FP8 && !wait_phase(sh, status, sh.bar(kV16Full), cc & 1, false, 25)) return false;
        fence_after_sync();
        const uint32_t v0 = FP8 ? v16_base : kv_base + ((cc % C::kStages) * C::kMaxBoxes) * kBoxKV;
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks) {
          const uint64_t bd = smem_desc_sw128(v0 + ks * 2048, kBoxKV, 1024);
          mma_ts(tbase + kTmemO, tbase + kTmemS + 64 * b + 8 * ks, bd, idesc_pv,
                 (cc | ks) != 0 ? 1u : 0u);
        }
        if (!FP8) mma_commit(sh.bar(kKvEmpty + cc % C::kStages));
        mma_commit(sh.bar(kPvDone + b));
        return true;
      };
      for (int c = 0; c < n_chunks && ok; ++c) {
        const int b = c & 1;
        const int st = c % C::kStages;
        if (!wait_phase(sh, status, sh.bar(kKvFull + st), (c / C::kStages) & 1, false, 23)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint32_t kv0 = kv_base + (st * C::kMaxBoxes) * kBoxKV;
        if constexpr (FP8) {
          for (int j = 0; j < nbox; ++j) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc_sw128(q_base + j * kBoxQ + k * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(kv0 + j * kBoxKV + k * 32, 16, 1024);
              mma_ss_f8(tbase + kTmemS + 64 * b, ad, bd, idesc_qk, (j | k) != 0 ? 1u : 0u);
            }
          }
        } else {
          // 256 latent dims: A = q in TMEM (8 columns per 16 dims)
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t bd = smem_desc_sw128(kv0 + j * kBoxKV + k * 32, 16, 1024);
              mma_ts(tbase + kTmemS + 64 * b, tbase + kTmemQ + 32 * j + 8 * k, bd, idesc_qk,
                     (j | k) != 0 ? 1u : 0u);
            }
          }
          if (crank == 1) {  // 64 rope dims: A = q's rope box in shared memory
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc_sw128(q_base + k * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(kv0 + 4 * kBoxKV + k * 32, 16, 1024);
              mma_ss(tbase + kTmemS + 64 * b, ad, bd, idesc_qk, 1u);
            }
          }
        }
        mma_commit(sh.bar(kSFull + b));
        if (FP8) mma_commit(sh.bar(kKvEmpty + st));
        if (c >= 1 && !issue_pv(c - 1)) ok = false;
      }
      if (ok && n_chunks >= 1 && issue_pv(n_chunks - 1)) mma_commit(sh.bar(kOFinal));
      // Drain every MMA this thread issued before TMEM is released.
      mma_commit(sh.bar(kDrain));
      drain_wait(status, sh.bar(kDrain), 0, 24);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ softmax warps
    const int q4 = warp & 3;                 // TMEM lane quarter of this warp
    const int r = q4 * 32 + lane;            // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int rho = row0 + r;
    const bool row_ok = rho < rows_total;
    const int vis = !row_ok ? 0 : (SPARSE ? INT_MAX : part_len - qlen + rho / H + 1);
    const float scale2 = p.score_scale_log2;
    const uint32_t recv_local = smem_u32(smem + C::kOffRecv);
    const uint32_t recv_peer = map_to_rank(recv_local, peer);
    const uint32_t bar_peer = map_to_rank(sh.bar0, peer);
    float m_ref = -INFINITY, m_true = -INFINITY, l = 0.f;
    if constexpr (!FP8) {
      // this row's 256 latent dims of q into TMEM (packed bf16 pairs)
      const int64_t qrow = static_cast<int64_t>(tok0) * H + row0 + r;
      const bool qok = qrow < static_cast<int64_t>(p.num_tokens) * H;
      const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                                         (qok ? qrow : 0) * kHeadDim + col0);
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 x = qok ? __ldg(qsrc + 8 * g + i) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * i] = x.x;
          v[4 * i + 1] = x.y;
          v[4 * i + 2] = x.z;
          v[4 * i + 3] = x.w;
        }
        tmem_st_32x32b_x32(tbase + lane_off + kTmemQ + 32 * g, v);
      }
      tmem_st_wait();
      fence_before_sync();
      mbar_arrive(sh.bar(kQTmem));
    }
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
      // the peer's partial scores for this chunk (its sender warps bulk-copy
      // them into this CTA's receive buffer)
      if (tid == 64) mbar_arrive_expect_tx(sh.bar(kRecvFull), kRecvBytes);
      ok = __all_sync(0xffffffffu, wait_phase(sh, status, sh.bar(kRecvFull), c & 1, true, 33));
      if (!ok) break;
      const uint8_t* src = smem + C::kOffRecv + r * 256;
      float s[64];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(src + ((q ^ (r & 15)) << 4));
        s[4 * q + 0] = __uint_as_float(sr[4 * q + 0]) + v.x;
        s[4 * q + 1] = __uint_as_float(sr[4 * q + 1]) + v.y;
        s[4 * q + 2] = __uint_as_float(sr[4 * q + 2]) + v.z;
        s[4 * q + 3] = __uint_as_float(sr[4 * q + 3]) + v.w;
      }
      // the receive buffer is consumed: one release arrive per warp on the
      // peer's barrier (the peer's next bulk copy overwrites it)
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(bar_peer + 8u * kPeerFree);

      // keys of the chunk that exist: inside the segment and, for the sparse
      // variant, with a valid slot (one ballot per 32 keys)
      const int c0 = seg_start + c * kKeys;
      const int nvalid = min(kKeys, seg_end - c0);
      uint64_t kmask = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1ull);
      if constexpr (SPARSE) {
        const bool v0 = lane < nvalid && p.slots[list_base + c0 + lane] >= 0;
        const bool v1 = lane + 32 < nvalid && p.slots[list_base + c0 + 32 + lane] >= 0;
        kmask = static_cast<uint64_t>(__ballot_sync(0xffffffffu, v0)) |
                (static_cast<uint64_t>(__ballot_sync(0xffffffffu, v1)) << 32);
      }
      // mask (only chunks with keys that do not exist or are causally hidden)
      // and the chunk maximum over the raw scores (scale2 > 0), 8-way tree
      const int lim = min(seg_end, vis) - c0;
      if (lim < 64 || kmask != ~0ull) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (!(j < lim && ((kmask >> j) & 1ull))) s[j] = -INFINITY;
      }
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
      for (int j = 8; j < 64; ++j) m8[j & 7] = fmaxf(m8[j & 7], s[j]);
      const float mraw = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const float mx = mraw * scale2;  // -inf stays -inf
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
          uint32_t o0[32], o1[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            o0[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            o1[j] = __float_as_uint(__uint_as_float(o[32 + j]) * alpha);
          }
          tmem_st_32x32b_x32(tbase + lane_off + kTmemO + 64 * g, o0);
          tmem_st_32x32b_x32(tbase + lane_off + kTmemO + 64 * g + 32, o1);
        }
        tmem_st_wait();
      }
      // P = 2^(s * scale2 - m_ref), into TMEM over the scores; 8 partial sums
      const float base = m_ref == -INFINITY ? 0.f : m_ref;
      uint32_t pk[32];
      float ps8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) ps8[i] = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float p0 = fast_exp2(fmaf(s[2 * j], scale2, -base));
        const float p1 = fast_exp2(fmaf(s[2 * j + 1], scale2, -base));
        ps8[j & 7] += p0 + p1;
        pk[j] = pack_p<FP8>(p0, p1);
      }
      l += ((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) + ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7]));
      // P overwrites the scores: the sender warps must have read them
      ok = __all_sync(0xffffffffu, wait_phase(sh, status, sh.bar(kSRead + b), par, false, 36));
      if (!ok) break;
      tmem_st_32x32b_x32(tbase + lane_off + kTmemS + 64 * b, pk);
      tmem_st_wait();
      if constexpr (!FP8) {
        // Zero the value rows of keys that do not exist (past the segment, or
        // an invalid sparse slot) so that whatever shared memory holds there
        // cannot reach O through P = 0.
        if (kmask != ~0ull) {
          uint8_t* vbase = smem + C::kOffKV + ((c % C::kStages) * C::kMaxBoxes) * kBoxKV;
          for (int i = tid - 64; i < 4 * kKeys * 8; i += 128) {
            const int box = i >> 9;
            const int row = (i >> 3) & 63;
            if (!((kmask >> row) & 1ull))
              *reinterpret_cast<uint4*>(vbase + box * kBoxKV + row * 128 + (i & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        }
      }
      fence_before_sync();
      mbar_arrive(sh.bar(kPFull + b));
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n_chunks > 0) {
      ok = __all_sync(0xffffffffu, wait_phase(sh, status, sh.bar(kOFinal), 0, false, 35));
      fence_after_sync();
    }
    // TMEM loads are warp-collective: every lane runs them, and only lanes
    // with a valid row store (ok is warp-uniform).
    if (ok) {
      const int tok = tok0 + (row_ok ? rho / H : 0);
      const int head = row_ok ? rho % H : 0;
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
        if (!row_ok) continue;
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
      if (crank == 0 && row_ok) {
        if (p.final_mode) {
          p.lse[th] = lse;
        } else {
          const int64_t ts = th * p.num_segments + seg;
          p.segm_max[ts] = l > 0.f ? m_true : -INFINITY;
          p.segm_expsum[ts] = l > 0.f ? l * exp2f(m_ref - m_true) : 0.f;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ sender (+ e4m3 values)
    // Each chunk's partial scores leave for the peer as soon as QK^T is done:
    // the rows of this warp's TMEM quarter are staged in shared memory and
    // one lane bulk-copies the 8 KB into the peer's receive buffer, counted
    // on the peer's barrier. For e4m3 the same warps then widen the chunk's
    // value columns to f16.
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t recv_peer = map_to_rank(smem_u32(smem + C::kOffRecv), peer);
    const uint32_t bar_peer = map_to_rank(sh.bar0, peer);
    const int ct = tid - 192;  // 0..127
    uint8_t* v16 = smem + C::kOffV16;
    bool ok = true;
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int b = c & 1;
      ok = __all_sync(0xffffffffu, wait_phase(sh, status, sh.bar(kSFull + b), (c >> 1) & 1, false, 51));
      if (!ok) break;
      fence_after_sync();
      if (lane == 0) bulk_wait_read_all();  // the previous copy has left the send buffer
      __syncwarp();
      uint8_t* snd = smem + C::kOffSend + r * 256;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t sr[32];
        tmem_ld_32x32b_x32(tbase + lane_off + kTmemS + 64 * b + 32 * h, sr);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(snd + (((8 * h + q) ^ (r & 15)) << 4)) =
              make_uint4(sr[4 * q], sr[4 * q + 1], sr[4 * q + 2], sr[4 * q + 3]);
      }
      fence_before_sync();
      mbar_arrive(sh.bar(kSRead + b));  // the softmax may overwrite the scores with P
      fence_proxy_async_smem();
      __syncwarp();
      if (c >= 1) {  // the peer has consumed the previous chunk's scores
        ok = __all_sync(0xffffffffu, wait_phase(sh, status, sh.bar(kPeerFree), (c - 1) & 1, true, 52));
        if (!ok) break;
      }
      if (lane == 0) {
        bulk_copy_to_cluster(recv_peer + q4 * 8192, smem_u32(smem + C::kOffSend + q4 * 8192), 8192,
                             bar_peer + 8u * kRecvFull);
        bulk_commit_group();
      }
      if constexpr (FP8) {
        const int st = c % C::kStages;
        ok = __all_sync(0xffffffffu,
                        wait_phase(sh, status, sh.bar(kKvFull + st), (c / C::kStages) & 1, false, 41));
        if (!ok) break;
        if (c >= 1) {
          // the previous chunk's P.V has finished reading the f16 values
          ok = __all_sync(0xffffffffu, wait_phase(sh, status, sh.bar(kPvDone + ((c - 1) & 1)),
                                                   ((c - 1) >> 1) & 1, false, 42));
          if (!ok) break;
        }
        const int nvalid = min(kKeys, seg_end - (seg_start + c * kKeys));
        const uint8_t* src = smem + C::kOffKV + (st * C::kMaxBoxes) * kBoxKV;
        // boxes 0 and 1 of the stage hold this CTA's 256 value columns
        for (int i = ct; i < 2 * kKeys * 8; i += 128) {
          const int box = i >> 9;
          const int rem = i & 511;
          const int row = rem >> 3;
          const int k = rem & 7;  // logical 16-byte chunk (16 e4m3 values)
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (row < nvalid)
            v = *reinterpret_cast<const uint4*>(src + box * kBoxKV + row * 128 + ((k ^ (row & 7)) << 4));
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          uint32_t hh[8];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            hh[2 * e2] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[e2] & 0xFFFF));
            hh[2 * e2 + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[e2] >> 16));
          }
          const int dbox = box * 2 + (k >> 2);
          const int lc = (k & 3) * 2;
          uint8_t* drow = v16 + dbox * kBoxKV + row * 128;
          *reinterpret_cast<uint4*>(drow + ((lc ^ (row & 7)) << 4)) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
          *reinterpret_cast<uint4*>(drow + (((lc + 1) ^ (row & 7)) << 4)) =
              make_uint4(hh[4], hh[5], hh[6], hh[7]);
        }
        fence_proxy_async_smem();
        mbar_arrive(sh.bar(kKvEmpty + st));
        mbar_arrive(sh.bar(kV16Full));
      }
    }
    if (lane == 0) bulk_wait_all();  // score copies complete before teardown
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
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

// 2-D map over a [rows, 576] tensor with 128-byte-wide boxes of box_rows rows.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows, bool fp8) {
  auto enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const uint32_t elt = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim) * elt};
  cuuint32_t box[2] = {128 / elt, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool FP8, bool SPARSE>
cudaError_t launch_variant(const TcMaps& maps, const DecodeParams& p, dim3 grid, int* status,
                           cudaStream_t stream) {
  using C = Cfg<FP8>;
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(decode_tc_kernel<FP8, SPARSE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_acq_rel);
  }
  decode_tc_kernel<FP8, SPARSE><<<grid, C::kThreads, C::kSmem, stream>>>(maps, p, status);
  return cudaGetLastError();
}

}  // namespace

int decode_tc_smem_bytes(bool fp8) { return fp8 ? Cfg<true>::kSmem : Cfg<false>::kSmem; }

cudaError_t launch_decode_tc(const DecodeParams& p, bool fp8, int64_t q_rows, int64_t kv_rows,
                             dim3 grid, int* status, cudaStream_t stream) {
  TcMaps maps;
  cudaError_t e = make_map(&maps.q, p.q, static_cast<uint64_t>(q_rows), kRows, fp8);
  if (e != cudaSuccess) return e;
  e = make_map(&maps.kv, p.kv, static_cast<uint64_t>(kv_rows), kKeys, fp8);
  if (e != cudaSuccess) return e;
  if (p.slots != nullptr) {
    if (fp8) return cudaErrorNotSupported;
    return launch_variant<false, true>(maps, p, grid, status, stream);
  }
  return fp8 ? launch_variant<true, false>(maps, p, grid, status, stream)
             : launch_variant<false, false>(maps, p, grid, status, stream);
}

}  // namespace mla
