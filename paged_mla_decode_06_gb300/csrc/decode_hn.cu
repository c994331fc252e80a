// decode_hn.cu -- split-K paged MLA decode on tcgen05 tensor cores with the
// query rows as the MMA N dimension (sm_103a): requests of at most 128 query
// rows (heads x tokens) over an e4m3 cache whose block size is a multiple
// of 64.
//
// A request of 16 heads padded to the 128-row M tile of the CTA-pair kernel
// spends 7/8 of every QK^T, softmax and P.V step on padding. Here a CTA owns
// NR <= 64 rows of a request and the operands swap roles, per chunk of 128
// keys:
//   S^T[keys, rows]  = K Q^T   M = 128 keys, N = NR, K = 576: 18 kind::f8f6f4
//                              instructions, A = the chunk's key rows (K-major,
//                              straight from the TMA ring), B = q;
//   O^T[cols, rows] += V^T P^T M = 128 value columns (four blocks of the 512),
//                              N = the rows, K = the 128 keys: A = the same key
//                              rows read MN-major, B = P^T, written by the
//                              softmax threads one key per thread (MN-major,
//                              8-key x 16-byte core matrices).
// P goes to the tensor core as two e4m3 terms, hi = e4m3(p) and
// lo = e4m3(p - hi), carrying ~8 significant bits of p (hi alone keeps 4,
// which would move rows of a few keys by several hundredths); both terms are
// one instruction of N = 2 NR (NR <= 48) or two of N = NR into the same
// accumulator. A tcgen05 instruction with N <= 64 costs about as much as one
// with N = 96 (measured), so the chunk costs ~34 instructions whatever NR is.
// Softmax: a thread owns one key (a TMEM lane of S^T) and half of the rows (a
// column each). A row's maximum over the chunk is a warp reduction
// (redux.sync.max.f32) and an exchange among the softmax warps through
// shared memory; p = 2^(s - m_ref + 4) with a reference max m_ref that moves
// only when a chunk max exceeds it by more than 4 (O^T is then rescaled in
// TMEM), so p <= 2^8 fits e4m3 and the bulk of the weights stays in its
// normal range; the true max is kept for the partials.
//
// Requests of 65..128 rows run on a thread-block cluster of CL = 2 CTAs, CTA
// r owning rows [r NR, (r + 1) NR) of the row tile: every key box is read
// from memory once, by one CTA of the cluster, and multicast by TMA to the
// ring slot of both, so that all heads of a request share one pass over its
// keys. A slot is refilled only after the consumers of every CTA released it
// (each commit arrives on the empty barrier of every CTA of the cluster); the
// loading CTA also arms the peer's full barrier with the box's bytes, so each
// CTA can tell, at teardown, when every box meant for it has landed.
//
// Work: with the balanced schedule, a worker (a CTA, or a cluster) walks a
// contiguous run of items (key ranges of row tiles) of about equal length,
// and the pipeline runs on across items: the ring, the S^T and P^T buffers
// and the barrier phases continue, the next item's boxes stream in while the
// current one finishes, and O^T is reused once the epilogue has read it.
// Without it, a CTA (cluster) runs one (row tile, segment, request) of the
// uniform partition.
//
// Warps: 0, 2 TMA producers (the key boxes through the block table), 1 q and
// QK^T issue, 3 P.V issue, 4-11 softmax and epilogue (a lane quarter of keys
// and half of the rows each, two warps per SM sub-partition). Every wait is
// bounded: a timeout records a code in the status word, stops the CTA's work,
// drains what was issued and exits.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "tc_ops.cuh"
#include "tma_map.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kKeys = 128;               // keys per chunk: M of QK^T, K of P.V
constexpr int kHalf = 64;                // keys per TMA box (rows of one block)
constexpr int kSlot = kKeys * 128;       // ring slot: one 128-byte column box of a chunk
constexpr int kRSlot = kKeys * 64;       // rope ring slot: the chunk's 64 rope columns
constexpr int kBoxes = 5;                // per chunk: 4 latent boxes (512 e4m3) + the rope box
constexpr int kThreads = 384;
constexpr int kProducers = 2;            // warps 0, 2
constexpr int kSoftWarps = 8;            // warps 4-11: four TMEM lane quarters x two row halves
constexpr int kMaxSlots = 14;
constexpr int kMaxRSlots = 4;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
constexpr float kPBias = 4.f;            // p = 2^(s - m_ref + kPBias) <= 2^(2 kPBias)
constexpr float kMove = 4.f;             // m_ref moves when a chunk max exceeds it by more

enum : int {
  kFull = 0,                    // [kMaxSlots] ring slot loaded
  kEmpty = kMaxSlots,           // [kMaxSlots] ring slot released by every CTA of the cluster
  kRFull = 2 * kMaxSlots,       // [kMaxRSlots] rope slot loaded
  kREmpty = kRFull + kMaxRSlots,  // [kMaxRSlots] rope slot released by every CTA of the cluster
  kQFull = kREmpty + kMaxRSlots,  // q of the current item loaded
  kQFree,                       // QK^T of the item complete: q may be replaced
  kSFull,                       // [2] S^T buffer written
  kSFree = kSFull + 2,          // [2] S^T buffer read
  kPFull = kSFree + 2,          // [2] P^T buffer written
  kPFree = kPFull + 2,          // [2] P.V of the buffer's chunk complete
  kXA = kPFree + 2,             // [2] softmax warps: chunk maxima posted
  kXE = kXA + 2,                // epilogue: row sums posted
  kXF = kXE + 1,                // epilogue: row factors posted
  kOFull = kXF + 1,             // last P.V of the item complete
  kOFree = kOFull + 1,          // epilogue read O^T: the next item may overwrite it
  kDrain = kOFree + 1,          // the QK^T issuer's MMAs complete
  kDrainPV = kDrain + 1,        // the P.V issuer's MMAs complete
  kNumBars = kDrainPV + 1
};

// Shared-memory header: barriers, TMEM address, abort flag, exchange arrays.
constexpr int kOffBar = 0;
constexpr int kOffTslot = 512;
constexpr int kOffAbort = 516;
constexpr int kOffIssued = 576;             // [kMaxSlots + kMaxRSlots + 1] int: last use issued
                                            // per ring slot, per rope slot, of q
constexpr int kIssuedQ = kMaxSlots + kMaxRSlots;
constexpr int kOffWmax = 1024;              // [2][4][64] warp maxima of a chunk
// per row and chunk parity (written for chunk c, read back at chunk c + 1):
constexpr int kOffMref = kOffWmax + 2048;   // [2][64] reference max
constexpr int kOffMtrue = kOffMref + 512;   // [2][64] true max
constexpr int kOffAlpha = kOffMtrue + 512;  // [2][64] rescale factor
constexpr int kOffVis = kOffAlpha + 512;    // [64] int: causal end of each row
constexpr int kOffLsum = kOffVis + 256;     // [4][64] row sums per warp
constexpr int kOffMult = kOffLsum + 1024;   // [64] output factor per row
constexpr int kHeader = 6144;
static_assert(kNumBars * 8 <= kOffTslot, "barrier space");
static_assert(kOffIssued + 4 * (kIssuedQ + 1) <= 1024, "issue record space");
static_assert(kOffMult + 256 <= kHeader, "header space");

constexpr int align1k(int v) { return (v + 1023) / 1024 * 1024; }

template <int NR>
struct HnCfg {
  static_assert(NR % 16 == 0 && NR >= 16 && NR <= 64, "16..64 rows in steps of 16");
  static constexpr bool kConcat = NR <= 48;         // hi and lo as one MMA of N = 2 NR
  static constexpr int kNpv = kConcat ? 2 * NR : NR;
  static constexpr int kOCols = 4 * kNpv;           // O^T: 4 blocks of kNpv columns
  static constexpr int kSCol = kOCols;              // S^T: 2 buffers of NR columns
  static constexpr int kCols = kOCols + 2 * NR;
  static constexpr uint32_t kTmemAlloc = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128
                                       : kCols <= 256 ? 256 : 512;
  static_assert(kCols <= 512, "TMEM columns");
  static constexpr int kQBox = NR * 128;            // one 128-byte column box of q
  static constexpr int kOffQ = kHeader;
  static constexpr int kPLbo = 16 * NR;             // P^T bytes per 8-key group (hi + lo cores)
  static constexpr int kPBytes = kKeys * 2 * NR;    // one P^T buffer
  // two P^T buffers: the softmax of chunk c + 1 writes while P.V of chunk c reads
  static constexpr int kPBufs = 2;
  static constexpr int kOffP = kOffQ + kBoxes * kQBox;
  // the P^T buffers double as the epilogue's output staging (2 KB per
  // softmax warp): P.V of the item is complete and the next item's first
  // P^T comes after the softmax warps' next exchange
  static constexpr int kStage = kSoftWarps * 2048;
  static constexpr int kPRegion = kPBufs * kPBytes > kStage ? kPBufs * kPBytes : kStage;
  static constexpr int kOffRing = align1k(kOffP + kPRegion);
  static constexpr int kUsable = 232448 - 1024;     // dynamic shared memory minus alignment slack
  // the rope columns (64 bytes of each key) have a ring of their own, of
  // 64-byte-wide boxes (in a 128-byte slot they would take twice the
  // space): the latent ring takes what leaves two rope slots, the rope ring
  // the rest
  static constexpr int kSlotsFit = (kUsable - kOffRing - 2 * kRSlot) / kSlot;
  static constexpr int kSlots = kSlotsFit < kMaxSlots ? kSlotsFit : kMaxSlots;
  static constexpr int kRSlotsFit = (kUsable - kOffRing - kSlots * kSlot) / kRSlot;
  static constexpr int kRSlots = kRSlotsFit < kMaxRSlots ? kRSlotsFit : kMaxRSlots;
  static constexpr int kOffRope = kOffRing + kSlots * kSlot;
  static constexpr int kSmem = kOffRope + kRSlots * kRSlot + 1024;
  // QK^T of chunk c + 1 is issued before P.V of chunk c, which holds the
  // ring indices of chunk c's value boxes: both chunks must fit the ring
  static_assert(kSlots >= 2 * (kBoxes - 1) && kRSlots >= 2, "ring slots");
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct HnMaps {
  CUtensorMap q;     // q viewed as [T*H rows, 576] e4m3, box 128 bytes x NR rows
  CUtensorMap kv;    // cache viewed as [NB*BS rows, 576] e4m3, box 128 bytes x 64 rows
  CUtensorMap kvr;   // the same, box 64 bytes x 64 rows (the rope columns)
  CUtensorMap out;   // out as [T*H, 1, 512] bf16, box 8 rows x 32 columns
  CUtensorMap part;  // segment partials as [slot rows, 1, 512] or [T*H, NS, 512] fp32
};

// One work item as this CTA sees it: a key range of a row tile.
struct Item {
  int unit, tok0, qlen, rows_total, row0, part_len;
  int seg, seg_start, seg_end, n_chunks, pslot;
  bool fin;
};

struct Ctx {
  uint8_t* smem;
  uint32_t bar0;
  volatile int* abort;
  int* status;
  uint64_t limit_ns;
  uint32_t tbase;
  int tid, warp, lane;
  int rank;               // CTA rank in the cluster: rows [rank NR, (rank + 1) NR) of the tile
  int it_begin, it_end;   // this worker's items (one item without the balanced schedule)
  __device__ uint32_t bar(int i) const { return bar0 + 8u * i; }
};

// Item `idx` of the balanced list, or (without one) the uniform partition's
// (row tile, segment, request) of this CTA's block index.
template <int NR, int CL>
__device__ Item item_at(const DecodeParams& p, int idx, int rank) {
  Item it;
  int tile, kb = 0, ke = 0;
  it.pslot = -1;
  if (p.items != nullptr) {
    const int4 a = reinterpret_cast<const int4*>(p.items)[2 * idx];
    const int4 b = reinterpret_cast<const int4*>(p.items)[2 * idx + 1];
    it.unit = a.x;
    tile = a.y;
    kb = a.z;
    ke = a.w;
    it.pslot = b.x;
    it.seg = 0;
    it.fin = it.pslot < 0;
  } else {
    tile = blockIdx.x / CL;
    it.seg = blockIdx.y;
    it.unit = blockIdx.z;
    it.fin = p.final_mode != 0;
  }
  it.qlen = 1;
  it.tok0 = it.unit;
  if (p.qo_indptr != nullptr) {
    it.tok0 = p.qo_indptr[it.unit];
    it.qlen = p.qo_indptr[it.unit + 1] - it.tok0;
  }
  it.part_len = p.seq_lens[it.unit];
  it.rows_total = it.qlen * p.num_heads;
  it.row0 = (tile * CL + rank) * NR;
  if (p.items != nullptr) {
    it.seg_start = kb;
    it.seg_end = min(ke, it.part_len);
  } else {
    const int span = p.num_segments * p.tile_size;
    const int tps = it.part_len > 0 ? cdiv(it.part_len, span) : 0;
    const int seg_len = tps * p.tile_size;
    it.seg_start = it.seg * seg_len;
    it.seg_end = min(it.seg_start + seg_len, it.part_len);
  }
  it.n_chunks = it.seg_end > it.seg_start ? cdiv(it.seg_end - it.seg_start, kKeys) : 0;
  // a row tile with no rows at all (a request with fewer tokens than the
  // longest) has nothing to read; the same for every CTA of the cluster
  if (tile * CL * NR >= it.rows_total) it.n_chunks = 0;
  return it;
}

// Causal end of row `r` of the CTA's rows in item `it`: keys before it are visible.
__device__ __forceinline__ int visible_end(const Item& it, int H, int r) {
  const int rho = it.row0 + r;
  return rho < it.rows_total ? it.part_len - it.qlen + rho / H + 1 : it.part_len;
}

__device__ __forceinline__ void report(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Bounded wait on a barrier phase; false on timeout (recorded) or abort. The
// thread sleeps in the wait (up to kSleepNs at a time, woken by the phase)
// rather than spinning, which would take issue slots from the MMA issuer.
// `cluster` selects cluster-scope acquire, for barriers that other CTAs of
// the cluster arrive on.
constexpr uint32_t kSleepNs = 20000;
template <bool kCluster = false>
__device__ bool wait_phase(const Ctx& x, uint32_t bar, uint32_t parity, int code) {
  if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  const uint32_t nap = x.limit_ns < kSleepNs ? static_cast<uint32_t>(x.limit_ns) : kSleepNs;
  while (!(kCluster ? mbar_try_wait_cluster_sleep(bar, parity, nap) : mbar_try_wait_sleep(bar, parity, nap))) {
    if (*x.abort) return false;
    if (global_timer_ns() - t0 > x.limit_ns) {
      report(x.status, code);
      *x.abort = 1;
      return false;
    }
  }
  return true;
}

// Every lane waits (each acquires what the phase published); warp-uniform result.
__device__ __forceinline__ bool warp_wait(const Ctx& x, uint32_t bar, uint32_t parity, int code) {
  return __all_sync(0xffffffffu, wait_phase(x, bar, parity, code)) != 0;
}

// Wait that ignores the abort flag (teardown drains), bounded by the default limit.
__device__ void drain_wait(const Ctx& x, uint32_t bar, uint32_t parity, int code) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_cluster_sleep(bar, parity, kSleepNs)) {
    if (global_timer_ns() - t0 > kDefaultWaitNs) {
      report(x.status, code);
      return;
    }
  }
}

// The softmax warps meet at barrier `idx` (one arrival per warp and phase):
// this warp's shared-memory writes are published, the others' acquired.
__device__ __forceinline__ bool cross_sync(const Ctx& x, int idx, uint32_t parity, int code) {
  __syncwarp();
  if (x.lane == 0) mbar_arrive(x.bar(idx));
  return warp_wait(x, x.bar(idx), parity, code);
}

// Release of a ring slot (or any barrier every CTA of the cluster counts) by
// this CTA's MMAs, once they complete.
template <int CL>
__device__ __forceinline__ void release(uint32_t bar) {
  if constexpr (CL == 1)
    mma_commit(bar);
  else
    mma_commit_mc(bar, static_cast<uint16_t>((1u << CL) - 1u));
}

// Cache row of key position pos (64 keys from a 64-aligned position lie in
// one block: the block size is a multiple of 64).
__device__ __forceinline__ int cache_row(const DecodeParams& p, const int32_t* bt_row, int pos) {
  const int bs = p.block_size;
  const int blk = pos / bs;
  return bt_row[blk] * bs + (pos - blk * bs);
}

// ------------------------------------------------------------------ producers
// Latent box j < 4 of the worker's g-th chunk (two 64-row TMA boxes from
// their blocks) goes to ring slot i % kSlots, i = 4 g + j, its rope box to
// rope slot g % kRSlots, the counts running on across the worker's items.
// Box b = 5 g + j is loaded by CTA b % CL of the cluster (the only one in a
// cluster of one) and there by producer warp (b / CL) % 2, which records
// the latest use issued per slot (the teardown waits for those loads). The whole warp looks up the cache rows of 16 chunks at a time
// (lane l: chunk l / 2, half l % 2), one window ahead of the chunks it
// issues, so that no TMA issue waits on a block-table read; lane 0 issues.
template <int NR, int CL>
__device__ void produce(const Ctx& x, const HnMaps& maps, const DecodeParams& p, int pidx) {
  using C = HnCfg<NR>;
  const int lane = x.lane;
  volatile int* issued = reinterpret_cast<volatile int*>(x.smem + kOffIssued);
  if (lane == 0) {
    tma_prefetch_desc(&maps.kv);
    tma_prefetch_desc(&maps.kvr);
  }
  const uint64_t pol = l2_evict_first();  // each key row is read once
  int gb = 0;                             // the worker's box count
  bool ok = true;
  for (int idx = x.it_begin; idx < x.it_end && ok; ++idx) {
    const Item it = item_at<NR, CL>(p, idx, x.rank);
    if (it.n_chunks == 0) continue;
    const int32_t* bt_row = p.block_table + static_cast<int64_t>(it.unit) * p.bt_stride;
    auto lookup = [&](int w0) {  // cache row of this lane's (chunk, half) in the window at w0
      const int pos = it.seg_start + (w0 + (lane >> 1)) * kKeys + (lane & 1) * kHalf;
      return pos < it.seg_end ? cache_row(p, bt_row, pos) : 0;
    };
    int cur = lookup(0);
    int nxt = lookup(16);
    for (int c = 0; c < it.n_chunks && ok; ++c, gb += kBoxes) {
      if (c > 0 && (c & 15) == 0) {
        cur = nxt;
        nxt = lookup(c + 16);
      }
      const int row0 = __shfl_sync(0xffffffffu, cur, 2 * (c & 15));
      const int row1 = __shfl_sync(0xffffffffu, cur, 2 * (c & 15) + 1);
      const bool two = it.seg_start + c * kKeys + kHalf < it.seg_end;
      if (lane == 0) {
        for (int j = 0; j < kBoxes; ++j) {
          const int bi = gb + j;
          if (bi % CL != x.rank || (bi / CL) % kProducers != pidx) continue;
          const bool rope = j == kBoxes - 1;
          const int i = rope ? gb / kBoxes : (gb / kBoxes) * (kBoxes - 1) + j;
          const int nslots = rope ? C::kRSlots : C::kSlots;
          const int slot = i % nslots;
          const int use = i / nslots;
          const int empty = rope ? kREmpty + slot : kEmpty + slot;
          if (use >= 1 && !wait_phase<(CL > 1)>(x, x.bar(empty), (use - 1) & 1, 11)) {
            ok = false;
            break;
          }
          const int box = rope ? kRSlot : kSlot;
          const uint32_t bytes = two ? box : box / 2;
          const uint32_t full = x.bar(rope ? kRFull + slot : kFull + slot);
          mbar_arrive_expect_tx(full, bytes);
          const uint32_t dst = smem_u32(x.smem + (rope ? C::kOffRope + slot * kRSlot : C::kOffRing + slot * kSlot));
          const CUtensorMap* map = rope ? &maps.kvr : &maps.kv;
          if constexpr (CL == 1) {
            tma_load_2d_hint(dst, map, 128 * j, row0, full, pol);
            if (two) tma_load_2d_hint(dst + box / 2, map, 128 * j, row1, full, pol);
          } else {
            // the peers' phases of this slot also wait for the box
            for (int r = 0; r < CL; ++r)
              if (r != x.rank) mbar_arrive_expect_tx_cluster(map_to_rank(full, r), bytes);
            constexpr uint16_t kAll = static_cast<uint16_t>((1u << CL) - 1u);
            tma_load_2d_mc_hint(dst, map, 128 * j, row0, full, kAll, pol);
            if (two) tma_load_2d_mc_hint(dst + box / 2, map, 128 * j, row1, full, kAll, pol);
          }
          atomicMax(const_cast<int*>(issued + (rope ? kMaxSlots + slot : slot)), use);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ MMA issue
// Two issuing threads on different SM sub-partitions: one loads each item's
// q and issues QK^T chunk after chunk as the boxes land (two S^T buffers
// ahead of the softmax), the other P.V as soon as a chunk's P^T is written.
// A tcgen05.mma with N <= 64 takes ~40 cycles of the tensor pipe but ~95 to
// issue from one thread that shares its sub-partition with busy softmax
// warps (measured); two issuers keep the pipe fed, and P.V of a chunk never
// waits behind the next chunk's loads, so its value boxes return to the
// ring at once.
template <int NR, int CL>
__device__ void qk_issue(const Ctx& x, const HnMaps& maps, const DecodeParams& p) {
  using C = HnCfg<NR>;
  if (x.lane != 0) return;
  constexpr uint32_t kIdQK = instr_desc(128, NR, 0, 0, false, false);
  const uint64_t q_desc = smem_desc_sw128(smem_u32(x.smem + C::kOffQ), 16, 1024);
  const uint64_t k_desc = smem_desc_sw128(smem_u32(x.smem + C::kOffRing), 16, 1024);  // K-major
  const uint64_t r_desc = smem_desc_sw64(smem_u32(x.smem + C::kOffRope), 512);         // K-major
  volatile int* issued = reinterpret_cast<volatile int*>(x.smem + kOffIssued);
  tma_prefetch_desc(&maps.q);
  int g = 0;   // the worker's chunk count
  int ne = 0;  // items with keys so far
  bool ok = true;
  for (int idx = x.it_begin; idx < x.it_end && ok; ++idx) {
    const Item it = item_at<NR, CL>(p, idx, x.rank);
    if (it.n_chunks == 0) continue;
    // this CTA's q rows of the item, once QK^T of the previous item has read q
    if (ne > 0 && !wait_phase(x, x.bar(kQFree), (ne - 1) & 1, 27)) break;
    mbar_arrive_expect_tx(x.bar(kQFull), kBoxes * C::kQBox);
    const int qrow = it.tok0 * p.num_heads + it.row0;
    for (int j = 0; j < kBoxes; ++j)
      tma_load_2d(smem_u32(x.smem + C::kOffQ + j * C::kQBox), &maps.q, 128 * j, qrow, x.bar(kQFull));
    issued[kIssuedQ] = ne;
    if (!wait_phase(x, x.bar(kQFull), ne & 1, 21)) break;
    for (int c = 0; c < it.n_chunks && ok; ++c, ++g) {
      const int b = g & 1;
      if (g >= 2 && !wait_phase(x, x.bar(kSFree + b), ((g - 2) >> 1) & 1, 22)) {
        ok = false;
        break;
      }
      const uint32_t d = x.tbase + C::kSCol + b * NR;
#pragma unroll
      for (int j = 0; j < kBoxes; ++j) {
        const bool rope = j == kBoxes - 1;
        const int i = rope ? g : g * (kBoxes - 1) + j;
        const int slot = i % (rope ? C::kRSlots : C::kSlots);
        const int use = i / (rope ? C::kRSlots : C::kSlots);
        if (!wait_phase<(CL > 1)>(x, x.bar(rope ? kRFull + slot : kFull + slot), use & 1, 23)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint64_t a = rope ? r_desc + static_cast<uint64_t>(slot * (kRSlot >> 4))
                                : k_desc + static_cast<uint64_t>(slot * (kSlot >> 4));
        const uint64_t qb = q_desc + static_cast<uint64_t>(j * (C::kQBox >> 4));
        // 32 e4m3 columns per instruction: 4 per latent box, 2 for the 64 rope columns
#pragma unroll
        for (int s = 0; s < (rope ? 2 : 4); ++s)
          mma_ss_f8(d, a + 2 * s, qb + 2 * s, kIdQK, (j | s) != 0 ? 1u : 0u);
        if (rope) release<CL>(x.bar(kREmpty + slot));  // the rope box's only read
      }
      if (!ok) break;
      mma_commit(x.bar(kSFull + b));
    }
    if (!ok) break;
    mma_commit(x.bar(kQFree));
    ++ne;
  }
  mma_commit(x.bar(kDrain));
  drain_wait(x, x.bar(kDrain), 0, 25);
}

template <int NR, int CL>
__device__ void pv_issue(const Ctx& x, const DecodeParams& p) {
  using C = HnCfg<NR>;
  if (x.lane != 0) return;
  constexpr uint32_t kIdPV = instr_desc(128, C::kNpv, 0, 0, true, true);
  const uint64_t v_desc = smem_desc_sw128(smem_u32(x.smem + C::kOffRing), kSlot, 1024);   // MN-major
  const uint64_t p_desc = smem_desc_interleave(smem_u32(x.smem + C::kOffP), C::kPLbo, 128);
  int g = 0, ne = 0;
  bool ok = true;
  for (int idx = x.it_begin; idx < x.it_end && ok; ++idx) {
    const Item it = item_at<NR, CL>(p, idx, x.rank);
    if (it.n_chunks == 0) continue;
    for (int c = 0; c < it.n_chunks; ++c, ++g) {
      const int b = g & 1;
      // O^T starts over: the previous item's epilogue must have read it
      if (c == 0 && ne > 0 && !wait_phase(x, x.bar(kOFree), (ne - 1) & 1, 28)) {
        ok = false;
        break;
      }
      // P^T of the chunk written; the softmax waited for S^T of the chunk,
      // whose QK^T waited for the very value boxes read here
      if (!wait_phase(x, x.bar(kPFull + b), (g >> 1) & 1, 24)) {
        ok = false;
        break;
      }
      fence_after_sync();
      const uint64_t pb = p_desc + static_cast<uint64_t>((g % C::kPBufs) * (C::kPBytes >> 4));
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int slot = (g * (kBoxes - 1) + m) % C::kSlots;
        const uint64_t a = v_desc + static_cast<uint64_t>(slot * (kSlot >> 4));
        const uint32_t dm = x.tbase + m * C::kNpv;
#pragma unroll
        for (int ks = 0; ks < kKeys / 32; ++ks) {
          const uint64_t av = a + static_cast<uint64_t>((ks * 32 * 128) >> 4);
          const uint64_t bv = pb + static_cast<uint64_t>((ks * 4 * C::kPLbo) >> 4);
          mma_ss_f8(dm, av, bv, kIdPV, (c | ks) != 0 ? 1u : 0u);
          if constexpr (!C::kConcat)  // the lo term: the next NR / 16 core matrices
            mma_ss_f8(dm, av, bv + static_cast<uint64_t>((NR / 16 * 128) >> 4), kIdPV, 1u);
        }
        release<CL>(x.bar(kEmpty + slot));  // the value box's last read
      }
      mma_commit(x.bar(kPFree + b));
    }
    if (!ok) break;
    mma_commit(x.bar(kOFull));
    ++ne;
  }
  mma_commit(x.bar(kDrainPV));
  drain_wait(x, x.bar(kDrainPV), 0, 26);
}

// ------------------------------------------------------------------ softmax + epilogue
// Loads NW consecutive 32-bit TMEM columns of this warp's lane quarter.
template <int NW>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[NW]) {
  static_assert(NW % 8 == 0, "8-column units");
#pragma unroll
  for (int u = 0; u < NW / 8; ++u) {
    uint32_t r[8];
    tmem_ld_32x32b_x8(taddr + 8 * u, r);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[8 * u + i] = __uint_as_float(r[i]);
  }
}

// p of two rows as two e4m3 code pairs: hi = e4m3(p), lo = e4m3(p - hi),
// formed in f16 (p rounded to 11 bits first; the difference is then exact).
__device__ __forceinline__ void p_terms(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  const __half2 ph = __floats2half2_rn(p0, p1);
  const uint32_t phb = *reinterpret_cast<const uint32_t*>(&ph);
  uint16_t h16, l16;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;\n" : "=h"(h16) : "r"(phb));
  uint32_t back;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(back) : "h"(h16));
  const __half2 d = __hsub2(ph, *reinterpret_cast<const __half2*>(&back));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;\n" : "=h"(l16) : "r"(*reinterpret_cast<const uint32_t*>(&d)));
  hi = h16;
  lo = l16;
}

// Eight warps: warp w owns the keys of TMEM lane quarter w % 4 and the rows
// [h NH, (h + 1) NH) of the CTA's rows, h = (w - 4) / 4, NH = NR / 2.
// Thread t8 < 64 (warps 4, 5) also owns row t8's reference and true maxima
// and causal end, which it resets for the next item in each epilogue.
template <int NR, int CL>
__device__ void softmax_rows(const Ctx& x, const HnMaps& maps, const DecodeParams& p) {
  using C = HnCfg<NR>;
  constexpr int NH = NR / 2;
  const int lane = x.lane;
  const int sw = x.warp - 4;                    // softmax warp 0..7
  const int q4 = x.warp & 3;                    // TMEM lane quarter of this warp
  const int r0 = (sw >> 2) * NH;                // first row of this warp
  const int k = q4 * 32 + lane;                 // the chunk key (S^T lane) this thread owns
  const int t8 = sw * 32 + lane;                // owner of row t8 in the exchanges
  const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
  float* wmax = reinterpret_cast<float*>(x.smem + kOffWmax);
  float* mref = reinterpret_cast<float*>(x.smem + kOffMref);
  float* mtrue = reinterpret_cast<float*>(x.smem + kOffMtrue);
  float* alpha = reinterpret_cast<float*>(x.smem + kOffAlpha);
  int* vis = reinterpret_cast<int*>(x.smem + kOffVis);
  float* lsum = reinterpret_cast<float*>(x.smem + kOffLsum);
  float* mult = reinterpret_cast<float*>(x.smem + kOffMult);
  const float scale2 = p.score_scale_log2;
  const int H = p.num_heads;
  uint8_t* pbuf0 = x.smem + C::kOffP + (k >> 3) * C::kPLbo + (k & 7) * 16;
  int g = 0;    // the worker's chunk count
  int ne = 0;   // items with keys so far
  int ni = 0;   // items so far
  bool ok = true;
  for (int idx = x.it_begin; idx < x.it_end && ok; ++idx, ++ni) {
    const Item it = item_at<NR, CL>(p, idx, x.rank);
    const int vis_min = vis[0];                 // row 0 of the CTA has the earliest causal end
    float l[NH];
#pragma unroll
    for (int n = 0; n < NH; ++n) l[n] = 0.f;
    for (int c = 0; c < it.n_chunks && ok; ++c, ++g) {
      const int b = g & 1;
      const uint32_t par = (g >> 1) & 1;
      ok = warp_wait(x, x.bar(kSFull + b), par, 31);
      if (!ok) break;
      fence_after_sync();
      float s[NH];  // raw scores q.k of this key for the warp's rows
      tmem_ld_cols<NH>(x.tbase + lane_off + C::kSCol + b * NR + r0, s);
      tmem_ld_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(x.bar(kSFree + b));  // QK^T two chunks on may overwrite it
      // keys that exist (inside the segment) and that each row may see; a
      // chunk inside the segment and before every row's causal end needs no mask
      const int pos = it.seg_start + c * kKeys + k;
      const bool key_ok = pos < it.seg_end;
      const int chunk_end = it.seg_start + (c + 1) * kKeys;
      const bool causal = it.qlen > 1 && chunk_end > vis_min;
      if (chunk_end > it.seg_end || causal) {
#pragma unroll
        for (int n = 0; n < NH; ++n)
          if (!(key_ok && (!causal || pos < vis[r0 + n]))) s[n] = -INFINITY;
      }
      // chunk max of every row over the raw scores (scale2 > 0): this warp's
      // 32 keys, then the four lane quarters
#pragma unroll
      for (int n = 0; n < NH; ++n) {
        const float r = warp_max_f32(s[n]);
        if (lane == (n & 31)) wmax[(b * 4 + q4) * 64 + r0 + n] = r;
      }
      ok = cross_sync(x, kXA + b, par, 32);
      if (!ok) break;
      // each warp moves the reference of its own rows (lane l: row r0 + l),
      // from the previous chunk's copy to this chunk's: the four warps of a
      // row half compute, and write, the same values
      float* mr = mref + b * 64;
      float* mt = mtrue + b * 64;
      float* al = alpha + b * 64;
      bool moved = false;
      if (lane < NH) {
        const int r = r0 + lane;
        const float* w = wmax + b * 256 + r;
        const float mc = fmaxf(fmaxf(w[0], w[64]), fmaxf(w[128], w[192])) * scale2;
        const float mo = mref[(b ^ 1) * 64 + r];
        mt[r] = fmaxf(mtrue[(b ^ 1) * 64 + r], mc);
        float a = 1.f, m = mo;
        if (mc > mo + kMove) {  // also when the row's first visible key arrives
          if (mo != -INFINITY) {
            a = fast_exp2(mo - mc);
            moved = true;
          }
          m = mc;
        }
        mr[r] = m;
        al[r] = a;
      }
      moved = __any_sync(0xffffffffu, moved);
      __syncwarp();
      if (moved) {
        // some of this warp's rows moved their reference: their sums and its
        // part of their O^T columns are rescaled
#pragma unroll
        for (int n = 0; n < NH; ++n) l[n] *= al[r0 + n];
        if (c > 0) {  // O^T holds P.V of the item's chunks < c: wait for the last of them
          ok = warp_wait(x, x.bar(kPFree + ((g - 1) & 1)), ((g - 1) >> 1) & 1, 34);
          if (!ok) break;
          fence_after_sync();
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int t = 0; t < (C::kConcat ? 2 : 1); ++t) {  // hi and lo columns
              const uint32_t ta = x.tbase + lane_off + m * C::kNpv + t * NR + r0;
#pragma unroll
              for (int u = 0; u < NH / 8; ++u) {
                uint32_t r[8];
                tmem_ld_32x32b_x8(ta + 8 * u, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  r[i] = __float_as_uint(__uint_as_float(r[i]) * al[r0 + 8 * u + i]);
                tmem_st_32x32b_x8(ta + 8 * u, r);
              }
            }
          }
          tmem_st_wait();
        }
      }
      // the P^T buffer is free once P.V of the chunk that used it last (two
      // chunks back, or one with a single buffer) has read it
      if (g >= C::kPBufs) {
        const int cp = g - C::kPBufs;
        ok = warp_wait(x, x.bar(kPFree + (cp & 1)), (cp >> 1) & 1, 35);
        if (!ok) break;
      }
      // p = 2^(s scale2 - m_ref + bias) as hi + lo e4m3 terms; rows in units of
      // 8 (an 8-byte half of a 16-row core matrix row)
      uint8_t* pk = pbuf0 + (g % C::kPBufs) * C::kPBytes;
#pragma unroll
      for (int u = 0; u < NH / 8; ++u) {
        const int R = r0 + 8 * u;  // first row of the unit
        uint32_t hw[2], lw[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t hc[2], lc[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int n = 8 * u + 4 * q + 2 * e;  // row index within the warp's rows
            const float2 m2 = *reinterpret_cast<const float2*>(mr + r0 + n);
            const float b0 = m2.x == -INFINITY ? 0.f : m2.x - kPBias;
            const float b1 = m2.y == -INFINITY ? 0.f : m2.y - kPBias;
            const float p0 = fast_exp2(fmaf(s[n], scale2, -b0));
            const float p1 = fast_exp2(fmaf(s[n + 1], scale2, -b1));
            l[n] += p0;
            l[n + 1] += p1;
            p_terms(p0, p1, hc[e], lc[e]);
          }
          hw[q] = hc[0] | (hc[1] << 16);
          lw[q] = lc[0] | (lc[1] << 16);
        }
        uint8_t* dst = pk + (R >> 4) * 128 + (R & 8);
        *reinterpret_cast<uint2*>(dst) = make_uint2(hw[0], hw[1]);
        *reinterpret_cast<uint2*>(dst + (NR / 16) * 128) = make_uint2(lw[0], lw[1]);
      }
      if (!key_ok) {
        // a key past the segment: its value row (stale or unloaded ring
        // contents, or cache rows past the sequence) must not reach O^T
        // through p = 0, so it is zeroed; each row half zeroes two of the
        // chunk's four value boxes
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
          const int m = 2 * (sw >> 2) + mm;
          uint4* row = reinterpret_cast<uint4*>(x.smem + C::kOffRing +
                                                ((g * (kBoxes - 1) + m) % C::kSlots) * kSlot + k * 128);
#pragma unroll
          for (int q = 0; q < 8; ++q) row[q] = z;
        }
      }
      fence_proxy_async_smem();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(x.bar(kPFull + b));
    }
    if (!ok) break;

    // ---------------------------------------------------------- epilogue
    if (it.n_chunks > 0) {
      ok = warp_wait(x, x.bar(kOFull), ne & 1, 36);
      if (!ok) break;
      fence_after_sync();
    }
#pragma unroll
    for (int n = 0; n < NH; ++n) {
      float v = l[n];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == (n & 31)) lsum[q4 * 64 + r0 + n] = v;
    }
    ok = cross_sync(x, kXE, ni & 1, 37);
    if (!ok) break;
    if (t8 < 64) {
      // the item's last chunk left the row state in buffer (g - 1) & 1,
      // which the next item's first chunk reads as its previous state
      const int lb = ((g - 1) & 1) * 64;
      if (t8 < NR) {
        const int rho = it.row0 + t8;
        const float L = (lsum[t8] + lsum[64 + t8]) + (lsum[128 + t8] + lsum[192 + t8]);
        const float base = mref[lb + t8] == -INFINITY ? 0.f : mref[lb + t8] - kPBias;  // the sums' reference
        float f = 0.f;
        if (rho < it.rows_total) {
          const int tok = it.tok0 + rho / H;
          const int head = rho % H;
          const int64_t th = static_cast<int64_t>(tok) * H + head;
          if (it.fin) {
            float lse = -INFINITY;
            if (p.sinks != nullptr) {
              const float s2 = p.sinks[head] * kLog2e;
              const float M = fmaxf(L > 0.f ? base : -INFINITY, s2);
              const float e = L > 0.f ? exp2f(base - M) : 0.f;
              const float W = L * e + exp2f(s2 - M);
              f = e / W;
              lse = kLn2 * (M + log2f(W));
            } else if (L > 0.f) {
              f = 1.f / L;
              lse = kLn2 * (base + log2f(L));
            }
            p.lse[th] = lse;
          } else {
            const int64_t ts = it.pslot >= 0 ? static_cast<int64_t>(it.pslot) * (CL * NR) + x.rank * NR + t8
                                             : th * p.num_segments + it.seg;
            const float mt = mtrue[lb + t8];
            p.segm_max[ts] = L > 0.f ? mt : -INFINITY;
            p.segm_expsum[ts] = L > 0.f ? L * exp2f(base - mt) : 0.f;
            f = L > 0.f ? 1.f / L : 0.f;
          }
        }
        mult[t8] = f * p.kv_scale;
      }
      // row t8's state for the next item (every warp's reads of this item's
      // state are behind the exchange above)
      mref[lb + t8] = -INFINITY;
      mtrue[lb + t8] = -INFINITY;
      if (idx + 1 < x.it_end) vis[t8] = visible_end(item_at<NR, CL>(p, idx + 1, x.rank), H, t8);
    }
    ok = cross_sync(x, kXF, ni & 1, 38);
    if (!ok) break;
    // O^T: lane = value column, column = row. A unit of 8 rows x this warp's
    // 32 columns is staged in shared memory (two buffers per warp) and
    // written by one TMA store, so that the warp never waits on global
    // stores; a unit cut by the end of the tile's rows is stored directly.
    const int rows_here = min(NR, it.rows_total - it.row0);
    uint8_t* stage = x.smem + C::kOffP + sw * 2048;
    int staged = 0;
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
      const int col = m * 128 + k;
#pragma unroll 1
      for (int u = 0; u < NH / 8; ++u) {
        const int ru = r0 + 8 * u;  // first row of the unit
        if (ru >= rows_here) break;
        float o[8];
        if (it.n_chunks > 0) {
          tmem_ld_cols<8>(x.tbase + lane_off + m * C::kNpv + ru, o);
          if constexpr (C::kConcat) {  // the lo terms' columns
            float o2[8];
            tmem_ld_cols<8>(x.tbase + lane_off + m * C::kNpv + NR + ru, o2);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] += o2[i];
          } else {
            tmem_ld_wait();
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = 0.f;
        }
        if (ru + 8 <= rows_here) {
          uint8_t* buf = stage + (staged & 1) * 1024;
          if (staged >= 2) {  // the store that read this buffer two units ago
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
          }
          if (it.fin) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              reinterpret_cast<__nv_bfloat16*>(buf + i * 64)[lane] = __float2bfloat16_rn(o[i] * mult[ru + i]);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) reinterpret_cast<float*>(buf + i * 128)[lane] = o[i] * mult[ru + i];
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            // rows of a tile are consecutive (token, head) rows, slot rows or
            // (token, head) rows of one segment
            const int x0 = m * 128 + q4 * 32;
            if (it.fin) {
              tma_store_3d(&maps.out, smem_u32(buf), x0, 0, it.tok0 * H + it.row0 + ru);
            } else if (it.pslot >= 0) {
              tma_store_3d(&maps.part, smem_u32(buf), x0, 0, it.pslot * (CL * NR) + x.rank * NR + ru);
            } else {
              tma_store_3d(&maps.part, smem_u32(buf), x0, it.seg, it.tok0 * H + it.row0 + ru);
            }
            bulk_commit_group();
          }
          ++staged;
          continue;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = ru + i;
          if (rr >= rows_here) break;
          const int rho = it.row0 + rr;
          const int64_t th = static_cast<int64_t>(it.tok0 + rho / H) * H + rho % H;
          const float v = o[i] * mult[rr];
          if (it.fin) {
            static_cast<__nv_bfloat16*>(p.out)[th * kRank + col] = __float2bfloat16_rn(v);
          } else {
            const int64_t ts = it.pslot >= 0 ? static_cast<int64_t>(it.pslot) * (CL * NR) + x.rank * NR + rr
                                             : th * p.num_segments + it.seg;
            p.segm_out[ts * kRank + col] = v;
          }
        }
      }
    }
    // the staging buffers are P^T space again from the next exchange on
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
    if (it.n_chunks > 0) {
      // O^T read: P.V of the next item may start over in it
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(x.bar(kOFree));
      ++ne;
    }
  }
  if (lane == 0) bulk_wait_all();  // the output stores have completed
  __syncwarp();
}

template <int NR, int CL>
__global__ void __launch_bounds__(kThreads, 1)
    decode_hn_kernel(const __grid_constant__ HnMaps maps, const DecodeParams p, int* status) {
  using C = HnCfg<NR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctx x;
  x.smem = smem;
  x.status = status;
  x.limit_ns = p.wait_ns != 0 ? p.wait_ns : kDefaultWaitNs;
  x.tid = threadIdx.x;
  x.warp = x.tid >> 5;
  x.lane = x.tid & 31;
  x.rank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  if (p.items != nullptr) {
    // balanced schedule: this worker's items, once the grid that wrote the
    // list has completed (a no-op unless launched as its programmatic dependent)
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    // the merge grid may launch once every CTA of this one has started
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int w = static_cast<int>(blockIdx.x) / CL;
    x.it_begin = p.worker_first[w];
    x.it_end = p.worker_first[w + 1];
  } else {
    x.it_begin = 0;
    x.it_end = 1;
  }

  x.bar0 = smem_u32(smem + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffTslot);
  x.abort = reinterpret_cast<volatile int*>(smem + kOffAbort);
  if (x.tid == 0) {
    *x.abort = 0;
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(x.bar(kFull + s), 1);
      mbar_init(x.bar(kEmpty + s), CL);
    }
    for (int s = 0; s < C::kRSlots; ++s) {
      mbar_init(x.bar(kRFull + s), 1);
      mbar_init(x.bar(kREmpty + s), CL);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(x.bar(kSFull + b), 1);
      mbar_init(x.bar(kSFree + b), kSoftWarps);
      mbar_init(x.bar(kPFull + b), kSoftWarps);
      mbar_init(x.bar(kPFree + b), 1);
      mbar_init(x.bar(kXA + b), kSoftWarps);
    }
    mbar_init(x.bar(kQFull), 1);
    mbar_init(x.bar(kQFree), 1);
    mbar_init(x.bar(kXE), kSoftWarps);
    mbar_init(x.bar(kXF), kSoftWarps);
    mbar_init(x.bar(kOFull), 1);
    mbar_init(x.bar(kOFree), kSoftWarps);
    mbar_init(x.bar(kDrain), 1);
    mbar_init(x.bar(kDrainPV), 1);
    fence_barrier_init();
  }
  if (x.tid <= kIssuedQ) reinterpret_cast<int*>(smem + kOffIssued)[x.tid] = -1;
  if (x.tid < 64) {
    // per-row state of the first item: reference and true maxima, causal end
    for (int b = 0; b < 2; ++b) {
      reinterpret_cast<float*>(smem + kOffMref)[b * 64 + x.tid] = -INFINITY;
      reinterpret_cast<float*>(smem + kOffMtrue)[b * 64 + x.tid] = -INFINITY;
    }
    if (x.it_begin < x.it_end)
      reinterpret_cast<int*>(smem + kOffVis)[x.tid] =
          visible_end(item_at<NR, CL>(p, x.it_begin, x.rank), p.num_heads, x.tid);
  }
  if (x.warp == 1) {
    tmem_alloc(smem_u32(tslot), C::kTmemAlloc);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if constexpr (CL > 1) cluster_sync();  // the peers' barriers exist before any remote arrive or load
  x.tbase = *tslot;

  if (x.warp == 0 || x.warp == 2) {
    produce<NR, CL>(x, maps, p, x.warp >> 1);
  } else if (x.warp == 1) {
    qk_issue<NR, CL>(x, maps, p);
  } else if (x.warp == 3) {
    pv_issue<NR, CL>(x, p);
  } else {
    softmax_rows<NR, CL>(x, maps, p);
  }

  __syncwarp();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (x.warp == 1) tmem_dealloc(x.tbase, C::kTmemAlloc);
  // every TMA load into this CTA's shared memory must have landed before the
  // CTA exits: per slot, the latest use armed here (by this CTA's loads or,
  // in a cluster, the peers', whose issue records are read once every CTA
  // has stopped issuing); all are consumed unless a wait gave up. Then q.
  if constexpr (CL > 1) cluster_sync();
  if (x.tid == 0) {
    const volatile int* issued = reinterpret_cast<const volatile int*>(smem + kOffIssued);
    for (int e = 0; e < kMaxSlots + kMaxRSlots; ++e) {
      const bool rope = e >= kMaxSlots;
      const int s = rope ? e - kMaxSlots : e;
      if (s >= (rope ? C::kRSlots : C::kSlots)) continue;
      int last = issued[e];
      if constexpr (CL > 1) {
        const uint32_t rec = smem_u32(smem + kOffIssued + 4 * e);
        for (int r = 0; r < CL; ++r)
          if (r != x.rank) last = max(last, ld_cluster_s32(map_to_rank(rec, r)));
      }
      if (last >= 0) drain_wait(x, x.bar(rope ? kRFull + s : kFull + s), last & 1, 12);
    }
    if (issued[kIssuedQ] >= 0) drain_wait(x, x.bar(kQFull), issued[kIssuedQ] & 1, 13);
  }
  // no CTA of the cluster exits while loads into another may still land
  if constexpr (CL > 1) cluster_sync();
}

template <int NR, int CL>
cudaError_t prepare(int* smem_bytes) {
  using C = HnCfg<NR>;
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(decode_hn_kernel<NR, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_acq_rel);
  }
  *smem_bytes = C::kSmem;
  return cudaSuccess;
}

template <int NR, int CL>
cudaError_t launch_rows(const HnMaps& maps, const DecodeParams& p, dim3 grid, int* status,
                        cudaStream_t stream) {
  int smem = 0;
  cudaError_t e = prepare<NR, CL>(&smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (CL > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = CL;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  // an ordinary launch after the schedule kernel: as a programmatic dependent
  // of it the 16-head e4m3 call measured 114.7 us against 110.6 us (the
  // kernel's griddepcontrol.wait is then a no-op)
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, decode_hn_kernel<NR, CL>, maps, p, status);
}

template <int NR>
cudaError_t max_pairs(int* n) {
  int smem = 0;
  cudaError_t e = prepare<NR, 2>(&smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, decode_hn_kernel<NR, 2>, &cfg);
}

}  // namespace

cudaError_t launch_decode_hn(const DecodeParams& p, int rows, int cluster, int64_t q_rows, int64_t kv_rows,
                             dim3 grid, int* status, cudaStream_t stream) {
  if (p.slots != nullptr) return cudaErrorNotSupported;
  if (p.items != nullptr && p.worker_first == nullptr) return cudaErrorInvalidValue;
  HnMaps maps{};
  cudaError_t e = make_row_map(&maps.q, p.q, static_cast<uint64_t>(q_rows), static_cast<uint32_t>(rows), true);
  if (e != cudaSuccess) return e;
  e = make_row_map(&maps.kv, p.kv, static_cast<uint64_t>(kv_rows), kHalf, true);
  if (e != cudaSuccess) return e;
  e = make_row_map(&maps.kvr, p.kv, static_cast<uint64_t>(kv_rows), kHalf, true, 64);
  if (e != cudaSuccess) return e;
  if (p.out != nullptr) {
    e = make_out_map(&maps.out, p.out, static_cast<uint64_t>(q_rows), 1, true);
    if (e != cudaSuccess) return e;
  }
  if (p.segm_out != nullptr) {
    e = p.items != nullptr ? make_out_map(&maps.part, p.segm_out, static_cast<uint64_t>(p.segm_rows), 1, false)
                           : make_out_map(&maps.part, p.segm_out, static_cast<uint64_t>(q_rows),
                                          static_cast<uint64_t>(p.num_segments), false);
    if (e != cudaSuccess) return e;
  }
  if (cluster == 1) {
    switch (rows) {
      case 16: return launch_rows<16, 1>(maps, p, grid, status, stream);
      case 32: return launch_rows<32, 1>(maps, p, grid, status, stream);
      case 48: return launch_rows<48, 1>(maps, p, grid, status, stream);
      case 64: return launch_rows<64, 1>(maps, p, grid, status, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (cluster == 2) {
    switch (rows) {
      case 48: return launch_rows<48, 2>(maps, p, grid, status, stream);
      case 64: return launch_rows<64, 2>(maps, p, grid, status, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t decode_hn_max_pairs(int rows, int* n) {
  switch (rows) {
    case 48: return max_pairs<48>(n);
    case 64: return max_pairs<64>(n);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
