// sched.cu -- the balanced work list of the tensor-core decode: split-K
// segments sized per batch from the device-resident lengths, so that every
// CTA pair gets about the same number of keys (a planner that fills the
// SMs). The "rocm_aiter_mla_sparse" page's ROCMAiterMLASparseImpl._forward_mla
// hands its decode call such a list (work_indptr, reduce_indptr,
// reduce_partial_map) on its persistent path.
//
// One block of 256 threads. A row is a (unit, row tile) pair, a unit being
// a request of the dense variant or a token of the sparse one, a row tile
// the query rows one CTA (pair) of the decode owns; a row covers
// the unit's g = cdiv(len, 128) key groups. The rows are laid end to end
// (unit-major) and the sequence of all their groups is cut every W =
// cdiv(total, workers) groups, as if each worker (a CTA pair of the
// 128-row kernel, a CTA of the rows-as-N kernel) took the next W groups;
// a cut closer than W / 8 to either end of its row is dropped, so that no
// piece is a sliver. Every row thus becomes k >= 1 pieces (one, of size 0,
// for an empty row, whose rows still get zeros and -inf). Items are written
// longest first: workers are handed out in launch order, so the ones that
// finish early take the short pieces (longest-processing-time list
// scheduling). Pieces of a split row write base-2 partials to consecutive
// partial slots; the unit table gives each row its first slot and its piece
// count, from which the merge finds them. Cuts number
// fewer than the workers, so the slots of split rows number at most two per
// worker and the items at most rows + workers.
// A unit of T > 1 row tiles (multi-token requests on the CTA pair) is cut
// once for all its tiles: the sequence is that of the units' g groups (W
// still the worker's share of all tiles' groups), so that the tiles' items
// cover the same keys. They are written next to each other, and their pairs
// read the keys together (one HBM pass, the other tiles hitting L2). Split
// units then own T k slots: at most 2 T_max per worker, and the items are at
// most rows + T_max workers. With one tile per unit this is the rule above.
//
// Contiguous mode (the rows-as-N kernel, whose workers run many items each):
// every multiple of W inside a row is a cut, so that worker w's share is
// exactly the groups [w W, (w + 1) W) of the sequence, and the items are
// written in sequence order with worker_first[w] = the first item of worker
// w (a piece belongs to the worker its first group falls to; an empty row,
// to the worker of its position).
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kGroupKeys = 128;   // piece boundaries fall on 128-key groups
constexpr int kSizeBins = 2048;   // ranking bins of piece sizes (in groups)
constexpr int kCacheUnits = 2048; // units whose sizes are kept in shared memory

struct UnitInfo {
  int groups;
  int tiles;
};

__device__ __forceinline__ UnitInfo unit_info_global(const SchedParams& p, int u) {
  int len, qlen = 1;
  if (p.sparse) {
    len = p.slot_indptr != nullptr ? p.slot_indptr[u + 1] - p.slot_indptr[u] : p.topk;
  } else {
    len = p.seq_lens[u];
    if (p.qo_indptr != nullptr) qlen = p.qo_indptr[u + 1] - p.qo_indptr[u];
  }
  UnitInfo i;
  i.groups = len > 0 ? cdiv(len, kGroupKeys) : 0;
  const int64_t rows = static_cast<int64_t>(qlen > 0 ? qlen : 0) * p.num_heads;
  const int64_t tiles = (rows + p.tile_rows - 1) / p.tile_rows;
  i.tiles = static_cast<int>(tiles < p.tiles_max ? tiles : p.tiles_max);
  return i;
}

// Block-wide sum over one value per thread.
__device__ long long block_sum(long long v, long long* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  long long s = 0;
  for (int w = 0; w < kThreads / 32; ++w) s += red[w];
  return s;
}

// Exclusive prefix of v over the block (thread order); *total gets the sum.
template <typename I>
__device__ I block_exclusive_scan(I v, long long* red, I* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  I inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const I n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  __syncthreads();
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  I before = 0, all = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    const I s = static_cast<I>(red[w]);
    if (w < warp) before += s;
    all += s;
  }
  *total = all;
  return before + inc - v;
}

// Cuts of the row occupying groups [a, a + g) of the sequence: multiples of
// W strictly inside, none within W / 8 of either end (unless `every`: all of
// them). Returns their number
// and the first one. I is int when the whole sequence fits (the usual case:
// 32-bit division is far cheaper), else long long.
template <typename I>
struct Cuts {
  I first;
  int count;
};

template <typename I>
__device__ __forceinline__ Cuts<I> row_cuts(I a, I g, I W, bool every = false) {
  const I d = every ? 0 : W / 8;
  const I lo = a + d + 1, hi = a + g - d - 1;  // allowed cut positions
  Cuts<I> c{0, 0};
  if (g > 0 && hi >= lo) {
    c.first = (lo + W - 1) / W * W;
    if (c.first <= hi) c.count = static_cast<int>((hi - c.first) / W + 1);
  }
  return c;
}

// Piece boundaries of a unit of g key groups at position a of the sequence
// of the units' groups: the multiples of W inside [a, a + g), none within
// W / 8 of its ends, as group offsets. All of the unit's row tiles are cut
// there. f(b) is called for each boundary in increasing order; returns
// their number.
template <typename I, typename F>
__device__ int unit_bounds(I a, int g, int T, I W, F f) {
  if (g <= 1 || T <= 0) return 0;
  const Cuts<I> c = row_cuts<I>(a, static_cast<I>(g), W);
  for (int j = 0; j < c.count; ++j) f(static_cast<int>(c.first + static_cast<I>(j) * W - a));
  return c.count;
}

// The histogram, the ranking and the items, with positions of type I. The
// T items of a piece (one per row tile) are written next to each other, so
// that the CTA pairs that read the same keys start together and the keys
// come from HBM once, the other tiles' reads hitting L2.
template <typename I, typename Info>
__device__ void schedule_items(const SchedParams& p, Info info, I W, long long* red, int* hist, int* start) {
  const int tid = threadIdx.x;
  const int U = p.num_units;
  auto bin_of = [](long long size) { return static_cast<int>(min(size, static_cast<long long>(kSizeBins - 1))); };
  // piece-size histogram (T items per piece); unit u starts at pos_u of
  // the sequence of the units' groups
  for (int b = tid; b < kSizeBins; b += kThreads) hist[b] = 0;
  I carry = 0;
  for (int u0 = 0; u0 < U; u0 += kThreads) {
    const int u = u0 + tid;
    UnitInfo i{0, 0};
    if (u < U) i = info(u);
    I sum;
    const I pos = carry + block_exclusive_scan<I>(static_cast<I>(i.groups), red, &sum);
    carry += sum;
    if (i.tiles > 0) {
      int prev = 0;
      unit_bounds<I>(pos, i.groups, i.tiles, W, [&](int b) {
        atomicAdd(&hist[bin_of(b - prev)], i.tiles);
        prev = b;
      });
      atomicAdd(&hist[bin_of(i.groups - prev)], i.tiles);
    }
  }
  __syncthreads();
  // start[b] = number of pieces in bins above b (kBinsPer bins per thread,
  // thread 0 taking the largest)
  {
    constexpr int kBinsPer = kSizeBins / kThreads;
    const int top = kSizeBins - 1 - kBinsPer * tid;
    int mine = 0;
#pragma unroll
    for (int j = 0; j < kBinsPer; ++j) mine += hist[top - j];
    int all;
    int before = block_exclusive_scan<int>(mine, red, &all);
#pragma unroll
    for (int j = 0; j < kBinsPer; ++j) {
      start[top - j] = before;
      before += hist[top - j];
    }
  }
  __syncthreads();
  for (int b = tid; b < kSizeBins; b += kThreads) hist[b] = 0;  // now the per-bin cursor
  __syncthreads();

  // items, unit table and partial slots (k per row tile of a split unit, tile-major)
  carry = 0;
  int slot_carry = 0;
  long long n_items = 0;
  for (int u0 = 0; u0 < U; u0 += kThreads) {
    const int u = u0 + tid;
    UnitInfo i{0, 0};
    if (u < U) i = info(u);
    I sum;
    const I pos = carry + block_exclusive_scan<I>(static_cast<I>(i.groups), red, &sum);
    carry += sum;
    const int k = i.tiles > 0 ? unit_bounds<I>(pos, i.groups, i.tiles, W, [](int) {}) + 1 : 0;
    const int nslots = k > 1 ? k * i.tiles : 0;
    int slot_sum;
    const int slot = slot_carry + block_exclusive_scan<int>(nslots, red, &slot_sum);
    slot_carry += slot_sum;
    if (i.tiles > 0) {
      for (int t = 0; t < i.tiles; ++t)
        reinterpret_cast<int2*>(p.unit_tab)[static_cast<int64_t>(u) * p.tiles_max + t] =
            make_int2(k > 1 ? slot + t * k : -1, k);
      int prev = 0, j = 0;
      auto emit = [&](int b) {
        const int at = start[bin_of(b - prev)] + atomicAdd(&hist[bin_of(b - prev)], i.tiles);
        const long long kb = static_cast<long long>(prev) * kGroupKeys;
        const long long ke = static_cast<long long>(b) * kGroupKeys;
        for (int t = 0; t < i.tiles; ++t) {
          int4* it = reinterpret_cast<int4*>(p.items) + 2 * static_cast<int64_t>(at + t);
          it[0] = make_int4(u, t, static_cast<int>(min(kb, static_cast<long long>(INT32_MAX))),
                            static_cast<int>(min(ke, static_cast<long long>(INT32_MAX))));
          it[1] = make_int4(k > 1 ? slot + t * k + j : -1, 0, 0, 0);
        }
        prev = b;
        ++j;
      };
      unit_bounds<I>(pos, i.groups, i.tiles, W, emit);
      emit(i.groups);
      n_items += static_cast<long long>(k) * i.tiles;
    }
  }
  n_items = block_sum(n_items, red);
  if (tid == 0) *p.n_items = static_cast<int32_t>(n_items);
}

// Exclusive prefixes of three per-thread counts over the block (thread
// order) and their totals.
__device__ int3 block_exclusive_scan3(int3 v, int3* red3, int3* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int3 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, inc.x, o);
    const int b = __shfl_up_sync(0xffffffffu, inc.y, o);
    const int c = __shfl_up_sync(0xffffffffu, inc.z, o);
    if (lane >= o) {
      inc.x += a;
      inc.y += b;
      inc.z += c;
    }
  }
  __syncthreads();
  if (lane == 31) red3[warp] = inc;
  __syncthreads();
  int3 before = make_int3(0, 0, 0), all = make_int3(0, 0, 0);
#pragma unroll 1
  for (int w = 0; w < kThreads / 32; ++w) {
    const int3 r = red3[w];
    if (w < warp) {
      before.x += r.x;
      before.y += r.y;
      before.z += r.z;
    }
    all.x += r.x;
    all.y += r.y;
    all.z += r.z;
  }
  *total = all;
  return make_int3(before.x + inc.x - v.x, before.y + inc.y - v.y, before.z + inc.z - v.z);
}

// The longest-first list when the units fit one per thread and their pieces
// fit kSmallPieces: each piece's place is counted directly (the items of
// the pieces larger than it, or as large and earlier in unit order), so the
// list is the same on every run and the kernel runs a few short phases (it
// is on the call's critical path, mostly waiting for its own code to load).
// Same pieces, slots and unit table as schedule_items. Returns false, having
// written nothing, when the pieces do not fit.
constexpr int kSmallPieces = 512;
static_assert(kSmallPieces <= 4096, "order keys hold the list position in 12 bits");

// Order key of piece q of the small list: its size in groups (clamped to 19
// bits: pieces that long are in any order among themselves), then its list
// position q < 4096 (earlier first). Distinct for distinct q.
__device__ __forceinline__ int order_key(int size, int q) {
  return (min(size, (1 << 19) - 1) << 12) | (4095 - q);
}

template <typename I>
__device__ bool schedule_items_small(const SchedParams& p, UnitInfo i, I W, long long* red, int4* pcs,
                                     int* scratch) {
  const int tid = threadIdx.x;
  const int u = tid;
  int* unit_k = scratch;                      // [kThreads] pieces of unit u
  int* unit_slot = scratch + kThreads;        // [kThreads] its first partial slot (-1)
  // [kSmallPieces + 4] order keys: larger = earlier in the list (size in
  // groups, then list order), -1 past the last piece
  int* pkey = scratch + 2 * kThreads;
  int* ptile = pkey + kSmallPieces + 4;       // [kSmallPieces + 4] row tiles (items) of each piece
  I sum;
  const I pos = block_exclusive_scan<I>(static_cast<I>(i.groups), red, &sum);
  Cuts<I> c{0, 0};
  if (i.tiles > 0 && i.groups > 1) c = row_cuts<I>(pos, static_cast<I>(i.groups), W);
  const int k = i.tiles > 0 ? c.count + 1 : 0;
  int3 tot;
  const int3 base = block_exclusive_scan3(make_int3(k, k > 1 ? k * i.tiles : 0, k * i.tiles),
                                          reinterpret_cast<int3*>(red + kThreads / 32), &tot);
  if (tot.x > kSmallPieces) return false;  // the same for every thread
  if (k > 0) {
    unit_k[u] = k;
    unit_slot[u] = k > 1 ? base.y : -1;
    int prev = 0;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
      const int next = j < c.count ? static_cast<int>(c.first + static_cast<I>(j) * W - pos) : i.groups;
      pcs[base.x + j] = make_int4(next - prev, u, prev, j);
      pkey[base.x + j] = order_key(next - prev, base.x + j);
      ptile[base.x + j] = i.tiles;
      prev = next;
    }
#pragma unroll 1
    for (int t = 0; t < i.tiles; ++t)
      reinterpret_cast<int2*>(p.unit_tab)[static_cast<int64_t>(u) * p.tiles_max + t] =
          make_int2(k > 1 ? base.y + t * k : -1, k);
  }
  const int P = tot.x;
  if (tid < 4) {  // pad to whole int4s: before no piece
    pkey[P + tid] = -1;
    ptile[P + tid] = 0;
  }
  __syncthreads();
  const int4* pk4 = reinterpret_cast<const int4*>(pkey);
  const int4* pt4 = reinterpret_cast<const int4*>(ptile);
#pragma unroll 1
  for (int q = tid; q < P; q += kThreads) {
    const int4 me = pcs[q];
    const int kq = pkey[q];
    // items of the pieces before this one (one compare per piece, no branch)
    int at = 0;
#pragma unroll 4
    for (int o = 0; o < P; o += 4) {
      const int4 a = pk4[o >> 2];
      const int4 b = pt4[o >> 2];
      at += a.x > kq ? b.x : 0;
      at += a.y > kq ? b.y : 0;
      at += a.z > kq ? b.z : 0;
      at += a.w > kq ? b.w : 0;
    }
    const int T = ptile[q], km = unit_k[me.y], slot0 = unit_slot[me.y];
    const int kb = static_cast<int>(min(static_cast<long long>(me.z) * kGroupKeys, static_cast<long long>(INT32_MAX)));
    const int ke =
        static_cast<int>(min(static_cast<long long>(me.z + me.x) * kGroupKeys, static_cast<long long>(INT32_MAX)));
#pragma unroll 1
    for (int t = 0; t < T; ++t) {
      int4* it = reinterpret_cast<int4*>(p.items) + 2 * static_cast<int64_t>(at + t);
      it[0] = make_int4(me.y, t, kb, ke);
      it[1] = make_int4(km > 1 ? slot0 + t * km + me.w : -1, 0, 0, 0);
    }
  }
  if (tid == 0) *p.n_items = tot.z;
  return true;
}

// Contiguous mode: items in sequence order and each worker's first item.
template <typename I, typename Info>
__device__ void schedule_contiguous(const SchedParams& p, Info info, I W, int workers, long long* red,
                                    int* owned) {
  const int tid = threadIdx.x;
  const int U = p.num_units;
  for (int w = tid; w < workers; w += kThreads) owned[w] = 0;
  __syncthreads();
  I carry = 0;
  int piece_carry = 0, slot_carry = 0;
  for (int u0 = 0; u0 < U; u0 += kThreads) {
    const int u = u0 + tid;
    UnitInfo i{0, 0};
    if (u < U) i = info(u);
    I sum;
    const I pos = carry + block_exclusive_scan<I>(static_cast<I>(i.tiles) * i.groups, red, &sum);
    carry += sum;
    int npieces = 0, nslots = 0;
    for (int t = 0; t < i.tiles; ++t) {
      const Cuts<I> c = row_cuts<I>(pos + static_cast<I>(t) * i.groups, i.groups, W, true);
      npieces += c.count + 1;
      if (c.count > 0) nslots += c.count + 1;
    }
    int piece_sum, slot_sum;
    int at = piece_carry + block_exclusive_scan<int>(npieces, red, &piece_sum);
    piece_carry += piece_sum;
    int slot = slot_carry + block_exclusive_scan<int>(nslots, red, &slot_sum);
    slot_carry += slot_sum;
    for (int t = 0; t < i.tiles; ++t) {
      const I a = pos + static_cast<I>(t) * i.groups;
      const Cuts<I> c = row_cuts<I>(a, i.groups, W, true);
      const int k = c.count + 1;
      const int pbase = k > 1 ? slot : -1;
      reinterpret_cast<int2*>(p.unit_tab)[static_cast<int64_t>(u) * p.tiles_max + t] = make_int2(pbase, k);
      I prev = a;
      for (int j = 0; j < k; ++j, ++at) {
        const I next = j < c.count ? c.first + j * W : a + i.groups;
        const long long owner = min(static_cast<long long>(prev / W), static_cast<long long>(workers - 1));
        atomicAdd(&owned[owner], 1);
        int4* it = reinterpret_cast<int4*>(p.items) + 2 * static_cast<int64_t>(at);
        const long long kb = static_cast<long long>(prev - a) * kGroupKeys;
        const long long ke = static_cast<long long>(next - a) * kGroupKeys;
        it[0] = make_int4(u, t, static_cast<int>(min(kb, static_cast<long long>(INT32_MAX))),
                          static_cast<int>(min(ke, static_cast<long long>(INT32_MAX))));
        it[1] = make_int4(k > 1 ? pbase + j : -1, 0, 0, 0);
        prev = next;
      }
      if (k > 1) slot += k;
    }
  }
  __syncthreads();
  // worker_first: exclusive scan of the pieces each worker owns
  int first = 0;
  for (int w0 = 0; w0 < workers; w0 += kThreads) {
    const int w = w0 + tid;
    int all;
    const int ex = block_exclusive_scan<int>(w < workers ? owned[w] : 0, red, &all);
    if (w < workers) p.worker_first[w] = first + ex;
    first += all;
  }
  if (tid == 0) {
    p.worker_first[workers] = first;
    *p.n_items = first;
  }
}

__global__ void __launch_bounds__(kThreads, 1) schedule_kernel(const SchedParams p) {
  // the decode kernel may launch now; it waits for this grid before reading
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  __shared__ long long red[kThreads / 32 * 3];  // block_exclusive_scan3 uses the last 16 as int3[8]
  __shared__ __align__(16) int hist[kSizeBins];
  __shared__ __align__(16) int start[kSizeBins];
  __shared__ int cache_g[kCacheUnits];
  __shared__ int cache_t[kCacheUnits];
  const int tid = threadIdx.x;
  const int U = p.num_units;
  const bool cached = U <= kCacheUnits;
  auto info = [&](int u) -> UnitInfo {
    if (cached) return UnitInfo{cache_g[u], cache_t[u]};
    return unit_info_global(p, u);
  };

  // total groups over all rows
  long long total = 0;
  for (int u = tid; u < U; u += kThreads) {
    const UnitInfo i = unit_info_global(p, u);
    if (cached) {
      cache_g[u] = i.groups;
      cache_t[u] = i.tiles;
    }
    total += static_cast<long long>(i.tiles) * i.groups;
  }
  total = block_sum(total, red);  // (its barriers also publish the cache)
  if (p.worker_first != nullptr) {
    const int workers = p.workers > 0 ? (p.workers < kSizeBins ? p.workers : kSizeBins) : 1;
    const long long W = total > 0 ? (total + workers - 1) / workers : 1;
    if (total < (1ll << 30))
      schedule_contiguous<int>(p, info, static_cast<int>(W), workers, red, hist);
    else
      schedule_contiguous<long long>(p, info, W, workers, red, hist);
    return;
  }
  const long long workers = p.workers > 0 ? p.workers : 1;
  const long long W = total > 0 ? (total + workers - 1) / workers : 1;
  if (U <= kThreads && total < (1ll << 30)) {
    static_assert(kSmallPieces * 16 <= kSizeBins * 4 && 2 * kThreads + 2 * (kSmallPieces + 4) <= kSizeBins,
                  "small-list scratch");
    const UnitInfo mine = tid < U ? UnitInfo{cache_g[tid], cache_t[tid]} : UnitInfo{0, 0};
    if (schedule_items_small<int>(p, mine, static_cast<int>(W), red, reinterpret_cast<int4*>(hist), start))
      return;
  }
  if (total < (1ll << 30))
    schedule_items<int>(p, info, static_cast<int>(W), red, hist, start);
  else
    schedule_items<long long>(p, info, W, red, hist, start);
}

}  // namespace

cudaError_t launch_schedule(const SchedParams& p, cudaStream_t stream) {
  schedule_kernel<<<1, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
