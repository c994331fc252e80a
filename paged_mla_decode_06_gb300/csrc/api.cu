// api.cu -- the C ABI declared in include/mla_decode.h: host-side argument
// checks, the planner, and the launches of the decode, merge and index
// kernels. Nothing here allocates device memory or synchronises a stream.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "mla_decode.h"

namespace {

constexpr int kHeadDim = 576;
constexpr int kRank = 512;
constexpr int kMaxHeads = 128;
constexpr int kMaxSegments = 64;
constexpr int kSparseTile = 64;
constexpr int64_t kRowsNMax = 128;  // query rows per request the rows-as-N kernel takes (a CTA pair)
constexpr int32_t kMaxWorkers = 1024;  // workers of the contiguous schedule
static_assert(sizeof(mla_problem_t) == 68 && sizeof(mla_plan_t) == 168,
              "the plan layout the bindings mirror");
constexpr size_t kWsAlign = 256;

thread_local const char* g_last_cuda_error = "";

mla_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MLA_OK;
  g_last_cuda_error = cudaGetErrorString(e);
  return MLA_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Largest power of two dividing the block, capped at 128
// (rocm_aiter_mla.py, _segmented_mla_page_size).
int32_t tile_for_block(int32_t bs) {
  const int32_t low = bs & -bs;
  return low < 128 ? low : 128;
}

mla_status_t check_problem(const mla_problem_t& p) {
  if (p.num_tokens < 0 || p.num_heads <= 0 || p.block_size <= 0) return MLA_ERR_INVALID_ARG;
  if (p.head_dim != kHeadDim || p.kv_lora_rank != kRank) return MLA_ERR_UNSUPPORTED;
  if (p.num_heads > kMaxHeads) return MLA_ERR_UNSUPPORTED;
  if (p.q_dtype != MLA_DTYPE_BF16 && p.q_dtype != MLA_DTYPE_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (p.kv_dtype != MLA_DTYPE_BF16 && p.kv_dtype != MLA_DTYPE_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (p.q_dtype != p.kv_dtype) return MLA_ERR_UNSUPPORTED;
  if (p.num_blocks <= 0) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(p.num_blocks) * p.block_size > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (p.num_segments < 0 || p.num_segments > kMaxSegments) return MLA_ERR_INVALID_ARG;
  if (p.num_sms < 0 || p.has_sinks < 0 || p.has_sinks > 1) return MLA_ERR_INVALID_ARG;
  if (p.topk < 0) return MLA_ERR_INVALID_ARG;
  if (p.kernel < MLA_KERNEL_AUTO || p.kernel > MLA_KERNEL_TCGEN05_ROWS_N) return MLA_ERR_INVALID_ARG;
  if (p.topk > 0) {
    if (p.topk % 128 != 0) return MLA_ERR_UNSUPPORTED;
    if (p.max_qlen > 1) return MLA_ERR_INVALID_ARG;  // sparse rows are single tokens
    if (p.num_tokens > 65535) return MLA_ERR_UNSUPPORTED;
  } else {
    if (p.num_reqs < 0 || p.max_blocks_per_req <= 0) return MLA_ERR_INVALID_ARG;
    if (p.max_seq_len < 0 || p.max_qlen < 1) return MLA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(p.max_seq_len) > static_cast<int64_t>(p.max_blocks_per_req) * p.block_size)
      return MLA_ERR_INVALID_ARG;
    if (p.num_reqs > 65535) return MLA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(p.max_qlen) * p.num_heads > (1 << 20)) return MLA_ERR_UNSUPPORTED;
  }
  return MLA_OK;
}

struct Inputs {
  const void* q;
  const void* kv;
  const int32_t* bt;
  int64_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* qo_indptr;
  const int32_t* slots;
  const int32_t* slot_indptr;
  float softmax_scale, q_scale, kv_scale;
};

mla_status_t check_inputs(const mla_plan_t* plan, const Inputs& in) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARG;
  const mla_problem_t& p = plan->prob;
  mla_status_t s = check_problem(p);
  if (s != MLA_OK) return s;
  if (plan->num_segments < 1 || plan->num_segments > kMaxSegments || plan->tile_size <= 0)
    return MLA_ERR_INVALID_ARG;
  if (p.num_tokens == 0) return MLA_OK;
  if (in.q == nullptr || in.kv == nullptr) return MLA_ERR_INVALID_ARG;
  if (!aligned(in.q, 16) || !aligned(in.kv, 16)) return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(in.softmax_scale) || !std::isfinite(in.q_scale) || !std::isfinite(in.kv_scale) ||
      !(in.softmax_scale > 0.f) || !(in.q_scale > 0.f) || !(in.kv_scale > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (p.topk > 0) {
    if (in.slots == nullptr || in.qo_indptr != nullptr) return MLA_ERR_INVALID_ARG;
    if (!aligned(in.slots, 4)) return MLA_ERR_INVALID_ARG;
  } else {
    if (in.bt == nullptr || in.seq_lens == nullptr || in.slots != nullptr) return MLA_ERR_INVALID_ARG;
    if (in.bt_stride < p.max_blocks_per_req) return MLA_ERR_INVALID_ARG;
    if (p.max_qlen > 1 && in.qo_indptr == nullptr) return MLA_ERR_INVALID_ARG;
    if (in.qo_indptr == nullptr && p.num_tokens != p.num_reqs) return MLA_ERR_INVALID_ARG;
    if (!aligned(in.bt, 4) || !aligned(in.seq_lens, 4)) return MLA_ERR_INVALID_ARG;
  }
  return MLA_OK;
}

mla::DecodeParams make_params(const mla_plan_t* plan, const Inputs& in) {
  const mla_problem_t& p = plan->prob;
  mla::DecodeParams d{};
  d.q = in.q;
  d.kv = in.kv;
  d.block_table = in.bt;
  d.bt_stride = in.bt_stride;
  d.seq_lens = in.seq_lens;
  d.qo_indptr = in.qo_indptr;
  d.slots = p.topk > 0 ? in.slots : nullptr;
  d.slot_indptr = p.topk > 0 ? in.slot_indptr : nullptr;
  d.num_tokens = p.num_tokens;
  d.num_reqs = p.num_reqs;
  d.num_heads = p.num_heads;
  d.block_size = p.block_size;
  d.topk = p.topk;
  d.num_segments = plan->num_segments;
  d.tile_size = plan->tile_size;
  d.row_tiles = plan->row_tiles;
  d.score_scale_log2 = in.softmax_scale * in.q_scale * in.kv_scale * 1.4426950408889634f;
  d.kv_scale = in.kv_scale;
  d.wait_ns = plan->wait_limit_us > 0 ? static_cast<uint64_t>(plan->wait_limit_us) * 1000ull : 0ull;
  return d;
}

mla::PartLens part_lens_for(const mla_plan_t* plan, const Inputs& in) {
  const mla_problem_t& p = plan->prob;
  mla::PartLens pl{};
  if (p.topk > 0) {
    if (in.slot_indptr != nullptr) {
      pl.mode = 2;
      pl.indptr = in.slot_indptr;
    } else {
      pl.mode = 3;
      pl.constant = p.topk;
    }
  } else {
    pl.mode = 1;
    pl.seq_lens = in.seq_lens;
    pl.qo_indptr = in.qo_indptr;
    pl.num_reqs = p.num_reqs;
  }
  return pl;
}

dim3 grid_of(const mla_plan_t* plan) {
  return dim3(static_cast<unsigned>(plan->grid_x), static_cast<unsigned>(plan->grid_y),
              static_cast<unsigned>(plan->grid_z));
}

// Workers of a balanced plan: split_items = 2 x workers partial slots (2 x
// workers x row tiles for the CTA pair, whose units' cuts split every tile).
int32_t plan_workers(const mla_plan_t* plan) {
  const int32_t per_cut = plan->kernel == mla::kTcPair128 && plan->row_tiles > 0 ? plan->row_tiles : 1;
  return plan->split_items / (2 * per_cut);
}

// Workspace pieces of the balanced schedule (after the status block):
// the item count, the items (32 bytes each), the unit table, each worker's
// first item (rows-as-N kernel), then the partial slots at the plan's
// segm_* offsets.
struct SchedLayout {
  size_t n_items, items, unit_tab, worker_first, end;
};

SchedLayout sched_layout(const mla_plan_t* plan) {
  const mla_problem_t& p = plan->prob;
  const size_t units = static_cast<size_t>(p.topk > 0 ? p.num_tokens : p.num_reqs);
  SchedLayout l;
  l.n_items = kWsAlign;
  l.items = 2 * kWsAlign;
  l.unit_tab = l.items + align_up(static_cast<size_t>(plan->max_items) * 32, kWsAlign);
  l.worker_first = l.unit_tab + align_up(units * static_cast<size_t>(plan->row_tiles) * 8, kWsAlign);
  l.end = l.worker_first + align_up((static_cast<size_t>(plan_workers(plan)) + 1) * 4, kWsAlign);
  return l;
}

// d.items selects the balanced grid: one CTA pair per item slot (CTA-pair
// kernel), one CTA or cluster per worker (rows-as-N kernel).
mla_status_t launch_decode(const mla_plan_t* plan, const mla::DecodeParams& d, int* status,
                           cudaStream_t stream) {
  if (plan->grid_z == 0) return MLA_OK;
  const mla_problem_t& p = plan->prob;
  const int64_t q_rows = static_cast<int64_t>(p.num_tokens) * p.num_heads;
  const int64_t kv_rows = static_cast<int64_t>(p.num_blocks) * p.block_size;
  const unsigned items = static_cast<unsigned>(plan->max_items);
  if (plan->kernel == mla::kTcPair128) {
    const dim3 grid = d.items != nullptr ? dim3(2u * items, 1u, 1u) : grid_of(plan);
    return cuda_status(mla::launch_decode_tc(d, p.kv_dtype == MLA_DTYPE_FP8_E4M3, q_rows, kv_rows,
                                             grid, status, stream));
  }
  if (plan->kernel == mla::kTcRowsN) {
    const int cluster = plan->tile_rows / plan->rows_per_cta;
    const unsigned workers = static_cast<unsigned>(plan_workers(plan));
    const dim3 grid = d.items != nullptr ? dim3(workers * cluster, 1u, 1u) : grid_of(plan);
    return cuda_status(mla::launch_decode_hn(d, plan->rows_per_cta, cluster, q_rows, kv_rows, grid,
                                             status, stream));
  }
  return cuda_status(mla::launch_decode_mma(plan->kernel, p.kv_dtype == MLA_DTYPE_FP8_E4M3, d,
                                            grid_of(plan), stream));
}

// ---- balanced schedule stages (plan->schedule == 1)

mla::SchedParams sched_params(const mla_plan_t* plan, const Inputs& in, uint8_t* ws) {
  const mla_problem_t& p = plan->prob;
  const SchedLayout l = sched_layout(plan);
  mla::SchedParams sp{};
  sp.seq_lens = in.seq_lens;
  sp.qo_indptr = in.qo_indptr;
  sp.slot_indptr = p.topk > 0 ? in.slot_indptr : nullptr;
  sp.topk = p.topk;
  sp.sparse = p.topk > 0 ? 1 : 0;
  sp.num_units = p.topk > 0 ? p.num_tokens : p.num_reqs;
  sp.num_heads = p.num_heads;
  sp.tiles_max = plan->row_tiles;
  sp.tile_rows = plan->tile_rows;
  sp.split_cap = plan->split_items;
  sp.items = reinterpret_cast<int32_t*>(ws + l.items);
  sp.n_items = reinterpret_cast<int32_t*>(ws + l.n_items);
  sp.unit_tab = reinterpret_cast<int32_t*>(ws + l.unit_tab);
  sp.workers = plan_workers(plan);
  if (plan->kernel == mla::kTcRowsN)  // workers run contiguous runs of items
    sp.worker_first = reinterpret_cast<int32_t*>(ws + l.worker_first);
  return sp;
}

mla_status_t check_scheduled(const mla_plan_t* plan, const void* workspace, size_t workspace_bytes) {
  if (plan == nullptr || plan->schedule != 1) return MLA_ERR_INVALID_ARG;
  if ((plan->kernel != mla::kTcPair128 && plan->kernel != mla::kTcRowsN) || plan->max_items <= 0 ||
      plan->split_items <= 0 || plan->row_tiles <= 0 || plan->rows_per_cta <= 0 ||
      plan->tile_rows < plan->rows_per_cta || plan_workers(plan) > kMaxWorkers || plan_workers(plan) < 1)
    return MLA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < plan->workspace_bytes) return MLA_ERR_WORKSPACE;
  if (!aligned(workspace, kWsAlign)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

mla_status_t run_schedule(const mla_plan_t* plan, const Inputs& in, uint8_t* ws, cudaStream_t stream) {
  return cuda_status(mla::launch_schedule(sched_params(plan, in, ws), stream));
}

mla_status_t run_items(const mla_plan_t* plan, const Inputs& in, const float* sinks, uint8_t* ws,
                       void* out, float* lse, cudaStream_t stream) {
  const mla::SchedParams sp = sched_params(plan, in, ws);
  mla::DecodeParams d = make_params(plan, in);
  d.items = sp.items;
  d.n_items = sp.n_items;
  d.worker_first = sp.worker_first;
  d.final_mode = 0;
  d.sinks = sinks;
  d.out = out;
  d.lse = lse;
  d.segm_out = reinterpret_cast<float*>(ws + plan->segm_output_offset);
  d.segm_rows = static_cast<int64_t>(plan->split_items) * plan->tile_rows;
  d.segm_max = reinterpret_cast<float*>(ws + plan->segm_max_offset);
  d.segm_expsum = reinterpret_cast<float*>(ws + plan->segm_expsum_offset);
  return launch_decode(plan, d, reinterpret_cast<int*>(ws + plan->status_offset), stream);
}

mla_status_t run_merge_items(const mla_plan_t* plan, const Inputs& in, const float* sinks, uint8_t* ws,
                             void* out, float* lse, cudaStream_t stream) {
  const mla_problem_t& p = plan->prob;
  const mla::SchedParams sp = sched_params(plan, in, ws);
  mla::MergeParams m{};
  m.segm_out = reinterpret_cast<float*>(ws + plan->segm_output_offset);
  m.segm_max = reinterpret_cast<float*>(ws + plan->segm_max_offset);
  m.segm_expsum = reinterpret_cast<float*>(ws + plan->segm_expsum_offset);
  m.part = part_lens_for(plan, in);
  m.num_tokens = p.num_tokens;
  m.num_heads = p.num_heads;
  m.num_segments = 1;
  m.rank = kRank;
  m.tile_size = plan->tile_size;
  m.sinks = sinks;
  m.out = out;
  m.lse = lse;
  m.unit_tab = sp.unit_tab;
  m.tiles_max = plan->row_tiles;
  m.tile_rows = plan->tile_rows;
  m.sparse = sp.sparse;
  return cuda_status(mla::launch_merge(m, stream));
}

}  // namespace

extern "C" {

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_DEVICE_STATUS: return "MLA_ERR_DEVICE_STATUS";
    default: return "MLA_ERR_UNKNOWN";
  }
}

const char* mla_last_cuda_error(void) { return g_last_cuda_error; }

int32_t mla_version(void) { return 101; }

mla_status_t mla_decode_plan(const mla_problem_t* prob, mla_plan_t* plan) {
  if (prob == nullptr || plan == nullptr) return MLA_ERR_INVALID_ARG;
  const mla_problem_t p = *prob;
  mla_status_t s = check_problem(p);
  if (s != MLA_OK) return s;
  std::memset(plan, 0, sizeof(*plan));
  plan->prob = p;

  int32_t sms = p.num_sms;
  if (sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_status(e);
  }
  plan->num_sms = sms;

  const bool sparse = p.topk > 0;
  const int32_t units = sparse ? p.num_tokens : p.num_reqs;
  const int64_t rows_per_unit = sparse ? p.num_heads : static_cast<int64_t>(p.num_heads) * p.max_qlen;
  // the CTA-pair kernel: 128-row tiles, dense (block size a multiple of 64) or sparse bf16;
  // the rows-as-N kernel: e4m3 dense (block size a multiple of 64), at most 64 rows
  const bool tc_ok = sparse ? p.kv_dtype == MLA_DTYPE_BF16 : p.block_size % 64 == 0;
  const bool rn_ok = !sparse && p.kv_dtype == MLA_DTYPE_FP8_E4M3 && p.block_size % 64 == 0 &&
                     rows_per_unit <= kRowsNMax;
  if (p.kernel == MLA_KERNEL_TCGEN05 && !tc_ok) return MLA_ERR_UNSUPPORTED;
  if (p.kernel == MLA_KERNEL_TCGEN05_ROWS_N && !rn_ok) return MLA_ERR_UNSUPPORTED;
  const bool use_rn = p.kernel == MLA_KERNEL_TCGEN05_ROWS_N || (p.kernel == MLA_KERNEL_AUTO && rn_ok);
  const bool use_pair = !use_rn && tc_ok && p.kernel != MLA_KERNEL_WARP_MMA;
  const bool use_tc = use_rn || use_pair;
  int32_t kernel, rows, cluster = 1;
  if (use_rn) {
    // up to 64 rows on one CTA; 65..128 rows on a cluster of two CTAs of
    // equal row counts, which share one pass over the request's keys
    kernel = mla::kTcRowsN;
    cluster = rows_per_unit > 64 ? 2 : 1;
    rows = static_cast<int32_t>(((rows_per_unit + cluster - 1) / cluster + 15) / 16 * 16);
    if (rows < 16) rows = 16;
  } else if (use_pair) {
    kernel = mla::kTcPair128;
    rows = 128;
  } else if (rows_per_unit <= 16) {
    kernel = mla::kMmaRows16;
    rows = 16;
  } else if (rows_per_unit <= 32) {
    kernel = mla::kMmaRows32;
    rows = 32;
  } else {
    kernel = mla::kMmaRows64;
    rows = 64;
  }
  const int32_t tile_rows = rows * cluster;  // rows of a row tile, one per CTA (cluster, pair)
  const int32_t row_tiles = static_cast<int32_t>((rows_per_unit + tile_rows - 1) / tile_rows);
  const int32_t tile = sparse ? kSparseTile : tile_for_block(p.block_size);
  const int32_t max_len = sparse ? p.topk : p.max_seq_len;

  int32_t ns = p.num_segments;
  // The tensor-core kernel with the planner's choice of segments takes the
  // balanced schedule: segment lengths follow the device-resident lengths
  // (sched.cu), at most two items per CTA pair when anything is split.
  const int64_t unit_tiles = static_cast<int64_t>(units) * row_tiles;
  const bool balanced = ns == 0 && use_tc && unit_tiles <= (1 << 20);
  if (balanced || (ns == 0 && use_tc)) {
    ns = 1;
  } else if (ns == 0) {
    // Enough CTAs for about two per SM, but no segment shorter than
    // ~512 keys: each extra segment costs a partial write and read.
    const int64_t per_seg = static_cast<int64_t>(units > 0 ? units : 1) * row_tiles;
    int64_t want = (2 * static_cast<int64_t>(sms) + per_seg - 1) / per_seg;
    const int64_t cap = max_len / 512 > 1 ? max_len / 512 : 1;
    if (want > cap) want = cap;
    if (want > 16) want = 16;
    ns = static_cast<int32_t>(want < 1 ? 1 : want);
  }

  plan->num_segments = ns;
  plan->tile_size = tile;
  plan->kernel = kernel;
  plan->rows_per_cta = rows;
  plan->tile_rows = tile_rows;
  plan->row_tiles = row_tiles;
  plan->grid_x = use_pair ? 2 * row_tiles : row_tiles * cluster;  // CTAs per row tile
  plan->grid_y = ns;
  plan->grid_z = units;
  plan->status_offset = 0;
  plan->workspace_bytes = kWsAlign;
  if (balanced) {
    // workers: CTA pairs of the 128-row kernel; CTAs or clusters of the
    // rows-as-N kernel, as many as can be resident at once
    int32_t workers = use_pair || cluster == 2 ? sms / 2 : sms;
    if (use_rn && cluster == 2 && p.num_sms == 0) {
      int pairs = 0;
      const cudaError_t e = mla::decode_hn_max_pairs(rows, &pairs);
      if (e != cudaSuccess) return cuda_status(e);
      if (pairs > 0 && pairs < workers) workers = pairs;
    }
    if (workers < 1) workers = 1;
    if (workers > kMaxWorkers) workers = kMaxWorkers;
    // the CTA pair cuts a unit of several row tiles once for all of them:
    // each cut then splits every tile (sched.cu)
    const int32_t per_cut = use_pair ? row_tiles : 1;
    const int32_t split_cap = 2 * workers * per_cut;
    plan->schedule = 1;
    plan->split_items = split_cap;
    plan->max_items = static_cast<int32_t>(unit_tiles + static_cast<int64_t>(workers) * per_cut);  // rows + cuts
    const SchedLayout l = sched_layout(plan);
    const size_t slot_rows = static_cast<size_t>(split_cap) * tile_rows;
    const size_t out_b = align_up(slot_rows * kRank * sizeof(float), kWsAlign);
    const size_t max_b = align_up(slot_rows * sizeof(float), kWsAlign);
    plan->segm_output_offset = l.end;
    plan->segm_max_offset = l.end + out_b;
    plan->segm_expsum_offset = l.end + out_b + max_b;
    plan->workspace_bytes = l.end + out_b + 2 * max_b;
  } else if (ns > 1) {
    const size_t th = static_cast<size_t>(p.num_tokens) * p.num_heads;
    const size_t out_b = align_up(th * ns * kRank * sizeof(float), kWsAlign);
    const size_t max_b = align_up(th * ns * sizeof(float), kWsAlign);
    plan->segm_output_offset = kWsAlign;
    plan->segm_max_offset = kWsAlign + out_b;
    plan->segm_expsum_offset = kWsAlign + out_b + max_b;
    plan->workspace_bytes = kWsAlign + out_b + 2 * max_b;
  }
  return MLA_OK;
}

mla_status_t mla_decode_segments(const mla_plan_t* plan, const void* q, const void* kv_cache,
                                 const int32_t* block_table, int64_t block_table_stride,
                                 const int32_t* seq_lens, const int32_t* qo_indptr,
                                 const int32_t* sparse_slots, const int32_t* sparse_indptr,
                                 float softmax_scale, float q_scale, float kv_scale,
                                 float* segm_output, float* segm_max, float* segm_expsum,
                                 cudaStream_t stream) {
  const Inputs in{q, kv_cache, block_table, block_table_stride, seq_lens, qo_indptr,
                  sparse_slots, sparse_indptr, softmax_scale, q_scale, kv_scale};
  mla_status_t s = check_inputs(plan, in);
  if (s != MLA_OK) return s;
  if (plan->prob.num_tokens == 0) return MLA_OK;
  if (segm_output == nullptr || segm_max == nullptr || segm_expsum == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(segm_output, 16) || !aligned(segm_max, 4) || !aligned(segm_expsum, 4))
    return MLA_ERR_INVALID_ARG;
  mla::DecodeParams d = make_params(plan, in);
  d.final_mode = 0;
  d.segm_out = segm_output;
  d.segm_max = segm_max;
  d.segm_expsum = segm_expsum;
  return launch_decode(plan, d, nullptr, stream);
}

mla_status_t mla_decode_fwd(const mla_plan_t* plan, const void* q, const void* kv_cache,
                            const int32_t* block_table, int64_t block_table_stride,
                            const int32_t* seq_lens, const int32_t* qo_indptr,
                            const int32_t* sparse_slots, const int32_t* sparse_indptr,
                            float softmax_scale, float q_scale, float kv_scale,
                            const float* sinks, void* workspace, size_t workspace_bytes,
                            void* out, float* lse, cudaStream_t stream) {
  const Inputs in{q, kv_cache, block_table, block_table_stride, seq_lens, qo_indptr,
                  sparse_slots, sparse_indptr, softmax_scale, q_scale, kv_scale};
  mla_status_t s = check_inputs(plan, in);
  if (s != MLA_OK) return s;
  const mla_problem_t& p = plan->prob;
  if ((sinks != nullptr) != (p.has_sinks == 1)) return MLA_ERR_INVALID_ARG;
  if (p.num_tokens == 0) return MLA_OK;
  if (out == nullptr || lse == nullptr || !aligned(out, 16) || !aligned(lse, 4))
    return MLA_ERR_INVALID_ARG;
  if (sinks != nullptr && !aligned(sinks, 4)) return MLA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < plan->workspace_bytes) return MLA_ERR_WORKSPACE;
  if (!aligned(workspace, kWsAlign)) return MLA_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws + plan->status_offset);
  mla::DecodeParams d = make_params(plan, in);
  if (plan->schedule == 1) {
    s = run_schedule(plan, in, ws, stream);
    if (s == MLA_OK) s = run_items(plan, in, sinks, ws, out, lse, stream);
    if (s == MLA_OK) s = run_merge_items(plan, in, sinks, ws, out, lse, stream);
    return s;
  }
  if (plan->num_segments == 1) {
    d.final_mode = 1;
    d.sinks = sinks;
    d.out = out;
    d.lse = lse;
    return launch_decode(plan, d, status, stream);
  }
  d.final_mode = 0;
  d.segm_out = reinterpret_cast<float*>(ws + plan->segm_output_offset);
  d.segm_max = reinterpret_cast<float*>(ws + plan->segm_max_offset);
  d.segm_expsum = reinterpret_cast<float*>(ws + plan->segm_expsum_offset);
  s = launch_decode(plan, d, status, stream);
  if (s != MLA_OK) return s;
  mla::MergeParams m{};
  m.segm_out = d.segm_out;
  m.segm_max = d.segm_max;
  m.segm_expsum = d.segm_expsum;
  m.part = part_lens_for(plan, in);
  m.num_tokens = p.num_tokens;
  m.num_heads = p.num_heads;
  m.num_segments = plan->num_segments;
  m.rank = kRank;
  m.tile_size = plan->tile_size;
  m.sinks = sinks;
  m.out = out;
  m.lse = lse;
  return cuda_status(mla::launch_merge(m, stream));
}

mla_status_t mla_workspace_status(const mla_plan_t* plan, const void* workspace, int32_t* code,
                                  int32_t clear, cudaStream_t stream) {
  if (plan == nullptr || workspace == nullptr || code == nullptr) return MLA_ERR_INVALID_ARG;
  if (!aligned(workspace, kWsAlign) || !aligned(code, 4)) return MLA_ERR_INVALID_ARG;
  uint8_t* word = static_cast<uint8_t*>(const_cast<void*>(workspace)) + plan->status_offset;
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess && clear != 0 && v != 0) e = cudaMemsetAsync(word, 0, sizeof(v), stream);
  if (e != cudaSuccess) return cuda_status(e);
  *code = v;
  return v == 0 ? MLA_OK : MLA_ERR_DEVICE_STATUS;
}

mla_status_t mla_decode_schedule(const mla_plan_t* plan, const int32_t* seq_lens,
                                 const int32_t* qo_indptr, const int32_t* sparse_indptr,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  mla_status_t s = check_scheduled(plan, workspace, workspace_bytes);
  if (s != MLA_OK) return s;
  s = check_problem(plan->prob);
  if (s != MLA_OK) return s;
  const mla_problem_t& p = plan->prob;
  if (p.num_tokens == 0) return MLA_OK;
  if (p.topk == 0) {
    if (seq_lens == nullptr || !aligned(seq_lens, 4)) return MLA_ERR_INVALID_ARG;
    if (p.max_qlen > 1 && qo_indptr == nullptr) return MLA_ERR_INVALID_ARG;
  }
  Inputs in{};
  in.seq_lens = seq_lens;
  in.qo_indptr = p.topk > 0 ? nullptr : qo_indptr;
  in.slot_indptr = p.topk > 0 ? sparse_indptr : nullptr;
  return run_schedule(plan, in, static_cast<uint8_t*>(workspace), stream);
}

mla_status_t mla_decode_items(const mla_plan_t* plan, const void* q, const void* kv_cache,
                              const int32_t* block_table, int64_t block_table_stride,
                              const int32_t* seq_lens, const int32_t* qo_indptr,
                              const int32_t* sparse_slots, const int32_t* sparse_indptr,
                              float softmax_scale, float q_scale, float kv_scale,
                              const float* sinks, void* workspace, size_t workspace_bytes,
                              void* out, float* lse, cudaStream_t stream) {
  const Inputs in{q, kv_cache, block_table, block_table_stride, seq_lens, qo_indptr,
                  sparse_slots, sparse_indptr, softmax_scale, q_scale, kv_scale};
  mla_status_t s = check_scheduled(plan, workspace, workspace_bytes);
  if (s != MLA_OK) return s;
  s = check_inputs(plan, in);
  if (s != MLA_OK) return s;
  const mla_problem_t& p = plan->prob;
  if ((sinks != nullptr) != (p.has_sinks == 1)) return MLA_ERR_INVALID_ARG;
  if (p.num_tokens == 0) return MLA_OK;
  if (out == nullptr || lse == nullptr || !aligned(out, 16) || !aligned(lse, 4))
    return MLA_ERR_INVALID_ARG;
  if (sinks != nullptr && !aligned(sinks, 4)) return MLA_ERR_INVALID_ARG;
  return run_items(plan, in, sinks, static_cast<uint8_t*>(workspace), out, lse, stream);
}

mla_status_t mla_merge_items(const mla_plan_t* plan, const int32_t* qo_indptr, const float* sinks,
                             void* workspace, size_t workspace_bytes, void* out, float* lse,
                             cudaStream_t stream) {
  mla_status_t s = check_scheduled(plan, workspace, workspace_bytes);
  if (s != MLA_OK) return s;
  s = check_problem(plan->prob);
  if (s != MLA_OK) return s;
  const mla_problem_t& p = plan->prob;
  if ((sinks != nullptr) != (p.has_sinks == 1)) return MLA_ERR_INVALID_ARG;
  if (p.num_tokens == 0) return MLA_OK;
  if (p.topk == 0 && p.max_qlen > 1 && qo_indptr == nullptr) return MLA_ERR_INVALID_ARG;
  if (out == nullptr || lse == nullptr || !aligned(out, 16) || !aligned(lse, 4))
    return MLA_ERR_INVALID_ARG;
  if (sinks != nullptr && !aligned(sinks, 4)) return MLA_ERR_INVALID_ARG;
  Inputs in{};
  in.qo_indptr = p.topk > 0 ? nullptr : qo_indptr;
  return run_merge_items(plan, in, sinks, static_cast<uint8_t*>(workspace), out, lse, stream);
}

mla_status_t mla_merge_segments(const float* segm_output, const float* segm_max,
                                const float* segm_expsum, const int32_t* part_lens,
                                int32_t num_tokens, int32_t num_heads, int32_t num_segments,
                                int32_t kv_lora_rank, int32_t tile_size, const float* sinks,
                                int32_t out_dtype, void* out, float* lse, cudaStream_t stream) {
  if (num_tokens < 0 || num_heads <= 0 || num_segments < 1 || num_segments > kMaxSegments ||
      tile_size <= 0)
    return MLA_ERR_INVALID_ARG;
  if (kv_lora_rank != 128 && kv_lora_rank != 256 && kv_lora_rank != 512) return MLA_ERR_INVALID_ARG;
  if (out_dtype != MLA_DTYPE_BF16) return MLA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return MLA_OK;
  if (segm_output == nullptr || segm_max == nullptr || segm_expsum == nullptr ||
      part_lens == nullptr || out == nullptr || lse == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(segm_output, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(segm_max, 4) || !aligned(segm_expsum, 4) || !aligned(part_lens, 4))
    return MLA_ERR_INVALID_ARG;
  if (sinks != nullptr && !aligned(sinks, 4)) return MLA_ERR_INVALID_ARG;
  mla::MergeParams m{};
  m.segm_out = segm_output;
  m.segm_max = segm_max;
  m.segm_expsum = segm_expsum;
  m.part.mode = 0;
  m.part.lens = part_lens;
  m.num_tokens = num_tokens;
  m.num_heads = num_heads;
  m.num_segments = num_segments;
  m.rank = kv_lora_rank;
  m.tile_size = tile_size;
  m.sinks = sinks;
  m.out = out;
  m.lse = lse;
  return cuda_status(mla::launch_merge(m, stream));
}

mla_status_t mla_merge_lse(const void* shard_out, const float* shard_lse, int32_t num_shards,
                           int32_t num_tokens, int32_t num_heads, int32_t kv_lora_rank,
                           const float* sinks, void* out, float* lse, cudaStream_t stream) {
  if (num_shards < 1 || num_tokens < 0 || num_heads <= 0) return MLA_ERR_INVALID_ARG;
  if (kv_lora_rank != 128 && kv_lora_rank != 256 && kv_lora_rank != 512) return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  if (shard_out == nullptr || shard_lse == nullptr || out == nullptr || lse == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(shard_out, 16) || !aligned(out, 16) || !aligned(shard_lse, 4) || !aligned(lse, 4) ||
      (sinks != nullptr && !aligned(sinks, 4)))
    return MLA_ERR_INVALID_ARG;
  mla::LseMergeParams m{};
  m.shard_out = shard_out;
  m.shard_lse = shard_lse;
  m.num_shards = num_shards;
  m.num_tokens = num_tokens;
  m.num_heads = num_heads;
  m.rank = kv_lora_rank;
  m.sinks = sinks;
  m.out = out;
  m.lse = lse;
  return cuda_status(mla::launch_merge_lse(m, stream));
}

mla_status_t mla_concat_quant_q(const void* ql_nope, int64_t nope_stride_t, int64_t nope_stride_h,
                                const void* q_pe, int64_t pe_stride_t, int64_t pe_stride_h,
                                int32_t num_tokens, int32_t num_heads, int32_t out_dtype,
                                float q_scale, void* out, cudaStream_t stream) {
  if (num_tokens < 0 || num_heads <= 0) return MLA_ERR_INVALID_ARG;
  if (out_dtype != MLA_DTYPE_BF16 && out_dtype != MLA_DTYPE_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (out_dtype == MLA_DTYPE_FP8_E4M3 && !(std::isfinite(q_scale) && q_scale > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  if (ql_nope == nullptr || q_pe == nullptr || out == nullptr) return MLA_ERR_INVALID_ARG;
  if (nope_stride_h < kRank || pe_stride_h < 64 || nope_stride_t < nope_stride_h * num_heads ||
      pe_stride_t < pe_stride_h * num_heads)
    return MLA_ERR_INVALID_ARG;
  // 16-byte vector loads of every 8-column group
  if (!aligned(ql_nope, 16) || !aligned(q_pe, 16) || !aligned(out, 16) || nope_stride_t % 8 ||
      nope_stride_h % 8 || pe_stride_t % 8 || pe_stride_h % 8)
    return MLA_ERR_INVALID_ARG;
  mla::QPrepParams q{};
  q.nope = ql_nope;
  q.nope_st = nope_stride_t;
  q.nope_sh = nope_stride_h;
  q.pe = q_pe;
  q.pe_st = pe_stride_t;
  q.pe_sh = pe_stride_h;
  q.num_tokens = num_tokens;
  q.num_heads = num_heads;
  q.fp8 = out_dtype == MLA_DTYPE_FP8_E4M3 ? 1 : 0;
  q.q_scale = q_scale;
  q.out = out;
  return cuda_status(mla::launch_concat_q(q, stream));
}

mla_status_t mla_sparse_seqlen(const int32_t* query_start_loc, const int32_t* seq_lens,
                               int32_t num_reqs, int32_t num_tokens, int32_t topk, int32_t* lens,
                               int32_t* indptr, cudaStream_t stream) {
  if (num_reqs < 0 || num_tokens < 0 || topk <= 0) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_tokens) * topk > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (indptr == nullptr || !aligned(indptr, 4)) return MLA_ERR_INVALID_ARG;
  if (lens != nullptr && !aligned(lens, 4)) return MLA_ERR_INVALID_ARG;
  if (query_start_loc == nullptr || !aligned(query_start_loc, 4)) return MLA_ERR_INVALID_ARG;
  if (num_reqs > 0 && (seq_lens == nullptr || !aligned(seq_lens, 4))) return MLA_ERR_INVALID_ARG;
  return cuda_status(mla::launch_sparse_seqlen(query_start_loc, seq_lens, num_reqs, num_tokens, topk, lens,
                                               indptr, stream));
}

mla_status_t mla_fit_kpool_indices(const int32_t* token_indices, int64_t ti_row_stride,
                                   int32_t num_tokens, int32_t width, int32_t topk, int32_t* out,
                                   int64_t out_row_stride, cudaStream_t stream) {
  if (num_tokens < 0 || topk <= 0 || width < topk) return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  if (token_indices == nullptr || out == nullptr || !aligned(token_indices, 4) || !aligned(out, 4))
    return MLA_ERR_INVALID_ARG;
  if (ti_row_stride < width || out_row_stride < topk) return MLA_ERR_INVALID_ARG;
  // the output must not overlap the input rows
  const uintptr_t in0 = reinterpret_cast<uintptr_t>(token_indices);
  const uintptr_t in1 = in0 + static_cast<uintptr_t>((num_tokens - 1) * ti_row_stride + width) * 4;
  const uintptr_t o0 = reinterpret_cast<uintptr_t>(out);
  const uintptr_t o1 = o0 + static_cast<uintptr_t>((num_tokens - 1) * out_row_stride + topk) * 4;
  if (o0 < in1 && in0 < o1) return MLA_ERR_INVALID_ARG;
  return cuda_status(mla::launch_fit_kpool(token_indices, ti_row_stride, num_tokens, width, topk, out,
                                           out_row_stride, stream));
}

mla_status_t mla_sparse_index_convert(const int32_t* req_id, const int32_t* block_table,
                                      int32_t bt_rows, int32_t bt_cols, int64_t bt_row_stride,
                                      const int32_t* token_indices, int64_t ti_row_stride,
                                      int32_t num_tokens, int32_t topk, int32_t block_size,
                                      const int32_t* cu_seqlens, int32_t* out,
                                      cudaStream_t stream) {
  if (num_tokens < 0 || topk <= 0 || topk % 128 != 0 || block_size <= 0) return MLA_ERR_INVALID_ARG;
  if (bt_rows <= 0 || bt_cols <= 0 || bt_row_stride < bt_cols || ti_row_stride < topk)
    return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_tokens) * (topk / 128) > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return MLA_OK;
  if (req_id == nullptr || block_table == nullptr || token_indices == nullptr || out == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(req_id, 4) || !aligned(block_table, 4) || !aligned(token_indices, 4) ||
      !aligned(out, 4) || (cu_seqlens != nullptr && !aligned(cu_seqlens, 4)))
    return MLA_ERR_INVALID_ARG;
  return cuda_status(mla::launch_index_convert(req_id, block_table, bt_rows, bt_cols, bt_row_stride,
                                               token_indices, ti_row_stride, num_tokens, topk,
                                               block_size, cu_seqlens, out, stream));
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the workspace is this file-scope device array.
// ---------------------------------------------------------------------------
}  // extern "C"

static __device__ __align__(256) unsigned char g_mla_static_scratch[MLA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_mla_static_scratch on the current device, looked up
// once per device and cached.
mla_status_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_mla_static_scratch);
    if (e != cudaSuccess) return cuda_status(e);
    if (p == nullptr) return MLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status_t mla_decode_fwd_static(const mla_plan_t* plan, const void* q, const void* kv_cache,
                                   const int32_t* block_table, int64_t block_table_stride,
                                   const int32_t* seq_lens, const int32_t* qo_indptr,
                                   const int32_t* sparse_slots, const int32_t* sparse_indptr,
                                   float softmax_scale, float q_scale, float kv_scale,
                                   const float* sinks, void* out, float* lse, int32_t* status_out,
                                   cudaStream_t stream) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARG;
  if (plan->workspace_bytes > MLA_STATIC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  if (plan->workspace_bytes < sizeof(int32_t) ||
      plan->status_offset > plan->workspace_bytes - sizeof(int32_t))
    return MLA_ERR_INVALID_ARG;
  if (status_out != nullptr && !aligned(status_out, 4)) return MLA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  mla_status_t s = static_scratch(&scratch);
  if (s != MLA_OK) return s;
  uint8_t* status = static_cast<uint8_t*>(scratch) + plan->status_offset;
  s = cuda_status(cudaMemsetAsync(status, 0, sizeof(int32_t), stream));
  if (s != MLA_OK) return s;
  s = mla_decode_fwd(plan, q, kv_cache, block_table, block_table_stride, seq_lens, qo_indptr,
                     sparse_slots, sparse_indptr, softmax_scale, q_scale, kv_scale, sinks,
                     scratch, MLA_STATIC_SCRATCH_BYTES, out, lse, stream);
  if (s != MLA_OK || status_out == nullptr) return s;
  return cuda_status(cudaMemcpyAsync(status_out, status, sizeof(int32_t),
                                     cudaMemcpyDeviceToDevice, stream));
}

}  // extern "C"
