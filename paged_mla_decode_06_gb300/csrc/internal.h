// internal.h -- parameter blocks and launchers shared between the C ABI
// layer (api.cu) and the kernels. Not part of the public interface.
#pragma once

#include <cstdint>
#include <cuda_runtime_api.h>

namespace mla {

// Decode kernel variants chosen by the planner.
enum KernelId : int32_t {
  kMmaRows16 = 1,   // warp-MMA split-K kernel, 16 query rows per CTA
  kMmaRows32 = 2,   // 32 rows per CTA
  kMmaRows64 = 3,   // 64 rows per CTA
  kTcPair128 = 4,   // tcgen05 CTA-pair kernel, 128 rows per pair
  kTcRowsN = 5,     // tcgen05 kernel with the query rows as N, 16..64 rows per CTA, 1-2 CTAs per tile
};

struct DecodeParams {
  const void* q;                 // [T, H, 576]
  const void* kv;                // [NB, BS, 576]
  const int32_t* block_table;    // dense
  int64_t bt_stride;
  const int32_t* seq_lens;       // dense [R]
  const int32_t* qo_indptr;      // dense [R+1] or null
  const int32_t* slots;          // sparse slot list or null
  const int32_t* slot_indptr;    // sparse [T+1] or null ([T, topk] layout)
  int32_t num_tokens, num_reqs, num_heads, block_size, topk;
  int32_t num_segments, tile_size, row_tiles;
  float score_scale_log2;        // softmax_scale * q_scale * kv_scale * log2(e)
  float kv_scale;
  const float* sinks;            // [H] or null (final mode only)
  int32_t final_mode;            // 1: write out/lse; 0: write segment partials
  float* segm_out;               // [T, H, NS, 512]; balanced schedule: [segm_rows, 512] slots
  int64_t segm_rows;
  float* segm_max;               // [T, H, NS]
  float* segm_expsum;            // [T, H, NS]
  void* out;                     // [T, H, 512] bf16
  float* lse;                    // [T, H]
  // balanced schedule (tensor-core kernel): item i = blockIdx.x / 2 is
  // {unit, tile, key begin, key end, partial slot or -1 (write out/lse)}
  // at items[8 i ..]; null selects the uniform NS partition
  const int32_t* items;
  const int32_t* n_items;
  // rows-as-N kernel: worker w (CTA or cluster) runs items
  // [worker_first[w], worker_first[w + 1]) in order
  const int32_t* worker_first;
  // bounded waits of the tensor-core kernels give up after this many
  // nanoseconds (0: the default, 2 s)
  uint64_t wait_ns;
};

// Balanced work list (sched.cu).
struct SchedParams {
  const int32_t* seq_lens;       // dense [R]
  const int32_t* qo_indptr;      // dense [R+1] or null
  const int32_t* slot_indptr;    // sparse [T+1] or null (topk per token)
  int32_t topk, sparse, num_units, num_heads, tiles_max;
  int32_t split_cap;             // item budget when segments are split
  int32_t tile_rows;             // query rows per row tile (and per partial slot)
  int32_t* items;                // [max_items, 8]
  int32_t* n_items;              // [1]
  int32_t* unit_tab;             // [num_units * tiles_max, 2]: first partial slot (-1), pieces
  // contiguous mode (non-null): items in sequence order, cut at every
  // multiple of cdiv(total, workers) groups, worker w's first item at
  // worker_first[w] ([workers + 1]); else longest first for one-item CTAs
  int32_t* worker_first;
  int32_t workers;               // the share of the groups is cdiv(total, workers)
};

cudaError_t launch_schedule(const SchedParams& p, cudaStream_t stream);

// Where the merge finds each token's partition length.
struct PartLens {
  const int32_t* lens;       // mode 0: lens[t]
  const int32_t* seq_lens;   // mode 1: seq_lens[request of t] via qo_indptr
  const int32_t* qo_indptr;
  const int32_t* indptr;     // mode 2: indptr[t+1] - indptr[t]
  int32_t num_reqs;
  int32_t constant;          // mode 3: constant
  int32_t mode;
};

struct MergeParams {
  const float* segm_out;
  const float* segm_max;
  const float* segm_expsum;
  PartLens part;
  int32_t num_tokens, num_heads, num_segments, rank, tile_size;
  const float* sinks;
  void* out;     // bf16
  float* lse;
  // balanced schedule: partials live in slots of 128 rows; unit_tab gives
  // each (unit, row tile) its first slot and piece count (null: uniform NS)
  const int32_t* unit_tab;
  int32_t tiles_max;
  int32_t tile_rows;   // rows per row tile and per partial slot
  int32_t sparse;
};

struct LseMergeParams {
  const void* shard_out;   // [W, T, H, rank] bf16
  const float* shard_lse;  // [W, T, H] natural log
  int32_t num_shards, num_tokens, num_heads, rank;
  const float* sinks;      // [H] or null
  void* out;               // [T, H, rank] bf16
  float* lse;              // [T, H]
};

cudaError_t launch_merge_lse(const LseMergeParams& p, cudaStream_t stream);

struct QPrepParams {
  const void* nope;          // [T, H, 512] bf16, strides in elements
  int64_t nope_st, nope_sh;
  const void* pe;            // [T, H, 64] bf16
  int64_t pe_st, pe_sh;
  int32_t num_tokens, num_heads;
  int32_t fp8;               // 1: e4m3 codes of q / q_scale; 0: bf16
  float q_scale;
  void* out;                 // [T, H, 576]
};

cudaError_t launch_concat_q(const QPrepParams& p, cudaStream_t stream);
cudaError_t launch_decode_mma(int32_t kernel, bool fp8, const DecodeParams& p, dim3 grid,
                              cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);
cudaError_t launch_index_convert(const int32_t* req_id, const int32_t* block_table,
                                 int32_t bt_rows, int32_t bt_cols, int64_t bt_stride,
                                 const int32_t* token_indices, int64_t ti_stride,
                                 int32_t num_tokens, int32_t topk, int32_t block_size,
                                 const int32_t* cu_seqlens, int32_t* out, cudaStream_t stream);

// Sparse front end (sparse_front.cu).
cudaError_t launch_sparse_seqlen(const int32_t* qsl, const int32_t* seq_lens, int32_t num_reqs,
                                 int32_t num_tokens, int32_t topk, int32_t* lens, int32_t* indptr,
                                 cudaStream_t stream);
cudaError_t launch_fit_kpool(const int32_t* ti, int64_t ti_stride, int32_t num_tokens, int32_t width,
                             int32_t topk, int32_t* out, int64_t out_stride, cudaStream_t stream);

// tcgen05 CTA-pair kernel: q_rows / kv_rows are the row counts of the q
// and cache tensors viewed as [rows, 576]; status (may be null) receives a
// nonzero code if a bounded wait times out.
cudaError_t launch_decode_tc(const DecodeParams& p, bool fp8, int64_t q_rows, int64_t kv_rows,
                             dim3 grid, int* status, cudaStream_t stream);

// tcgen05 kernel with the query rows as the MMA N dimension (e4m3, dense,
// block size a multiple of 64): rows = 16, 32, 48 or 64 query rows per CTA,
// `cluster` (1, or 2 with 48 or 64 rows) CTAs per row tile sharing its key
// boxes. With the balanced schedule the grid holds one CTA (cluster) per
// worker.
cudaError_t launch_decode_hn(const DecodeParams& p, int rows, int cluster, int64_t q_rows, int64_t kv_rows,
                             dim3 grid, int* status, cudaStream_t stream);
// Clusters of two CTAs of `rows` rows that can be resident at once on the
// current device.
cudaError_t decode_hn_max_pairs(int rows, int* n);

// Shared memory bytes a decode variant needs (host query for validation).
int decode_mma_smem_bytes(int32_t kernel, bool fp8);
int decode_tc_smem_bytes(bool fp8);

}  // namespace mla
