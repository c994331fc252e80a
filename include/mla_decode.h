/*
 * mla_decode.h -- C ABI of the paged MLA decode library for GB300 (sm_103a).
 *
 * Multi-head latent attention decode over a paged latent KV cache. Every
 * cache slot holds one 576-wide row: c_kv (kv_lora_rank = 512 columns)
 * followed by k_pe (64 rope columns). Scores use all 576 columns; the values
 * are the first 512 columns of the same row. The KV sequence of every row is
 * split into segments (split-K); each segment produces base-2 partials
 * (max, expsum, normalised partial output) and a merge produces the output
 * plus a natural-log LSE. Optional per-head fp32 sink logits, e4m3 fp8 q/KV
 * with per-tensor scales, multi-token causal rows and a sparse top-k variant
 * whose per-request positions are mapped through the block table.
 *
 * Sources (vLLM pages on the ROCm AITER MLA backend):
 *   [merge]  "vllm.v1.attention.ops.rocm_aiter_mla_merge", module docstring
 *            and merge_mla_segments_triton (partition, base-2 partials,
 *            natural-log LSE, shapes).
 *   [sparse] "vllm.v1.attention.backends.mla.rocm_aiter_mla_sparse":
 *            ROCMAiterMLASparseImpl.__init__ (sinks must be fp32 [H]),
 *            _forward_mla (sink fold, empty rows), forward_mqa (q layout,
 *            fp8 per-tensor scales), triton_convert_req_index_to_global_index
 *            (index formula, -1 rules, topk % 128 == 0).
 *   [dense]  "vllm/v1/attention/backends/mla/rocm_aiter_mla.py" (source
 *            listing): forward_mqa (q [T, H, 576], cache view), the
 *            segmented call in _forward_segmented_dcp_verify,
 *            _segmented_mla_page_size (tile rule) and
 *            dcp_local_verify_row_lens (causal bound of multi-token rows).
 *
 * Conventions shared by every entry point:
 *   - The caller owns all memory. Every pointer argument except the plan and
 *     problem structs is a DEVICE pointer. The library allocates nothing and
 *     never synchronises the stream; all work is enqueued on `stream`.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns an error status and launches nothing. Nothing is
 *     thrown across the ABI.
 *   - MLA_ERR_CUDA means a launch failed (cudaGetLastError after the launch);
 *     mla_last_cuda_error() gives the CUDA error string of the calling thread.
 *   - Contiguous layouts unless a stride is given. Rows of q and of the cache
 *     are 576 elements; q, kv_cache and out must be 16-byte aligned,
 *     workspace 256-byte aligned, lse and the float/int arrays 4-byte aligned.
 *   - Values the host cannot see (block-table entries, seq_lens, slots) are
 *     trusted to be in range: block_table entries in [0, num_blocks),
 *     0 <= seq_lens[r] <= max_blocks_per_req * block_size, seq_lens[r] >=
 *     qlen_r, slots in [-1, num_blocks * block_size).
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* a shape, pointer, alignment or enum is invalid */
  MLA_ERR_UNSUPPORTED = 2,   /* valid but not built (e.g. head_dim != 576) */
  MLA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than the plan needs */
  MLA_ERR_CUDA = 4,          /* a CUDA launch failed; see mla_last_cuda_error() */
  MLA_ERR_DEVICE_STATUS = 5  /* a kernel's bounded internal wait ran out: its status
                                word in the workspace is set (mla_workspace_status) */
} mla_status_t;

typedef enum {
  MLA_DTYPE_BF16 = 0,        /* bfloat16 */
  MLA_DTYPE_FP8_E4M3 = 1     /* OCP e4m3fn, value = code * per-tensor scale */
} mla_dtype_t;

/* Host-side description of one decode call ([dense] forward_mqa, [sparse]
 * forward_mqa). */
typedef struct {
  int32_t num_tokens;          /* T: rows of q, out and lse */
  int32_t num_reqs;            /* R: dense requests (rows of block_table, seq_lens);
                                  ignored by the sparse variant */
  int32_t num_heads;           /* H, 1..128 */
  int32_t head_dim;            /* 576 (512 + 64); other values are unsupported */
  int32_t kv_lora_rank;        /* 512 */
  int32_t block_size;          /* tokens per physical cache block (> 0) */
  int32_t max_blocks_per_req;  /* columns of block_table that may be read */
  int32_t num_blocks;          /* physical blocks in the cache */
  int32_t max_seq_len;         /* host upper bound of seq_lens (dense) */
  int32_t max_qlen;            /* max tokens per request; 1 when qo_indptr is NULL */
  int32_t topk;                /* 0 = dense; > 0 = sparse, longest slot list per token */
  int32_t q_dtype;             /* mla_dtype_t */
  int32_t kv_dtype;            /* mla_dtype_t; must equal q_dtype */
  int32_t has_sinks;           /* 1 when a sinks array will be passed */
  int32_t num_segments;        /* split-K segments per row; 0 lets the planner choose */
  int32_t num_sms;             /* SMs to plan for; 0 queries the current device */
  int32_t kernel;              /* 0 lets the planner choose the decode kernel; else a
                                  mla_kernel_t value (MLA_ERR_UNSUPPORTED if it cannot
                                  run this problem) */
} mla_problem_t;

/* Decode kernel variants. MLA_KERNEL_AUTO takes MLA_KERNEL_TCGEN05_ROWS_N
 * where it can run, else MLA_KERNEL_TCGEN05, else MLA_KERNEL_WARP_MMA. */
typedef enum {
  MLA_KERNEL_AUTO = 0,
  MLA_KERNEL_WARP_MMA = 1,     /* warp-level MMA split-K kernel: every shape */
  MLA_KERNEL_TCGEN05 = 2,      /* tcgen05/TMEM CTA-pair kernel, 128 query rows
                                  per pair as the MMA M dimension: dense bf16
                                  or e4m3 with block_size a multiple of 64, or
                                  sparse bf16 */
  MLA_KERNEL_TCGEN05_ROWS_N = 3 /* tcgen05/TMEM kernel with the query rows as
                                  the MMA N dimension, one CTA per 16..64 rows
                                  (a cluster of two CTAs sharing each key box
                                  for 65..128 rows):
                                  dense e4m3 with block_size a multiple of 64
                                  and num_heads * max_qlen <= 128 */
} mla_kernel_t;

/* Filled by mla_decode_plan; pass it unchanged to mla_decode_fwd or
 * mla_decode_segments. */
typedef struct {
  mla_problem_t prob;
  int32_t num_segments;        /* NS actually used (>= 1) */
  int32_t tile_size;           /* partition unit: tiles_per_segment =
                                  cdiv(len, NS * tile_size) ([merge] docstring) */
  int32_t kernel;              /* decode kernel variant (internal id) */
  int32_t rows_per_cta;        /* query rows (token x head) one CTA owns (the
                                  CTA-pair kernel: one pair) */
  int32_t row_tiles;           /* row tiles per request (dense) or token (sparse) */
  int32_t grid_x, grid_y, grid_z;
  int32_t num_sms;
  int32_t schedule;            /* 1: balanced schedule (see mla_decode_plan), else 0 */
  int32_t max_items;           /* balanced: work items the decode grid holds */
  int32_t split_items;         /* balanced: partial slots of tile_rows rows,
                                  two per worker: 2 * (num_sms / 2) for the
                                  CTA-pair kernel, 2 * num_sms for the
                                  rows-as-N kernel (2 * the clusters of two
                                  that fit at once, for 65..128 rows) */
  int32_t wait_limit_us;       /* bound on every internal wait of the tensor-core
                                  kernels, in microseconds; the planner sets 0,
                                  which means 2 s. A caller may lower it after
                                  planning. A wait that runs out sets the
                                  workspace status word and the kernel exits
                                  without writing its outputs. */
  int32_t tile_rows;           /* query rows of a row tile: rows_per_cta times
                                  the CTAs that share the tile's keys (1 or 2),
                                  or 128 for the CTA-pair kernel */
  size_t workspace_bytes;      /* bytes mla_decode_fwd needs (>= 256) */
  size_t status_offset;        /* workspace layout, 256-B aligned pieces: a device */
  size_t segm_output_offset;   /* status word (int32) at offset 0, then, when */
  size_t segm_max_offset;      /* NS > 1, segm_output, segm_max and segm_expsum */
  size_t segm_expsum_offset;
} mla_plan_t;

/*
 * mla_decode_plan -- choose segments, tile and launch shape for a problem.
 * Host only: no device call other than (when prob->num_sms == 0) a query of
 * the current device's SM count, no synchronisation.
 * tile_size = min(128, largest power of two dividing block_size)
 * ([dense] _segmented_mla_page_size); the sparse variant has no page
 * structure and uses a 64-entry tile.
 * Balanced schedule: when a tensor-core kernel runs, prob->num_segments
 * is 0 and units x row tiles is at most 2^20 (else NS = 1 with the uniform
 * partition), the plan sets schedule = 1 and num_segments = 1, and mla_decode_fwd
 * sizes the segments on the device from the lengths of the call (the work
 * list of [sparse] _forward_mla's persistent path, work_indptr /
 * reduce_indptr / reduce_partial_map). Rows (a unit, i.e. a dense request or
 * a sparse token, times its tiles of tile_rows query rows) of
 * g = cdiv(len, 128) key groups are laid end to end and the sequence of all
 * groups is cut every W = cdiv(total, workers) groups. CTA-pair kernel:
 * workers = num_sms / 2 pairs, cuts within W / 8 of a row's ends dropped,
 * one item per pair, the pieces longest first (pieces of equal size in
 * unit order when the units number at most 256, so the list is the same on
 * every call; larger batches order them arbitrarily). Rows-as-N kernel: workers =
 * num_sms CTAs (or the clusters of two that fit), every cut kept, and
 * worker w runs the pieces of groups [w W, (w + 1) W) one after another.
 * max_items = rows + workers. Unsplit rows are written by the decode kernel
 * itself; split rows write base-2 partials to slots of tile_rows rows in the
 * workspace (split_items = 2 * workers of them) and mla_merge_items combines
 * them. Workspace layout: status block, item count at 256, items (32 bytes
 * each, max_items of them) at 512, the unit table (int32 pairs {first slot
 * or -1, pieces} per unit and row tile) at the next 256-byte boundary, each
 * worker's first item (int32, workers + 1) at the next, then segm_output
 * [split_items * tile_rows, 512], segm_max and segm_expsum
 * [split_items * tile_rows] at the plan's offsets.
 * Errors: MLA_ERR_INVALID_ARG for NULL pointers or inconsistent sizes,
 * MLA_ERR_UNSUPPORTED for head_dim != 576, kv_lora_rank != 512,
 * num_heads > 128, q_dtype != kv_dtype, or topk not a multiple of 128.
 */
MLA_API mla_status_t mla_decode_plan(const mla_problem_t* prob, mla_plan_t* plan);

/*
 * mla_decode_fwd -- the whole decode: split-K segments, then the merge
 * (skipped when NS == 1: the segment kernel then writes out and lse itself).
 * Under a balanced plan: mla_decode_schedule, mla_decode_items and
 * mla_merge_items in turn.
 *
 *   q            [T, H, 576] in q_dtype ([dense] forward_mqa: ql_nope || q_pe)
 *   kv_cache     [num_blocks, block_size, 576] in kv_dtype
 *   block_table  [R, >= max_blocks_per_req] int32, row stride
 *                block_table_stride elements (dense; may be NULL if sparse)
 *   seq_lens     [R] int32 KV length of each request including its new
 *                tokens (dense; may be NULL if sparse)
 *   qo_indptr    [R + 1] int32 token offsets of the requests, or NULL for one
 *                token per request. Row j of a qlen-token request sees
 *                positions [0, seq_len - qlen + j] ([dense]
 *                dcp_local_verify_row_lens).
 *   sparse_slots global cache slots (output of mla_sparse_index_convert),
 *                -1 = unused entry; [T, topk] when sparse_indptr is NULL,
 *                else a flat list where token t owns
 *                [sparse_indptr[t], sparse_indptr[t + 1]) (at most topk).
 *                NULL for the dense variant. Mutually exclusive with qo_indptr.
 *   softmax_scale, q_scale, kv_scale: score = softmax_scale * q_scale *
 *                kv_scale * (q . k) over 576 columns; values are scaled by
 *                kv_scale. All three must be finite and > 0 (1 for the
 *                q/kv scales of bf16).
 *   sinks        [H] fp32 natural-log sink logits or NULL ([sparse]
 *                _forward_mla): a sink adds e^sink to the softmax denominator
 *                and nothing to the output.
 *   workspace    plan->workspace_bytes of device memory, 256-byte aligned.
 *                Its first int32 is a device status word that must be zero
 *                before the first call (zero it once after allocating): the
 *                tensor-core kernels write a nonzero code there, and leave
 *                their outputs unwritten, if one of their bounded internal
 *                waits runs out (plan->wait_limit_us; read it, and reset it,
 *                with mla_workspace_status). The rest needs no
 *                initialisation.
 *   out          [T, H, 512] bf16; lse [T, H] fp32 natural log. Every element
 *                is written; a row with no visible key gets out = 0 and
 *                lse = -inf (or its sink).
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_WORKSPACE, MLA_ERR_CUDA.
 */
MLA_API mla_status_t mla_decode_fwd(const mla_plan_t* plan, const void* q, const void* kv_cache,
                            const int32_t* block_table, int64_t block_table_stride,
                            const int32_t* seq_lens, const int32_t* qo_indptr,
                            const int32_t* sparse_slots, const int32_t* sparse_indptr,
                            float softmax_scale, float q_scale, float kv_scale,
                            const float* sinks, void* workspace, size_t workspace_bytes,
                            void* out, float* lse, cudaStream_t stream);

/*
 * The three stages of mla_decode_fwd under a balanced plan (schedule == 1),
 * for callers that compute the work list once per step (it depends only on
 * the lengths) or time the stages apart. Each returns MLA_ERR_INVALID_ARG for a plan without the
 * balanced schedule and MLA_ERR_WORKSPACE for a missing or short workspace.
 *
 * mla_decode_schedule -- the work list of the plan's balanced schedule into
 *   the workspace, from seq_lens / qo_indptr (dense) or sparse_indptr
 *   (sparse; NULL means topk entries per token). One block on `stream`.
 */
MLA_API mla_status_t mla_decode_schedule(const mla_plan_t* plan, const int32_t* seq_lens,
                                         const int32_t* qo_indptr, const int32_t* sparse_indptr,
                                         void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream);

/*
 * mla_decode_items -- the decode kernel over the work list in the
 *   workspace, written by mla_decode_schedule for the same lengths (one list
 *   serves any number of calls): out and lse of unsplit rows, base-2
 *   partials of split rows in the workspace's slots. Arguments as
 *   mla_decode_fwd.
 */
MLA_API mla_status_t mla_decode_items(const mla_plan_t* plan, const void* q, const void* kv_cache,
                                      const int32_t* block_table, int64_t block_table_stride,
                                      const int32_t* seq_lens, const int32_t* qo_indptr,
                                      const int32_t* sparse_slots, const int32_t* sparse_indptr,
                                      float softmax_scale, float q_scale, float kv_scale,
                                      const float* sinks, void* workspace, size_t workspace_bytes,
                                      void* out, float* lse, cudaStream_t stream);

/*
 * mla_merge_items -- out and lse of the split rows from their partial slots
 *   ([merge] merge_mla_segments_triton weights, sinks folded as there);
 *   rows of unsplit units are left untouched. qo_indptr as given to the
 *   decode (dense multi-token requests), else NULL.
 */
MLA_API mla_status_t mla_merge_items(const mla_plan_t* plan, const int32_t* qo_indptr,
                                     const float* sinks, void* workspace, size_t workspace_bytes,
                                     void* out, float* lse, cudaStream_t stream);

/*
 * mla_decode_segments -- the split-K stage alone: base-2 partials of every
 * segment ([merge] module docstring, "each segment emits base-2 partials").
 * Same inputs as mla_decode_fwd; sinks are not used here (the merge folds
 * them). For segment s of token t, head h, over the keys of the segment the
 * row may see, with s2 = score * log2(e):
 *   segm_max   [T, H, NS]      m2 = max s2          (-inf if no key)
 *   segm_expsum[T, H, NS]      l  = sum 2^(s2 - m2) (0 if no key)
 *   segm_output[T, H, NS, 512] o  = sum 2^(s2 - m2) v / l (0 if no key)
 * The partition of token t is [s*tps*tile, min((s+1)*tps*tile, len)) with
 * tps = cdiv(len, NS * tile), len = seq_len of its request (shared by all
 * rows of a multi-token request) or the length of its slot list.
 * Every element of the three arrays is written, empty segments included.
 */
MLA_API mla_status_t mla_decode_segments(const mla_plan_t* plan, const void* q, const void* kv_cache,
                                 const int32_t* block_table, int64_t block_table_stride,
                                 const int32_t* seq_lens, const int32_t* qo_indptr,
                                 const int32_t* sparse_slots, const int32_t* sparse_indptr,
                                 float softmax_scale, float q_scale, float kv_scale,
                                 float* segm_output, float* segm_max, float* segm_expsum,
                                 cudaStream_t stream);

/*
 * mla_merge_segments -- merge base-2 partials into out and natural-log lse
 * ([merge] merge_mla_segments_triton). For token t the segments whose start
 * lies inside [0, part_lens[t]) (partition as above, from part_lens and
 * tile_size) and whose expsum is > 0 take part. With M = max(m2_s,
 * sink * log2 e) and W = sum_s l_s 2^(m2_s - M) + 2^(sink log2 e - M):
 *   out = sum_s l_s 2^(m2_s - M) o_s / W,   lse = ln 2 * (M + log2 W).
 * No contributing segment and no sink: out = 0, lse = -inf.
 *   segm_output [T, H, NS, kv_lora_rank] fp32, segm_max / segm_expsum
 *   [T, H, NS] fp32, part_lens [T] int32, sinks [H] fp32 or NULL,
 *   out [T, H, kv_lora_rank] in out_dtype (BF16 only), lse [T, H] fp32.
 * kv_lora_rank must be a positive multiple of 128; num_segments 1..64.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (out_dtype), MLA_ERR_CUDA.
 */
MLA_API mla_status_t mla_merge_segments(const float* segm_output, const float* segm_max,
                                const float* segm_expsum, const int32_t* part_lens,
                                int32_t num_tokens, int32_t num_heads, int32_t num_segments,
                                int32_t kv_lora_rank, int32_t tile_size, const float* sinks,
                                int32_t out_dtype, void* out, float* lse, cudaStream_t stream);

/*
 * mla_sparse_seqlen -- per-token lengths of the sparse slot lists and their
 * exclusive prefix sum, ready to serve as cu_seqlens of
 * mla_sparse_index_convert and sparse_indptr of the decode ([sparse]
 * ROCMAiterMLASparseMetadataBuilder.build: generate_sparse_seqlen_triton,
 * then the cumsum into paged_kv_indptr). The page gives no kernel body; the
 * reading taken: token j of request r (qlen = query_start_loc[r + 1] -
 * query_start_loc[r] tokens) sees its causal prefix (the bound of [dense]
 * dcp_local_verify_row_lens) and selects at most topk positions:
 *   lens[t] = clamp(seq_lens[r] - qlen + j + 1, 0, topk).
 * Tokens before query_start_loc[0] or at or past query_start_loc[num_reqs]
 * get length 0.
 *   query_start_loc [num_reqs + 1] int32, nondecreasing; seq_lens [num_reqs]
 *   lens [num_tokens] int32 or NULL; indptr [num_tokens + 1] int32
 * One block on `stream`. Errors: MLA_ERR_INVALID_ARG for negative sizes,
 * topk <= 0, NULL or misaligned pointers; MLA_ERR_UNSUPPORTED when
 * num_tokens * topk exceeds INT32_MAX.
 */
MLA_API mla_status_t mla_sparse_seqlen(const int32_t* query_start_loc, const int32_t* seq_lens,
                                       int32_t num_reqs, int32_t num_tokens, int32_t topk,
                                       int32_t* lens, int32_t* indptr, cudaStream_t stream);

/*
 * mla_fit_kpool_indices -- the indexer's [T, width] rows (width >= topk)
 * fitted to the fixed width topk ([sparse] fit_kpool_indices_to_aiter,
 * which keeps the kpool tail's live entries). The page gives no kernel
 * body; the reading taken: columns [0, topk) are the selected positions,
 * columns [topk, width) the kpool tail, an entry is live when >= 0; with n
 * the number of live tail entries (the first topk of them at most), output
 * row t is the first topk - n selected entries followed by the n live tail
 * entries in their order. Nothing is de-duplicated; width == topk copies.
 *   token_indices [T, width] int32, row stride ti_row_stride (>= width)
 *   out [T, topk] int32, row stride out_row_stride (>= topk), not
 *   overlapping the input
 * One warp per row. Errors: MLA_ERR_INVALID_ARG for width < topk, topk <= 0,
 * short strides, NULL, misaligned or overlapping buffers.
 */
MLA_API mla_status_t mla_fit_kpool_indices(const int32_t* token_indices, int64_t ti_row_stride,
                                           int32_t num_tokens, int32_t width, int32_t topk,
                                           int32_t* out, int64_t out_row_stride,
                                           cudaStream_t stream);

/*
 * mla_sparse_index_convert -- per-request top-k positions to global slots
 * ([sparse] triton_convert_req_index_to_global_index):
 *   out[t, i] = block_table[req_id[t], idx / block_size] * block_size
 *               + idx % block_size,   idx = token_indices[t, i],
 * and -1 when idx < 0, when idx / block_size >= bt_cols, or when req_id[t]
 * is not in [0, bt_rows). Block-table values are not range-checked.
 * Integer arithmetic in int32; the caller keeps num_blocks * block_size
 * below 2^31.
 *   req_id        [T] int32
 *   block_table   [bt_rows, bt_cols] int32 with row stride bt_row_stride
 *   token_indices [T, topk] int32 with row stride ti_row_stride
 *   cu_seqlens    NULL: out is [T, topk]. Else [T + 1] int32 and the first
 *                 cu_seqlens[t+1] - cu_seqlens[t] (<= topk) entries of row t
 *                 are written to out[cu_seqlens[t] + i]; nothing else in out
 *                 is touched.
 * topk must be a positive multiple of 128; block_size > 0.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_CUDA.
 */
MLA_API mla_status_t mla_sparse_index_convert(const int32_t* req_id, const int32_t* block_table,
                                      int32_t bt_rows, int32_t bt_cols, int64_t bt_row_stride,
                                      const int32_t* token_indices, int64_t ti_row_stride,
                                      int32_t num_tokens, int32_t topk, int32_t block_size,
                                      const int32_t* cu_seqlens, int32_t* out,
                                      cudaStream_t stream);

/*
 * mla_merge_lse -- combine the (out, lse) of W key shards of the same rows,
 * the cross-rank merge that consumes the natural-log LSE of
 * mla_decode_fwd / mla_merge_segments under decode context parallelism
 * ([merge] module docstring: "the natural-log LSE it returns is what the
 * cross-rank DCP merge consumes"). With M = max_w lse_w:
 *   out = sum_w e^(lse_w - M) out_w / Z,  lse = M + ln Z,
 *   Z = sum_w e^(lse_w - M) (+ e^(sink - M)).
 * Shards with lse = -inf take no part; no shard and no sink gives out = 0,
 * lse = -inf. A sink is folded here once, so shards are decoded without it.
 *   shard_out [W, T, H, kv_lora_rank] bf16, shard_lse [W, T, H] fp32,
 *   sinks [H] fp32 or NULL, out [T, H, kv_lora_rank] bf16, lse [T, H] fp32.
 * kv_lora_rank must be 128, 256 or 512.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_CUDA.
 */
MLA_API mla_status_t mla_merge_lse(const void* shard_out, const float* shard_lse,
                                   int32_t num_shards, int32_t num_tokens, int32_t num_heads,
                                   int32_t kv_lora_rank, const float* sinks, void* out,
                                   float* lse, cudaStream_t stream);

/*
 * mla_concat_quant_q -- the q pre-step of forward_mqa ([sparse] and [dense]
 * forward_mqa: q = ql_nope || q_pe, and for fp8 attention the static
 * per-tensor quantisation with layer._q_scale):
 *   out[t, h, 0:512] = ql_nope[t, h, :], out[t, h, 512:576] = q_pe[t, h, :]
 * as bf16, or as e4m3 codes of (value / q_scale) rounded to nearest even
 * with magnitudes above 448 saturated (the division is fp32).
 *   ql_nope [T, H, 512] bf16, strides (elements) nope_stride_t, nope_stride_h
 *   q_pe    [T, H, 64]  bf16, strides pe_stride_t, pe_stride_h
 *   out     [T, H, 576] contiguous, in out_dtype
 * The last dims are contiguous; pointers 16-byte aligned, strides multiples
 * of 8 elements. Errors: MLA_ERR_INVALID_ARG, MLA_ERR_CUDA.
 */
MLA_API mla_status_t mla_concat_quant_q(const void* ql_nope, int64_t nope_stride_t,
                                        int64_t nope_stride_h, const void* q_pe,
                                        int64_t pe_stride_t, int64_t pe_stride_h,
                                        int32_t num_tokens, int32_t num_heads, int32_t out_dtype,
                                        float q_scale, void* out, cudaStream_t stream);

/* Largest plan->workspace_bytes that mla_decode_fwd_static accepts. */
#define MLA_STATIC_SCRATCH_BYTES ((size_t)64 << 20) /* 64 MiB */

/*
 * mla_decode_fwd_static -- mla_decode_fwd for callers that cannot allocate
 * device memory. The pages have no counterpart: it exists for serving
 * engines that reserve nearly all HBM for the paged KV cache at start-up and
 * route every later allocation through their own pool, whose op interface
 * offers no workspace argument, so a decode-time cudaMalloc would fail or is
 * not allowed.
 *
 * Arguments, outputs and errors are those of mla_decode_fwd, except that the
 * workspace is a file-scope device array of MLA_STATIC_SCRATCH_BYTES inside
 * this library instead of a caller buffer. Nothing here calls cudaMalloc,
 * cudaFree or an allocating library routine.
 *   - Set-up: the first call on a device (the current one) looks up that
 *     array's device address once and caches it; make that first call before
 *     any stream capture begins.
 *   - Size limit: a plan whose workspace_bytes exceeds
 *     MLA_STATIC_SCRATCH_BYTES is rejected with MLA_ERR_WORKSPACE before any
 *     device work. Only plans requested with prob.num_segments = 1 are sure
 *     to fit (they need 256 bytes); a planner-chosen balanced plan needs its
 *     work list and partial slots (about 41 MB for 64 requests of 128 heads on
 *     a 152-SM part) and, for very many requests, can exceed the limit and
 *     is then refused.
 *   - Sharing: every call on a device uses the same array, which keeps the
 *     last call's partials. Each call first clears the array's status word
 *     (stream-ordered memset); nothing else must start at zero. Calls whose
 *     GPU work overlaps (different streams or host threads without ordering
 *     between them) race on the array and give undefined results; calls on
 *     one stream are ordered and safe.
 *   - status_out: NULL, or a device int32 that receives (stream-ordered) the
 *     status word after the kernels: 0, or the nonzero code of a bounded
 *     internal wait that timed out.
 */
MLA_API mla_status_t mla_decode_fwd_static(const mla_plan_t* plan, const void* q,
                                           const void* kv_cache, const int32_t* block_table,
                                           int64_t block_table_stride, const int32_t* seq_lens,
                                           const int32_t* qo_indptr, const int32_t* sparse_slots,
                                           const int32_t* sparse_indptr, float softmax_scale,
                                           float q_scale, float kv_scale, const float* sinks,
                                           void* out, float* lse, int32_t* status_out,
                                           cudaStream_t stream);

/*
 * mla_workspace_status -- the device status word of a workspace, after the
 * work enqueued on `stream` so far (the stream is synchronised: call it
 * between steps, not inside a captured graph). The tensor-core decode
 * kernels write a nonzero code there, and leave their outputs unwritten,
 * when one of their bounded internal waits runs out (plan->wait_limit_us);
 * nothing else writes it. *code receives the word; with clear != 0 a nonzero
 * word is reset to 0 (stream-ordered), so that the workspace can serve the
 * next call.
 * Returns MLA_OK when the word was 0, MLA_ERR_DEVICE_STATUS when it was not,
 * MLA_ERR_INVALID_ARG for NULL or misaligned pointers, MLA_ERR_CUDA.
 */
MLA_API mla_status_t mla_workspace_status(const mla_plan_t* plan, const void* workspace,
                                          int32_t* code, int32_t clear, cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
MLA_API const char* mla_status_string(mla_status_t status);

/* CUDA error string recorded by the last MLA_ERR_CUDA on the calling thread,
 * or "" (static / thread-local storage). */
MLA_API const char* mla_last_cuda_error(void);

/* Library version as major * 10000 + minor * 100 + patch. */
MLA_API int32_t mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
