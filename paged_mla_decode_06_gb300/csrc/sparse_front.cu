// sparse_front.cu -- the sparse path's front end on the rocm_aiter_mla_sparse
// page, ahead of the index conversion:
//   * the metadata builder's per-token list lengths (generate_sparse_seqlen
//     there) and their prefix sum (paged_kv_indptr): token j of a request
//     with qlen tokens sees its causal prefix seq_len - qlen + j + 1 (the
//     dense page's bound for multi-token rows) and selects at most topk of
//     those positions;
//   * the fit of the indexer's [T, W] rows to AITER's fixed width topk
//     (fit_kpool_indices_to_aiter there): the first topk - n selected
//     entries, then the n live (>= 0) entries of the kpool tail (columns
//     [topk, W)) in order, n capped at topk. The page gives no kernel body;
//     this is the reading both functions implement.
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kSeqThreads = 1024;
constexpr int kFitWarps = 4;

// One block. Pass 1, one thread per request: the lengths of the request's
// tokens go to indptr[t + 1] (scratch). Pass 2, tokens in chunks of 1024:
// each thread reads its length (before any write of the chunk: the scan's
// barriers separate them), then indptr[t] = the exclusive prefix.
__global__ void __launch_bounds__(kSeqThreads, 1) sparse_seqlen_kernel(
    const int32_t* __restrict__ qsl, const int32_t* __restrict__ seq_lens, int32_t num_reqs,
    int32_t num_tokens, int32_t topk, int32_t* __restrict__ lens, int32_t* __restrict__ indptr) {
  __shared__ int warp_sum[kSeqThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int r = tid; r < num_reqs; r += kSeqThreads) {
    const int q0 = qsl[r], q1 = qsl[r + 1];
    const int qlen = q1 - q0;
    const int64_t base = static_cast<int64_t>(seq_lens[r]) - qlen + 1;
    for (int j = 0; j < qlen; ++j) {
      const int t = q0 + j;
      if (t < 0 || t >= num_tokens) continue;
      const int64_t visible = base + j;
      indptr[t + 1] = static_cast<int>(visible < 0 ? 0 : (visible > topk ? topk : visible));
    }
  }
  // tokens before the first request or past the last one get length 0
  const int first = num_reqs > 0 ? max(qsl[0], 0) : 0;
  const int covered = num_reqs > 0 ? min(qsl[num_reqs], num_tokens) : 0;
  __syncthreads();  // pass 1's global writes are visible to the whole block
  int carry = 0;
  for (int t0 = 0; t0 < num_tokens; t0 += kSeqThreads) {
    const int t = t0 + tid;
    const int len = t >= first && t < covered ? indptr[t + 1] : 0;
    int inc = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    __syncthreads();
    if (lane == 31) warp_sum[warp] = inc;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kSeqThreads / 32; ++w) {
      const int s = warp_sum[w];
      if (w < warp) before += s;
      total += s;
    }
    if (t < num_tokens) {
      indptr[t] = carry + before + inc - len;
      if (lens != nullptr) lens[t] = len;
    }
    carry += total;
  }
  if (tid == 0) indptr[num_tokens] = carry;
}

// One warp per row: count the live tail, copy the head, compact the tail.
__global__ void __launch_bounds__(kFitWarps * 32) fit_kpool_kernel(
    const int32_t* __restrict__ ti, int64_t ti_stride, int32_t num_tokens, int32_t width,
    int32_t topk, int32_t* __restrict__ out, int64_t out_stride) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kFitWarps + (threadIdx.x >> 5);
  if (t >= num_tokens) return;
  const int32_t* row = ti + static_cast<int64_t>(t) * ti_stride;
  int32_t* orow = out + static_cast<int64_t>(t) * out_stride;
  const int tail = width - topk;
  int live = 0;
  for (int c = 0; c < tail; c += 32) {
    const bool ok = c + lane < tail && row[topk + c + lane] >= 0;
    live += __popc(__ballot_sync(0xffffffffu, ok));
  }
  const int n = live < topk ? live : topk;
  for (int i = lane; i < topk - n; i += 32) orow[i] = row[i];
  int pos = 0;  // live tail entries placed so far
  for (int c = 0; c < tail && pos < n; c += 32) {
    const int v = c + lane < tail ? row[topk + c + lane] : -1;
    const unsigned m = __ballot_sync(0xffffffffu, v >= 0);
    const int rank = pos + __popc(m & ((1u << lane) - 1u));
    if (v >= 0 && rank < n) orow[topk - n + rank] = v;
    pos += __popc(m);
  }
}

}  // namespace

cudaError_t launch_sparse_seqlen(const int32_t* qsl, const int32_t* seq_lens, int32_t num_reqs,
                                 int32_t num_tokens, int32_t topk, int32_t* lens, int32_t* indptr,
                                 cudaStream_t stream) {
  sparse_seqlen_kernel<<<1, kSeqThreads, 0, stream>>>(qsl, seq_lens, num_reqs, num_tokens, topk, lens,
                                                      indptr);
  return cudaGetLastError();
}

cudaError_t launch_fit_kpool(const int32_t* ti, int64_t ti_stride, int32_t num_tokens, int32_t width,
                             int32_t topk, int32_t* out, int64_t out_stride, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((num_tokens + kFitWarps - 1) / kFitWarps);
  fit_kpool_kernel<<<blocks, kFitWarps * 32, 0, stream>>>(ti, ti_stride, num_tokens, width, topk, out,
                                                          out_stride);
  return cudaGetLastError();
}

}  // namespace mla
