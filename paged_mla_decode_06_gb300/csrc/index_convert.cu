// index_convert.cu -- per-request top-k positions to global cache slots
// (rocm_aiter_mla_sparse page, triton_convert_req_index_to_global_index):
//   out[t, i] = block_table[req_id[t], idx / BS] * BS + idx % BS,
// -1 for idx < 0, for a block column past the table, or for a request id
// outside the table. One CTA per (token, 128-entry column tile); every
// thread converts one entry. With cu_seqlens the first
// cu[t+1] - cu[t] entries of row t go to out[cu[t] + i].
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kTileN = 128;

__global__ void __launch_bounds__(kTileN) index_convert_kernel(
    const int32_t* __restrict__ req_id, const int32_t* __restrict__ block_table, int32_t bt_rows,
    int32_t bt_cols, int64_t bt_stride, const int32_t* __restrict__ token_indices,
    int64_t ti_stride, int32_t topk, int32_t bs, const int32_t* __restrict__ cu_seqlens,
    int32_t* __restrict__ out) {
  const int tiles_per_row = topk / kTileN;
  const int t = blockIdx.x / tiles_per_row;
  const int i = (blockIdx.x % tiles_per_row) * kTileN + threadIdx.x;
  int n = topk;
  int64_t dst = static_cast<int64_t>(t) * topk + i;
  if (cu_seqlens != nullptr) {
    n = min(cu_seqlens[t + 1] - cu_seqlens[t], topk);
    dst = static_cast<int64_t>(cu_seqlens[t]) + i;
  }
  if (i >= n) return;
  const int r = req_id[t];
  const int idx = token_indices[static_cast<int64_t>(t) * ti_stride + i];
  int v = -1;
  if (idx >= 0 && r >= 0 && r < bt_rows) {
    const int blk = idx / bs;
    if (blk < bt_cols) {
      v = block_table[static_cast<int64_t>(r) * bt_stride + blk] * bs + (idx - blk * bs);
    }
  }
  out[dst] = v;
}

}  // namespace

cudaError_t launch_index_convert(const int32_t* req_id, const int32_t* block_table,
                                 int32_t bt_rows, int32_t bt_cols, int64_t bt_stride,
                                 const int32_t* token_indices, int64_t ti_stride,
                                 int32_t num_tokens, int32_t topk, int32_t block_size,
                                 const int32_t* cu_seqlens, int32_t* out, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>(num_tokens) * static_cast<unsigned>(topk / kTileN);
  index_convert_kernel<<<blocks, kTileN, 0, stream>>>(req_id, block_table, bt_rows, bt_cols,
                                                       bt_stride, token_indices, ti_stride, topk,
                                                       block_size, cu_seqlens, out);
  return cudaGetLastError();
}

}  // namespace mla
