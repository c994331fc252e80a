// tma_map.cuh -- host-side TMA tensor maps over [rows, 576] row tensors (q
// and the KV cache viewed as rows), 128-byte-wide boxes with the 128-byte
// swizzle the tcgen05 shared-memory descriptors of the decode kernels expect;
// and over the [rows, mid, 512] outputs the decode stores.
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime_api.h>

namespace mla {

inline PFN_cuTensorMapEncodeTiled_v12000 tma_encode_fn() {
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

// 2-D map over a [rows, 576] tensor of bf16 or e4m3 elements with boxes 128
// bytes wide (or 64, with the 64-byte swizzle) and box_rows rows high; reads
// past the last row or column fill zeros.
inline cudaError_t make_row_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows,
                                bool fp8, uint32_t box_bytes = 128) {
  auto enc = tma_encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const uint32_t elt = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(576), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(576) * elt};
  cuuint32_t box[2] = {box_bytes / elt, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D map over an output tensor [rows, mid, 512] of fp32 (or bf16 with
// `bf16`) values, row stride mid * 512 elements, for stores of boxes of
// box_rows rows x box_cols columns (one box column at a time along `mid`):
// by default 8 x 32 without swizzle; with `sw128` the shared-memory tile is
// in the 128-byte swizzle (box_cols x element size must then be 128 bytes).
inline cudaError_t make_out_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t mid, bool bf16,
                                uint32_t box_cols = 32, uint32_t box_rows = 8, bool sw128 = false) {
  auto enc = tma_encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const uint64_t elt = bf16 ? 2 : 4;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(512), static_cast<cuuint64_t>(mid), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(512 * elt), static_cast<cuuint64_t>(512 * elt * mid)};
  cuuint32_t box[3] = {box_cols, 1, box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace mla
