// tmap.h — host-side TMA tensor-map encoding for [B, N, H, d] bf16 or fp16 tensors.
//
// The map views a [B, N, H, d] tensor as 4-D with dims (d, H, N, B) and byte
// strides (2, 2d, 2Hd, 2NHd).  The box is 64 x 1 x 128 x 1: 128 rows (tokens)
// of one head, 64 head-dim columns (128 bytes) with the 128-byte swizzle.
// Columns >= d and rows >= N are filled with zeros by the hardware, which is
// how head dims that are not multiples of 64 and ragged N are handled.
// cuTensorMapEncodeTiled is looked up through the runtime's driver
// entry-point query, so the library does not link against libcuda.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace fa {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// rows_box: tokens per box (128); cols_box: head-dim columns per box (64).
inline cudaError_t make_bhnd_tmap(CUtensorMap* map, const void* base, int B, int N, int H, int d,
                                  int rows_box = 128, int cols_box = 64, bool f16 = false) {
  auto fn = encode_tiled_fn();
  if (fn == nullptr) return cudaErrorSymbolNotFound;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(H) * d * 2,
                                 static_cast<cuuint64_t>(N) * H * d * 2};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(cols_box), 1u,
                             static_cast<cuuint32_t>(rows_box), 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace fa
