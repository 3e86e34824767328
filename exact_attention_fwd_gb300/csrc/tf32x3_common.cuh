// tf32x3_common.cuh — pieces shared by the float32 tensor-core kernels
// (3xTF32 forward and backward): tcgen05 kind::tf32 MMAs, their instruction
// descriptor, float32 tensor maps, rounding to tf32, and the split passes
// that write the hi / lo copies of the inputs.
//
// A float32 x is split into hi = x rounded to the nearest tf32 value and
// lo = (x - hi) rounded to the nearest tf32 value; a product is taken as
// hi*hi + hi*lo + lo*hi (3xTF32).  Every tf32 MMA operand is K-major, so a
// tensor that is contracted over its rows is also split into a transposed
// copy [B, H, d, Np].
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "sm103_ptx.cuh"
#include "tmap.h"

namespace fa {
namespace {

// D[tmem] (+)= A * B with tf32 operands (32-bit elements, fp32 accumulate):
// A from shared memory (SS) or TMEM (TS), B from shared memory.
__device__ __forceinline__ void mma_ss_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_tf32(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for kind::tf32: D format F32 (bits 4-5 = 1), A and B
// format TF32 (code 2 in bits 7-9 and 10-12), both K-major, N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// 4-D float32 tensor map with the 128-byte swizzle (box inner extent 32
// floats = 128 bytes); elements outside `dims` read as zero.
cudaError_t make_f32_tmap(CUtensorMap* map, const void* base, const cuuint64_t dims[4],
                          const cuuint64_t strides[3], const cuuint32_t box[4]) {
  auto fn = encode_tiled_fn();
  if (fn == nullptr) return cudaErrorSymbolNotFound;
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Nearest tf32 value (ties away from zero) of a finite float32 of magnitude
// below 2^127: add half of the dropped 13-bit field, then clear it.
__device__ __forceinline__ float tf32_rn(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

// Split pass, Q and K: 4 elements per thread with 16-byte loads and stores.
__global__ void __launch_bounds__(256) split_qk_kernel(const float4* q, const float4* k,
                                                       float4* qh, float4* ql, float4* kh,
                                                       float4* kl, size_t n4) {
  for (size_t x = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < n4;
       x += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 a = q[x], bk = k[x];
    const float4 ah = make_float4(tf32_rn(a.x), tf32_rn(a.y), tf32_rn(a.z), tf32_rn(a.w));
    const float4 bh = make_float4(tf32_rn(bk.x), tf32_rn(bk.y), tf32_rn(bk.z), tf32_rn(bk.w));
    qh[x] = ah;
    ql[x] = make_float4(tf32_rn(a.x - ah.x), tf32_rn(a.y - ah.y), tf32_rn(a.z - ah.z),
                        tf32_rn(a.w - ah.w));
    kh[x] = bh;
    kl[x] = make_float4(tf32_rn(bk.x - bh.x), tf32_rn(bk.y - bh.y), tf32_rn(bk.z - bh.z),
                        tf32_rn(bk.w - bh.w));
  }
}

// V^T split: [B, N, H, d] -> hi / lo as [B, H, d, Np] (Np = N rounded up to
// 4; rows n >= N are written as zeros).  A CTA transposes 32 rows (n) by 64
// columns (c) of one (b, h) through one shared-memory tile: 16-byte loads of
// V rows, 16-byte stores of V^T rows, index arithmetic once per CTA.
__global__ void __launch_bounds__(256) split_vt_kernel(const float* v, float* vth, float* vtl,
                                                       int N, int H, int d, int Np) {
  __shared__ float tile[32][65];
  const int n0 = blockIdx.x * 32, c0 = blockIdx.y * 64, bh = blockIdx.z;
  const int b = bh / H, h = bh % H;
  const size_t rs = static_cast<size_t>(H) * d;   // floats between V rows
  const float* vb = v + (static_cast<size_t>(b) * N * H + h) * d;
  for (int i = threadIdx.x; i < 32 * 16; i += 256) {
    const int r = i >> 4, c4 = (i & 15) * 4, n = n0 + r, c = c0 + c4;
    float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (n < N && c < d) x = *reinterpret_cast<const float4*>(vb + n * rs + c);
    tile[r][c4] = x.x;
    tile[r][c4 + 1] = x.y;
    tile[r][c4 + 2] = x.z;
    tile[r][c4 + 3] = x.w;
  }
  __syncthreads();
  const size_t ob = (static_cast<size_t>(bh) * d + c0) * Np + n0;
  for (int i = threadIdx.x; i < 64 * 8; i += 256) {
    const int c = i >> 3, n4 = (i & 7) * 4;
    if (c0 + c < d && n0 + n4 < Np) {
      float xs[4], hs[4], ls[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xs[j] = tile[n4 + j][c];
        hs[j] = tf32_rn(xs[j]);
        ls[j] = tf32_rn(xs[j] - hs[j]);
      }
      const size_t o = ob + static_cast<size_t>(c) * Np + n4;
      *reinterpret_cast<float4*>(vth + o) = make_float4(hs[0], hs[1], hs[2], hs[3]);
      *reinterpret_cast<float4*>(vtl + o) = make_float4(ls[0], ls[1], ls[2], ls[3]);
    }
  }
}


// K-step offsets (8 tf32 = 32 bytes) inside a 2-chunk K-major tile, in the
// descriptor's 16-byte units.
__device__ __forceinline__ uint64_t kstep(int kk, int chunk_bytes) {
  return static_cast<uint64_t>(((kk >> 2) * chunk_bytes + (kk & 3) * 32) >> 4);
}

}  // namespace
}  // namespace fa
