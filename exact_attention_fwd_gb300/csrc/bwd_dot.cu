// bwd_dot.cu — the backward pre-pass D_i = <dO_i, O_i> ("Flash Attention 2 —
// backward pass notes", section "The math (FA2 backward with recompute)",
// first line, and option 1 of "Why the WGSL kernel isn't shipped this turn":
// compute D once into a [B, H, N] buffer).
//
// Memory-bound: it reads O and dO once and writes 4 bytes per row.  Rows of
// [B, N, H, d] tensors with consecutive (n, h) are contiguous, so a warp takes
// 32 consecutive flattened rows and its lanes read consecutive 16-byte chunks
// of them: every load instruction of the warp is one contiguous 512-byte span.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_common.cuh"

namespace fa {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerWarp = 32;

// elt: 0 float32, 1 bf16, 2 fp16
template <int kElt>
__device__ __forceinline__ float dot_chunk(const uint4& a, const uint4& b) {
  if (kElt == 2) {
    const __half2* x = reinterpret_cast<const __half2*>(&a);
    const __half2* y = reinterpret_cast<const __half2*>(&b);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 fx = __half22float2(x[i]);
      const float2 fy = __half22float2(y[i]);
      s = fmaf(fx.x, fy.x, s);
      s = fmaf(fx.y, fy.y, s);
    }
    return s;
  }
  if (kElt == 1) {
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 fx = __bfloat1622float2(x[i]);
      const float2 fy = __bfloat1622float2(y[i]);
      s = fmaf(fx.x, fy.x, s);
      s = fmaf(fx.y, fy.y, s);
    }
    return s;
  }
  const float* x = reinterpret_cast<const float*>(&a);
  const float* y = reinterpret_cast<const float*>(&b);
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) s = fmaf(x[i], y[i], s);
  return s;
}

template <int kElt>
__global__ void __launch_bounds__(kThreads) dot_do_o_kernel(BwdParams p) {
  // partial sums of one warp's rows: 32 rows x at most 32 chunks (fp32, d = 128)
  __shared__ float part[kThreads / 32][kRowsPerWarp * 32];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int elt = kElt ? 2 : 4;
  const int cpr = p.d * elt / 16;                       // 16-byte chunks per row
  const long long rows = static_cast<long long>(p.B) * p.N * p.H;
  const uint4* O = static_cast<const uint4*>(p.o);
  const uint4* G = static_cast<const uint4*>(p.dO);
  const long long groups = (rows + kRowsPerWarp - 1) / kRowsPerWarp;
  const long long stride = static_cast<long long>(gridDim.x) * (kThreads / 32);
  for (long long g = static_cast<long long>(blockIdx.x) * (kThreads / 32) + warp; g < groups;
       g += stride) {
    const long long r0 = g * kRowsPerWarp;
    const int nrows = static_cast<int>(rows - r0 < kRowsPerWarp ? rows - r0 : kRowsPerWarp);
    const int nchunks = nrows * cpr;
    const long long c0 = r0 * cpr;
    for (int i = lane; i < nchunks; i += 32) {
      const uint4 a = __ldg(O + c0 + i);
      const uint4 b = __ldg(G + c0 + i);
      part[warp][i] = dot_chunk<kElt>(a, b);
    }
    __syncwarp();
    if (lane < nrows) {
      float s = 0.0f;
      for (int c = 0; c < cpr; ++c) s += part[warp][lane * cpr + c];
      // flattened row r = (b * N + n) * H + h  ->  D[(b * H + h) * N + n]
      const long long r = r0 + lane;
      const int h = static_cast<int>(r % p.H);
      const long long bn = r / p.H;
      const int n = static_cast<int>(bn % p.N);
      const long long b = bn / p.N;
      p.D[(b * p.H + h) * p.N + n] = s;
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_bwd_dot(const BwdParams& p, int elt, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long rows = static_cast<long long>(p.B) * p.N * p.H;
  const long long groups = (rows + kRowsPerWarp - 1) / kRowsPerWarp;
  long long blocks = (groups + (kThreads / 32) - 1) / (kThreads / 32);
  const long long cap = static_cast<long long>(sms > 0 ? sms : 148) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  void* args[] = {const_cast<BwdParams*>(&p)};
  const void* kern = elt == 2   ? reinterpret_cast<const void*>(dot_do_o_kernel<2>)
                     : elt == 1 ? reinterpret_cast<const void*>(dot_do_o_kernel<1>)
                                : reinterpret_cast<const void*>(dot_do_o_kernel<0>);
  return cudaLaunchKernel(kern, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), args, 0, s);
}

}  // namespace fa
