// bwd_dot.cu — the backward pre-pass D_i = <dO_i, O_i> ("Flash Attention 2 —
// backward pass notes", section "The math (FA2 backward with recompute)",
// first line, and option 1 of "Why the WGSL kernel isn't shipped this turn":
// compute D once into a [B, H, N] buffer).
//
// Memory-bound: it reads O and dO once and writes 4 bytes per row.  Rows of
// [B, N, H, d] tensors with consecutive (n, h) are contiguous, so the lanes of
// a warp read consecutive 16-byte chunks of consecutive rows: every load
// instruction of the warp is one contiguous 512-byte span.  When a row is a
// power-of-two number of chunks (d = 8, 16, 32, 64, 128), each row belongs to
// a fixed group of lanes, the row's partial dot products are summed with warp
// shuffles, and every lane keeps 2 rows' chunks of both tensors in flight (more
// raised the register count and lowered the resident warps: measured slower);
// other head sizes stage the partial sums in shared memory.  The grid is the
// number of blocks that fit on the SMs at once, each striding over the rows.
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

// Row = kCpr lanes (kCpr 16-byte chunks); a warp covers 32 / kCpr rows per
// pass and kUnroll passes per iteration.
template <int kElt, int kCpr>
__global__ void __launch_bounds__(kThreads) dot_shfl_kernel(BwdParams p) {
  constexpr int kRowsPass = 32 / kCpr;
  constexpr int kUnroll = 2;
  constexpr int kRowsIter = kRowsPass * kUnroll;
  const int lane = threadIdx.x & 31, sub = lane % kCpr, rr = lane / kCpr;
  const long long rows = static_cast<long long>(p.B) * p.N * p.H;
  const uint4* O = static_cast<const uint4*>(p.o);
  const uint4* G = static_cast<const uint4*>(p.dO);
  const long long w0 = static_cast<long long>(blockIdx.x) * (kThreads / 32) + threadIdx.x / 32;
  const long long nw = static_cast<long long>(gridDim.x) * (kThreads / 32);
  for (long long r0 = w0 * kRowsIter; r0 < rows; r0 += nw * kRowsIter) {
    uint4 a[kUnroll], b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long r = r0 + u * kRowsPass + rr;
      if (r < rows) {
        a[u] = __ldg(O + r * kCpr + sub);
        b[u] = __ldg(G + r * kCpr + sub);
      } else {
        a[u] = make_uint4(0u, 0u, 0u, 0u);
        b[u] = a[u];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float s = dot_chunk<kElt>(a[u], b[u]);
#pragma unroll
      for (int off = kCpr / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      const long long r = r0 + u * kRowsPass + rr;
      if (sub == 0 && r < rows) {
        // flattened row r = (b * N + n) * H + h  ->  D[(b * H + h) * N + n]
        // (32-bit division where the row count allows: fewer registers)
        if (rows <= 0x7fffffffLL) {
          const unsigned ru = static_cast<unsigned>(r), Hu = static_cast<unsigned>(p.H),
                         Nu = static_cast<unsigned>(p.N);
          const unsigned h = ru % Hu, bn = ru / Hu, n = bn % Nu, bb = bn / Nu;
          p.D[(static_cast<size_t>(bb) * Hu + h) * Nu + n] = s;
        } else {
          const int h = static_cast<int>(r % p.H);
          const long long bn = r / p.H;
          const int n = static_cast<int>(bn % p.N);
          const long long bb = bn / p.N;
          p.D[(bb * p.H + h) * p.N + n] = s;
        }
      }
    }
  }
}

template <int kElt>
const void* dot_kernel_for(int cpr) {
  switch (cpr) {
    case 1: return reinterpret_cast<const void*>(dot_shfl_kernel<kElt, 1>);
    case 2: return reinterpret_cast<const void*>(dot_shfl_kernel<kElt, 2>);
    case 4: return reinterpret_cast<const void*>(dot_shfl_kernel<kElt, 4>);
    case 8: return reinterpret_cast<const void*>(dot_shfl_kernel<kElt, 8>);
    case 16: return reinterpret_cast<const void*>(dot_shfl_kernel<kElt, 16>);
    case 32: return reinterpret_cast<const void*>(dot_shfl_kernel<kElt, 32>);
    default: return reinterpret_cast<const void*>(dot_do_o_kernel<kElt>);
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
  void* args[] = {const_cast<BwdParams*>(&p)};
  const int cpr = p.d * (elt == 0 ? 4 : 2) / 16;   // 16-byte chunks per row
  const void* kern = elt == 2   ? dot_kernel_for<2>(cpr)
                     : elt == 1 ? dot_kernel_for<1>(cpr)
                                : dot_kernel_for<0>(cpr);
  // as many blocks as are resident at once (each strides over the rows)
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const long long cap = static_cast<long long>(sms > 0 ? sms : 148) * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return cudaLaunchKernel(kern, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), args, 0, s);
}

}  // namespace fa
