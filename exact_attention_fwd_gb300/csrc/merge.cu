// merge.cu — split-KV merge: per-slice attention results -> output and L.
//
// Source: "Flash Attention 2 — forward pass notes", section "Loop (per
// (b, h, Q-tile))" (the softmax of concatenated key blocks is the merge of
// the blocks' (m, l) states), and the "Lesson K23, fused attention" facts
// page, `sources.onlineSoftmax.claims[2]` (the merge is associative and
// commutative, so the slices may be reduced in any order).
//
// A slice result normalised over its own keys, (O_s, L_s), is the state
// (m = L_s, l = 1, O = O_s).  Merging all of them at once:
//   M = max_s L_s,  W = sum_s 2^((L_s - M) log2 e),  L = M + log W,
//   O = sum_s 2^((L_s - M) log2 e) O_s / W.
// Slices whose L_s is -inf, and slices a row does not read (causal: slice s
// starts after the row), are skipped without reading O_s.
//
// HBM-bound: one thread per 4 output columns of a row, rows in [B, N, H]
// order, so a warp's loads of each slice and its output stores are
// contiguous 16-byte accesses.  The grid is a multiple of the SM count and
// strides over the columns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "fa_common.cuh"

namespace fa {
namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

template <int kOut>   // 0 float32, 1 bf16, 2 fp16
__device__ __forceinline__ void store4(void* o, size_t idx4, float4 v) {
  if constexpr (kOut == 0) {
    reinterpret_cast<float4*>(o)[idx4] = v;
  } else if constexpr (kOut == 1) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(o)[idx4] = u;
  } else {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(o)[idx4] = u;
  }
}

template <int kOut>
__global__ void __launch_bounds__(kThreads) merge_kernel(const MergeParams p) {
  const int d4 = p.d / 4;
  const size_t total = static_cast<size_t>(p.B) * p.N * p.H * d4;
  const size_t slice_o = static_cast<size_t>(p.B) * p.N * p.H * d4;   // float4s per slice
  const size_t slice_l = static_cast<size_t>(p.B) * p.H * p.N;
  const float4* op = reinterpret_cast<const float4*>(p.o_part);
  for (size_t x = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < total;
       x += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int c4 = static_cast<int>(x % d4);
    const size_t row = x / d4;   // (b, n, h)
    const int h = static_cast<int>(row % p.H);
    const size_t bn = row / p.H;
    const int n = static_cast<int>(bn % p.N);
    const int b = static_cast<int>(bn / p.N);
    // slices this row reads
    int ns = p.nsplit;
    if (p.causal) ns = min(ns, n / p.keys_per_split + 1);
    const size_t lrow = (static_cast<size_t>(b) * p.H + h) * p.N + n;
    float M = -INFINITY;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, p.lse_part[s * slice_l + lrow]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = -INFINITY;
    if (M != -INFINITY) {
      float W = 0.0f;
      for (int s = 0; s < ns; ++s) {
        const float ls = p.lse_part[s * slice_l + lrow];
        if (ls == -INFINITY) continue;
        const float w = exp2f((ls - M) * kLog2e);
        const float4 v = op[s * slice_o + x];
        W += w;
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
      const float inv = 1.0f / W;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
      L = M + log2f(W) * kLn2;
    }
    store4<kOut>(p.o, x, acc);
    if (c4 == 0) p.lse[lrow] = L;
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, int out_elt, cudaStream_t s) {
  if (p.d % 4 != 0 || p.nsplit < 1 || p.keys_per_split < 1) return cudaErrorInvalidValue;
  const size_t total = static_cast<size_t>(p.B) * p.N * p.H * (p.d / 4);
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  // 8 resident blocks of 256 threads per SM, at most one pass over the columns
  const size_t want = (total + kThreads - 1) / kThreads;
  const size_t cap = static_cast<size_t>(sms) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  MergeParams pc = p;
  if (out_elt == 0) merge_kernel<0><<<grid, kThreads, 0, s>>>(pc);
  else if (out_elt == 1) merge_kernel<1><<<grid, kThreads, 0, s>>>(pc);
  else merge_kernel<2><<<grid, kThreads, 0, s>>>(pc);
  return cudaGetLastError();
}

}  // namespace fa
