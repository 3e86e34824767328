// simt_f32.cu — float32 attention forward and backward on the FMA pipes.
//
// Float32 storage needs float32 arithmetic: the tensor cores' tf32 mode keeps
// 10 mantissa bits and cannot hold O to 1e-5, so the float32 entry points run
// the same FlashAttention-2 loops on CUDA cores.
//
// Forward ("Flash Attention 2 — forward pass notes", "Loop (per (b, h,
// Q-tile))"): a CTA owns kBR query rows of one (b, h) and walks K/V blocks of
// kBC keys staged in shared memory, keeping (m, l, O) per row in registers
// with the rescale alpha = exp(m_old - m_new); causal blocks past the tile's
// last row are skipped; keys >= N and above the diagonal score -inf.  Each
// warp owns kRowsPerWarp rows; for the scores, lane j takes key j of the
// block; for the output, lane c owns columns c, c+32, c+64, c+96.
//
// Backward ("Flash Attention 2 — backward pass notes", "The math (FA2 backward
// with recompute)" and option 3 of "Why the WGSL kernel isn't shipped this
// turn"): a dK/dV kernel whose CTA owns kBC keys and walks the query blocks at
// or below the diagonal, and a dQ kernel whose CTA owns kBR queries and walks
// the key blocks up to the diagonal.  P = exp(S - L) is recomputed from the
// saved log-sum-exp; no float atomics.
#include <cfloat>
#include <cmath>

#include "fa_common.cuh"

namespace fa {
namespace {

constexpr int kBR = 32;            // query rows per CTA
constexpr int kBC = 32;            // keys per block (= warp width)
constexpr int kWarps = 4;
constexpr int kRowsPerWarp = kBR / kWarps;
constexpr int kMaxD = 128;
constexpr int kColsPerLane = kMaxD / 32;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Element (b, n, h, c) of a [B, N, H, d] tensor.
__device__ __forceinline__ size_t idx4(int b, int n, int h, int c, int N, int H, int d) {
  return ((static_cast<size_t>(b) * N + n) * H + h) * d + c;
}

// Load rows [r0, r0 + rows) of one head into smem with row stride `ld`,
// zero-filling rows >= N.
__device__ __forceinline__ void load_rows(float* dst, int ld, const float* src, int b, int h,
                                          int r0, int rows, int N, int H, int d) {
  for (int e = threadIdx.x; e < rows * d; e += blockDim.x) {
    const int r = e / d, c = e % d;
    const int n = r0 + r;
    dst[r * ld + c] = (n < N) ? src[idx4(b, n, h, c, N, H, d)] : 0.0f;
  }
}

template <bool kCausal>
__global__ void __launch_bounds__(kWarps * 32) fwd_simt_kernel(FwdParams p) {
  extern __shared__ float sm[];
  const int d = p.d, N = p.N, H = p.H;
  const int ldk = d + 1;                      // padded: lane j reads row j
  float* sQ = sm;                             // [kBR][d]
  float* sK = sQ + kBR * d;                   // [kBC][d + 1]
  float* sV = sK + kBC * ldk;                 // [kBC][d]
  const int bh = blockIdx.y, b = bh / H, h = bh % H;
  const int q0 = blockIdx.x * kBR;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float* Q = static_cast<const float*>(p.q);
  const float* K = static_cast<const float*>(p.k);
  const float* V = static_cast<const float*>(p.v);

  load_rows(sQ, d, Q, b, h, q0, kBR, N, H, d);

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kColsPerLane];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.0f;
#pragma unroll
    for (int c = 0; c < kColsPerLane; ++c) acc[r][c] = 0.0f;
  }

  const int q_last = min(q0 + kBR, N) - 1;
  for (int k0 = 0; k0 < N; k0 += kBC) {
    if (kCausal && k0 > q_last) break;         // causal block skip
    __syncthreads();
    load_rows(sK, ldk, K, b, h, k0, kBC, N, H, d);
    load_rows(sV, d, V, b, h, k0, kBC, N, H, d);
    __syncthreads();
    const int key = k0 + lane;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int row = warp * kRowsPerWarp + r;
      const int qi = q0 + row;
      float s = 0.0f;
      for (int c = 0; c < d; ++c) s = fmaf(sQ[row * d + c], sK[lane * ldk + c], s);
      s *= p.scale;
      const bool masked = (key >= N) || (kCausal && key > qi);
      if (masked) s = -INFINITY;
      const float m_new = fmaxf(m[r], warp_max(s));
      if (m_new == -INFINITY) continue;         // nothing visible yet
      const float alpha = (m[r] == -INFINITY) ? 0.0f : expf(m[r] - m_new);
      const float pj = masked ? 0.0f : expf(s - m_new);
      l[r] = l[r] * alpha + warp_sum(pj);
#pragma unroll
      for (int c = 0; c < kColsPerLane; ++c) acc[r][c] *= alpha;
      for (int j = 0; j < kBC; ++j) {
        const float pb = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
        for (int c = 0; c < kColsPerLane; ++c) {
          const int col = lane + 32 * c;
          if (col < d) acc[r][c] = fmaf(pb, sV[j * d + col], acc[r][c]);
        }
      }
      m[r] = m_new;
    }
  }

  float* O = static_cast<float*>(p.o);
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int qi = q0 + warp * kRowsPerWarp + r;
    if (qi >= N) continue;
    const bool live = l[r] > 0.0f;
    const float inv = live ? 1.0f / l[r] : 0.0f;
#pragma unroll
    for (int c = 0; c < kColsPerLane; ++c) {
      const int col = lane + 32 * c;
      if (col < d) O[idx4(b, qi, h, col, N, H, d)] = acc[r][c] * inv;
    }
    if (lane == 0)
      p.lse[static_cast<size_t>(bh) * N + qi] = live ? m[r] + logf(l[r]) : -INFINITY;
  }
}

// dK, dV for kBC keys per CTA.  Lane i takes query i of the current block.
template <bool kCausal>
__global__ void __launch_bounds__(kWarps * 32) bwd_dkdv_simt_kernel(BwdParams p) {
  extern __shared__ float sm[];
  const int d = p.d, N = p.N, H = p.H;
  const int ldq = d + 1;
  float* sK = sm;                       // [kBC][d]
  float* sV = sK + kBC * d;             // [kBC][d]
  float* sQ = sV + kBC * d;             // [kBR][d + 1]
  float* sdO = sQ + kBR * ldq;          // [kBR][d + 1]
  float* sL = sdO + kBR * ldq;          // [kBR]
  float* sD = sL + kBR;                 // [kBR]
  const int bh = blockIdx.y, b = bh / H, h = bh % H;
  const int k0 = blockIdx.x * kBC;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float* Q = static_cast<const float*>(p.q);
  const float* Kp = static_cast<const float*>(p.k);
  const float* Vp = static_cast<const float*>(p.v);
  const float* dO = static_cast<const float*>(p.dO);

  load_rows(sK, d, Kp, b, h, k0, kBC, N, H, d);
  load_rows(sV, d, Vp, b, h, k0, kBC, N, H, d);

  float dk[kRowsPerWarp][kColsPerLane], dv[kRowsPerWarp][kColsPerLane];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int c = 0; c < kColsPerLane; ++c) dk[r][c] = dv[r][c] = 0.0f;

  const int q_start = kCausal ? k0 : 0;         // queries i >= first key of the tile
  for (int q0 = (q_start / kBR) * kBR; q0 < N; q0 += kBR) {
    __syncthreads();
    load_rows(sQ, ldq, Q, b, h, q0, kBR, N, H, d);
    load_rows(sdO, ldq, dO, b, h, q0, kBR, N, H, d);
    for (int i = threadIdx.x; i < kBR; i += blockDim.x) {
      const int qi = q0 + i;
      sL[i] = (qi < N) ? p.lse[static_cast<size_t>(bh) * N + qi] : -INFINITY;
      sD[i] = (qi < N) ? p.D[static_cast<size_t>(bh) * N + qi] : 0.0f;
    }
    __syncthreads();
    const int qi = q0 + lane;
    const float Li = sL[lane], Di = sD[lane];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int kr = warp * kRowsPerWarp + r;
      const int kj = k0 + kr;
      float s = 0.0f, dp = 0.0f;
      for (int c = 0; c < d; ++c) {
        s = fmaf(sK[kr * d + c], sQ[lane * ldq + c], s);
        dp = fmaf(sV[kr * d + c], sdO[lane * ldq + c], dp);
      }
      const bool masked = (qi >= N) || (kj >= N) || (kCausal && kj > qi) || (Li == -INFINITY);
      const float pij = masked ? 0.0f : expf(s * p.scale - Li);
      const float ds = pij * (dp - Di);
      for (int i = 0; i < kBR; ++i) {
        const float pb = __shfl_sync(0xffffffffu, pij, i);
        const float db = __shfl_sync(0xffffffffu, ds, i);
#pragma unroll
        for (int c = 0; c < kColsPerLane; ++c) {
          const int col = lane + 32 * c;
          if (col < d) {
            dv[r][c] = fmaf(pb, sdO[i * ldq + col], dv[r][c]);
            dk[r][c] = fmaf(db, sQ[i * ldq + col], dk[r][c]);
          }
        }
      }
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int kj = k0 + warp * kRowsPerWarp + r;
    if (kj >= N) continue;
#pragma unroll
    for (int c = 0; c < kColsPerLane; ++c) {
      const int col = lane + 32 * c;
      if (col >= d) continue;
      const size_t e = idx4(b, kj, h, col, N, H, d);
      static_cast<float*>(p.dk)[e] = dk[r][c] * p.scale;
      static_cast<float*>(p.dv)[e] = dv[r][c];
    }
  }
}

// dQ for kBR queries per CTA.  Lane j takes key j of the current block.
template <bool kCausal>
__global__ void __launch_bounds__(kWarps * 32) bwd_dq_simt_kernel(BwdParams p) {
  extern __shared__ float sm[];
  const int d = p.d, N = p.N, H = p.H;
  const int ldk = d + 1;
  float* sQ = sm;                       // [kBR][d]
  float* sdO = sQ + kBR * d;            // [kBR][d]
  float* sK = sdO + kBR * d;            // [kBC][d + 1]
  float* sV = sK + kBC * ldk;           // [kBC][d + 1]
  const int bh = blockIdx.y, b = bh / H, h = bh % H;
  const int q0 = blockIdx.x * kBR;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float* Q = static_cast<const float*>(p.q);
  const float* Kp = static_cast<const float*>(p.k);
  const float* Vp = static_cast<const float*>(p.v);
  const float* dO = static_cast<const float*>(p.dO);

  load_rows(sQ, d, Q, b, h, q0, kBR, N, H, d);
  load_rows(sdO, d, dO, b, h, q0, kBR, N, H, d);

  float L[kRowsPerWarp], Dr[kRowsPerWarp], dq[kRowsPerWarp][kColsPerLane];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int qi = q0 + warp * kRowsPerWarp + r;
    L[r] = (qi < N) ? p.lse[static_cast<size_t>(bh) * N + qi] : -INFINITY;
    Dr[r] = (qi < N) ? p.D[static_cast<size_t>(bh) * N + qi] : 0.0f;
#pragma unroll
    for (int c = 0; c < kColsPerLane; ++c) dq[r][c] = 0.0f;
  }

  const int q_last = min(q0 + kBR, N) - 1;
  for (int k0 = 0; k0 < N; k0 += kBC) {
    if (kCausal && k0 > q_last) break;
    __syncthreads();
    load_rows(sK, ldk, Kp, b, h, k0, kBC, N, H, d);
    load_rows(sV, ldk, Vp, b, h, k0, kBC, N, H, d);
    __syncthreads();
    const int kj = k0 + lane;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int row = warp * kRowsPerWarp + r;
      const int qi = q0 + row;
      float s = 0.0f, dp = 0.0f;
      for (int c = 0; c < d; ++c) {
        s = fmaf(sQ[row * d + c], sK[lane * ldk + c], s);
        dp = fmaf(sdO[row * d + c], sV[lane * ldk + c], dp);
      }
      const bool masked = (qi >= N) || (kj >= N) || (kCausal && kj > qi) || (L[r] == -INFINITY);
      const float pij = masked ? 0.0f : expf(s * p.scale - L[r]);
      const float ds = pij * (dp - Dr[r]);
      for (int j = 0; j < kBC; ++j) {
        const float db = __shfl_sync(0xffffffffu, ds, j);
#pragma unroll
        for (int c = 0; c < kColsPerLane; ++c) {
          const int col = lane + 32 * c;
          if (col < d) dq[r][c] = fmaf(db, sK[j * ldk + col], dq[r][c]);
        }
      }
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int qi = q0 + warp * kRowsPerWarp + r;
    if (qi >= N) continue;
#pragma unroll
    for (int c = 0; c < kColsPerLane; ++c) {
      const int col = lane + 32 * c;
      if (col < d) static_cast<float*>(p.dq)[idx4(b, qi, h, col, N, H, d)] = dq[r][c] * p.scale;
    }
  }
}

template <typename Kern>
cudaError_t launch(Kern kern, dim3 grid, size_t smem, cudaStream_t s, const void* params_ptr) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<void*>(params_ptr)};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kern), grid, dim3(kWarps * 32), args,
                          smem, s);
}

}  // namespace

cudaError_t launch_fwd_simt_f32(const FwdParams& p, cudaStream_t s, bool causal) {
  const dim3 grid((p.N + kBR - 1) / kBR, p.B * p.H);
  const size_t smem = sizeof(float) * (kBR * p.d + kBC * (p.d + 1) + kBC * p.d);
  return causal ? launch(fwd_simt_kernel<true>, grid, smem, s, &p)
                : launch(fwd_simt_kernel<false>, grid, smem, s, &p);
}

// phase 1: dQ kernel; phase 2: dK/dV kernel (either order works for fp32).
cudaError_t launch_bwd_simt_f32(const BwdParams& p, cudaStream_t s, bool causal, int phase) {
  if (phase == 2) {
    const dim3 gk((p.N + kBC - 1) / kBC, p.B * p.H);
    const size_t smem_k = sizeof(float) * (2 * kBC * p.d + 2 * kBR * (p.d + 1) + 2 * kBR);
    return causal ? launch(bwd_dkdv_simt_kernel<true>, gk, smem_k, s, &p)
                  : launch(bwd_dkdv_simt_kernel<false>, gk, smem_k, s, &p);
  }
  if (phase != 1) return cudaErrorInvalidValue;
  const dim3 gq((p.N + kBR - 1) / kBR, p.B * p.H);
  const size_t smem_q = sizeof(float) * (2 * kBR * p.d + 2 * kBC * (p.d + 1));
  return causal ? launch(bwd_dq_simt_kernel<true>, gq, smem_q, s, &p)
                : launch(bwd_dq_simt_kernel<false>, gq, smem_q, s, &p);
}

}  // namespace fa
