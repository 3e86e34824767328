// unfused.cu — the unfused forward (Algorithm 0) as a comparison path.
//
// Source: the "Lesson K23, fused attention" facts page, `sources.flashAttention`
// (Algorithm 0: S = Q K^T written to global memory, a row softmax reads S and
// writes P, then O = P V) and its `traffic` block (the unfused form moves the
// N x N matrices through global memory: 4 N^2 bytes of extra memory per head).
// It exists to measure what the fused kernel saves, on the same hardware.
//
// Three launches per call, all on the caller's stream:
//   1. S = scale Q K^T per head, float32 [B, H, N, N] in the workspace: a
//      plain batched GEMM (cuBLAS, 16-bit inputs, float32 accumulate).
//   2. row softmax (this file): one warp per query row reads its S row, takes
//      the masked max m and sum l, writes exp(S - m) as 16-bit values in place
//      over the first half of the same row (row pitch stays 4 N bytes), and
//      writes l and L = m + log l.
//   3. O' = exp(S - m) V per head: a plain batched GEMM (cuBLAS), float32.
//   4. O = O' / l, rounded once to 16 bits (this file).
// The division by l comes after the product, as in the fused kernel: the
// row's largest weight is then exactly 1 before rounding, and P / l is never
// rounded to 16 bits (with peaked rows that would cost up to half a 16-bit
// ulp of the dominant weight).
// cuBLAS is loaded on first use (dlopen), so the rest of the library does not
// depend on it; its workspace is a fixed part of the caller's workspace, so
// no call allocates device memory (the first call on a device creates the
// cuBLAS handle).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cublas_v2.h>
#include <dlfcn.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa_common.cuh"

namespace {

constexpr size_t kGemmWorkspace = 32u << 20;   // cuBLAS workspace inside ours
constexpr int kRowsPerBlock = 8;               // one warp per row

template <bool kF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (kF16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <bool kF16>
__device__ __forceinline__ void store16(void* p, size_t idx, float x) {
  if constexpr (kF16) reinterpret_cast<__half*>(p)[idx] = __float2half_rn(x);
  else reinterpret_cast<__nv_bfloat16*>(p)[idx] = __float2bfloat16_rn(x);
}

// Masked row softmax in place.  Row r = (b, h, i) of S starts at float offset
// r N; its P row starts at 16-bit offset 2 r N (the same bytes).  Pass 1 keeps
// a running (max, sum) per lane over the lane's columns and merges the lanes;
// pass 2 re-reads S (the row is still in L2) and writes P.  In pass 2, the P
// values of columns [32t, 32t + 32) overwrite S columns [16t, 16t + 16), which
// every lane has read by iteration t (a warp barrier separates each
// iteration's reads from its writes).
template <bool kF16>
__global__ void __launch_bounds__(32 * kRowsPerBlock) row_softmax_kernel(float* S, float* lse,
                                                                        float* lsum,
                                                                        long long rows, int N,
                                                                        int causal) {
  const long long r = static_cast<long long>(blockIdx.x) * kRowsPerBlock + threadIdx.x / 32;
  if (r >= rows) return;   // whole warps only: rows are per warp
  const int lane = threadIdx.x & 31;
  const int i = static_cast<int>(r % N);             // query index within the head
  const int lim = causal ? i : N - 1;                // last visible key
  const float* srow = S + static_cast<size_t>(r) * N;
  float m = -INFINITY, l = 0.0f;
  for (int j = lane; j <= lim; j += 32) {
    const float s = srow[j];
    if (s > m) {
      l = l * expf(m - s) + 1.0f;
      m = s;
    } else {
      l += expf(s - m);
    }
  }
  // merge the lanes' (m, l) states
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, l, off);
    const float mn = fmaxf(m, mo);
    l = (mn == -INFINITY) ? 0.0f : l * expf(m - mn) + lo * expf(mo - mn);
    m = mn;
  }
  void* prow = reinterpret_cast<uint16_t*>(S) + static_cast<size_t>(r) * 2 * N;
  for (int j0 = 0; j0 < N; j0 += 32) {
    const int j = j0 + lane;
    float s = -INFINITY;
    if (j <= lim) s = srow[j];
    __syncwarp();   // every lane has read this iteration's S before any P lands
    if (j < N) store16<kF16>(prow, j, (j <= lim) ? expf(s - m) : 0.0f);
  }
  if (lane == 0) {
    lse[r] = (l > 0.0f) ? m + logf(l) : -INFINITY;
    lsum[r] = l;
  }
}

// O = O' / l per row, rounded once; 4 columns per thread, rows in [B, N, H]
// order (O' and O share the [B, N, H, d] layout; l is [B, H, N]).
template <bool kF16>
__global__ void __launch_bounds__(256) normalize_kernel(const float4* o32, uint2* o,
                                                        const float* lsum, int N, int H, int d4,
                                                        size_t total) {
  for (size_t x = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < total;
       x += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t row = x / d4;   // (b, n, h)
    const int h = static_cast<int>(row % H);
    const size_t bn = row / H;
    const int n = static_cast<int>(bn % N);
    const size_t b = bn / N;
    const float l = lsum[(b * H + h) * N + n];
    const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
    const float4 v = o32[x];
    o[x] = make_uint2(pack2<kF16>(v.x * inv, v.y * inv), pack2<kF16>(v.z * inv, v.w * inv));
  }
}

}  // namespace

namespace {

// cuBLAS entry points, resolved once from the shared library (the GEMM is
// the C symbol with 32-bit sizes and 64-bit batch strides).
using GemmFn = cublasStatus_t (*)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int,
                                  int, const void*, const void*, cudaDataType, int, long long,
                                  const void*, cudaDataType, int, long long, const void*, void*,
                                  cudaDataType, int, long long, int, cublasComputeType_t,
                                  cublasGemmAlgo_t);
struct Cublas {
  decltype(&cublasCreate_v2) create = nullptr;
  decltype(&cublasSetStream_v2) set_stream = nullptr;
  decltype(&cublasSetWorkspace_v2) set_workspace = nullptr;
  GemmFn gemm = nullptr;
  bool tried = false, ok = false;
};
Cublas g_cublas;
constexpr int kMaxDevices = 64;
cublasHandle_t g_handle[kMaxDevices] = {};
std::mutex g_cublas_mu;

bool load_cublas() {
  if (g_cublas.tried) return g_cublas.ok;
  g_cublas.tried = true;
  void* h = dlopen("libcublas.so.13", RTLD_NOW | RTLD_LOCAL);
  if (h == nullptr) h = dlopen("libcublas.so", RTLD_NOW | RTLD_LOCAL);
  if (h == nullptr) return false;
  g_cublas.create = reinterpret_cast<decltype(g_cublas.create)>(dlsym(h, "cublasCreate_v2"));
  g_cublas.set_stream =
      reinterpret_cast<decltype(g_cublas.set_stream)>(dlsym(h, "cublasSetStream_v2"));
  g_cublas.set_workspace =
      reinterpret_cast<decltype(g_cublas.set_workspace)>(dlsym(h, "cublasSetWorkspace_v2"));
  g_cublas.gemm =
      reinterpret_cast<decltype(g_cublas.gemm)>(dlsym(h, "cublasGemmStridedBatchedEx"));
  g_cublas.ok = g_cublas.create && g_cublas.set_stream && g_cublas.set_workspace && g_cublas.gemm;
  return g_cublas.ok;
}

size_t scores_bytes(int B, int H, int N) {
  return static_cast<size_t>(B) * H * N * N * sizeof(float);
}
size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
size_t o32_bytes(int B, int H, int N, int d) {
  return static_cast<size_t>(B) * N * H * d * sizeof(float);
}
size_t rows_bytes(int B, int H, int N) { return static_cast<size_t>(B) * H * N * sizeof(float); }

}  // namespace

extern "C" {

size_t fa_fwd_unfused_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  return up256(scores_bytes(B, H, N)) + up256(o32_bytes(B, H, N, d)) +
         up256(rows_bytes(B, H, N)) + kGemmWorkspace;
}

fa_status fa_fwd_unfused(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, float scale, int causal, fa_dtype dtype,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16)
    return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1 || d < 1 || d % 8 != 0 || !std::isfinite(scale))
    return FA_ERR_INVALID_ARG;
  if (d > 128 || dtype == FA_DTYPE_F32) return FA_ERR_UNSUPPORTED;
  if (static_cast<long double>(B) * H * N * N * 4 >= static_cast<long double>(1ULL << 40))
    return FA_ERR_UNSUPPORTED;
  if (workspace_bytes < fa_fwd_unfused_workspace_size(B, H, N, d)) return FA_ERR_INVALID_ARG;
  const uintptr_t ws = reinterpret_cast<uintptr_t>(workspace);
  if ((ws & 255) != 0) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) & 15)
    return FA_ERR_INVALID_ARG;

  std::lock_guard<std::mutex> lock(g_cublas_mu);
  if (!load_cublas()) return FA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  if (g_handle[dev] == nullptr && g_cublas.create(&g_handle[dev]) != CUBLAS_STATUS_SUCCESS) {
    g_handle[dev] = nullptr;
    return FA_ERR_CUDA;
  }
  cublasHandle_t hd = g_handle[dev];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // workspace: S, then O' (float32 [B, N, H, d]), l ([B, H, N]), the GEMMs' scratch
  char* wsp = static_cast<char*>(workspace);
  float* S = reinterpret_cast<float*>(wsp);
  float* o32 = reinterpret_cast<float*>(wsp + up256(scores_bytes(B, H, N)));
  float* lsum = reinterpret_cast<float*>(reinterpret_cast<char*>(o32) + up256(o32_bytes(B, H, N, d)));
  void* gemm_ws = reinterpret_cast<char*>(lsum) + up256(rows_bytes(B, H, N));
  if (g_cublas.set_stream(hd, s) != CUBLAS_STATUS_SUCCESS ||
      g_cublas.set_workspace(hd, gemm_ws, kGemmWorkspace) != CUBLAS_STATUS_SUCCESS)
    return FA_ERR_CUDA;

  const cudaDataType_t t16 = (dtype == FA_DTYPE_F16) ? CUDA_R_16F : CUDA_R_16BF;
  const int ld = H * d;                      // row pitch of q, k, v, o
  const long long seq = static_cast<long long>(N) * H * d;
  const long long nn = static_cast<long long>(N) * N;
  const float zero = 0.0f, one = 1.0f;
  // Column-major views: a head's q, k, v, o are d x N with leading dimension
  // H d; heads of one sequence are d elements apart.
  for (int b = 0; b < B; ++b) {
    // S^T (col-major N x N, ld N) = K_h^T Q_h: S[i][j] = scale q_i . k_j
    const char* qb = static_cast<const char*>(q) + static_cast<size_t>(b) * seq * 2;
    const char* kb = static_cast<const char*>(k) + static_cast<size_t>(b) * seq * 2;
    if (g_cublas.gemm(hd, CUBLAS_OP_T, CUBLAS_OP_N, N, N, d, &scale, kb, t16, ld, d, qb, t16, ld,
                      d, &zero, S + static_cast<size_t>(b) * H * nn, CUDA_R_32F, N, nn, H,
                      CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
      return FA_ERR_CUDA;
  }
  const long long rows = static_cast<long long>(B) * H * N;
  const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (blocks > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (dtype == FA_DTYPE_F16)
    row_softmax_kernel<true><<<static_cast<unsigned>(blocks), 32 * kRowsPerBlock, 0, s>>>(
        S, lse, lsum, rows, N, causal != 0);
  else
    row_softmax_kernel<false><<<static_cast<unsigned>(blocks), 32 * kRowsPerBlock, 0, s>>>(
        S, lse, lsum, rows, N, causal != 0);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  for (int b = 0; b < B; ++b) {
    // O'_h (col-major d x N, ld H d) = V_h P_h^T, P row i at 16-bit pitch 2 N
    const char* vb = static_cast<const char*>(v) + static_cast<size_t>(b) * seq * 2;
    float* ob = o32 + static_cast<size_t>(b) * seq;
    const uint16_t* P = reinterpret_cast<const uint16_t*>(S) + static_cast<size_t>(b) * H * 2 * nn;
    if (g_cublas.gemm(hd, CUBLAS_OP_N, CUBLAS_OP_N, d, N, N, &one, vb, t16, ld, d, P, t16, 2 * N,
                      2 * nn, &zero, ob, CUDA_R_32F, ld, d, H, CUBLAS_COMPUTE_32F,
                      CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
      return FA_ERR_CUDA;
  }
  const size_t total4 = static_cast<size_t>(B) * N * H * (d / 4);
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return FA_ERR_CUDA;
  const size_t want = (total4 + 255) / 256, cap = static_cast<size_t>(sms) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (dtype == FA_DTYPE_F16)
    normalize_kernel<true><<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(o32),
                                                 static_cast<uint2*>(o), lsum, N, H, d / 4, total4);
  else
    normalize_kernel<false><<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(o32),
                                                  static_cast<uint2*>(o), lsum, N, H, d / 4, total4);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
