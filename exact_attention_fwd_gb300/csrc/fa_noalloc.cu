// fa_noalloc.cu — fa_bwd_noalloc: the attention backward without a caller-
// supplied workspace, for callers that must not allocate device memory when
// they call us.
//
// fa_bwd needs B*H*N floats of scratch (the per-row D values).  Most callers
// pass a workspace they allocated; some cannot allocate at call time, for
// example code whose device memory is owned by a host framework's own pool
// and that is not allowed to call cudaMalloc itself, or latency-critical code
// that cannot afford cudaMalloc (which may synchronise the device).  For them
// the scratch lives in a fixed array in this library's device image instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its own copy of kNoAllocMaxRows floats (16 MiB) until the
// process exits.  Host code cannot use the array's name as a device address;
// the device address is looked up once per device with cudaGetSymbolAddress
// (with that device current) on the first call made on that device, and then
// passed to the kernels like any other pointer.  That first call per device
// should therefore come before any stream capture.
//
// All calls on a device share the one array and it keeps the previous call's
// contents.  Nothing in it needs to start at zero: the backward's first kernel
// writes every entry it later reads.  Calls whose work overlaps on the GPU
// (different streams, or different host threads without ordering) race on
// the array and give wrong gradients; serialise them.
#include <cstdint>
#include <mutex>

#include "fa_common.cuh"

namespace {

constexpr size_t kNoAllocMaxRows = static_cast<size_t>(FA_BWD_NOALLOC_MAX_ROWS);

static __device__ __align__(256) float g_bwd_scratch[kNoAllocMaxRows];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of this device's scratch array, looked up on first use.
fa_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || ptr == nullptr)
      return FA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dO, void* dq, void* dk,
                                    void* dv, int B, int H, int N, int d, float scale, int causal,
                                    fa_dtype dtype, fa_dtype grad_dtype, void* stream) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  const unsigned long long rows = static_cast<unsigned long long>(B) *
                                  static_cast<unsigned long long>(H) *
                                  static_cast<unsigned long long>(N);
  if (rows > kNoAllocMaxRows) return FA_ERR_UNSUPPORTED;   // beyond the fixed scratch
  void* scratch = nullptr;
  const fa_status st = scratch_for_current_device(&scratch);
  if (st != FA_OK) return st;
  return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, dtype, grad_dtype,
                scratch, kNoAllocMaxRows * sizeof(float), stream);
}
