// fa_api.cu — the C ABI declared in include/fa.h: argument validation, the
// device status word, and dispatch to the float32 SIMT kernels or the bf16
// tcgen05 kernels.  No call here allocates device memory.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "fa_common.cuh"

namespace {

// One status word per device; kernels record FA_ERR_TIMEOUT here.
__device__ int g_fa_status = 0;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;

// Device address of this device's status word (looked up once per device,
// with that device current).
int* status_word(fa_status* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = FA_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fa_status) != cudaSuccess) {
      *err = FA_ERR_CUDA;
      return nullptr;
    }
    g_status_ptr[dev] = static_cast<int*>(ptr);
  }
  return g_status_ptr[dev];
}

bool probe_timeout_requested() {
  const char* v = std::getenv("FA_SELFTEST_WAIT_TIMEOUT");
  return v != nullptr && v[0] == '1';
}

size_t elt_size(fa_dtype t) { return t == FA_DTYPE_F32 ? 4 : 2; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// [a, a + na) and [b, b + nb) overlap
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

fa_status check_shape(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (d < 1 || d % 8 != 0) return FA_ERR_INVALID_ARG;
  if (d > 128) return FA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  // element count and byte strides must stay far inside 64-bit / TMA limits
  const long double elems = static_cast<long double>(B) * N * H * d;
  if (elems * 4 >= static_cast<long double>(1ULL << 40)) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

}  // namespace

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

size_t fa_bwd_workspace_size(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  const size_t bytes = static_cast<size_t>(B) * H * N * sizeof(float);
  return (bytes + 255) & ~static_cast<size_t>(255);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, fa_dtype dtype, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16)
    return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  const size_t tbytes = static_cast<size_t>(B) * N * H * d * elt_size(dtype);
  const size_t lbytes = static_cast<size_t>(B) * H * N * sizeof(float);
  for (const void* in : {q, k, v}) {
    if (overlaps(o, tbytes, in, tbytes) || overlaps(lse, lbytes, in, tbytes))
      return FA_ERR_INVALID_ARG;
  }
  if (overlaps(o, tbytes, lse, lbytes)) return FA_ERR_INVALID_ARG;

  fa_status err = FA_OK;
  int* status = status_word(&err);
  if (status == nullptr) return err;

  fa::FwdParams p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
  p.B = B; p.H = H; p.N = N; p.d = d;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  p.probe_timeout = probe_timeout_requested() ? 1 : 0;
  p.f16 = (dtype == FA_DTYPE_F16) ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = (dtype == FA_DTYPE_F32) ? fa::launch_fwd_simt_f32(p, s, causal != 0)
                                          : fa::launch_fwd_tc16(p, s, causal != 0);
  if (e == cudaErrorNotSupported) return FA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"

namespace {

// Validates fa_bwd's arguments and fills the launch parameters.
fa_status prepare_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                      float scale, fa_dtype dtype, fa_dtype grad_dtype, void* workspace,
                      size_t workspace_bytes, fa::BwdParams* out) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !workspace)
    return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16)
    return FA_ERR_INVALID_ARG;
  if (grad_dtype != dtype && grad_dtype != FA_DTYPE_F32) return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (workspace_bytes < fa_bwd_workspace_size(B, H, N)) return FA_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, o, dO, static_cast<const void*>(dq),
                          static_cast<const void*>(dk), static_cast<const void*>(dv)})
    if (!aligned(ptr, 16)) return FA_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || !aligned(workspace, 256)) return FA_ERR_INVALID_ARG;
  const size_t in_bytes = static_cast<size_t>(B) * N * H * d * elt_size(dtype);
  const size_t g_bytes = static_cast<size_t>(B) * N * H * d * elt_size(grad_dtype);
  const size_t l_bytes = static_cast<size_t>(B) * H * N * sizeof(float);
  const void* outs[] = {dq, dk, dv};
  const void* ins[] = {q, k, v, o, dO};
  for (const void* outp : outs) {
    for (const void* in : ins)
      if (overlaps(outp, g_bytes, in, in_bytes)) return FA_ERR_INVALID_ARG;
    if (overlaps(outp, g_bytes, lse, l_bytes) || overlaps(outp, g_bytes, workspace, workspace_bytes))
      return FA_ERR_INVALID_ARG;
  }
  if (overlaps(dq, g_bytes, dk, g_bytes) || overlaps(dq, g_bytes, dv, g_bytes) ||
      overlaps(dk, g_bytes, dv, g_bytes))
    return FA_ERR_INVALID_ARG;
  for (const void* in : ins)
    if (overlaps(workspace, workspace_bytes, in, in_bytes)) return FA_ERR_INVALID_ARG;
  if (overlaps(workspace, workspace_bytes, lse, l_bytes)) return FA_ERR_INVALID_ARG;

  fa_status err = FA_OK;
  int* status = status_word(&err);
  if (status == nullptr) return err;

  fa::BwdParams& p = *out;
  p = fa::BwdParams{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.dO = dO;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.D = static_cast<float*>(workspace);
  p.B = B; p.H = H; p.N = N; p.d = d;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.grad_f32 = (grad_dtype == FA_DTYPE_F32) ? 1 : 0;
  p.status = status;
  p.probe_timeout = probe_timeout_requested() ? 1 : 0;
  p.f16 = (dtype == FA_DTYPE_F16) ? 1 : 0;
  return FA_OK;
}

// 16-bit inputs with d <= 64: the dQ kernel forms D's first estimate from the
// O and dO rows it loads, so phase 0 launches nothing
bool bwd_prepass(int d, fa_dtype dtype) { return dtype == FA_DTYPE_F32 || d > 64; }

fa_status run_bwd_phase(const fa::BwdParams& p, int phase, fa_dtype dtype, bool causal,
                        cudaStream_t s) {
  cudaError_t e;
  if (phase == 0) {
    if (!bwd_prepass(p.d, dtype)) return FA_OK;
    e = fa::launch_bwd_dot(p, dtype == FA_DTYPE_F32 ? 0 : (dtype == FA_DTYPE_BF16 ? 1 : 2), s);
  } else if (dtype == FA_DTYPE_F32) {
    e = fa::launch_bwd_simt_f32(p, s, causal, phase);
  } else {
    e = fa::launch_bwd_tc16(p, s, causal, phase);
  }
  if (e == cudaErrorNotSupported) return FA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, fa_dtype grad_dtype, void* workspace,
                 size_t workspace_bytes, void* stream) {
  fa::BwdParams p;
  fa_status st = prepare_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, dtype,
                             grad_dtype, workspace, workspace_bytes, &p);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int phase = 0; phase < 3 && st == FA_OK; ++phase)
    st = run_bwd_phase(p, phase, dtype, causal != 0, s);
  return st;
}

int fa_bwd_prepass(int d, fa_dtype dtype) { return bwd_prepass(d, dtype) ? 1 : 0; }

fa_status fa_bwd_phase(int phase, const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                       int H, int N, int d, float scale, int causal, fa_dtype dtype,
                       fa_dtype grad_dtype, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (phase < 0 || phase > 2) return FA_ERR_INVALID_ARG;
  fa::BwdParams p;
  fa_status st = prepare_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, dtype,
                             grad_dtype, workspace, workspace_bytes, &p);
  if (st != FA_OK) return st;
  return run_bwd_phase(p, phase, dtype, causal != 0, static_cast<cudaStream_t>(stream));
}

fa_status fa_sync_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return static_cast<fa_status>(v);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// split-KV forward
// ---------------------------------------------------------------------------

namespace {

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t part_o_bytes(int B, int H, int N, int d, int nsplit) {
  return static_cast<size_t>(nsplit) * B * N * H * d * sizeof(float);
}
size_t part_l_bytes(int B, int H, int N, int nsplit) {
  return static_cast<size_t>(nsplit) * B * H * N * sizeof(float);
}

int slices_of(int N, int keys_per_split) { return (N + keys_per_split - 1) / keys_per_split; }

fa_status run_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                      int B, int H, int N, int d, float scale, int causal, fa_dtype dtype,
                      int keys_per_split, cudaStream_t s) {
  int* status = nullptr;
  fa_status err = FA_OK;
  status = status_word(&err);
  if (status == nullptr) return err;
  fa::FwdParams p{};
  p.q = q; p.k = k; p.v = v; p.o = nullptr; p.lse = nullptr;
  p.B = B; p.H = H; p.N = N; p.d = d;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  p.probe_timeout = probe_timeout_requested() ? 1 : 0;
  p.f16 = (dtype == FA_DTYPE_F16) ? 1 : 0;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.split_blocks = keys_per_split / 128;
  p.nsplit = slices_of(N, keys_per_split);
  cudaError_t e = fa::launch_fwd_tc16_partial(p, s, causal != 0);
  if (e == cudaErrorNotSupported) return FA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status run_merge(const float* o_part, const float* lse_part, int nsplit, int keys_per_split,
                    int causal, void* o, float* lse, int B, int H, int N, int d, fa_dtype dtype,
                    cudaStream_t s) {
  fa::MergeParams m{};
  m.o_part = o_part; m.lse_part = lse_part; m.o = o; m.lse = lse;
  m.B = B; m.H = H; m.N = N; m.d = d;
  m.nsplit = nsplit;
  m.keys_per_split = keys_per_split;
  m.causal = causal != 0;
  const int elt = dtype == FA_DTYPE_F32 ? 0 : (dtype == FA_DTYPE_BF16 ? 1 : 2);
  return fa::launch_merge(m, elt, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_fwd_splitkv_keys_per_split(int N, int num_splits) {
  if (N < 1 || num_splits < 1) return 0;
  const long long per = (static_cast<long long>(N) + 256LL * num_splits - 1) / (256LL * num_splits);
  return static_cast<int>(256 * per);
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int num_splits) {
  if (B < 1 || H < 1 || N < 1 || d < 1 || num_splits < 1) return 0;
  const int ns = slices_of(N, fa_fwd_splitkv_keys_per_split(N, num_splits));
  return round256(part_o_bytes(B, H, N, d, ns)) + round256(part_l_bytes(B, H, N, ns));
}

fa_status fa_fwd_partial(const void* q, const void* k, const void* v, float* o_part,
                         float* lse_part, int B, int H, int N, int d, float scale, int causal,
                         fa_dtype dtype, int keys_per_split, void* stream) {
  if (!q || !k || !v || !o_part || !lse_part) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16)
    return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (keys_per_split < 256 || keys_per_split % 256 != 0) return FA_ERR_INVALID_ARG;
  if (dtype == FA_DTYPE_F32) return FA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o_part, 16) ||
      !aligned(lse_part, 4))
    return FA_ERR_INVALID_ARG;
  const int ns = slices_of(N, keys_per_split);
  const size_t tbytes = static_cast<size_t>(B) * N * H * d * elt_size(dtype);
  const size_t ob = part_o_bytes(B, H, N, d, ns), lb = part_l_bytes(B, H, N, ns);
  if (static_cast<long double>(ob) >= static_cast<long double>(1ULL << 40)) return FA_ERR_UNSUPPORTED;
  for (const void* in : {q, k, v})
    if (overlaps(o_part, ob, in, tbytes) || overlaps(lse_part, lb, in, tbytes))
      return FA_ERR_INVALID_ARG;
  if (overlaps(o_part, ob, lse_part, lb)) return FA_ERR_INVALID_ARG;
  return run_partial(q, k, v, o_part, lse_part, B, H, N, d, scale, causal, dtype, keys_per_split,
                     static_cast<cudaStream_t>(stream));
}

fa_status fa_merge(const float* o_part, const float* lse_part, int num_splits, int keys_per_split,
                   int causal, void* o, float* lse, int B, int H, int N, int d, fa_dtype dtype,
                   void* stream) {
  if (!o_part || !lse_part || !o || !lse) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16)
    return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d, 1.0f);
  if (st != FA_OK) return st;
  if (num_splits < 1 || keys_per_split < 1) return FA_ERR_INVALID_ARG;
  if (!aligned(o_part, 16) || !aligned(o, 16) || !aligned(lse_part, 4) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  const size_t ob = part_o_bytes(B, H, N, d, num_splits), lb = part_l_bytes(B, H, N, num_splits);
  if (static_cast<long double>(ob) >= static_cast<long double>(1ULL << 40)) return FA_ERR_UNSUPPORTED;
  const size_t tbytes = static_cast<size_t>(B) * N * H * d * elt_size(dtype);
  const size_t l1 = static_cast<size_t>(B) * H * N * sizeof(float);
  if (overlaps(o, tbytes, o_part, ob) || overlaps(o, tbytes, lse_part, lb) ||
      overlaps(lse, l1, o_part, ob) || overlaps(lse, l1, lse_part, lb) ||
      overlaps(o, tbytes, lse, l1))
    return FA_ERR_INVALID_ARG;
  return run_merge(o_part, lse_part, num_splits, keys_per_split, causal, o, lse, B, H, N, d, dtype,
                   static_cast<cudaStream_t>(stream));
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, float scale, int causal, fa_dtype dtype,
                         int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16)
    return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (num_splits < 1) return FA_ERR_INVALID_ARG;
  if (dtype == FA_DTYPE_F32) return FA_ERR_UNSUPPORTED;
  const size_t need = fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits);
  if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 256))
    return FA_ERR_INVALID_ARG;
  const size_t tbytes = static_cast<size_t>(B) * N * H * d * elt_size(dtype);
  const size_t lbytes = static_cast<size_t>(B) * H * N * sizeof(float);
  for (const void* in : {q, k, v}) {
    if (overlaps(o, tbytes, in, tbytes) || overlaps(lse, lbytes, in, tbytes) ||
        overlaps(workspace, workspace_bytes, in, tbytes))
      return FA_ERR_INVALID_ARG;
  }
  if (overlaps(o, tbytes, lse, lbytes) || overlaps(workspace, workspace_bytes, o, tbytes) ||
      overlaps(workspace, workspace_bytes, lse, lbytes))
    return FA_ERR_INVALID_ARG;
  const int kps = fa_fwd_splitkv_keys_per_split(N, num_splits);
  const int ns = slices_of(N, kps);
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             round256(part_o_bytes(B, H, N, d, ns)));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = run_partial(q, k, v, o_part, lse_part, B, H, N, d, scale, causal, dtype, kps, s);
  if (st != FA_OK) return st;
  return run_merge(o_part, lse_part, ns, kps, causal, o, lse, B, H, N, d, dtype, s);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// float32 forward on the tensor cores (3xTF32)
// ---------------------------------------------------------------------------

extern "C" {

size_t fa_bwd_tf32x3_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  return fa::tf32x3_bwd_workspace_bytes(B, H, N, d);
}

fa_status fa_bwd_tf32x3(const float* q, const float* k, const float* v, const float* o,
                        const float* lse, const float* dO, float* dq, float* dk, float* dv,
                        int B, int H, int N, int d, float scale, int causal, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (d > 64 && check_shape(B, H, N, d, scale) == FA_OK) return FA_ERR_UNSUPPORTED;
  if (workspace_bytes < fa_bwd_tf32x3_workspace_size(B, H, N, d)) return FA_ERR_INVALID_ARG;
  fa::BwdParams p;
  fa_status st = prepare_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, FA_DTYPE_F32,
                             FA_DTYPE_F32, workspace, workspace_bytes, &p);
  if (st != FA_OK) return st;
  cudaError_t e = fa::launch_bwd_tf32x3(p, workspace, static_cast<cudaStream_t>(stream),
                                        causal != 0);
  if (e == cudaErrorNotSupported) return FA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_fwd_tf32x3_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  return fa::tf32x3_workspace_bytes(B, H, N, d);
}

fa_status fa_fwd_tf32x3(const float* q, const float* k, const float* v, float* o, float* lse,
                        int B, int H, int N, int d, float scale, int causal, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (workspace_bytes < fa_fwd_tf32x3_workspace_size(B, H, N, d)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 256))
    return FA_ERR_INVALID_ARG;
  const size_t tbytes = static_cast<size_t>(B) * N * H * d * 4;
  const size_t lbytes = static_cast<size_t>(B) * H * N * sizeof(float);
  for (const void* in : {static_cast<const void*>(q), static_cast<const void*>(k),
                         static_cast<const void*>(v)}) {
    if (overlaps(o, tbytes, in, tbytes) || overlaps(lse, lbytes, in, tbytes) ||
        overlaps(workspace, workspace_bytes, in, tbytes))
      return FA_ERR_INVALID_ARG;
  }
  if (overlaps(o, tbytes, lse, lbytes) || overlaps(workspace, workspace_bytes, o, tbytes) ||
      overlaps(workspace, workspace_bytes, lse, lbytes))
    return FA_ERR_INVALID_ARG;
  fa_status err = FA_OK;
  int* status = status_word(&err);
  if (status == nullptr) return err;
  fa::FwdParams p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
  p.B = B; p.H = H; p.N = N; p.d = d;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  p.probe_timeout = probe_timeout_requested() ? 1 : 0;
  cudaError_t e = fa::launch_fwd_tf32x3(p, workspace, static_cast<cudaStream_t>(stream),
                                        causal != 0);
  if (e == cudaErrorNotSupported) return FA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
