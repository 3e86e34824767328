// fa_common.cuh — shared definitions of the attention kernels: status codes,
// the device status word, bounded-wait budgets and kernel launch parameters.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace fa {

// Budget of one bounded device wait, in SM clock cycles (~2 s at 2 GHz).
constexpr long long kWaitBudget = 4000000000LL;
// Budget of the waits that drain in-flight copies after a failure.
constexpr long long kDrainBudget = 2000000000LL;
// Budget of the deliberate never-satisfied wait used by the timeout self-test.
constexpr long long kProbeBudget = 200000LL;

// Record a device-side failure in the status word (first writer wins).
__device__ __forceinline__ void record_error(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Forward launch parameters shared by the fp32 and bf16 paths.
struct FwdParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, N, d;
  float scale;        // multiplier of the raw dot products
  float scale_log2;   // scale * log2(e)
  int* status;        // device status word
  int probe_timeout;  // nonzero: run the bounded-wait self-test and exit
};

struct BwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  float* D;           // [B, H, N] workspace: rowsum(dO * O)
  int B, H, N, d;
  float scale;
  float scale_log2;
  int grad_f32;       // 1: gradients stored as float32
  int* status;
  int probe_timeout;
};

// Host-side launchers (defined in the kernel translation units).
cudaError_t launch_fwd_simt_f32(const FwdParams& p, cudaStream_t s, bool causal);
cudaError_t launch_bwd_simt_f32(const BwdParams& p, cudaStream_t s, bool causal, int phase);
cudaError_t launch_bwd_dot(const BwdParams& p, bool bf16, cudaStream_t s);
// bf16 tensor-core path; returns cudaErrorNotSupported for shapes it does not
// take.  Tensor maps are built inside from the raw pointers.
cudaError_t launch_fwd_tc_bf16(const FwdParams& p, cudaStream_t s, bool causal);
// phase 1: dQ kernel (also refines D in the workspace); phase 2: dK/dV kernel.
cudaError_t launch_bwd_tc_bf16(const BwdParams& p, cudaStream_t s, bool causal, int phase);

}  // namespace fa
