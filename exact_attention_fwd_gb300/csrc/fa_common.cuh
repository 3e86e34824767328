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

// Forward launch parameters shared by the fp32 and 16-bit paths.
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
  int f16;            // 16-bit storage is fp16 (else bf16)
  // split-KV partial pass (launch_fwd_tc16_partial); unused otherwise
  float* o_part;      // [nsplit, B, N, H, d] float32
  float* lse_part;    // [nsplit, B, H, N] float32
  int split_blocks;   // 128-key blocks per key slice (even)
  int nsplit;         // key slices: ceil(N / (128 split_blocks))
};

// fa_merge's launch parameters.
struct MergeParams {
  const float* o_part;
  const float* lse_part;
  void* o;
  float* lse;
  int B, H, N, d;
  int nsplit;          // slices present
  int keys_per_split;
  int causal;
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
  int f16;            // 16-bit storage (inputs, 16-bit gradients) is fp16 (else bf16)
};

// Host-side launchers (defined in the kernel translation units).
cudaError_t launch_fwd_simt_f32(const FwdParams& p, cudaStream_t s, bool causal);
cudaError_t launch_bwd_simt_f32(const BwdParams& p, cudaStream_t s, bool causal, int phase);
// elt: 0 float32, 1 bf16, 2 fp16 storage of O and dO
cudaError_t launch_bwd_dot(const BwdParams& p, int elt, cudaStream_t s);
// 16-bit (bf16 or fp16, p.f16) tensor-core path; returns
// cudaErrorNotSupported for shapes it does not take.  Tensor maps are built
// inside from the raw pointers.
cudaError_t launch_fwd_tc16(const FwdParams& p, cudaStream_t s, bool causal);
// split-KV partial pass of the tensor-core forward (writes p.o_part, p.lse_part)
cudaError_t launch_fwd_tc16_partial(const FwdParams& p, cudaStream_t s, bool causal);
// out_elt: 0 float32, 1 bf16, 2 fp16 storage of the merged O
cudaError_t launch_merge(const MergeParams& p, int out_elt, cudaStream_t s);
// float32 forward on the tensor cores (3xTF32), d <= 64; workspace of
// tf32x3_workspace_bytes() holds the hi/lo split of q, k, v
size_t tf32x3_workspace_bytes(int B, int H, int N, int d);
cudaError_t launch_fwd_tf32x3(const FwdParams& p, void* workspace, cudaStream_t s, bool causal);
// phase 1: dQ kernel (also refines D in the workspace); phase 2: dK/dV kernel.
cudaError_t launch_bwd_tc16(const BwdParams& p, cudaStream_t s, bool causal, int phase);
// float32 backward on the tensor cores (3xTF32), d <= 64: split passes, the D
// pre-pass (into the workspace), the dQ kernel and the dK/dV kernel; the
// workspace of tf32x3_bwd_workspace_bytes() holds D and the hi / lo copies
size_t tf32x3_bwd_workspace_bytes(int B, int H, int N, int d);
cudaError_t launch_bwd_tf32x3(const BwdParams& p, void* workspace, cudaStream_t s, bool causal);

}  // namespace fa
