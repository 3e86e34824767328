// tc_bwd.cu — bf16 attention backward on the sm_103a tensor cores (pending).
#include "fa_common.cuh"

namespace fa {

cudaError_t launch_bwd_tc_bf16(const BwdParams&, cudaStream_t, bool) {
  return cudaErrorNotSupported;
}

}  // namespace fa
