// Backward attention on the tcgen05 tensor cores (written next).
#include "kernels.h"

namespace attn {

cudaError_t launch_bwd_tc(const Problem&, const CUtensorMap&, const CUtensorMap&,
                          const CUtensorMap&, const CUtensorMap&, const float*, const float*,
                          __nv_bfloat16*, __nv_bfloat16*, __nv_bfloat16*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace attn
