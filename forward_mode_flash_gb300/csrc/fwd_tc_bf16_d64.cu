// Tensor-core forward + JVP kernels for bf16 inputs, head dimension 64.
#include "fwd_dual_tc.cuh"

namespace jvp {
cudaError_t launch_fwd_tc_bf16_d64(int mask_kind, bool tangent, const TcMaps& maps,
                                   const FwdParams& p, cudaStream_t stream) {
  return launch_tc_dispatch<__nv_bfloat16, 64>(mask_kind, tangent, maps, p, stream);
}
}  // namespace jvp
