// Tensor-core backward kernels for bf16 inputs, head dimension 128.
#include "bwd_dual_tc.cuh"

namespace jvp {
cudaError_t launch_bwd_tc_bf16_d128(int mask_kind, const BwdTcMaps& qmaps, const BwdTcMaps& kmaps,
                                   const BwdParams& p, int num_sms, unsigned int* status,
                                   cudaStream_t stream, cudaStream_t kstream) {
  return launch_bwd_tc_dispatch<__nv_bfloat16, 128>(mask_kind, qmaps, kmaps, p, num_sms, status, stream,
                                                 kstream);
}
}  // namespace jvp
