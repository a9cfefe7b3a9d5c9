// Tensor-core backward kernels for f16 inputs, head dimension 64.
#include "bwd_dual_tc.cuh"

namespace jvp {
cudaError_t launch_bwd_tc_f16_d64(int mask_kind, const BwdTcMaps& qmaps, const BwdTcMaps& kmaps,
                                   const BwdParams& p, int num_sms, unsigned int* status,
                                   cudaStream_t stream, cudaStream_t kstream) {
  return launch_bwd_tc_dispatch<__half, 64>(mask_kind, qmaps, kmaps, p, num_sms, status, stream,
                                                 kstream);
}
}  // namespace jvp
