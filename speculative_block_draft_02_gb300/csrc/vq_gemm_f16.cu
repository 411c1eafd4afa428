// Instantiations of the W4 projection kernels for f16 activations.
#include "vq_gemm.cuh"
#include "vq_tc.cuh"

namespace vq {
int launch_gemm_f16(const GemmLaunch& L) { return launch_gemm_act<VQ_F16>(L); }
}  // namespace vq
