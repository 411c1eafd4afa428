// Instantiations of the W4 projection kernels for bf16 activations.
#include "vq_gemm.cuh"
#include "vq_tc.cuh"

namespace vq {
int launch_gemm_bf16(const GemmLaunch& L) { return launch_gemm_act<VQ_BF16>(L); }
}  // namespace vq
