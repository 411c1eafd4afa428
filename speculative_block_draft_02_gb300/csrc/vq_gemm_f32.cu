// Instantiations of the W4 projection kernels for f32 activations.
#include "vq_gemm.cuh"

namespace vq {
int launch_gemm_f32(const GemmLaunch& L) { return launch_gemm_act<VQ_F32>(L); }
}  // namespace vq
