// affine_gemv_f32.cu -- instantiations of the CUDA-core affine GEMV for f32 activations.
#include "affine_gemv.cuh"

namespace gai4 {
cudaError_t launch_affine_gemv_f32(const AffineGemvLaunch& L, cudaStream_t s) {
    return launch_affine_gemv_dtype<F32>(L, s);
}
}  // namespace gai4
