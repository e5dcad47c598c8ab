// Limits and host launchers of the radial edge-scalar kernels (radial.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace e3gb {

constexpr int kRadialMaxBasis = 16, kRadialMaxHidden = 16;

cudaError_t radial_hidden(int64_t E, const float* vec, const float* W1, int nb, int H, float rc, float* h,
                          cudaStream_t s);
cudaError_t radial_backward(int64_t E, const float* vec, const float* W1, int nb, int H, float rc, const float* dh,
                            float* dvec, int accumulate, cudaStream_t s);

}  // namespace e3gb
