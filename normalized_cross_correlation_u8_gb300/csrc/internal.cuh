// internal.cuh -- declarations shared by the translation units of libcorr.so
// (not part of the C ABI; include/corr.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace corr {

// Launches the u8 normalized cross-correlation on `stream`.  Arguments are
// already validated by the C ABI layer (corr_api.cu).
cudaError_t ncc_u8_launch(const uint8_t *image, int w, int h,
                          const uint8_t *tmpl, int wt, int ht,
                          uint32_t *sums_out, float *coef_out,
                          cudaStream_t stream);

// Launches the f32 full cross-correlation on `stream` (validated arguments).
cudaError_t xcorr_f32_launch(const float *left, int nl, const float *right,
                             int nr, int H, int W, float *out,
                             cudaStream_t stream);

}  // namespace corr
