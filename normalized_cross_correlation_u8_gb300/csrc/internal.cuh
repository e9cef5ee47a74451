// internal.cuh -- declarations shared by the translation units of libcorr.so
// (not part of the C ABI; include/corr.h is).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace corr {

// Number of SMs of the current device (queried once per device).
int device_sm_count();

// Let `kernel` use up to the device's opt-in shared memory (less its static
// shared memory).  The attribute persists, so the driver is called once per
// (device, kernel).
cudaError_t allow_dynamic_smem(const void *kernel);


// Stream-ordered temporary device memory from the library's pool on the
// current device (scratch.cu); release it with cudaFreeAsync on `stream`.
cudaError_t scratch_alloc(void **ptr, size_t bytes, cudaStream_t stream);

// Device memory the library's pool on the current device holds right now
// (0 if it has none).
cudaError_t scratch_reserved(size_t *bytes);

// Methods of the u8 fast path (corr.h: CORR_NCC_METHOD_*).
constexpr int kMethodDp4a = 0;   // SumI, SumISq, SumIT all by dp4a in the tiled kernel
constexpr int kMethodBox = 1;    // SumI, SumISq as box sums of the tile; SumIT by dp4a

// Launches the u8 normalized cross-correlation on `stream`.  Arguments are
// already validated by the C ABI layer (corr_api.cu).
cudaError_t ncc_u8_launch(const uint8_t *image, int w, int h, size_t pitch,
                          const uint8_t *tmpl, int wt, int ht,
                          uint32_t *sums_out, float *coef_out, int method,
                          cudaStream_t stream);

// Launches the f32 full cross-correlation on `stream` (validated arguments).
cudaError_t xcorr_f32_launch(const float *left, int nl, const float *right,
                             int nr, int H, int W, float *out,
                             cudaStream_t stream);

// Which kernel corr_xcorr_f32 runs for this shape (corr.h:
// CORR_XCORR_KERNEL_*).
int xcorr_f32_kernel_kind(int nl, int nr, int H, int W);

// Bytes of split-row scratch corr_xcorr_f32 would take for this shape (0
// when the chosen kernel needs none).
size_t xcorr_f32_scratch_bytes(const float *left, int nl, const float *right, int nr,
                               int H, int W, size_t max_scratch = ~size_t(0));

// As xcorr_f32_launch, but split-row partial sums go to `scratch` (at least
// xcorr_f32_scratch_bytes long; cudaErrorInvalidValue otherwise) instead of
// the library's pool: nothing is allocated.
cudaError_t xcorr_f32_launch_scratch(const float *left, int nl, const float *right,
                                     int nr, int H, int W, float *out, float *scratch,
                                     size_t scratch_bytes, cudaStream_t stream);

// Entry of the no-allocation variant (xcorr_noalloc.cu): scratch from the
// library's fixed device array.  Returns cudaErrorInvalidValue if the shape
// needs more than that array holds.
cudaError_t xcorr_f32_noalloc_launch(const float *left, int nl, const float *right,
                                     int nr, int H, int W, float *out,
                                     cudaStream_t stream);

// Tensor-core form of the f32 cross-correlation for small matrices
// (xcorr_tc.cu): H, W <= 16.
namespace tc {
bool supported(int nl, int nr, int H, int W);
cudaError_t launch(const float *left, int nl, const float *right, int nr, int H, int W,
                   float *out, cudaStream_t stream);
// Reads and clears the flag the kernel sets when a bounded wait gave up.
cudaError_t take_status(int *gave_up);
}  // namespace tc

// Tensor-core form for larger matrices (xcorr_tcl.cu): partial sums of
// K units in `scratch` (scratch_bytes long), added by a second kernel.
namespace tcl {
size_t scratch_bytes(int nl, int nr, int H, int W);
cudaError_t launch(const float *left, int nl, const float *right, int nr, int H, int W,
                   float *out, float *scratch, cudaStream_t stream);
cudaError_t take_status(int *gave_up);
}  // namespace tcl

// One warp per overlap with an in-warp reduction (xcorr_warp.cu).
namespace warp {
cudaError_t launch(const float *left, int nl, const float *right, int nr, int H, int W,
                   float *out, cudaStream_t stream);
}  // namespace warp

}  // namespace corr
