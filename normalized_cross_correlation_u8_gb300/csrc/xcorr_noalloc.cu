// xcorr_noalloc.cu -- the f32 cross-correlation for callers that cannot
// allocate device memory.
//
// corr_xcorr_f32 takes the split-row partial sums of large matrices from a
// stream-ordered memory pool, which allocates from the driver the first time
// a shape needs more than the pool holds.  Some callers may not let a library
// do that: an application that reserves all device memory up front for its
// own allocator, a plug-in hosted by a framework that forbids driver
// allocations inside its calls, or a real-time loop that must never wait on
// the allocator.  For them this file holds the scratch in a fixed device
// array that is part of the library image, so the call allocates nothing.
//
// The array is CORR_XCORR_NOALLOC_SCRATCH_BYTES (16 MiB) long.  Every GPU on
// which the library's device code is loaded holds it until the process exits;
// its memory is committed when the driver loads this file's module, which
// under lazy module loading is the first cudaGetSymbolAddress below (the
// first call on a device whose shape needs scratch).
// All calls on all streams share it: calls that overlap on the GPU race on it,
// so a caller must order them (one stream, or events).  Nothing in it needs to
// start at zero -- every partial sum a call reads was written earlier in the
// same call -- so it is never cleared.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/corr.h"
#include "internal.cuh"

namespace corr {
namespace {

constexpr size_t kScratchFloats = CORR_XCORR_NOALLOC_SCRATCH_BYTES / sizeof(float);

static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float *g_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (host code cannot use the symbol itself: on the host its name
// denotes a shadow variable, not device memory).
cudaError_t scratch_address(float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess) return e;
    g_addr[dev] = static_cast<float *>(p);
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

cudaError_t xcorr_f32_noalloc_launch(const float *left, int nl, const float *right,
                                     int nr, int H, int W, float *out,
                                     cudaStream_t stream) {
  const size_t need =
      xcorr_f32_scratch_bytes(left, nl, right, nr, H, W, CORR_XCORR_NOALLOC_SCRATCH_BYTES);
  if (need > CORR_XCORR_NOALLOC_SCRATCH_BYTES) return cudaErrorInvalidValue;
  float *scratch = nullptr;
  if (need > 0) {
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return e;
  }
  return xcorr_f32_launch_scratch(left, nl, right, nr, H, W, out, scratch,
                                  CORR_XCORR_NOALLOC_SCRATCH_BYTES, stream);
}

}  // namespace corr
