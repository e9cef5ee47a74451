// scratch.cu -- temporary device memory for the kernels of libcorr.so:
// stream-ordered allocations from one library-owned pool per device whose
// release threshold is unlimited, so blocks freed by one call are reused by
// the next without going back to the driver.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.cuh"

namespace corr {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxDevices] = {};

cudaError_t scratch_pool(cudaMemPool_t *pool) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  if (!g_pools[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t p;
    if ((e = cudaMemPoolCreate(&p, &props)) != cudaSuccess) return e;
    uint64_t keep = ~uint64_t(0);
    if ((e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep)) !=
        cudaSuccess) {
      cudaMemPoolDestroy(p);
      return e;
    }
    g_pools[dev] = p;
  }
  *pool = g_pools[dev];
  return cudaSuccess;
}

}  // namespace

cudaError_t scratch_alloc(void **ptr, size_t bytes, cudaStream_t stream) {
  cudaMemPool_t pool;
  cudaError_t e = scratch_pool(&pool);
  if (e != cudaSuccess) return e;
  return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

}  // namespace corr
