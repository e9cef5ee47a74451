// scratch.cu -- temporary device memory for the kernels of libcorr.so:
// stream-ordered allocations from one library-owned pool per device.  The
// pool's release threshold is zero, so the library keeps nothing between
// calls: a block freed by one call is reused by the next call queued before
// the stream (or device) is synchronised, and handed back to the driver at
// that synchronisation.
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
    uint64_t keep = 0;
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

cudaError_t scratch_reserved(size_t *bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  *bytes = 0;
  if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lock(g_pool_mu);
    pool = g_pools[dev];
  }
  if (!pool) return cudaSuccess;
  uint64_t v = 0;
  if ((e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &v)) != cudaSuccess)
    return e;
  *bytes = size_t(v);
  return cudaSuccess;
}

cudaError_t scratch_alloc(void **ptr, size_t bytes, cudaStream_t stream) {
  cudaMemPool_t pool;
  cudaError_t e = scratch_pool(&pool);
  if (e != cudaSuccess) return e;
  return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

}  // namespace corr
