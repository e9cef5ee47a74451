// device.cu -- per-device launch attributes shared by the kernels of
// libcorr.so: the SM count and the shared-memory opt-in, each queried once
// and cached (per device, per kernel) under a mutex.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <set>

#include "internal.cuh"

namespace corr {
namespace {

constexpr int kAttrDevices = 64;
std::mutex g_attr_mu;
int g_sms[kAttrDevices] = {};
int g_smem_optin[kAttrDevices] = {};
std::set<const void *> g_smem_done[kAttrDevices];

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kAttrDevices) return -1;
  return dev;
}

cudaError_t device_attrs_locked(int dev) {
  if (g_smem_optin[dev]) return cudaSuccess;
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  g_smem_optin[dev] = optin;
  return cudaSuccess;
}

}  // namespace

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (!g_sms[dev]) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
      return 1;
    g_sms[dev] = sms;
  }
  return g_sms[dev];
}

cudaError_t allow_dynamic_smem(const void *kernel) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (g_smem_done[dev].count(kernel)) return cudaSuccess;
  cudaError_t e = device_attrs_locked(dev);
  if (e != cudaSuccess) return e;
  // dynamic + the kernel's static shared memory may not exceed the opt-in limit
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kernel)) != cudaSuccess) return e;
  const int dyn = g_smem_optin[dev] - int(fa.sharedSizeBytes);
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn)) !=
      cudaSuccess)
    return e;
  g_smem_done[dev].insert(kernel);
  return cudaSuccess;
}

}  // namespace corr
