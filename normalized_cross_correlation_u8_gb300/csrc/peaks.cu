// peaks.cu -- issue-rate probes (include/corr_peaks.h): saturating kernels of
// unsigned __dp4a and of FP32 FMA, timed with CUDA events.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/corr.h"
#include "../../include/corr_peaks.h"

namespace {

__device__ uint32_t g_sink_u32;
__device__ float g_sink_f32;

constexpr int kChains = 8;
constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;

// kChains independent dp4a chains per thread; SHF funnel shifts per 8 dp4a.
template <int SHF>
__global__ void __launch_bounds__(kThreads) dp4a_probe(int iters, uint32_t seed) {
  uint32_t acc[kChains], x[kChains];
#pragma unroll
  for (int k = 0; k < kChains; ++k) {
    acc[k] = seed + threadIdx.x + k;
    x[k] = (seed * 2654435761u) ^ (threadIdx.x * 40503u + k);
  }
  const uint32_t y = seed | 0x80808080u;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int k = 0; k < kChains; ++k) acc[k] = __dp4a(acc[k], y, acc[k]);
#pragma unroll
      for (int k = 0; k < SHF; ++k) x[k] = __funnelshift_r(x[k], x[k + 1], 8);
    }
  }
  uint32_t s = 0;
#pragma unroll
  for (int k = 0; k < kChains; ++k) s ^= acc[k] ^ x[k];
  if (s == 0x9e3779b9u) g_sink_u32 = s;
}

__global__ void __launch_bounds__(kThreads) ffma_probe(int iters, float seed) {
  float acc[kChains];
#pragma unroll
  for (int k = 0; k < kChains; ++k) acc[k] = seed + float(threadIdx.x + k);
  const float a = 0.999f + seed * 1e-9f, b = 1e-7f * seed;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int k = 0; k < kChains; ++k) acc[k] = fmaf(acc[k], a, b);
  }
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kChains; ++k) s += acc[k];
  if (s == 1234.5f) g_sink_f32 = s;
}

template <typename Launch>
int time_probe(Launch launch, double ops_per_launch, double *rate,
               double *seconds) {
  cudaStream_t stream = static_cast<cudaStream_t>(corr_get_stream());
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return CORR_ECUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return CORR_ECUDA;
  }
  float best = 1e30f;
  cudaError_t err = cudaSuccess;
  for (int rep = 0; rep < 4 && err == cudaSuccess; ++rep) {  // rep 0 warms up
    cudaEventRecord(e0, stream);
    launch(stream);
    cudaEventRecord(e1, stream);
    err = cudaEventSynchronize(e1);
    if (err == cudaSuccess) err = cudaGetLastError();
    float ms = 0.f;
    if (err == cudaSuccess) cudaEventElapsedTime(&ms, e0, e1);
    if (rep > 0 && ms < best) best = ms;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (err != cudaSuccess) return CORR_ECUDA;
  if (rate) *rate = ops_per_launch / (best * 1e-3);
  if (seconds) *seconds = best * 1e-3;
  return CORR_OK;
}

int grid_blocks() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  return sms * kBlocksPerSm;
}

}  // namespace

extern "C" {

int corr_peak_dp4a(int shf_per_8, double *dp4a_per_s, double *seconds) {
  if (shf_per_8 != 0 && shf_per_8 != 1 && shf_per_8 != 2 && shf_per_8 != 4)
    return CORR_EINVAL;
  const int blocks = grid_blocks();
  if (blocks <= 0) return CORR_ECUDA;
  const int iters = 4096;
  const double ops = double(blocks) * kThreads * iters * 4 * kChains;
  auto launch = [&](cudaStream_t s) {
    switch (shf_per_8) {
      case 0: dp4a_probe<0><<<blocks, kThreads, 0, s>>>(iters, 12345u); break;
      case 1: dp4a_probe<1><<<blocks, kThreads, 0, s>>>(iters, 12345u); break;
      case 2: dp4a_probe<2><<<blocks, kThreads, 0, s>>>(iters, 12345u); break;
      default: dp4a_probe<4><<<blocks, kThreads, 0, s>>>(iters, 12345u); break;
    }
  };
  return time_probe(launch, ops, dp4a_per_s, seconds);
}

int corr_peak_ffma(double *ffma_per_s, double *seconds) {
  const int blocks = grid_blocks();
  if (blocks <= 0) return CORR_ECUDA;
  const int iters = 4096;
  const double ops = double(blocks) * kThreads * iters * 4 * kChains;
  auto launch = [&](cudaStream_t s) {
    ffma_probe<<<blocks, kThreads, 0, s>>>(iters, 1.0f);
  };
  return time_probe(launch, ops, ffma_per_s, seconds);
}

}  // extern "C"
