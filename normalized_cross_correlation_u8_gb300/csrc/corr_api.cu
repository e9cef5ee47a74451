// corr_api.cu -- the C ABI of libcorr.so (include/corr.h): argument checks,
// per-thread stream and error state, dispatch to the kernel launchers.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/corr.h"
#include "internal.cuh"

namespace {

thread_local cudaStream_t tls_stream = nullptr;
thread_local int tls_cuda_error = 0;
thread_local int tls_ncc_method = CORR_NCC_METHOD_BOX;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return CORR_OK;
  tls_cuda_error = int(e);
  return CORR_ECUDA;
}

// The calling thread's current device, or -1 (error cleared) if there is
// none.
int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return dev;
}

// The address at which device `dev`'s kernels reach a caller buffer:
// device or managed memory of this device as is; page-locked host memory
// mapped into the device's address space by its device alias.  Anything
// else (pageable host memory, another device's memory, an unknown address)
// is refused with CORR_EINVAL before any launch.
template <typename T>
int device_view(int dev, T *p, T **out) {
  if (dev < 0) return CORR_EINVAL;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();   // clear the sticky-free error of an unknown pointer
    return CORR_EINVAL;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice:
      if (at.device != dev) return CORR_EINVAL;
      *out = p;
      return CORR_OK;
    case cudaMemoryTypeManaged:
      *out = p;
      return CORR_OK;
    case cudaMemoryTypeHost:
      if (!at.devicePointer) return CORR_EINVAL;
      *out = static_cast<T *>(at.devicePointer);
      return CORR_OK;
    default:
      return CORR_EINVAL;
  }
}

// device_view of the three f32 buffers, each still 4-byte aligned.
int device_views(const float **left, const float **right, float **out) {
  const int dev = current_device();
  int rc;
  if ((rc = device_view(dev, *left, left)) != CORR_OK ||
      (rc = device_view(dev, *right, right)) != CORR_OK ||
      (rc = device_view(dev, *out, out)) != CORR_OK)
    return rc;
  if ((reinterpret_cast<uintptr_t>(*left) | reinterpret_cast<uintptr_t>(*right) |
       reinterpret_cast<uintptr_t>(*out)) & 3)
    return CORR_EINVAL;
  return CORR_OK;
}

}  // namespace

extern "C" {

int corr_ncc_u8(const uint8_t *image, int w, int h, const uint8_t *tmpl,
                int wt, int ht, uint32_t *sums_out, float *coef_out) {
  if (w <= 0) return CORR_EINVAL;
  return corr_ncc_u8_pitched(image, w, h, size_t(w), tmpl, wt, ht, sums_out, coef_out);
}

int corr_ncc_u8_pitched(const uint8_t *image, int w, int h, size_t pitch,
                        const uint8_t *tmpl, int wt, int ht, uint32_t *sums_out,
                        float *coef_out) {
  if (!image || !tmpl || (!sums_out && !coef_out)) return CORR_EINVAL;
  if (w <= 0 || h <= 0 || wt <= 0 || ht <= 0) return CORR_EINVAL;
  if (pitch < size_t(w)) return CORR_EINVAL;
  if (wt > w || ht > h) return CORR_EINVAL;
  if (int64_t(wt) * ht > CORR_NCC_MAX_TEMPLATE_PIXELS) return CORR_EUNSUPPORTED;
  if (int64_t(ht) * ((wt + 3) / 4) > CORR_NCC_MAX_GENERAL_TEMPLATE_WORDS)
    return CORR_EUNSUPPORTED;
  const int dev = current_device();
  int rc;
  if ((rc = device_view(dev, image, &image)) != CORR_OK ||
      (rc = device_view(dev, tmpl, &tmpl)) != CORR_OK ||
      (sums_out && (rc = device_view(dev, sums_out, &sums_out)) != CORR_OK) ||
      (coef_out && (rc = device_view(dev, coef_out, &coef_out)) != CORR_OK))
    return rc;
  // output planes are addressed with size_t, coordinates with int
  const int method = tls_ncc_method == CORR_NCC_METHOD_BOX ? corr::kMethodBox
                                                            : corr::kMethodDp4a;
  return cuda_status(corr::ncc_u8_launch(image, w, h, pitch, tmpl, wt, ht, sums_out,
                                         coef_out, method, tls_stream));
}

int corr_ncc_set_method(int method) {
  if (method != CORR_NCC_METHOD_DP4A && method != CORR_NCC_METHOD_BOX) return CORR_EINVAL;
  tls_ncc_method = method;
  return CORR_OK;
}

int corr_ncc_get_method(void) { return tls_ncc_method; }

int corr_xcorr_f32(const float *left, int nl, const float *right, int nr,
                   int H, int W, float *out) {
  if (!left || !right || !out) return CORR_EINVAL;
  if (nl <= 0 || nr <= 0 || H <= 0 || W <= 0) return CORR_EINVAL;
  if ((reinterpret_cast<uintptr_t>(left) | reinterpret_cast<uintptr_t>(right) |
       reinterpret_cast<uintptr_t>(out)) & 3)
    return CORR_EINVAL;
  // pair and coordinate indices are int: keep every count inside int range
  if (int64_t(nl) * nr > 0x7fffffffLL) return CORR_EUNSUPPORTED;
  if (int64_t(2) * H - 1 > 0x7fffffffLL || int64_t(2) * W - 1 > 0x7fffffffLL)
    return CORR_EUNSUPPORTED;
  int rc;
  if ((rc = device_views(&left, &right, &out)) != CORR_OK) return rc;
  return cuda_status(
      corr::xcorr_f32_launch(left, nl, right, nr, H, W, out, tls_stream));
}

int corr_xcorr_f32_noalloc(const float *left, int nl, const float *right, int nr,
                           int H, int W, float *out) {
  if (!left || !right || !out) return CORR_EINVAL;
  if (nl <= 0 || nr <= 0 || H <= 0 || W <= 0) return CORR_EINVAL;
  if ((reinterpret_cast<uintptr_t>(left) | reinterpret_cast<uintptr_t>(right) |
       reinterpret_cast<uintptr_t>(out)) & 3)
    return CORR_EINVAL;
  if (int64_t(nl) * nr > 0x7fffffffLL) return CORR_EUNSUPPORTED;
  if (int64_t(2) * H - 1 > 0x7fffffffLL || int64_t(2) * W - 1 > 0x7fffffffLL)
    return CORR_EUNSUPPORTED;
  if (corr::xcorr_f32_scratch_bytes(left, nl, right, nr, H, W,
                                    CORR_XCORR_NOALLOC_SCRATCH_BYTES) >
      CORR_XCORR_NOALLOC_SCRATCH_BYTES)
    return CORR_EUNSUPPORTED;
  int rc;
  if ((rc = device_views(&left, &right, &out)) != CORR_OK) return rc;
  return cuda_status(
      corr::xcorr_f32_noalloc_launch(left, nl, right, nr, H, W, out, tls_stream));
}

int corr_xcorr_f32_kernel(int nl, int nr, int H, int W, int *kind) {
  if (!kind || nl <= 0 || nr <= 0 || H <= 0 || W <= 0) return CORR_EINVAL;
  if (int64_t(nl) * nr > 0x7fffffffLL) return CORR_EUNSUPPORTED;
  if (int64_t(2) * H - 1 > 0x7fffffffLL || int64_t(2) * W - 1 > 0x7fffffffLL)
    return CORR_EUNSUPPORTED;
  *kind = corr::xcorr_f32_kernel_kind(nl, nr, H, W);
  return CORR_OK;
}

int corr_device_status(void) {
  cudaError_t e = cudaStreamSynchronize(tls_stream);
  if (e != cudaSuccess) return cuda_status(e);
  int gave_up = 0, gave_up_l = 0;
  if ((e = corr::tc::take_status(&gave_up)) != cudaSuccess) return cuda_status(e);
  if ((e = corr::tcl::take_status(&gave_up_l)) != cudaSuccess) return cuda_status(e);
  return gave_up || gave_up_l ? CORR_ETIMEOUT : CORR_OK;
}

int corr_scratch_reserved(size_t *bytes) {
  if (!bytes) return CORR_EINVAL;
  return cuda_status(corr::scratch_reserved(bytes));
}

int corr_set_stream(void *stream) {
  tls_stream = static_cast<cudaStream_t>(stream);
  return CORR_OK;
}

void *corr_get_stream(void) { return static_cast<void *>(tls_stream); }

const char *corr_strerror(int code) {
  switch (code) {
    case CORR_OK: return "ok";
    case CORR_EINVAL: return "invalid argument";
    case CORR_EUNSUPPORTED: return "unsupported size";
    case CORR_ECUDA: return "CUDA runtime error";
    case CORR_ETIMEOUT: return "a kernel gave up a bounded wait";
    default: return "unknown error code";
  }
}

int corr_last_cuda_error(void) { return tls_cuda_error; }

int corr_version(void) { return 100; }

}  // extern "C"
