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

}  // namespace

extern "C" {

int corr_ncc_u8(const uint8_t *image, int w, int h, const uint8_t *tmpl,
                int wt, int ht, uint32_t *sums_out, float *coef_out) {
  if (!image || !tmpl || (!sums_out && !coef_out)) return CORR_EINVAL;
  if (w <= 0 || h <= 0 || wt <= 0 || ht <= 0) return CORR_EINVAL;
  if (wt > w || ht > h) return CORR_EINVAL;
  if (int64_t(wt) * ht > CORR_NCC_MAX_TEMPLATE_PIXELS) return CORR_EUNSUPPORTED;
  // output planes are addressed with size_t, coordinates with int
  const int method = tls_ncc_method == CORR_NCC_METHOD_BOX ? corr::kMethodBox
                                                            : corr::kMethodDp4a;
  return cuda_status(corr::ncc_u8_launch(image, w, h, tmpl, wt, ht, sums_out,
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
  if (corr::xcorr_f32_scratch_bytes(left, nl, right, nr, H, W) >
      CORR_XCORR_NOALLOC_SCRATCH_BYTES)
    return CORR_EUNSUPPORTED;
  return cuda_status(
      corr::xcorr_f32_noalloc_launch(left, nl, right, nr, H, W, out, tls_stream));
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
    default: return "unknown error code";
  }
}

int corr_last_cuda_error(void) { return tls_cuda_error; }

int corr_version(void) { return 100; }

}  // extern "C"
