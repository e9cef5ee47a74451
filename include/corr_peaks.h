/*
 * corr_peaks.h -- issue-rate probes of libcorr.so, used to state the
 * arithmetic roofline of the correlation kernels on the device they run on.
 *
 * Not an operation of the pages: the u8 path is bound by unsigned __dp4a
 * issue (The CUDA Handbook ch. 15, section 15.5 moves the kernel from
 * latency-bound to arithmetic-bound) and the f32 path by FP32 fused
 * multiply-add issue, and neither rate is published for this GPU, so the
 * library measures them.  Each probe launches a saturating kernel on the
 * current device (every SM, full occupancy, independent chains), times it
 * with CUDA events on the calling thread's stream (corr_set_stream) and
 * synchronises that stream before returning.  No caller buffers.
 *
 * Return codes as in corr.h.
 */
#ifndef CORR_PEAKS_H_
#define CORR_PEAKS_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Unsigned dp4a per second.  shf_per_8: funnel shifts issued per 8 dp4a
 * (0, 1, 2 or 4) to show whether shifts share the dp4a pipe.  *seconds gets
 * the timed kernel's duration.  Either out pointer may be NULL. */
int corr_peak_dp4a(int shf_per_8, double *dp4a_per_s, double *seconds);

/* FP32 fused multiply-adds per second (one FMA = 2 flops). */
int corr_peak_ffma(double *ffma_per_s, double *seconds);

#ifdef __cplusplus
}
#endif

#endif /* CORR_PEAKS_H_ */
