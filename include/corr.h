/*
 * corr.h -- C ABI of libcorr.so, GB300 (sm_103a) sliding-window 2D
 * correlation in two forms.
 *
 * Plain C types only.  Every buffer pointer is a DEVICE pointer (memory the
 * caller allocated on the current CUDA device, e.g. a torch tensor's
 * data_ptr(), or managed memory); page-locked host memory mapped into the
 * device's address space is also accepted (through its device alias; the
 * kernels then read and write across the host link, which is far slower
 * than copying).  Pageable host memory and other devices' memory are
 * refused with CORR_EINVAL.  The library never frees, keeps or reallocates
 * a caller buffer.  Calls are asynchronous on the calling thread's stream (see
 * corr_set_stream) and run on the calling thread's current CUDA device.
 * Every argument is checked before anything is launched: a call that returns
 * an error has written nothing.
 *
 * Return codes: CORR_OK or one of the negative CORR_E* codes below;
 * corr_strerror() names them.  After CORR_ECUDA, corr_last_cuda_error()
 * returns the cudaError_t value that caused it.
 */
#ifndef CORR_H_
#define CORR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CORR_OK 0
#define CORR_EINVAL (-1)        /* null pointer, size <= 0, template larger than image */
#define CORR_EUNSUPPORTED (-2)  /* a size the kernels do not handle (see each call) */
#define CORR_ECUDA (-3)         /* CUDA runtime error (no device, launch failure, ...) */
#define CORR_ETIMEOUT (-4)      /* a kernel gave up a bounded wait (corr_device_status) */

/* Largest template (pixels) whose SumISq and SumIT (at most N * 255^2)
 * still fit the unsigned 32-bit accumulators: 66051 * 65025 < 2^32 <=
 * 66052 * 65025. */
#define CORR_NCC_MAX_TEMPLATE_PIXELS 66051

/* Templates wider than 128 pixels, or too tall for the tiled kernel's
 * shared memory, take a general kernel that holds the template as packed
 * 32-bit words, ceil(wt/4) per row: ht * ceil(wt/4) may not exceed this
 * (only 1-pixel-wide templates taller than it are affected). */
#define CORR_NCC_MAX_GENERAL_TEMPLATE_WORDS 58000

/*
 * corr_ncc_u8 -- 8-bit normalized cross-correlation (template matching).
 *
 * Defined by The CUDA Handbook, ch. 15 "Image Processing: Normalized
 * Correlation", section 15.5 "Instruction-Level Parallelism and DP4A": for
 * every valid offset (x, y), 0 <= x <= w-wt, 0 <= y <= h-ht, the exact
 * unsigned 32-bit sums over the template window
 *     SumI   = sum_{j<ht,i<wt} I[y+j][x+i]
 *     SumISq = sum I[y+j][x+i]^2
 *     SumIT  = sum I[y+j][x+i] * T[j][i]
 * and the normalized coefficient (N = wt*ht, SumT / SumTSq the template's
 * sum and sum of squares)
 *     coef = (N*SumIT - SumI*SumT) / sqrt((N*SumISq - SumI^2)(N*SumTSq - SumT^2)),
 * with coef = 0 where either variance term is zero (flat window or flat
 * template).  Numerator and variance terms are exact 64-bit integers; the
 * final ratio is single precision (within 1e-5 absolute of the exact value).
 *
 *   image     device, w*h bytes, row-major, row pitch w bytes, any alignment
 *             (16- or 8-byte aligned rows are staged with vector loads).
 *             Templates up to 128 wide take the tiled fast kernel; wider ones
 *             a general kernel with the same results.
 *   w, h      image width and height in pixels, > 0.
 *   tmpl      device, wt*ht bytes, row-major, pitch wt.
 *   wt, ht    template size, 0 < wt <= w, 0 < ht <= h, and
 *             wt*ht <= CORR_NCC_MAX_TEMPLATE_PIXELS and
 *             ht*ceil(wt/4) <= CORR_NCC_MAX_GENERAL_TEMPLATE_WORDS, else
 *             CORR_EUNSUPPORTED.
 *             Any width: the template packs into 32-bit words with the last
 *             word of a row zero-padded, and that word's SumI / SumISq take
 *             only its template bytes.
 *   sums_out  device, 3 planes [3][oh][ow] of uint32 (SumI, SumISq, SumIT),
 *             ow = w-wt+1, oh = h-ht+1, dense, y-major; or NULL to skip.
 *   coef_out  device, [oh][ow] float32, dense; or NULL to skip.
 *             At least one of sums_out / coef_out must be non-NULL.
 */
int corr_ncc_u8(const uint8_t *image, int w, int h, const uint8_t *tmpl,
                int wt, int ht, uint32_t *sums_out, float *coef_out);

/*
 * corr_ncc_u8_pitched -- corr_ncc_u8 on an image whose rows are `pitch`
 * bytes apart (pitch >= w, else CORR_EINVAL): a pitched allocation or a
 * crop of a larger image.  Only the w bytes of each row are read; the
 * outputs stay dense.  corr_ncc_u8 is this call with pitch = w.  Vector
 * staging of the tile needs the image pointer, w and pitch all 16- (or 8-)
 * byte multiples; other images are staged with byte loads, same results.
 */
int corr_ncc_u8_pitched(const uint8_t *image, int w, int h, size_t pitch,
                        const uint8_t *tmpl, int wt, int ht, uint32_t *sums_out,
                        float *coef_out);

/*
 * corr_ncc_set_method / corr_ncc_get_method -- how corr_ncc_u8 forms SumI
 * and SumISq on its tiled fast kernel (templates up to 128 wide; wider or
 * very tall ones always use the first method).  Thread-local, like the
 * stream.  Both methods give bit-identical sums and coefficients, and
 * neither allocates memory.
 *
 *   CORR_NCC_METHOD_DP4A  the section's method: all three sums by unsigned
 *                         dp4a in the tiled kernel.
 *   CORR_NCC_METHOD_BOX   SumI and SumISq as box filters of I and I^2,
 *                         formed in the kernel from its staged tile by
 *                         sliding column and row sums (exact in unsigned
 *                         32-bit arithmetic), so the dp4a loop runs one
 *                         dp4a per 4 pixels (SumIT) instead of three.  A
 *                         reformulation that is not on the pages.
 *
 * corr_ncc_set_method returns CORR_EINVAL for any other value (the method
 * is then unchanged).  The default is CORR_NCC_METHOD_BOX.
 */
#define CORR_NCC_METHOD_DP4A 0
#define CORR_NCC_METHOD_BOX 1
int corr_ncc_set_method(int method);
int corr_ncc_get_method(void);

/*
 * corr_xcorr_f32 -- float32 full 2D cross-correlation, all overlaps.
 *
 * Defined by the "Efficient GPU-accelerated Parallel Cross-correlation"
 * artifact README (kernel overview: each output is one overlap of a left and
 * a right matrix; all overlaps are computed; one-to-one, one-to-many and
 * n-to-m batches).  For every pair (li, ri) and shift (dy, dx) with
 * |dy| < H, |dx| < W:
 *     out[li][ri][dy+H-1][dx+W-1] = sum_{y,x} L_li[y][x] * R_ri[y-dy][x-dx]
 * over the (y, x) where both matrices are indexed inside their bounds (the
 * same convention as scipy.signal.correlate2d(L, R, mode="full")).  Sums are
 * accumulated in float32; each output is within 1e-5 * sum |L*R| (over the
 * same overlap) of the exact value.
 *
 *   left      device, nl matrices [nl][H][W] float32, contiguous, 4-byte aligned.
 *   nl        number of left matrices, > 0 (1 for one-to-one and one-to-many).
 *   right     device, [nr][H][W] float32, contiguous, 4-byte aligned.
 *   nr        number of right matrices, > 0.
 *   H, W      matrix height and width, > 0.
 *   out       device, [nl][nr][2H-1][2W-1] float32, dense; pair li*nr+ri.
 *
 * Shapes it splits across blocks (row bands of more than 128 overlap rows
 * in a small batch, or x segments of rows wider than about 770 floats) take
 * temporary device memory for the partial sums, stream-ordered on the
 * current stream from a pool the library keeps per device; CORR_ECUDA if
 * that allocation fails.  The library holds none of it between calls: a
 * block freed by one call is reused by calls queued before the next
 * synchronisation of the stream or device, which hands it back to the
 * driver (see corr_scratch_reserved).
 */
int corr_xcorr_f32(const float *left, int nl, const float *right, int nr,
                   int H, int W, float *out);

/*
 * corr_xcorr_f32_kernel -- which of the library's kernels corr_xcorr_f32
 * runs for a batch of this shape on the current device (*kind gets one of
 * the values below); CORR_EINVAL for non-positive sizes or a NULL kind.
 * Launches nothing.  The choice also follows the environment variables
 * CORR_XCORR_TC, CORR_XCORR_TCL and CORR_XCORR_WARP ("1" / "0": take /
 * never take that kernel where it applies), read on every call.
 */
#define CORR_XCORR_KERNEL_ROWS 0      /* rows kernel, whole rows staged */
#define CORR_XCORR_KERNEL_ROWS_WIN 1  /* rows kernel, column windows */
#define CORR_XCORR_KERNEL_BCAST 2     /* rights in lanes (one-to-many) */
#define CORR_XCORR_KERNEL_TINY 3      /* small matrices, FP32 FMA */
#define CORR_XCORR_KERNEL_TENSOR 4    /* small matrices, tensor cores (split TF32) */
#define CORR_XCORR_KERNEL_WARP 5      /* one warp per overlap */
#define CORR_XCORR_KERNEL_TENSOR_LARGE 6   /* larger matrices, tensor cores (split TF32) */
int corr_xcorr_f32_kernel(int nl, int nr, int H, int W, int *kind);

/*
 * corr_xcorr_f32_noalloc -- corr_xcorr_f32 for callers that cannot allocate.
 *
 * No counterpart on the pages: this is a deployment variant of
 * corr_xcorr_f32 with the same arguments, layouts and error codes.  It runs
 * the kernel corr_xcorr_f32 would run whenever that kernel's scratch fits
 * the array below, with bit-identical results (the larger-matrix
 * tensor-core kernel's partial tiles and item counter included: 1 x 32 of
 * 64x64 needs 8 MiB); otherwise (larger one-to-one or one-to-many batches,
 * e.g. one 256x256 pair, whose tensor-core partial tiles take 16 MiB and
 * more) it runs the scalar kernel that fits, whose results meet the same
 * per-element bound but may differ in the last bits.
 * corr_xcorr_f32 takes temporary device memory for the partial sums of large
 * matrices from a stream-ordered pool that may call the driver's allocator.
 * Some callers cannot allow that -- an application that reserves all device
 * memory up front for its own allocator, a plug-in whose host framework
 * forbids driver allocations during its calls, a real-time loop that must
 * never wait on an allocator.  This call allocates nothing: its scratch is a
 * fixed array of CORR_XCORR_NOALLOC_SCRATCH_BYTES inside the library image,
 * which every GPU that loads the library's device code holds until the
 * process exits.
 *
 *   * Shapes whose partial sums need more than that return
 *     CORR_EUNSUPPORTED before anything is launched.  Of the scalar
 *     kernels only the large-matrix ones use scratch, when they split the
 *     overlap rows into bands
 *     (more than 128 rows in a small batch: one 256x256 pair needs 2 MiB)
 *     or the rows into x segments (rows wider than about 770 floats: about
 *     48 bytes per matrix element, so one 1024x1024 pair needs 48 MiB and
 *     is rejected).
 *   * The array's device memory is committed when the driver loads the
 *     library's module that holds it.  Under CUDA's lazy module loading (the
 *     default) that happens during the first call on a device that needs
 *     scratch, which also looks the array's device address up on that
 *     device: that call can fail with CORR_ECUDA if the caller has already
 *     reserved all device memory.  So make one warm-up call on each device
 *     with a shape that uses scratch (one 256x256 pair does) before
 *     reserving memory or beginning a stream capture, or load modules
 *     eagerly (environment CUDA_MODULE_LOADING=EAGER).
 *   * Every call, on every stream and thread, shares the one array: calls
 *     that overlap on the GPU race and corrupt each other's results, so
 *     order them (one stream, or events between streams).
 */
#define CORR_XCORR_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int corr_xcorr_f32_noalloc(const float *left, int nl, const float *right, int nr,
                           int H, int W, float *out);

/* Synchronises this thread's stream, then reports whether any of the
 * library's kernels gave up a bounded wait since the previous call
 * (CORR_ETIMEOUT: the outputs of the call that did are incomplete) or
 * CORR_OK.  Only the tensor-core cross-correlation kernel waits on other
 * units (the tensor cores' completion barriers); each wait ends after about
 * a second, so a fault there returns an error instead of hanging the GPU. */
int corr_device_status(void);

/* Bytes of device memory the library's scratch pool holds on the current
 * device right now: nonzero only while calls that use scratch are queued or
 * running (none after the stream or device has been synchronised). */
int corr_scratch_reserved(size_t *bytes);

/* Stream for this thread's following calls (a cudaStream_t; NULL = the
 * legacy default stream).  Thread-local; never fails. */
int corr_set_stream(void *stream);
void *corr_get_stream(void);

/* Human-readable name of a return code (static string). */
const char *corr_strerror(int code);

/* cudaError_t behind this thread's most recent CORR_ECUDA (0 if none). */
int corr_last_cuda_error(void);

/* Library ABI version (major*100 + minor). */
int corr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CORR_H_ */
