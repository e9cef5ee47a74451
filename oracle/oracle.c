/*
 * oracle.c -- plain, slow, obviously correct CPU definitions of the two
 * sliding-window correlations.  TEST INFRASTRUCTURE ONLY: nothing on the
 * product path may include, link or call this file.  It shares no code,
 * header, table or helper with the CUDA library; it is built on its own by
 * gcc (oracle/build.py) and loaded by the tests and by the bench's CPU
 * baseline leg through ctypes.
 *
 * Sources (web pages, cited by title and section):
 *
 *  [H15] The CUDA Handbook, ch. 15 "Image Processing: Normalized Correlation",
 *        section 15.5 "Instruction-Level Parallelism and DP4A".  Defines the
 *        three per-offset accumulations SumI (sum of window pixels), SumISq
 *        (sum of squared window pixels) and SumIT (sum of window pixel times
 *        template pixel), over unsigned 8-bit pixels, in unsigned 32-bit
 *        accumulators.  The section prints only the sums; the coefficient is
 *        the textbook normalized correlation written over those sums (the
 *        chapter's subject), with N = template pixel count:
 *            (N*SumIT - SumI*SumT) / sqrt((N*SumISq - SumI^2)(N*SumTSq - SumT^2))
 *
 *  [JPDC] "Efficient GPU-accelerated Parallel Cross-correlation" replication
 *        package README (jpdc23-artifact), kernel overview paragraphs: every
 *        output is one overlap (relative shift) of a left and a right matrix,
 *        computed for all shifts ("full" cross-correlation), in one-to-one,
 *        one-to-many and n-to-m batches.  The page states no index
 *        convention; the reading used here is
 *            out[dy+H-1][dx+W-1] = sum_{y,x} L[y][x] * R[y-dy][x-dx]
 *        over the (y,x) where both indices are inside the matrices.
 *
 * Every function below is a direct transcription of these definitions with
 * plain loops: no blocking, no reordering, no shared work between outputs.
 * Floating point is accumulated in IEEE double.
 *
 * Return codes: 0 ok, -1 invalid argument, -2 unsupported size.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_EUNSUPPORTED (-2)

/* N*255^2 must fit the unsigned 32-bit accumulators [H15] use. */
#define ORACLE_MAX_TEMPLATE_PIXELS 66051L

/* ---------------------------------------------------------------------- */
/* u8 normalized cross-correlation [H15]                                   */
/* ---------------------------------------------------------------------- */

/* Sums of the template itself: SumT and SumTSq. */
static void tmpl_sums(const uint8_t *tmpl, int wt, int ht, uint32_t *sum_t,
                      uint32_t *sum_t_sq) {
    uint32_t s = 0, sq = 0;
    for (int j = 0; j < ht; j++)
        for (int i = 0; i < wt; i++) {
            uint32_t t = tmpl[(size_t)j * wt + i];
            s += t;
            sq += t * t;
        }
    *sum_t = s;
    *sum_t_sq = sq;
}

/* The three sums at one offset (x, y): window pixel (x+i, y+j) meets
 * template pixel (i, j). */
static void ncc_sums_at(const uint8_t *image, int w, const uint8_t *tmpl,
                        int wt, int ht, int x, int y, uint32_t *sum_i,
                        uint32_t *sum_i_sq, uint32_t *sum_it) {
    uint32_t si = 0, sq = 0, st = 0;
    for (int j = 0; j < ht; j++)
        for (int i = 0; i < wt; i++) {
            uint32_t p = image[(size_t)(y + j) * w + (x + i)];
            uint32_t t = tmpl[(size_t)j * wt + i];
            si += p;
            sq += p * p;
            st += p * t;
        }
    *sum_i = si;
    *sum_i_sq = sq;
    *sum_it = st;
}

/* Coefficient from exact sums.  Numerator and both variance terms are
 * formed in 64-bit integers (exact); only the final ratio is in double.
 * A flat window or a flat template (zero variance term) gives 0. */
static double ncc_coef(long n, uint32_t sum_i, uint32_t sum_i_sq,
                       uint32_t sum_it, uint32_t sum_t, uint32_t sum_t_sq) {
    int64_t num = (int64_t)n * sum_it - (int64_t)sum_i * sum_t;
    int64_t d_i = (int64_t)n * sum_i_sq - (int64_t)sum_i * sum_i;
    int64_t d_t = (int64_t)n * sum_t_sq - (int64_t)sum_t * sum_t;
    if (d_i <= 0 || d_t <= 0) return 0.0;
    return (double)num / sqrt((double)d_i * (double)d_t);
}

static int ncc_check(const uint8_t *image, int w, int h, const uint8_t *tmpl,
                     int wt, int ht) {
    if (!image || !tmpl || w <= 0 || h <= 0 || wt <= 0 || ht <= 0)
        return ORACLE_EINVAL;
    if (wt > w || ht > h) return ORACLE_EINVAL;
    if ((long)wt * ht > ORACLE_MAX_TEMPLATE_PIXELS) return ORACLE_EUNSUPPORTED;
    return ORACLE_OK;
}

/* All valid offsets.  sums_out: three planes [3][oh][ow] (SumI, SumISq,
 * SumIT), oh = h-ht+1, ow = w-wt+1.  coef_f64 / coef_f32: [oh][ow], either
 * may be NULL.  nthreads > 1 splits output rows across OpenMP threads. */
int oracle_ncc_u8(const uint8_t *image, int w, int h, const uint8_t *tmpl,
                  int wt, int ht, uint32_t *sums_out, double *coef_f64,
                  float *coef_f32, int nthreads) {
    int rc = ncc_check(image, w, h, tmpl, wt, ht);
    if (rc) return rc;
    if (!sums_out) return ORACLE_EINVAL;
    const int ow = w - wt + 1, oh = h - ht + 1;
    const size_t plane = (size_t)ow * oh;
    const long n = (long)wt * ht;
    uint32_t sum_t, sum_t_sq;
    tmpl_sums(tmpl, wt, ht, &sum_t, &sum_t_sq);
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int y = 0; y < oh; y++)
        for (int x = 0; x < ow; x++) {
            uint32_t si, sq, st;
            ncc_sums_at(image, w, tmpl, wt, ht, x, y, &si, &sq, &st);
            size_t o = (size_t)y * ow + x;
            sums_out[o] = si;
            sums_out[plane + o] = sq;
            sums_out[2 * plane + o] = st;
            double c = ncc_coef(n, si, sq, st, sum_t, sum_t_sq);
            if (coef_f64) coef_f64[o] = c;
            if (coef_f32) coef_f32[o] = (float)c;
        }
    return ORACLE_OK;
}

/* Selected offsets only: (xs[k], ys[k]) for k < count.  sums_out: [3][count]
 * planes; coef_f64: [count] (may be NULL). */
int oracle_ncc_u8_at(const uint8_t *image, int w, int h, const uint8_t *tmpl,
                     int wt, int ht, long count, const int *xs, const int *ys,
                     uint32_t *sums_out, double *coef_f64) {
    int rc = ncc_check(image, w, h, tmpl, wt, ht);
    if (rc) return rc;
    if (count < 0 || (count > 0 && (!xs || !ys || !sums_out)))
        return ORACLE_EINVAL;
    const long n = (long)wt * ht;
    uint32_t sum_t, sum_t_sq;
    tmpl_sums(tmpl, wt, ht, &sum_t, &sum_t_sq);
    for (long k = 0; k < count; k++) {
        if (xs[k] < 0 || ys[k] < 0 || xs[k] > w - wt || ys[k] > h - ht)
            return ORACLE_EINVAL;
        uint32_t si, sq, st;
        ncc_sums_at(image, w, tmpl, wt, ht, xs[k], ys[k], &si, &sq, &st);
        sums_out[k] = si;
        sums_out[count + k] = sq;
        sums_out[2 * count + k] = st;
        if (coef_f64) coef_f64[k] = ncc_coef(n, si, sq, st, sum_t, sum_t_sq);
    }
    return ORACLE_OK;
}

/* Template-only sums, exposed so tests can check SumT/SumTSq directly. */
int oracle_template_sums(const uint8_t *tmpl, int wt, int ht, uint32_t *out2) {
    if (!tmpl || !out2 || wt <= 0 || ht <= 0) return ORACLE_EINVAL;
    tmpl_sums(tmpl, wt, ht, &out2[0], &out2[1]);
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------- */
/* f32 full 2D cross-correlation [JPDC], accumulated in double             */
/* ---------------------------------------------------------------------- */

/* One overlap: shift (dy, dx) of right matrix R against left matrix L.
 * *abs_sum receives sum |L*R| over the same overlap (the error scale). */
static double xcorr_at(const float *L, const float *R, int H, int W, int dy,
                       int dx, double *abs_sum) {
    double s = 0.0, a = 0.0;
    for (int y = 0; y < H; y++) {
        int yr = y - dy;
        if (yr < 0 || yr >= H) continue;
        for (int x = 0; x < W; x++) {
            int xr = x - dx;
            if (xr < 0 || xr >= W) continue;
            double p = (double)L[(size_t)y * W + x] * (double)R[(size_t)yr * W + xr];
            s += p;
            a += fabs(p);
        }
    }
    *abs_sum = a;
    return s;
}

static int xcorr_check(const float *left, int nl, const float *right, int nr,
                       int H, int W) {
    if (!left || !right || nl <= 0 || nr <= 0 || H <= 0 || W <= 0)
        return ORACLE_EINVAL;
    return ORACLE_OK;
}

/* Every pair (li, ri) and every shift.  left: [nl][H][W], right: [nr][H][W].
 * out / abs_out: [nl][nr][2H-1][2W-1] (pair index li*nr+ri; abs_out may be
 * NULL).  nthreads > 1 splits pairs x output rows across OpenMP threads. */
int oracle_xcorr_f32(const float *left, int nl, const float *right, int nr,
                     int H, int W, double *out, double *abs_out,
                     int nthreads) {
    int rc = xcorr_check(left, nl, right, nr, H, W);
    if (rc) return rc;
    if (!out) return ORACLE_EINVAL;
    const int oh = 2 * H - 1, ow = 2 * W - 1;
    const size_t mat = (size_t)H * W, plane = (size_t)oh * ow;
    const long rows = (long)nl * nr * oh;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (long row = 0; row < rows; row++) {
        long pair = row / oh;
        int oy = (int)(row % oh);
        int li = (int)(pair / nr), ri = (int)(pair % nr);
        const float *L = left + (size_t)li * mat;
        const float *R = right + (size_t)ri * mat;
        for (int ox = 0; ox < ow; ox++) {
            double a;
            double s = xcorr_at(L, R, H, W, oy - (H - 1), ox - (W - 1), &a);
            size_t o = (size_t)pair * plane + (size_t)oy * ow + ox;
            out[o] = s;
            if (abs_out) abs_out[o] = a;
        }
    }
    return ORACLE_OK;
}

/* Selected outputs: pair ls[k]*nr+rs[k], output index (oys[k], oxs[k]) in
 * [0,2H-1) x [0,2W-1).  out / abs_out: [count] (abs_out may be NULL). */
int oracle_xcorr_f32_at(const float *left, int nl, const float *right, int nr,
                        int H, int W, long count, const int *ls, const int *rs,
                        const int *oys, const int *oxs, double *out,
                        double *abs_out) {
    int rc = xcorr_check(left, nl, right, nr, H, W);
    if (rc) return rc;
    if (count < 0 || (count > 0 && (!ls || !rs || !oys || !oxs || !out)))
        return ORACLE_EINVAL;
    const size_t mat = (size_t)H * W;
    for (long k = 0; k < count; k++) {
        if (ls[k] < 0 || ls[k] >= nl || rs[k] < 0 || rs[k] >= nr ||
            oys[k] < 0 || oys[k] >= 2 * H - 1 || oxs[k] < 0 || oxs[k] >= 2 * W - 1)
            return ORACLE_EINVAL;
        double a;
        out[k] = xcorr_at(left + (size_t)ls[k] * mat, right + (size_t)rs[k] * mat,
                          H, W, oys[k] - (H - 1), oxs[k] - (W - 1), &a);
        if (abs_out) abs_out[k] = a;
    }
    return ORACLE_OK;
}
