// ncc_u8_kernels.cuh -- 8-bit normalized cross-correlation on sm_103a:
// kernels and launch helpers shared by ncc_u8.cu, ncc_u8_wide.cu and the
// box-form translation units ncc_u8_box.cu / ncc_u8_box_wide.cu.
//
// Method (The CUDA Handbook, ch. 15 "Image Processing: Normalized
// Correlation", section 15.5 "Instruction-Level Parallelism and DP4A"):
// four pixels are packed into one 32-bit word and each of the three sums
// advances by one *unsigned* __dp4a per word (SumI against 0x01010101,
// SumISq against the word itself, SumIT against the packed template word).
// Consecutive output columns slide the window by one byte, so a thread's
// window words are cut out of two aligned image words with __funnelshift_r;
// the template packs directly into words (a width that is not a multiple of
// four zero-pads each row's last word, whose SumI / SumISq then take only
// the template bytes: a generalization the section does not state).  Several
// independent output columns (and rows) per thread keep many accumulation
// chains in flight (the section's instruction-level parallelism).
//
// GB300 layout of the work (fast path: wt up to 128, any image alignment;
// wider templates take the general path below):
//   * a CTA owns 128 output columns x TY output rows; it copies the image
//     tile plus its halo (TY+ht-1 rows x 128+wt+8 bytes) into shared memory
//     with independent 16-byte vector loads (one memory latency per tile,
//     out-of-image bytes zero), and stages the template as packed words;
//   * each half-warp owns R output rows, each lane 8 adjacent columns whose
//     words start 8-byte aligned; the half-warp walks its R+ht-1 tile rows
//     once, cutting each row into the lane's 8 windows with funnel shifts
//     (windows of columns 4..7 at word i equal those of columns 0..3 at word
//     i+1, so 3 shifts per word serve 8 columns) and pairing it with
//     template row k-r for each of its R output rows;
//   * the template row is read as warp-uniform 16-byte shared broadcasts;
//     each CTA also reduces SumT / SumTSq from it;
//   * the epilogue forms N*SumIT - SumI*SumT and N*SumISq - SumI^2 exactly in
//     64-bit integers before the single-precision ratio, and writes each
//     output plane through a warp-private staging area (coalesced stores)
//     or, for large box-form templates, straight from the lanes.
// Box form (BOX = true, the library's default; not on the pages): SumI and
// SumISq are box filters of the staged tile -- sliding column sums over ht
// rows, then sliding row sums over wt columns, exact in unsigned 32-bit
// arithmetic -- so the dp4a loop accumulates SumIT alone (box_columns,
// box_rows).
// Measured on GB300: with the three sums the unsigned dp4a pipe (64 per SM
// per clock) is 80-93 % busy with dp4a on 32-128-wide templates; the box
// form does the same steps 1.9-2.6x faster.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <array>
#include <type_traits>
#include <utility>

#include "internal.cuh"

namespace corr {
namespace ncc {

constexpr int kCols = 8;                   // output columns per lane
constexpr int kUnitCols = 32 * kCols;      // output columns per warp unit (general path)
constexpr int kHalfUnitCols = 16 * kCols;  // output columns per warp unit (fast path)
// Warps per CTA and output rows per half-warp (compile-time tuning knobs).
#ifndef CORR_NCC_WARPS
#define CORR_NCC_WARPS 2
#endif
#ifndef CORR_NCC_ROWS
#define CORR_NCC_ROWS 1
#endif
#ifndef CORR_NCC_MINB
#define CORR_NCC_MINB 1
#endif
#ifndef CORR_NCC_KSPLIT
#define CORR_NCC_KSPLIT 2
#endif
// Output rows per half-warp of the box-sum form: CORR_NCC_BOX_ROWS, or 1
// for templates of up to CORR_NCC_BOX_NARROW_WORDS words on images whose
// tiles would fill fewer than CORR_NCC_BOX_NARROW_TILES_PER_SM tiles per SM
// (smaller tiles then fill the SMs more evenly).
#ifndef CORR_NCC_BOX_ROWS
#define CORR_NCC_BOX_ROWS 2
#endif
#ifndef CORR_NCC_BOX_NARROW_WORDS
#define CORR_NCC_BOX_NARROW_WORDS 4
#endif
#ifndef CORR_NCC_BOX_NARROW_TILES_PER_SM
#define CORR_NCC_BOX_NARROW_TILES_PER_SM 16
#endif
// Minimum resident CTAs per SM asked of the compiler for the box form:
// templates of up to 16 words, and wider ones.
#ifndef CORR_NCC_BOX_MINB
#define CORR_NCC_BOX_MINB 8
#endif
#ifndef CORR_NCC_BOX_MINB_WIDE
#define CORR_NCC_BOX_MINB_WIDE 1
#endif
// Template-row ranges (warp groups) per tile of the SumIT-only kernel.
// Fast kernel: write outputs through a warp-private staging area
// (coalesced stores) rather than each lane's own 8 columns -- always for the
// three-dp4a method, and for the box form while the template has at most
// CORR_NCC_STAGED_BOX_WORDS words (wtw * ht): beyond that the staging's
// instructions cost more than the scattered stores.
#ifndef CORR_NCC_STAGED_STORES
#define CORR_NCC_STAGED_STORES 1
#endif
#ifndef CORR_NCC_STAGED_BOX_WORDS
#define CORR_NCC_STAGED_BOX_WORDS 200
#endif
// Warps per template-row group (row groups of the tile) of the box form.
#ifndef CORR_NCC_BOX_WARPS
#define CORR_NCC_BOX_WARPS 2
#endif
#ifndef CORR_NCC_BOX_KSPLIT
#define CORR_NCC_BOX_KSPLIT 2
#endif
constexpr int kWarpsPerCta = CORR_NCC_WARPS;
constexpr int kThreads = 32 * kWarpsPerCta;
// Fast path: the template rows of a tile are split into kSplit ranges, one
// per group of kWarpsPerCta warps; the groups' partial sums are added in
// shared memory (integer sums: exact in any order).
constexpr int kSplit = CORR_NCC_KSPLIT;
constexpr int kBoxRows = CORR_NCC_BOX_ROWS;
constexpr int kBoxNarrowWords = CORR_NCC_BOX_NARROW_WORDS;
constexpr int kBoxSplit = CORR_NCC_BOX_KSPLIT;
constexpr int kBoxWarps = CORR_NCC_BOX_WARPS;
// Warp groups and threads of the fast kernel (BOX: the SumIT-only form).
template <bool BOX>
struct FixedShape {
  static constexpr int kWarps = BOX ? kBoxWarps : kWarpsPerCta;   // per group
  static constexpr int kGroups = BOX ? kBoxSplit : kSplit;
  static constexpr int kThreadsPerCta = 32 * kWarps * kGroups;
};


// Shared memory of a fast-path tile: the packed template (ht rows of wtp
// words), the image tile plus halo (TY+ht-1 rows of 128+4*wtw+8 bytes,
// rounded to 16) and the exchange area of the template-row split (groups
// warp groups, ns sums per output).
// Box-sum form: the column sums of the tile's TY output rows (row stride
// box_v_stride words, column x stored at box_v_col(x) = x + x/8) and the
// finished SumI / SumISq of its TY x 128 outputs (16-byte chunk q of a row
// stored at box_s_chunk(q)), each for I and I^2.
//
// The row pass reads the column sums as 16 runs of 8 (columns 8 k + j) from
// two rows at once: column 8 k + j lands in bank 9 k + j + j/8 (mod 32), 16
// distinct banks, and a row stride of 16 mod 32 puts the second row on the
// other 16.
__host__ __device__ inline int box_v_col(int x) { return x + (x >> 3); }
__host__ __device__ inline int box_v_stride(int wt) {
  const int nv = kHalfUnitCols + wt - 1;              // columns a tile's windows reach
  const int last = box_v_col(nv - 1);                 // skewed index of the last one
  return ((last + 1 - 16 + 31) & ~31) + 16;           // = 16 mod 32: conflict-free rows
}
// Finished sums are written and read as two 16-byte chunks 2k, 2k + 1 per
// thread, 8 threads (k = 8 g .. 8 g + 7) per shared-memory phase: flipping
// the low bit of every chunk in the upper half of each group of 16 spreads
// those 8 chunks over all 32 banks.
__host__ __device__ inline int box_s_chunk(int q) { return q ^ ((q >> 3) & 1); }
// The box-sum form reuses dead regions: once the dp4a loop is done, the
// column sums overwrite the template and the finished SumI / SumISq the
// tile, so its layout is [tile | exchange | template], each of the first
// and last at least as large as what later takes its place.
struct TileLayout {
  size_t tile, part, tmpl, total;   // byte offsets of the regions, total size
};
inline TileLayout fixed_tile_layout(int ht, int wtw, int wtp, int rows, int warps,
                                    int groups, int ns, bool box, int wt) {
  const int ty = 2 * rows * warps;
  const size_t rb = (kHalfUnitCols + 4 * wtw + 8 + 15) & ~15;
  const size_t tile = size_t(ty + ht - 1) * rb;
  const size_t part = size_t(groups - 1) * warps * 32 * ns * rows * kCols * 4;
  const size_t tmpl = size_t(ht) * wtp * 4;
  TileLayout l;
  if (!box) {
    l.tmpl = 0;
    l.tile = tmpl;
    l.part = tmpl + tile;
    l.total = tmpl + tile + part;
  } else {
    const size_t s = size_t(2) * ty * kHalfUnitCols * 4;
    const size_t v = size_t(2) * ty * box_v_stride(wt) * 4;
    l.tile = 0;
    l.part = tile > s ? tile : s;
    l.tmpl = l.part + part;
    l.total = l.tmpl + (tmpl > v ? tmpl : v);
  }
  return l;
}
constexpr uint32_t kOnes = 0x01010101u;
constexpr int kStageBatch = 4;       // tile chunks per thread loaded ahead of the template

struct NccArgs {
  const uint8_t *image;
  const uint8_t *tmpl;
  uint32_t *sums;
  float *coef;
  size_t plane;      // ow * oh
  int w, h, wt, ht;
  size_t pitch;      // bytes from one image row to the next (>= w)
  int wtw;           // template words per row (ceil(wt / 4))
  int tail;          // wt % 4: bytes of the last word that are template pixels (0: all)
  uint32_t tail_ones;  // SumI multiplier of the last word (0x01 in its template bytes)
  uint32_t tail_mask;  // SumISq mask of the last word (0xff in its template bytes)
  int wtp;           // shared-memory template row stride in words (multiple of 4)
  int ow, oh;
  int rows;          // fast path: output rows per half-warp (the kernel's R)
  int staged;        // fast path: coalesced stores through shared memory
  int tiles_x;       // units across a row of outputs
  int units;         // warp units (fast path: 128 cols x 2R rows)
};

__device__ __forceinline__ uint32_t fshr(uint32_t lo, uint32_t hi, int bytes) {
  return __funnelshift_r(lo, hi, 8 * bytes);
}

// Four bytes of image row `row` starting at byte `off`; bytes at or past w
// read as zero (they only ever feed columns past the last valid offset).
__device__ __forceinline__ uint32_t load_word_bytes(const uint8_t *row, int off,
                                                    int w) {
  uint32_t v = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b)
    if (off + b < w) v |= uint32_t(__ldg(row + off + b)) << (8 * b);
  return v;
}

// Stage the template into shared memory as 32-bit words (row stride wtp,
// zero padded) and reduce SumT, SumTSq over the CTA.
__device__ __forceinline__ void stage_template(const NccArgs &a, uint32_t *tmpl_s,
                                               uint32_t *red, uint32_t &sum_t,
                                               uint32_t &sum_t_sq) {
  if (threadIdx.x < 2) red[threadIdx.x] = 0;
  __syncthreads();
  const bool aligned4 = (reinterpret_cast<uintptr_t>(a.tmpl) & 3) == 0 && a.tail == 0;
  uint32_t s = 0, q = 0;
  const int total = a.ht * a.wtp;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int j = idx / a.wtp, i = idx - j * a.wtp;
    uint32_t v = 0;
    if (i < a.wtw) {
      const int byte = j * a.wt + 4 * i;
      if (aligned4) {
        v = __ldg(reinterpret_cast<const uint32_t *>(a.tmpl + byte));
      } else {
#pragma unroll
        for (int b = 0; b < 4; ++b)
          if (4 * i + b < a.wt) v |= uint32_t(__ldg(a.tmpl + byte + b)) << (8 * b);
      }
    }
    tmpl_s[idx] = v;
    s = __dp4a(v, kOnes, s);
    q = __dp4a(v, v, q);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    q += __shfl_xor_sync(0xffffffffu, q, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&red[0], s);
    atomicAdd(&red[1], q);
  }
  __syncthreads();
  sum_t = red[0];
  sum_t_sq = red[1];
}

// Three unsigned dp4a per window: the section's inner step.
template <int R>
__device__ __forceinline__ void accum_window(uint32_t (&sI)[R][kCols],
                                             uint32_t (&sQ)[R][kCols],
                                             uint32_t (&sT)[R][kCols], int r,
                                             int c, uint32_t win, uint32_t tw) {
  sI[r][c] = __dp4a(win, kOnes, sI[r][c]);
  sQ[r][c] = __dp4a(win, win, sQ[r][c]);
  sT[r][c] = __dp4a(win, tw, sT[r][c]);
}

// The last word of a template row whose width is not a multiple of 4: its
// pad bytes are zero in the template word (SumIT needs nothing more), while
// SumI and SumISq take only the template bytes of the window.
template <int R>
__device__ __forceinline__ void accum_window_tail(uint32_t (&sI)[R][kCols],
                                                  uint32_t (&sQ)[R][kCols],
                                                  uint32_t (&sT)[R][kCols], int r,
                                                  int c, uint32_t win, uint32_t tw,
                                                  uint32_t ones, uint32_t mask) {
  sI[r][c] = __dp4a(win, ones, sI[r][c]);
  sQ[r][c] = __dp4a(win & mask, win, sQ[r][c]);
  sT[r][c] = __dp4a(win, tw, sT[r][c]);
}

// Single-precision value of an integer |v| < 2^55 from two 32-bit
// conversions: v = hi * 2^24 + lo with lo < 2^24 exact in float, hi rounded
// once and the sum once (relative error below 2^-23).  A direct 64-bit
// conversion would issue on the FP64 unit, which this part provides at a few
// lanes per clock.
__device__ __forceinline__ float i64_to_f32(int64_t v) {
  const int32_t hi = int32_t(v >> 24);
  const uint32_t lo = uint32_t(v) & 0xffffffu;
  return fmaf(float(hi), 16777216.f, float(lo));
}

// Write the sums and the coefficient of one lane's R x 8 block.  The
// numerator and the window variance term are exact 64-bit integers; the
// ratio is num * rsqrt(dI) * rsqrt(dT) in single precision (a few ulp of
// |coef| <= 1, far inside the 1e-5 bound).  rs_t = rsqrt(dT) is per template.
template <int R>
__device__ __forceinline__ void epilogue(const NccArgs &a, int x0, int y0,
                                         const uint32_t (&sI)[R][kCols],
                                         const uint32_t (&sQ)[R][kCols],
                                         const uint32_t (&sT)[R][kCols],
                                         uint32_t sum_t, float rs_t) {
  const int64_t n = int64_t(a.wt) * a.ht;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int y = y0 + r;
    if (y >= a.oh) break;
#pragma unroll
    for (int c = 0; c < kCols; ++c) {
      const int x = x0 + c;
      if (x >= a.ow) break;
      const size_t o = size_t(y) * a.ow + x;
      const uint32_t vi = sI[r][c], vq = sQ[r][c];
      if (a.sums) {
        a.sums[o] = vi;
        a.sums[a.plane + o] = vq;
        a.sums[2 * a.plane + o] = sT[r][c];
      }
      if (a.coef) {
        const int64_t si = vi;
        const int64_t num = n * int64_t(sT[r][c]) - si * int64_t(sum_t);
        const int64_t d_i = n * int64_t(vq) - si * si;
        a.coef[o] = d_i > 0 ? i64_to_f32(num) * rsqrtf(i64_to_f32(d_i)) * rs_t : 0.f;
      }
    }
  }
}

// The same outputs for a whole warp of the tiled kernel, written through a
// warp-private staging area so that the global stores are coalesced.  A
// lane owns 8 adjacent columns, so storing its own values makes every store
// instruction touch 16 sectors for 64 bytes; staging one plane at a time
// ([2 halves][R][128] words, half h's row r at (h*R + r)*128) lets each
// store instruction write 32 consecutive outputs of one row instead.  The
// warp's rows are yw .. yw+2R-1 and its columns xt .. xt+127.
template <int R>
__device__ __forceinline__ void epilogue_staged(const NccArgs &a, int xt, int yw, int lane,
                                                const uint32_t (&sI)[R][kCols],
                                                const uint32_t (&sQ)[R][kCols],
                                                const uint32_t (&sT)[R][kCols],
                                                uint32_t sum_t, float rs_t,
                                                uint32_t *stage) {
  const int64_t n = int64_t(a.wt) * a.ht;
  const int half = lane >> 4, hl = lane & 15;
  // value(r, c) of one plane -> staging area -> coalesced rows of dst
  auto put = [&](auto value, uint32_t *dst) {
    __syncwarp();                           // the area's previous reads are done
#pragma unroll
    for (int r = 0; r < R; ++r) {
      uint4 *row = reinterpret_cast<uint4 *>(stage + (half * R + r) * kHalfUnitCols +
                                             hl * kCols);
      row[0] = make_uint4(value(r, 0), value(r, 1), value(r, 2), value(r, 3));
      row[1] = make_uint4(value(r, 4), value(r, 5), value(r, 6), value(r, 7));
    }
    __syncwarp();
#pragma unroll
    for (int rr = 0; rr < 2 * R; ++rr) {
      const int y = yw + rr;
      if (y >= a.oh) break;
      uint32_t *out = dst + size_t(y) * a.ow + xt;
#pragma unroll
      for (int k = 0; k < kHalfUnitCols / 32; ++k) {
        const int col = 32 * k + lane;
        if (xt + col < a.ow) out[col] = stage[rr * kHalfUnitCols + col];
      }
    }
  };
  if (a.sums) {
    put([&](int r, int c) { return sI[r][c]; }, a.sums);
    put([&](int r, int c) { return sQ[r][c]; }, a.sums + a.plane);
    put([&](int r, int c) { return sT[r][c]; }, a.sums + 2 * a.plane);
  }
  if (a.coef) {
    put([&](int r, int c) {
          const int64_t si = sI[r][c];
          const int64_t num = n * int64_t(sT[r][c]) - si * int64_t(sum_t);
          const int64_t d_i = n * int64_t(sQ[r][c]) - si * si;
          return __float_as_uint(
              d_i > 0 ? i64_to_f32(num) * rsqrtf(i64_to_f32(d_i)) * rs_t : 0.f);
        },
        reinterpret_cast<uint32_t *>(a.coef));
  }
}

// rsqrt of the template variance term N*SumTSq - SumT^2, or 0 for a flat
// template (which makes every coefficient 0).
__device__ __forceinline__ float template_rsqrt(const NccArgs &a, uint32_t sum_t,
                                                uint32_t sum_t_sq) {
  const int64_t n = int64_t(a.wt) * a.ht;
  const int64_t d_t = n * int64_t(sum_t_sq) - int64_t(sum_t) * int64_t(sum_t);
  return d_t > 0 ? rsqrtf(float(d_t)) : 0.f;
}

// One image row (tile-relative index rel = k - y0) against template rows
// rel - r for the R output rows r of the unit; `mask` selects the rows r for
// which 0 <= rel - r < ht (all of them when FULL).
// Words of one staged image row a lane holds: the WT + 1 words its 8
// windows reach, read as 8-byte pairs.
template <int WT>
struct RowWords {
  static constexpr int kPairs = (WT + 3) / 2;
  static constexpr int kWords = 2 * kPairs;
};

template <int R, int WT, bool FULL, bool BOX>
__device__ __forceinline__ void row_fixed(const uint32_t (&wv)[RowWords<WT>::kWords],
                                          const uint32_t *tmpl_s, int rel,
                                          unsigned mask, uint32_t (&sI)[R][kCols],
                                          uint32_t (&sQ)[R][kCols],
                                          uint32_t (&sT)[R][kCols], const NccArgs &a) {
  constexpr int WTP = (WT + 3) & ~3;
#pragma unroll
  for (int ib = 0; ib < WT; ib += 4) {
    uint4 tq[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (FULL || ((mask >> r) & 1u))
        tq[r] = *reinterpret_cast<const uint4 *>(tmpl_s + (rel - r) * WTP + ib);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int i = ib + m;
      if (i >= WT) break;
      uint32_t win[kCols];
#pragma unroll
      for (int c = 0; c < kCols; ++c) {
        const int k = i + (c >> 2), s = c & 3;
        win[c] = s == 0 ? wv[k] : fshr(wv[k], wv[k + 1], s);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (!(FULL || ((mask >> r) & 1u))) continue;
        const uint32_t tw = m == 0 ? tq[r].x : m == 1 ? tq[r].y : m == 2 ? tq[r].z : tq[r].w;
        if (BOX) {                      // SumIT only; pad template bytes are zero
#pragma unroll
          for (int c = 0; c < kCols; ++c) sT[r][c] = __dp4a(win[c], tw, sT[r][c]);
        } else if (i == WT - 1 && a.tail) {   // partial last word (warp-uniform)
#pragma unroll
          for (int c = 0; c < kCols; ++c)
            accum_window_tail<R>(sI, sQ, sT, r, c, win[c], tw, a.tail_ones, a.tail_mask);
        } else {
#pragma unroll
          for (int c = 0; c < kCols; ++c) accum_window<R>(sI, sQ, sT, r, c, win[c], tw);
        }
      }
    }
  }
}

// Box-sum form, column step: for each tile column x that a window of the
// tile reaches (x < 128 + wt - 1) and each output row y < TY of the tile,
// v[y][x] = sum_{i<ht} tile[y+i][x] and the same of squares; the first
// window is summed directly, the next TY-1 slide down by one row (exact in
// unsigned 32-bit arithmetic).  Rows of the tile past the image were not
// staged; they only reach outputs past oh, which are never stored.
template <int TY, int RB>
__device__ __forceinline__ void box_columns(const uint8_t *tile, int ht, int nv, int vs,
                                            uint32_t *v_i, uint32_t *v_q, int tid,
                                            int nthreads) {
  for (int x = tid; x < nv; x += nthreads) {
    const uint8_t *col = tile + x;
    uint32_t s = 0, q = 0;
#pragma unroll 4
    for (int i = 0; i < ht; ++i) {
      const uint32_t b = col[i * RB];
      s += b;
      q += b * b;
    }
    const int xs = box_v_col(x);
    v_i[xs] = s;
    v_q[xs] = q;
#pragma unroll
    for (int y = 1; y < TY; ++y) {
      const uint32_t bi = col[(y + ht - 1) * RB], bo = col[(y - 1) * RB];
      s += bi - bo;
      q += bi * bi - bo * bo;
      v_i[y * vs + xs] = s;
      v_q[y * vs + xs] = q;
    }
  }
}

// Box-sum form, row step: SumI[y][c] = sum_{j<wt} v[y][c+j] (and SumISq)
// for the tile's TY x 128 outputs, a thread per run of 8 columns (the first
// sum direct, the next 7 sliding by one column), into s_i / s_q [TY][128]
// (written as 16-byte vectors).
template <int TY>
__device__ __forceinline__ void box_rows(const uint32_t *v_i, const uint32_t *v_q, int wt,
                                         int vs, uint32_t *s_i, uint32_t *s_q, int tid,
                                         int nthreads) {
  constexpr int kRuns = kHalfUnitCols / kCols;
  for (int u = tid; u < TY * kRuns; u += nthreads) {
    const int y = u / kRuns, c0 = (u - y * kRuns) * kCols;
    const uint32_t *ri = v_i + y * vs, *rq = v_q + y * vs;
    uint32_t s = 0, q = 0;
#pragma unroll 4
    for (int j = 0; j < wt; ++j) {
      const int x = c0 + j, xs = box_v_col(x);
      s += ri[xs];
      q += rq[xs];
    }
    uint32_t oi[kCols], oq[kCols];
    oi[0] = s;
    oq[0] = q;
#pragma unroll
    for (int c = 1; c < kCols; ++c) {
      const int xo = c0 + c - 1, xi = xo + wt;
      s += ri[box_v_col(xi)] - ri[box_v_col(xo)];
      q += rq[box_v_col(xi)] - rq[box_v_col(xo)];
      oi[c] = s;
      oq[c] = q;
    }
    uint4 *di = reinterpret_cast<uint4 *>(s_i + y * kHalfUnitCols);
    uint4 *dq = reinterpret_cast<uint4 *>(s_q + y * kHalfUnitCols);
#pragma unroll
    for (int c = 0; c < kCols; c += 4) {
      const int ch = box_s_chunk((c0 + c) >> 2);
      di[ch] = make_uint4(oi[c], oi[c + 1], oi[c + 2], oi[c + 3]);
      dq[ch] = make_uint4(oq[c], oq[c + 1], oq[c + 2], oq[c + 3]);
    }
  }
}

// Fast path: template width WT words known at compile time, any image
// alignment (the staging unit VB follows it).
//
// A CTA owns a tile of 128 output columns x TY = 2*R*kWarps output
// rows.  It first copies the image tile plus halo -- TY+ht-1 rows of
// 128+4*WT+8 bytes (rounded to 16) -- into shared memory with 16-byte (or
// 8-byte) vector loads that are all independent, so the tile costs one
// memory latency instead of one per image row.  Then half-warp h of warp w
// takes output rows w*2R + h*R .. +R-1 (each lane 8 adjacent columns) and
// walks its R+ht-1 tile rows from shared memory; each row is cut into
// windows once and paired with template row k-r for each of its R rows.
// Words of the next tile row are read while the current one is consumed.
template <int WT>
struct TileGeom {
  static constexpr int kRowBytes = (kHalfUnitCols + 4 * WT + 8 + 15) & ~15;
};

// Tile staging unit by image alignment: VB = 16 or 8 when the image pointer
// and width are that aligned (whole vector loads, a chunk lies wholly inside
// or outside the image), VB = 1 otherwise (4-byte chunks assembled from byte
// loads, each byte checked against w).
template <int VB>
struct StageChunk {
  using type = typename std::conditional<VB == 16, uint4,
               typename std::conditional<VB == 8, uint2, uint32_t>::type>::type;
  static constexpr int kBytes = int(sizeof(type));
};

template <int R, int WT, int VB, bool BOX>
__global__ void __launch_bounds__(FixedShape<BOX>::kThreadsPerCta,
                                  !BOX ? CORR_NCC_MINB
                                  : WT <= 16 ? CORR_NCC_BOX_MINB : CORR_NCC_BOX_MINB_WIDE)
    ncc_u8_fixed_kernel(const NccArgs a) {
  constexpr int KS = FixedShape<BOX>::kGroups;
  constexpr int WPC = FixedShape<BOX>::kWarps;
  constexpr int kFixedThreads = FixedShape<BOX>::kThreadsPerCta;
  constexpr int WTP = (WT + 3) & ~3;
  constexpr int RB = TileGeom<WT>::kRowBytes;
  constexpr int TY = 2 * R * WPC;
  extern __shared__ uint4 smem_u4[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(smem_u4);
  constexpr int NS = BOX ? 1 : 3;                     // sums exchanged per column
  constexpr int E = NS * R * kCols;
  const size_t tile_bytes = size_t(TY + a.ht - 1) * RB;
  const size_t part_bytes = size_t(KS - 1) * WPC * E * 32 * 4;
  const size_t s_bytes = size_t(2) * TY * kHalfUnitCols * 4;
  // regions as fixed_tile_layout places them
  uint8_t *tile = BOX ? smem : smem + size_t(a.ht) * WTP * 4;
  uint32_t *part = reinterpret_cast<uint32_t *>(
      BOX ? smem + (tile_bytes > s_bytes ? tile_bytes : s_bytes) : tile + tile_bytes);
  uint32_t *tmpl_s = BOX ? reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(part) +
                                                        part_bytes)
                         : reinterpret_cast<uint32_t *>(smem);
  __shared__ uint32_t red[2];

  const int tx = blockIdx.x % a.tiles_x, ty = blockIdx.x / a.tiles_x;
  const int xt = tx * kHalfUnitCols, yt = ty * TY;
  const int trows = min(TY + a.ht - 1, a.h - yt);   // tile rows inside the image

  // ---- tile + halo -> shared memory (out-of-image bytes become zero) ----
  // The first kStageBatch chunks per thread are loaded into registers and
  // the template is staged while they are in flight, so a tile costs about
  // one memory latency; taller tiles copy the rest afterwards.
  using Chunk = typename StageChunk<VB>::type;
  constexpr int CB = StageChunk<VB>::kBytes;          // bytes per chunk
  constexpr int C = RB / CB;                          // chunks per tile row
  const int nchunks = trows * C;
  auto chunk_load = [&](int i) {
    Chunk v;
    memset(&v, 0, sizeof(v));
    const int r = i / C, c = i - r * C;
    const int x = xt + CB * c;
    const uint8_t *row = a.image + size_t(yt + r) * a.pitch;
    if constexpr (VB == 1) {
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (x + b < a.w) v |= uint32_t(__ldg(row + x + b)) << (8 * b);
    } else {
      if (x < a.w) v = __ldg(reinterpret_cast<const Chunk *>(row + x));   // w, pitch % CB == 0
    }
    return v;
  };
  auto chunk_store = [&](int i, const Chunk &v) {
    const int r = i / C, c = i - r * C;
    *reinterpret_cast<Chunk *>(tile + r * RB + CB * c) = v;
  };
  Chunk first[kStageBatch];
#pragma unroll
  for (int k = 0; k < kStageBatch; ++k) {
    const int i = threadIdx.x + k * kFixedThreads;
    if (i < nchunks) first[k] = chunk_load(i);
  }
  uint32_t sum_t, sum_t_sq;
  stage_template(a, tmpl_s, red, sum_t, sum_t_sq);   // ends with __syncthreads
#pragma unroll
  for (int k = 0; k < kStageBatch; ++k) {
    const int i = threadIdx.x + k * kFixedThreads;
    if (i < nchunks) chunk_store(i, first[k]);
  }
  for (int i = threadIdx.x + kStageBatch * kFixedThreads; i < nchunks; i += kFixedThreads)
    chunk_store(i, chunk_load(i));
  __syncthreads();

  // BOX: column sums over the template, SumI / SumISq over the tile, each
  // once the region is dead
  const int vs = BOX ? box_v_stride(a.wt) : 0;
  uint32_t *v_i = tmpl_s, *v_q = v_i + TY * vs;
  uint32_t *s_i = reinterpret_cast<uint32_t *>(tile), *s_q = s_i + TY * kHalfUnitCols;

  const int warp_id = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int warp = warp_id % WPC;            // row group of the tile
  const int ks = warp_id / WPC;              // template-row range
  const int j_lo = ks * a.ht / KS, j_hi = (ks + 1) * a.ht / KS;
  const int half = lane >> 4, hl = lane & 15;
  const int yr0 = warp * 2 * R + half * R;           // tile-relative first row
  const int x0 = xt + hl * kCols;
  const int y0 = yt + yr0;

  uint32_t sI[R][kCols], sQ[R][kCols], sT[R][kCols];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int c = 0; c < kCols; ++c) sI[r][c] = sQ[r][c] = sT[r][c] = 0;

  // Warp-uniform row count: rows of the lower half past the tile's rows in
  // the image read the last staged row (their outputs are past oh and are
  // never stored).
  const int nrows = max(0, min(R + a.ht - 1, trows - warp * 2 * R));
  const uint8_t *lane_base = tile + hl * kCols;
  constexpr int NW = RowWords<WT>::kWords;
  auto load_row = [&](int rel, uint32_t (&dst)[NW]) {
    const int r = min(yr0 + rel, trows - 1);
    const uint8_t *row = lane_base + r * RB;
#pragma unroll
    for (int p = 0; p < RowWords<WT>::kPairs; ++p) {
      const uint2 v = *reinterpret_cast<const uint2 *>(row + 8 * p);
      dst[2 * p] = v.x;
      dst[2 * p + 1] = v.y;
    }
  };
  // Tile row yr0 + rel meets template row rel - r for output row r; this
  // warp group takes template rows [j_lo, j_hi).  Rows [body_lo, body_hi)
  // meet all R output rows and run unmasked, two at a time with the next
  // row's words read ahead (load_row clamps its row, so reading one row
  // past the end is harmless); the first and last R-1 rows are masked.
  const int rel_end = min(nrows, j_hi + R - 1);
  const int body_lo = min(j_lo + R - 1, rel_end);
  const int body_hi = max(body_lo, min(j_hi, rel_end));
  auto masked_row = [&](int rel) {
    uint32_t wv[NW];
    load_row(rel, wv);
    unsigned mask = 0;
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (rel - r >= j_lo && rel - r < j_hi) mask |= 1u << r;
    row_fixed<R, WT, false, BOX>(wv, tmpl_s, rel, mask, sI, sQ, sT, a);
  };
  for (int rel = j_lo; rel < body_lo; ++rel) masked_row(rel);
  {
    uint32_t wa[NW], wb[NW];
    int rel = body_lo;
    load_row(rel, wa);
    for (; rel + 1 < body_hi; rel += 2) {
      load_row(rel + 1, wb);
      row_fixed<R, WT, true, BOX>(wa, tmpl_s, rel, 0u, sI, sQ, sT, a);
      load_row(rel + 2, wa);
      row_fixed<R, WT, true, BOX>(wb, tmpl_s, rel + 1, 0u, sI, sQ, sT, a);
    }
    if (rel < body_hi) row_fixed<R, WT, true, BOX>(wa, tmpl_s, rel, 0u, sI, sQ, sT, a);
  }
  for (int rel = body_hi; rel < rel_end; ++rel) masked_row(rel);
  if (KS > 1 || BOX) {
    // groups 1.. hand their partial sums to group 0 through shared memory;
    // BOX: all threads form the column sums from the tile (into the
    // template's place), then the box sums (into the tile's)
    __syncthreads();                        // template and tile reads done
    if (ks > 0) {
      uint32_t *dst = part + ((ks - 1) * WPC + warp) * E * 32 + lane;
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const int e = (r * kCols + c) * NS;
          if (BOX) {
            dst[e * 32] = sT[r][c];
          } else {
            dst[(e + 0) * 32] = sI[r][c];
            dst[(e + 1) * 32] = sQ[r][c];
            dst[(e + 2) * 32] = sT[r][c];
          }
        }
    }
    if constexpr (BOX) {
      box_columns<TY, RB>(tile, a.ht, kHalfUnitCols + a.wt - 1, vs, v_i, v_q, threadIdx.x,
                          kFixedThreads);
      __syncthreads();                      // column sums done, tile dead
      box_rows<TY>(v_i, v_q, a.wt, vs, s_i, s_q, threadIdx.x, kFixedThreads);
    }
    __syncthreads();
    if (ks > 0) return;
#pragma unroll 1
    for (int g = 1; g < KS; ++g) {
      const uint32_t *src = part + ((g - 1) * WPC + warp) * E * 32 + lane;
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const int e = (r * kCols + c) * NS;
          if (BOX) {
            sT[r][c] += src[e * 32];
          } else {
            sI[r][c] += src[(e + 0) * 32];
            sQ[r][c] += src[(e + 1) * 32];
            sT[r][c] += src[(e + 2) * 32];
          }
        }
    }
    if constexpr (BOX) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < kCols; c += 4) {
          const int o = (yr0 + r) * kHalfUnitCols + 4 * box_s_chunk((hl * kCols + c) >> 2);
          const uint4 vi = *reinterpret_cast<const uint4 *>(s_i + o);
          const uint4 vq = *reinterpret_cast<const uint4 *>(s_q + o);
          sI[r][c] = vi.x; sI[r][c + 1] = vi.y; sI[r][c + 2] = vi.z; sI[r][c + 3] = vi.w;
          sQ[r][c] = vq.x; sQ[r][c + 1] = vq.y; sQ[r][c + 2] = vq.z; sQ[r][c + 3] = vq.w;
        }
    }
  }
  if constexpr (KS > 1 && CORR_NCC_STAGED_STORES) {
    if (a.staged) {                         // warp-uniform
      // this warp's partial-sum area (read above) holds 2R x 128 words
      static_assert(NS * R * kCols * 32 >= 2 * R * kHalfUnitCols, "staging area too small");
      epilogue_staged<R>(a, xt, yt + warp * 2 * R, lane, sI, sQ, sT, sum_t,
                         template_rsqrt(a, sum_t, sum_t_sq), part + warp * E * 32);
      return;
    }
  }
  epilogue<R>(a, x0, y0, sI, sQ, sT, sum_t, template_rsqrt(a, sum_t, sum_t_sq));
}

// General path: any template width (multiple of 4) and any image alignment.
// Same decomposition; words are assembled from bytes and the template row is
// walked one word at a time.
template <int R>
__global__ void __launch_bounds__(kThreads)
    ncc_u8_general_kernel(const NccArgs a) {
  extern __shared__ uint4 smem_u4[];
  uint32_t *tmpl_s = reinterpret_cast<uint32_t *>(smem_u4);
  __shared__ uint32_t red[2];
  uint32_t sum_t, sum_t_sq;
  stage_template(a, tmpl_s, red, sum_t, sum_t_sq);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x * kWarpsPerCta + warp;
  if (unit >= a.units) return;
  const int tx = unit % a.tiles_x, rb = unit / a.tiles_x;
  const int x0 = tx * kUnitCols + lane * kCols;
  const int y0 = rb * R;

  uint32_t sI[R][kCols], sQ[R][kCols], sT[R][kCols];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int c = 0; c < kCols; ++c) sI[r][c] = sQ[r][c] = sT[r][c] = 0;

  const int nrows = min(R + a.ht - 1, a.h - y0);
  for (int rel = 0; rel < nrows; ++rel) {
    const uint8_t *row = a.image + size_t(y0 + rel) * a.pitch;
    unsigned mask = 0;
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (rel - r >= 0 && rel - r < a.ht) mask |= 1u << r;
    uint32_t w0 = load_word_bytes(row, x0, a.w);
    uint32_t w1 = load_word_bytes(row, x0 + 4, a.w);
    for (int i = 0; i < a.wtw; ++i) {
      const uint32_t w2 = load_word_bytes(row, x0 + 4 * (i + 2), a.w);
      uint32_t win[kCols];
      win[0] = w0;
      win[1] = fshr(w0, w1, 1);
      win[2] = fshr(w0, w1, 2);
      win[3] = fshr(w0, w1, 3);
      win[4] = w1;
      win[5] = fshr(w1, w2, 1);
      win[6] = fshr(w1, w2, 2);
      win[7] = fshr(w1, w2, 3);
      const bool tail = a.tail && i == a.wtw - 1;   // partial last word (warp-uniform)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (!((mask >> r) & 1u)) continue;
        const uint32_t tw = tmpl_s[(rel - r) * a.wtp + i];
        if (tail) {
#pragma unroll
          for (int c = 0; c < kCols; ++c)
            accum_window_tail<R>(sI, sQ, sT, r, c, win[c], tw, a.tail_ones, a.tail_mask);
        } else {
#pragma unroll
          for (int c = 0; c < kCols; ++c) accum_window<R>(sI, sQ, sT, r, c, win[c], tw);
        }
      }
      w0 = w1;
      w1 = w2;
    }
  }
  epilogue<R>(a, x0, y0, sI, sQ, sT, sum_t, template_rsqrt(a, sum_t, sum_t_sq));
}

template <typename Kernel>
cudaError_t set_smem(Kernel kernel, size_t smem) {
  if (smem > 48 * 1024) return allow_dynamic_smem(reinterpret_cast<const void *>(kernel));
  return cudaSuccess;
}

template <typename Kernel>
cudaError_t launch(Kernel kernel, const NccArgs &a, size_t smem,
                   cudaStream_t stream) {
  cudaError_t e = set_smem(kernel, smem);
  if (e != cudaSuccess) return e;
  const int blocks = (a.units + kWarpsPerCta - 1) / kWarpsPerCta;
  kernel<<<blocks, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

// One CTA of `threads` per tile.
template <typename Kernel>
cudaError_t launch_tiles(Kernel kernel, const NccArgs &a, size_t smem, int threads,
                         cudaStream_t stream) {
  cudaError_t e = set_smem(kernel, smem);
  if (e != cudaSuccess) return e;
  kernel<<<a.units, threads, smem, stream>>>(a);
  return cudaGetLastError();
}

// Fast-path launchers for template widths of 1 .. kMaxFixedWords words:
// words 1 .. kNarrowWords are instantiated in ncc_u8.cu, the rest in
// ncc_u8_wide.cu (two translation units compile in parallel).
constexpr int kMaxFixedWords = 32;
constexpr int kNarrowWords = 16;
using FixedLauncher = cudaError_t (*)(const NccArgs &, size_t, int, cudaStream_t);

template <int R, int WT, bool BOX>
cudaError_t launch_fixed(const NccArgs &a, size_t smem, int vb, cudaStream_t stream) {
  constexpr int T = FixedShape<BOX>::kThreadsPerCta;
  return vb == 16 ? launch_tiles(ncc_u8_fixed_kernel<R, WT, 16, BOX>, a, smem, T, stream)
       : vb == 8  ? launch_tiles(ncc_u8_fixed_kernel<R, WT, 8, BOX>, a, smem, T, stream)
                  : launch_tiles(ncc_u8_fixed_kernel<R, WT, 1, BOX>, a, smem, T, stream);
}

// Launchers of template words FIRST + 0 .. FIRST + sizeof...(Ks) - 1.
template <int R, bool BOX, int FIRST, int... Ks>
constexpr std::array<FixedLauncher, sizeof...(Ks)> fixed_launchers(
    std::integer_sequence<int, Ks...>) {
  return {{launch_fixed<R, FIRST + Ks, BOX>...}};
}

}  // namespace ncc

// Fast path for templates of kNarrowWords + 1 .. kMaxFixedWords words
// (ncc_u8_wide.cu), and its SumIT-only form (ncc_u8_box_wide.cu).
cudaError_t ncc_u8_launch_fixed_wide(const ncc::NccArgs &a, size_t smem, int vb,
                                     cudaStream_t stream);
cudaError_t ncc_u8_launch_fixed_box_wide(const ncc::NccArgs &a, size_t smem, int vb,
                                         cudaStream_t stream);

// Box-sum form of the fast path (ncc_u8_box.cu): SumI / SumISq as box
// filters of the staged tile, SumIT alone by dp4a.
cudaError_t ncc_u8_launch_box(const ncc::NccArgs &a, size_t smem, int vb,
                              cudaStream_t stream);

}  // namespace corr
