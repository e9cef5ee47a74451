// ncc_u8_box.cu -- the box-sum variant of the 8-bit NCC: SumI and SumISq
// from separable sliding sums, so the tiled dp4a kernel accumulates SumIT
// alone (one unsigned dp4a per 4 pixels instead of three).
//
// SumI and SumISq do not depend on the template, only on its size: they are
// box filters of I and I^2.  A box filter separates into a horizontal pass
// (each image row, windows of wt pixels) and a vertical pass (each output
// column, windows of ht horizontal sums); each pass slides its window by
// adding the entering and subtracting the leaving element.  All arithmetic
// is unsigned 32-bit: every partial and final sum is a sum of at most
// wt*ht <= 66052 terms of at most 255^2, below 2^32, so the differences of
// the slides are exact and the results equal the direct sums bit for bit.
// This is not the section's method (The CUDA Handbook, ch. 15, section 15.5
// forms all three sums with dp4a); it is a reformulation of the same sums
// that moves two thirds of the dp4a work into two O(wt + ht) passes.
#include "ncc_u8_kernels.cuh"

namespace corr {
namespace ncc {
namespace {

constexpr int kBoxThreads = 128;
constexpr int kBoxSeg = 512;       // horizontal pass: output columns per warp
constexpr int kBoxLaneBytes = kBoxSeg / 32;
constexpr int kBoxStrip = 32;      // vertical pass: output rows per thread
constexpr int kBoxBatch = 16;      // vertical pass: rows whose loads are in flight together

// Horizontal pass: for image row r and output columns x < ow,
// hi[r][x] = sum_{j<wt} I[r][x+j] and hq[r][x] = sum_{j<wt} I[r][x+j]^2,
// as differences of running sums along the row: with P(k) the sum of the
// row's pixels xs .. xs+k-1, hi[r][x] = P(x-xs+wt) - P(x-xs).  A warp owns
// kBoxSeg output columns from xs: lane l sums 16 pixels from xs+16l (and 4
// of the wt pixels past the segment from xs+kBoxSeg+4l), a warp scan turns
// the lane totals into offsets, the running sums go to shared memory, and
// the outputs are read back as differences and stored coalesced.  Pixels
// at or past w read as zero; they only reach P beyond the last valid x.
// The fast path keeps wt <= 128, so 4 pixels per lane cover the overhang.
// VEC: rows 16-byte aligned (image pointer and w), so a lane's 16 pixels
// are one vector load and its 4 overhang pixels one word.
// Running sums are stored at index k + k/32 (one pad word per 32), so the
// lanes' stride-16 writes fall in distinct banks.
__device__ __forceinline__ int box_pidx(int k) { return k + (k >> 5); }

template <bool VEC>
__global__ void __launch_bounds__(kBoxThreads)
    ncc_u8_box_rows_kernel(const uint8_t *image, int w, int wt, int ow, int segs,
                           int items, uint32_t *hi, uint32_t *hq) {
  constexpr int kP = kBoxSeg + 128 + 1 + (kBoxSeg + 128) / 32 + 1;
  __shared__ uint32_t ps_i[kBoxThreads / 32][kP], ps_q[kBoxThreads / 32][kP];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * (kBoxThreads / 32) + warp;
  if (item >= items) return;                  // warp-uniform
  const int r = item / segs, xs = (item - r * segs) * kBoxSeg;
  const uint8_t *row = image + size_t(r) * w;
  uint32_t *pi = ps_i[warp], *pq = ps_q[warp];

  // 16 segment pixels and 4 overhang pixels per lane, all loads independent
  uint32_t px[kBoxLaneBytes], ov[4];
  const int xa = xs + kBoxLaneBytes * lane, xb = xs + kBoxSeg + 4 * lane;
  if constexpr (VEC) {
    uint4 v = make_uint4(0, 0, 0, 0);
    uint32_t o = 0;
    if (xa < w) v = __ldg(reinterpret_cast<const uint4 *>(row + xa));
    if (xb < w) o = __ldg(reinterpret_cast<const uint32_t *>(row + xb));
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < kBoxLaneBytes; ++k) px[k] = (words[k >> 2] >> (8 * (k & 3))) & 0xffu;
#pragma unroll
    for (int k = 0; k < 4; ++k) ov[k] = (o >> (8 * k)) & 0xffu;
  } else {
#pragma unroll
    for (int k = 0; k < kBoxLaneBytes; ++k) px[k] = xa + k < w ? __ldg(row + xa + k) : 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) ov[k] = xb + k < w ? __ldg(row + xb + k) : 0u;
  }
  uint32_t ts = 0, tq = 0, os = 0, oq = 0;
#pragma unroll
  for (int k = 0; k < kBoxLaneBytes; ++k) { ts += px[k]; tq += px[k] * px[k]; }
#pragma unroll
  for (int k = 0; k < 4; ++k) { os += ov[k]; oq += ov[k] * ov[k]; }
  // inclusive warp scans of the lane totals (segment, then overhang)
  uint32_t es = ts, eq = tq, fs = os, fq = oq;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t a = __shfl_up_sync(0xffffffffu, es, d), b = __shfl_up_sync(0xffffffffu, eq, d);
    const uint32_t c = __shfl_up_sync(0xffffffffu, fs, d), e = __shfl_up_sync(0xffffffffu, fq, d);
    if (lane >= d) { es += a; eq += b; fs += c; fq += e; }
  }
  const uint32_t seg_s = __shfl_sync(0xffffffffu, es, 31), seg_q = __shfl_sync(0xffffffffu, eq, 31);
  es -= ts; eq -= tq;                         // exclusive
  fs += seg_s - os; fq += seg_q - oq;         // exclusive, after the segment
  if (lane == 0) { pi[0] = 0; pq[0] = 0; }
#pragma unroll
  for (int k = 0; k < kBoxLaneBytes; ++k) {
    es += px[k];
    eq += px[k] * px[k];
    const int j = box_pidx(kBoxLaneBytes * lane + k + 1);
    pi[j] = es;
    pq[j] = eq;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    fs += ov[k];
    fq += ov[k] * ov[k];
    const int j = box_pidx(kBoxSeg + 4 * lane + k + 1);
    pi[j] = fs;
    pq[j] = fq;
  }
  __syncwarp();
  uint32_t *oi = hi + size_t(r) * ow, *oq2 = hq + size_t(r) * ow;
#pragma unroll 4
  for (int k = lane; k < kBoxSeg; k += 32) {
    const int x = xs + k;
    if (x >= ow) break;
    const int j1 = box_pidx(k + wt), j0 = box_pidx(k);
    oi[x] = pi[j1] - pi[j0];                  // exact modulo 2^32
    oq2[x] = pq[j1] - pq[j0];
  }
}

// Vertical pass: for output column x and output rows y of strip blockIdx.y,
// si[y][x] = sum_{i<ht} hi[y+i][x] (and sq from hq): the first window is
// summed directly, the next ones slide by one row.  Threads of a warp take
// adjacent columns (coalesced), and the loads of kBoxBatch rows are issued
// together so that a strip costs a few memory latencies, not one per row.
__global__ void __launch_bounds__(kBoxThreads)
    ncc_u8_box_cols_kernel(const uint32_t *hi, const uint32_t *hq, int ow, int oh,
                           int ht, uint32_t *si, uint32_t *sq) {
  const int x = blockIdx.x * kBoxThreads + threadIdx.x;
  if (x >= ow) return;
  const int y0 = blockIdx.y * kBoxStrip;
  const int y1 = min(y0 + kBoxStrip, oh);
  const uint32_t *pi = hi + x, *pq = hq + x;
  uint32_t s = 0, q = 0;
  int j = 0;
  for (; j + kBoxBatch <= ht; j += kBoxBatch) {
    uint32_t a[kBoxBatch], b[kBoxBatch];
#pragma unroll
    for (int k = 0; k < kBoxBatch; ++k) {
      const size_t o = size_t(y0 + j + k) * ow;
      a[k] = __ldg(pi + o);
      b[k] = __ldg(pq + o);
    }
#pragma unroll
    for (int k = 0; k < kBoxBatch; ++k) { s += a[k]; q += b[k]; }
  }
  for (; j < ht; ++j) {
    const size_t o = size_t(y0 + j) * ow;
    s += __ldg(pi + o);
    q += __ldg(pq + o);
  }
  for (int y = y0; y < y1; y += kBoxBatch) {
    // rows y+k+ht enter and rows y+k leave for k with y+k+1 < y1 (then
    // y+k+ht <= h-1)
    uint32_t ai[kBoxBatch], ao[kBoxBatch], bi[kBoxBatch], bo[kBoxBatch];
#pragma unroll
    for (int k = 0; k < kBoxBatch; ++k) {
      if (y + k + 1 < y1) {
        const size_t oin = size_t(y + k + ht) * ow, oout = size_t(y + k) * ow;
        ai[k] = __ldg(pi + oin);
        ao[k] = __ldg(pi + oout);
        bi[k] = __ldg(pq + oin);
        bo[k] = __ldg(pq + oout);
      } else {
        ai[k] = ao[k] = bi[k] = bo[k] = 0;
      }
    }
#pragma unroll
    for (int k = 0; k < kBoxBatch; ++k) {
      if (y + k >= y1) break;
      const size_t o = size_t(y + k) * ow + x;
      si[o] = s;
      sq[o] = q;
      s += ai[k] - ao[k];                     // exact modulo 2^32
      q += bi[k] - bo[k];
    }
  }
}

}  // namespace
}  // namespace ncc

cudaError_t ncc_u8_launch_box(ncc::NccArgs a, size_t smem, int vb, cudaStream_t stream) {
  using namespace ncc;
  constexpr int R = kBoxRows;
  if (a.wtw < 1 || a.wtw > kMaxFixedWords) return cudaErrorInvalidValue;
  const size_t hplane = size_t(a.h) * a.ow;
  const size_t bytes = (2 * hplane + (a.sums ? 0 : 2 * a.plane)) * sizeof(uint32_t);
  void *scratch = nullptr;
  cudaError_t e = scratch_alloc(&scratch, bytes, stream);
  if (e != cudaSuccess) return e;
  uint32_t *hi = static_cast<uint32_t *>(scratch), *hq = hi + hplane;
  uint32_t *si = a.sums ? a.sums : hq + hplane;
  uint32_t *sq = si + a.plane;
  {
    constexpr int kWarps = kBoxThreads / 32;
    const int segs = (a.ow + kBoxSeg - 1) / kBoxSeg;
    const long long items = (long long)segs * a.h;
    const long long blocks = (items + kWarps - 1) / kWarps;
    if (blocks > 0x7fffffffLL) {
      e = cudaErrorInvalidConfiguration;
    } else {
      const bool vec = (reinterpret_cast<uintptr_t>(a.image) & 15) == 0 && (a.w & 15) == 0;
      auto kern = vec ? ncc_u8_box_rows_kernel<true> : ncc_u8_box_rows_kernel<false>;
      kern<<<unsigned(blocks), kBoxThreads, 0, stream>>>(a.image, a.w, a.wt, a.ow, segs,
                                                         int(items), hi, hq);
      e = cudaGetLastError();
    }
  }
  if (e == cudaSuccess) {
    const dim3 grid((a.ow + kBoxThreads - 1) / kBoxThreads,
                    (a.oh + kBoxStrip - 1) / kBoxStrip);
    ncc_u8_box_cols_kernel<<<grid, kBoxThreads, 0, stream>>>(hi, hq, a.ow, a.oh, a.ht, si, sq);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    a.box_i = si;
    a.box_q = sq;
    if (a.wtw > kNarrowWords) {
      e = ncc_u8_launch_fixed_box_wide(a, smem, vb, stream);
    } else {
      static constexpr auto table =
          fixed_launchers<R, true, 1>(std::make_integer_sequence<int, kNarrowWords>{});
      e = table[a.wtw - 1](a, smem, vb, stream);
    }
  }
  const cudaError_t f = cudaFreeAsync(scratch, stream);
  return e != cudaSuccess ? e : f;
}

}  // namespace corr
