// xcorr_warp.cu -- float32 full 2D cross-correlation, one warp per overlap.
//
// The artifact README ("Efficient GPU-accelerated Parallel
// Cross-correlation", kernel overview: warp-per-shift) lists a kernel in
// which a whole warp computes one overlap (one relative shift of a left and
// a right matrix): its lanes share the overlap's products and a reduction
// inside the warp forms the output.  It suits shapes whose overlaps are few
// and long (very wide, very short matrices: one-dimensional signals), where
// the tiled kernels have too few overlap rows to give every lane its own.
//
// Here a warp walks its overlap row by row; the lanes take consecutive
// columns (coalesced loads of both rows), wrapping onto the next rows when
// the overlap is narrower than the warp, and keep two independent partial
// sums.  The lanes' sums are added by a fixed butterfly of shuffles, so the
// result does not depend on scheduling.  Warps take overlaps in order of
// decreasing size within each pair (the centre first), so the longest ones
// start early.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"

namespace corr {
namespace warp {
namespace {

constexpr int kWarps = 8;   // warps per CTA

// k-th of n positions in order of distance from the middle (the middle,
// then alternately right and left of it).
__device__ __forceinline__ int centered(int k, int n) {
  const int m = (n - 1) >> 1;
  if (k == 0) return m;
  return (k & 1) ? m + ((k + 1) >> 1) : m - (k >> 1);
}

__global__ void __launch_bounds__(32 * kWarps) xcorr_warp_kernel(
    const float *__restrict__ left, const float *__restrict__ right, float *__restrict__ out,
    int nr, int H, int W, long long units) {
  const int lane = threadIdx.x & 31;
  const int ndy = 2 * H - 1, ndx = 2 * W - 1;
  const long long per_pair = (long long)ndy * ndx;
  const long long nwarps = (long long)gridDim.x * kWarps;
  for (long long u = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); u < units;
       u += nwarps) {
    const long long pair = u / per_pair;
    const int k = int(u - pair * per_pair);
    // k-th overlap of the pair, centre (largest) first
    const int oy = centered(k % ndy, ndy), ox = centered(k / ndy, ndx);
    const int dy = oy - (H - 1), dx = ox - (W - 1);
    const int l = int(pair / nr), r = int(pair - (long long)l * nr);
    const int ylo = dy > 0 ? dy : 0, yhi = dy < 0 ? H + dy : H;
    const int xlo = dx > 0 ? dx : 0, xhi = dx < 0 ? W + dx : W;
    const int w = xhi - xlo;
    const float *lrow = left + ((size_t)l * H + ylo) * W + xlo;
    const float *rrow = right + ((size_t)r * H + (ylo - dy)) * W + (xlo - dx);
    // lane's first element (row, col) of the flattened overlap, and its step
    const int srow = 32 / w, scol = 32 % w;
    int row = lane / w, col = lane % w;
    const int rows = yhi - ylo;
    float acc0 = 0.f, acc1 = 0.f;
    while (row < rows) {
      const size_t o = (size_t)row * W + col;
      acc0 = fmaf(__ldg(lrow + o), __ldg(rrow + o), acc0);
      row += srow;
      col += scol;
      if (col >= w) {
        col -= w;
        ++row;
      }
      if (row >= rows) break;
      const size_t o2 = (size_t)row * W + col;
      acc1 = fmaf(__ldg(lrow + o2), __ldg(rrow + o2), acc1);
      row += srow;
      col += scol;
      if (col >= w) {
        col -= w;
        ++row;
      }
    }
    float acc = acc0 + acc1;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) out[pair * per_pair + (size_t)oy * ndx + ox] = acc;
  }
}

}  // namespace

cudaError_t launch(const float *left, int nl, const float *right, int nr, int H, int W,
                   float *out, cudaStream_t stream) {
  const long long units = (long long)nl * nr * (2LL * H - 1) * (2LL * W - 1);
  // enough warps for several per SM scheduler, no more than the work
  const long long want = (units + kWarps - 1) / kWarps;
  const long long cap = 64LL * device_sm_count();
  const long long blocks = want < cap ? want : cap;
  xcorr_warp_kernel<<<unsigned(blocks), 32 * kWarps, 0, stream>>>(left, right, out, nr, H, W,
                                                                    units);
  return cudaGetLastError();
}

}  // namespace warp
}  // namespace corr
