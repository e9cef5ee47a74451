// xcorr_f32.cu -- float32 full 2D cross-correlation on sm_103a.
//
// Method ("Efficient GPU-accelerated Parallel Cross-correlation" artifact
// README, kernel overview): every output is one overlap (relative shift) of
// a left and a right matrix; a thread keeps a register buffer of one matrix
// row that slides along x while the other matrix's values stream past
// (grouped overlaps: one buffer feeds several neighbouring shifts), and
// batches of pairs share the same code path (one-to-one, one-to-many,
// n-to-m).
//
//   out[pair][dy+H-1][dx+W-1] = sum_{y,x} L[y][x] * R[y-dy][x-dx]
//
// Decomposition used here:
//   * a warp owns one output unit: a group of G pairs x one shift row dy x
//     P neighbouring shifts dx0 .. dx0+P-1;
//   * the 32 lanes are G pair slots x (32/G) row phases: lane (g, ph) sums the
//     overlap rows y = ylo+ph, ylo+ph+32/G, ... for pair g, so every lane of
//     the warp runs the same x loop (same shifts -> same x range) and the
//     y rows split the reduction;
//   * per row, a lane holds R[y-dy][x-dx0-p] for p < P in a register ring
//     that advances one element per x step, so each pair of loads feeds P
//     multiply-adds; the ring is indexed with compile-time positions by
//     unrolling the x loop by P;
//   * a butterfly of shuffles adds the row phases; each lane then stores
//     some of the group's P outputs.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"

namespace corr {
namespace {

constexpr int kP = 8;              // neighbouring shifts per lane
constexpr int kWarpsPerCta = 4;
constexpr int kThreads = 32 * kWarpsPerCta;

struct XcArgs {
  const float *left;
  const float *right;
  float *out;
  int nl, nr, H, W;
  int pairs;
  int G;          // pair slots per warp (power of two, 1..32)
  int log_ph;     // log2(32 / G)
  int groups_x;   // dx groups per output row: ceil((2W-1) / kP)
  int pair_blocks;
  long long units;
};

template <int P>
__global__ void __launch_bounds__(kThreads) xcorr_rows_kernel(const XcArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long unit = (long long)blockIdx.x * kWarpsPerCta + warp;
  if (unit >= a.units) return;
  const int oh = 2 * a.H - 1, ow = 2 * a.W - 1;
  // unit -> (pair block, output row, dx group)
  const int gx = int(unit % a.groups_x);
  const long long rest = unit / a.groups_x;
  const int oy = int(rest % oh);
  const int pb = int(rest / oh);
  const int dy = oy - (a.H - 1);
  const int dx0 = gx * P - (a.W - 1);

  const int ph_count = 1 << a.log_ph;
  const int g = lane >> a.log_ph, ph = lane & (ph_count - 1);
  const int pair = pb * a.G + g;
  const bool pair_ok = pair < a.pairs;
  const int li = pair_ok ? pair / a.nr : 0, ri = pair_ok ? pair % a.nr : 0;
  const size_t mat = size_t(a.H) * a.W;
  const float *L = a.left + li * mat;
  const float *R = a.right + ri * mat;

  const int ylo = max(0, dy), yhi = min(a.H, a.H + dy);
  const int xlo = max(0, dx0), xhi = min(a.W, a.W + dx0 + P - 1);
  const int W = a.W;

  float acc[P];
#pragma unroll
  for (int p = 0; p < P; ++p) acc[p] = 0.f;

  if (pair_ok) {
    for (int y = ylo + ph; y < yhi; y += ph_count) {
      const float *Lrow = L + size_t(y) * W;
      const float *Rrow = R + size_t(y - dy) * W;
      // ring position of the element for shift p at x step s: (s - p) mod P
      float buf[P];
      buf[0] = 0.f;
#pragma unroll
      for (int p = 1; p < P; ++p) {
        const int v = xlo - dx0 - p;
        buf[P - p] = (v >= 0 && v < W) ? __ldg(Rrow + v) : 0.f;
      }
      int x = xlo;
      for (; x + P <= xhi; x += P) {
#pragma unroll
        for (int s = 0; s < P; ++s) {
          const int v = x + s - dx0;
          buf[s] = v < W ? __ldg(Rrow + v) : 0.f;
          const float l = __ldg(Lrow + x + s);
#pragma unroll
          for (int p = 0; p < P; ++p) acc[p] = fmaf(l, buf[(s - p + P) % P], acc[p]);
        }
      }
#pragma unroll
      for (int s = 0; s < P; ++s) {
        if (x + s < xhi) {
          const int v = x + s - dx0;
          buf[s] = v < W ? __ldg(Rrow + v) : 0.f;
          const float l = __ldg(Lrow + x + s);
#pragma unroll
          for (int p = 0; p < P; ++p) acc[p] = fmaf(l, buf[(s - p + P) % P], acc[p]);
        }
      }
    }
  }
  // add the row phases of each pair slot (lanes differ in their low bits)
  for (int o = 1; o < ph_count; o <<= 1) {
#pragma unroll
    for (int p = 0; p < P; ++p) acc[p] += __shfl_xor_sync(0xffffffffu, acc[p], o);
  }
  if (!pair_ok) return;
  float *orow = a.out + size_t(pair) * oh * ow + size_t(oy) * ow;
  // every lane of the slot now holds the totals; lane ph stores p = ph mod 32/G
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const int dx = dx0 + p;
    if ((p & (ph_count - 1)) == ph && dx < a.W) orow[dx + a.W - 1] = acc[p];
  }
}

int ilog2(int v) {
  int r = 0;
  while ((1 << (r + 1)) <= v) ++r;
  return r;
}

}  // namespace

cudaError_t xcorr_f32_launch(const float *left, int nl, const float *right,
                             int nr, int H, int W, float *out,
                             cudaStream_t stream) {
  XcArgs a;
  a.left = left;
  a.right = right;
  a.out = out;
  a.nl = nl;
  a.nr = nr;
  a.H = H;
  a.W = W;
  a.pairs = nl * nr;
  // enough pair slots that each lane sums about four rows of a full overlap
  int G = 1;
  while (G < 32 && (32 / G) * 4 > H) G <<= 1;
  while (G > 1 && G / 2 >= a.pairs) G >>= 1;
  a.G = G;
  a.log_ph = ilog2(32 / G);
  a.groups_x = (2 * W - 1 + kP - 1) / kP;
  a.pair_blocks = (a.pairs + G - 1) / G;
  a.units = (long long)a.pair_blocks * (2 * H - 1) * a.groups_x;
  const long long blocks = (a.units + kWarpsPerCta - 1) / kWarpsPerCta;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  xcorr_rows_kernel<kP><<<unsigned(blocks), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace corr
