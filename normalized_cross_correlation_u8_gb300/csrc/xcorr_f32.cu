// xcorr_f32.cu -- float32 full 2D cross-correlation on sm_103a.
//
// Method ("Efficient GPU-accelerated Parallel Cross-correlation" artifact
// README, kernel overview): every output is one overlap (relative shift) of
// a left and a right matrix,
//
//   out[pair][dy+H-1][dx+W-1] = sum_{y,x} L[y][x] * R[y-dy][x-dx],
//
// and the fast kernels keep a register buffer of one matrix that slides
// along x while the other matrix streams past (warp-shuffle family), compute
// several neighbouring overlaps per thread from shared buffers (grouped
// overlap), and reuse one left matrix against several right matrices
// (multi-matrix-right).  The same ideas, laid out for sm_103a:
//
//   * A CTA owns a block of outputs: Q output rows (mode "rows": Q shifts dy
//     of one pair; mode "rights": Q right matrices at one dy) x NW warps x P
//     neighbouring shifts dx, for G pair slots.  Every warp takes P shifts.
//   * The rows y of the overlap are the reduction: lane (g, ph) of a warp
//     sums rows y = ph, ph + 32/G, ... of pair slot g, so all lanes run the
//     same x loop (same shifts, same x range) and no lane idles in x.
//   * The rows a chunk needs are staged from global memory into shared
//     memory with zero padding, so every shift reads in-bounds values with
//     no branches: out-of-range products become 0 * x.
//   * Per lane and per overlap row: a float4 of L feeds 4 x steps; for each
//     q a float4 of R enters a 12-entry register ring that holds the
//     R[x-dx0-p] values of the P = 8 shifts, indexed at compile-time
//     positions by unrolling three 4-step blocks; 5 shared loads feed
//     4 * P * Q = 128 FMAs.
//   * A shuffle butterfly adds the row phases; lanes then store.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"

namespace corr {
namespace {

constexpr int kP = 8;                // neighbouring shifts dx per lane
constexpr int kQ = 4;                // output rows per lane
constexpr int kRing = kP + 4;        // ring of R values (multiple of 4)
constexpr int kPadL = kP;            // zero columns left of a staged row
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

struct RowArgs {
  const float *left;
  const float *right;
  float *out;
  int nl, nr, H, W;
  int G, log_ph, ph;      // pair slots, log2(rows per chunk), rows per chunk
  int S;                  // shared row stride (floats), S % 8 == 4
  int dxbase;             // first shift of group 0 (multiple of 4, <= 1-W)
  int ngroups;            // dx groups of kP
  int nsuper;             // ceil(ngroups / kWarps)
  int ndy;                // row blocks: ceil((2H-1)/kQ) (rows) or 2H-1 (rights)
  int nslots_blocks;      // pair-slot blocks
  int rights_mode;        // 0: Q shifts dy of one pair; 1: Q right matrices
  int vec4;               // global rows can be read as float4
  int per_slot_rows;      // staged rows per pair slot
};

// k-th block in order of distance from the middle of n blocks.
__device__ __forceinline__ int centered(int k, int n) {
  const int m = (n - 1) >> 1;
  if (k == 0) return m;
  return (k & 1) ? m + ((k + 1) >> 1) : m - (k >> 1);
}

__device__ __forceinline__ void stage_row(float *dst, const float *src, int W,
                                          bool valid, bool vec4) {
  // dst points at column 0 of the staged row (kPadL zeros precede it).
  if (!valid) {
    for (int x = threadIdx.x & 31; x < W; x += 32) dst[x] = 0.f;
    return;
  }
  if (vec4) {
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    for (int x = threadIdx.x & 31; x < (W >> 2); x += 32) d4[x] = __ldg(s4 + x);
  } else {
    for (int x = threadIdx.x & 31; x < W; x += 32) dst[x] = __ldg(src + x);
  }
}

// One 4-step block of the x loop: a float4 of L, and for each q a float4 of
// R entering ring positions 4J..4J+3 (J = block index mod 3).  The ring
// position of R[u0 + j] is j mod kRing, so shift p at step s reads position
// (4J + s - p) mod kRing.
template <int J>
__device__ __forceinline__ void ring_block(float (&acc)[kQ][kP],
                                           float (&ring)[kQ][kRing],
                                           const float *lp,
                                           const float *const (&Rq)[kQ], int ub) {
  const float4 l4 = *reinterpret_cast<const float4 *>(lp);
#pragma unroll
  for (int q = 0; q < kQ; ++q) {
    const float4 r4 = *reinterpret_cast<const float4 *>(Rq[q] + ub);
    ring[q][4 * J + 0] = r4.x;
    ring[q][4 * J + 1] = r4.y;
    ring[q][4 * J + 2] = r4.z;
    ring[q][4 * J + 3] = r4.w;
  }
  const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int p = 0; p < kP; ++p)
#pragma unroll
      for (int q = 0; q < kQ; ++q)
        acc[q][p] = fmaf(lv[s], ring[q][(4 * J + s - p + 2 * kRing) % kRing], acc[q][p]);
}

// One overlap row of one lane: acc[q][p] += sum_x L[x] * Rq[x - dx0 - p],
// x over [xlo, xlo + 4 nb); u0 = xlo - dx0 (a multiple of 4).  Lrow / Rq
// point at column 0 of zero-padded staged rows.
__device__ __forceinline__ void lane_row(float (&acc)[kQ][kP], const float *Lrow,
                                         const float *const (&Rq)[kQ], int xlo,
                                         int u0, int nb) {
  static_assert(kP == 8 && kRing == 12, "ring preload assumes P = 8");
  float ring[kQ][kRing];
#pragma unroll
  for (int q = 0; q < kQ; ++q) {
    // R[u0-8 .. u0-1] -> positions 4..11
    const float4 a = *reinterpret_cast<const float4 *>(Rq[q] + u0 - 8);
    const float4 b = *reinterpret_cast<const float4 *>(Rq[q] + u0 - 4);
    ring[q][4] = a.x; ring[q][5] = a.y; ring[q][6] = a.z; ring[q][7] = a.w;
    ring[q][8] = b.x; ring[q][9] = b.y; ring[q][10] = b.z; ring[q][11] = b.w;
#pragma unroll
    for (int i = 0; i < 4; ++i) ring[q][i] = 0.f;
  }
  const float *lp = Lrow + xlo;
  int ub = u0;
  int b = 0;
  for (; b + 3 <= nb; b += 3) {
    ring_block<0>(acc, ring, lp, Rq, ub);
    ring_block<1>(acc, ring, lp + 4, Rq, ub + 4);
    ring_block<2>(acc, ring, lp + 8, Rq, ub + 8);
    lp += 12;
    ub += 12;
  }
  if (b < nb) ring_block<0>(acc, ring, lp, Rq, ub);
  if (b + 1 < nb) ring_block<1>(acc, ring, lp + 4, Rq, ub + 4);
}

__global__ void __launch_bounds__(kThreads, 2) xcorr_rows_kernel(const RowArgs a) {
  extern __shared__ float4 smem4[];
  float *sm = reinterpret_cast<float *>(smem4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- which outputs this CTA owns (costly blocks first) ----
  int item = blockIdx.x;
  const int sb = item % a.nslots_blocks;
  item /= a.nslots_blocks;
  const int dyb = centered(item % a.ndy, a.ndy);
  const int dxs = centered(item / a.ndy, a.nsuper);
  const int H = a.H, W = a.W, S = a.S;

  const int g = lane >> a.log_ph;          // pair slot of this lane
  const int ph = lane & (a.ph - 1);        // row phase of this lane
  const int slot = sb * a.G + g;           // global slot index

  // slot -> pair(s).  rows mode: slot = pair; rights mode: slot = (left,
  // block of kQ rights)
  int li, r0, nrq;
  if (!a.rights_mode) {
    li = slot / a.nr;
    r0 = slot % a.nr;
    nrq = 1;
  } else {
    const int rblocks = (a.nr + kQ - 1) / kQ;
    li = slot / rblocks;
    r0 = (slot % rblocks) * kQ;
    nrq = min(kQ, a.nr - r0);
  }
  const bool slot_ok = li < a.nl;

  int dy0, ylo, yhi;
  if (!a.rights_mode) {
    dy0 = dyb * kQ - (H - 1);
    ylo = max(0, dy0);
    yhi = min(H, H + dy0 + kQ - 1);
  } else {
    dy0 = dyb - (H - 1);
    ylo = max(0, dy0);
    yhi = min(H, H + dy0);
  }
  const int group = dxs * kWarps + warp;
  const int dx0 = a.dxbase + group * kP;
  const bool group_ok = group < a.ngroups;
  const int xlo = max(0, dx0);
  const int xhi = min(W, W + dx0 + kP - 1);
  const int nb = xhi > xlo ? (xhi - xlo + 3) >> 2 : 0;

  // ---- zero the whole staging area once (padding columns stay zero) ----
  const int rows_total = a.G * a.per_slot_rows;
  for (int i = threadIdx.x; i < rows_total * S; i += kThreads) sm[i] = 0.f;

  float acc[kQ][kP];
#pragma unroll
  for (int q = 0; q < kQ; ++q)
#pragma unroll
    for (int p = 0; p < kP; ++p) acc[q][p] = 0.f;

  const size_t mat = size_t(H) * W;
  const int rows_per_slot = a.per_slot_rows;
  const int lrows = a.ph;                            // L rows per slot
  for (int yc = ylo; yc < yhi; yc += a.ph) {
    __syncthreads();
    // stage: per slot, L rows yc..yc+ph-1, then R rows
    for (int r = warp; r < rows_total; r += kWarps) {
      const int gs = r / rows_per_slot, k = r - gs * rows_per_slot;
      const int sl = sb * a.G + gs;
      int sli, sr0;
      if (!a.rights_mode) {
        sli = sl / a.nr;
        sr0 = sl % a.nr;
      } else {
        const int rblocks = (a.nr + kQ - 1) / kQ;
        sli = sl / rblocks;
        sr0 = (sl % rblocks) * kQ;
      }
      float *dst = sm + size_t(r) * S + kPadL;
      if (sli >= a.nl) {
        stage_row(dst, nullptr, W, false, false);
        continue;
      }
      if (k < lrows) {
        const int y = yc + k;
        stage_row(dst, a.left + sli * mat + size_t(y) * W, W, y < yhi, a.vec4);
      } else if (!a.rights_mode) {
        // R rows yr = yc - dy0 - (kQ-1) + (k - lrows)
        const int yr = yc - dy0 - (kQ - 1) + (k - lrows);
        stage_row(dst, a.right + sr0 * mat + size_t(yr) * W, W, yr >= 0 && yr < H,
                  a.vec4);
      } else {
        const int kk = k - lrows, rq = kk / lrows, yr = yc + (kk % lrows) - dy0;
        const bool ok = sr0 + rq < a.nr && yr >= 0 && yr < H && yc + (kk % lrows) < yhi;
        stage_row(dst, a.right + (sr0 + rq) * mat + size_t(yr) * W, W, ok, a.vec4);
      }
    }
    __syncthreads();
    const int y = yc + ph;
    if (!slot_ok || !group_ok || y >= yhi || nb == 0) continue;
    const float *base = sm + size_t(g) * rows_per_slot * S + kPadL;
    const float *Lrow = base + size_t(ph) * S;
    const float *Rq[kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      if (!a.rights_mode)
        Rq[q] = base + size_t(lrows + ph + (kQ - 1) - q) * S;
      else
        Rq[q] = base + size_t(lrows + q * lrows + ph) * S;
    }
    lane_row(acc, Lrow, Rq, xlo, xlo - dx0, nb);
  }

  // ---- add the row phases; every lane of a slot then holds the sums ----
  for (int o = 1; o < a.ph; o <<= 1) {
#pragma unroll
    for (int q = 0; q < kQ; ++q)
#pragma unroll
      for (int p = 0; p < kP; ++p)
        acc[q][p] += __shfl_xor_sync(0xffffffffu, acc[q][p], o);
  }
  if (!slot_ok || !group_ok) return;
  const int oh = 2 * H - 1, ow = 2 * W - 1;
#pragma unroll
  for (int q = 0; q < kQ; ++q) {
#pragma unroll
    for (int p = 0; p < kP; ++p) {
      if (((q * kP + p) & (a.ph - 1)) != ph) continue;
      const int dx = dx0 + p;
      if (dx <= -W || dx >= W) continue;
      int dy, ri;
      if (!a.rights_mode) {
        dy = dy0 + q;
        ri = r0;
        if (dy >= H) continue;
      } else {
        dy = dy0;
        ri = r0 + q;
        if (q >= nrq) continue;
      }
      const size_t pair = size_t(li) * a.nr + ri;
      a.out[(pair * oh + (dy + H - 1)) * ow + (dx + W - 1)] = acc[q][p];
    }
  }
}

// ---------------------------------------------------------------------------
// General fallback for matrices too wide to stage (shared rows beyond the
// per-CTA limit): same unit decomposition, operands read through L1 with
// bounds predicates instead of zero-padded shared rows.
// ---------------------------------------------------------------------------
constexpr int kDirectP = 8;
constexpr int kDirectWarps = 4;

struct DirectArgs {
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
__global__ void __launch_bounds__(32 * kDirectWarps) xcorr_direct_kernel(const DirectArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long unit = (long long)blockIdx.x * kDirectWarps + warp;
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

namespace {

cudaError_t launch_direct(const float *left, int nl, const float *right, int nr,
                          int H, int W, float *out, cudaStream_t stream) {
  DirectArgs a;
  a.left = left;
  a.right = right;
  a.out = out;
  a.nl = nl;
  a.nr = nr;
  a.H = H;
  a.W = W;
  a.pairs = nl * nr;
  int G = 1;
  while (G < 32 && (32 / G) * 4 > H) G <<= 1;
  while (G > 1 && G / 2 >= a.pairs) G >>= 1;
  a.G = G;
  a.log_ph = ilog2(32 / G);
  a.groups_x = (2 * W - 1 + kDirectP - 1) / kDirectP;
  a.pair_blocks = (a.pairs + G - 1) / G;
  a.units = (long long)a.pair_blocks * (2 * H - 1) * a.groups_x;
  const long long blocks = (a.units + kDirectWarps - 1) / kDirectWarps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  xcorr_direct_kernel<kDirectP><<<unsigned(blocks), 32 * kDirectWarps, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

// Largest shared staging area the row kernel takes (two CTAs per SM fit).
constexpr size_t kMaxRowSmem = 110 * 1024;

cudaError_t xcorr_f32_launch(const float *left, int nl, const float *right,
                             int nr, int H, int W, float *out,
                             cudaStream_t stream) {
  RowArgs a;
  a.left = left;
  a.right = right;
  a.out = out;
  a.nl = nl;
  a.nr = nr;
  a.H = H;
  a.W = W;
  // several rights per left: kQ rights share each staged L row; otherwise
  // kQ neighbouring shifts dy of one pair
  a.rights_mode = nr >= kQ ? 1 : 0;
  const long long slots = a.rights_mode ? (long long)nl * ((nr + kQ - 1) / kQ)
                                        : (long long)nl * nr;
  // enough row phases that a lane sums several rows, but not more than H
  int G = 1;
  while (G < 32 && (32 / G) * 4 > H) G <<= 1;
  while (G > 1 && G / 2 >= slots) G >>= 1;
  a.G = G;
  a.ph = 32 / G;
  a.log_ph = ilog2(a.ph);
  a.per_slot_rows = a.rights_mode ? a.ph * (1 + kQ) : (2 * a.ph + kQ - 1);
  const int need = kPadL + ((W + 3) & ~3) + kP + 8;
  a.S = ((need + 7) & ~7) + 4;
  a.dxbase = -(((W - 1) + 3) & ~3);
  a.ngroups = ((W - 1) - a.dxbase) / kP + 1;
  a.nsuper = (a.ngroups + kWarps - 1) / kWarps;
  a.ndy = a.rights_mode ? 2 * H - 1 : (2 * H - 1 + kQ - 1) / kQ;
  a.nslots_blocks = int((slots + G - 1) / G);
  a.vec4 = ((W & 3) == 0 && (reinterpret_cast<uintptr_t>(left) & 15) == 0 &&
            (reinterpret_cast<uintptr_t>(right) & 15) == 0) ? 1 : 0;
  const size_t smem = size_t(G) * a.per_slot_rows * a.S * sizeof(float);
  const long long blocks = (long long)a.nslots_blocks * a.ndy * a.nsuper;
  if (smem > kMaxRowSmem || blocks > 0x7fffffffLL)
    return launch_direct(left, nl, right, nr, H, W, out, stream);
  cudaError_t e = cudaFuncSetAttribute(
      xcorr_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  xcorr_rows_kernel<<<unsigned(blocks), kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace corr
