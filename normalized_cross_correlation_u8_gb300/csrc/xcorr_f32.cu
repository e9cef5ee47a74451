// xcorr_f32.cu -- float32 full 2D cross-correlation on sm_103a.
//
// Method ("Efficient GPU-accelerated Parallel Cross-correlation" artifact
// README, kernel overview): every output is one overlap (relative shift) of
// a left and a right matrix,
//
//   out[pair][dy+H-1][dx+W-1] = sum_{y,x} L[y][x] * R[y-dy][x-dx],
//
// computed for all shifts.  The page's fast kernels keep a register buffer
// of one matrix that slides along x while the other streams past (warp-
// shuffle family), compute several neighbouring overlaps per thread
// (grouped overlap), reuse one matrix against several others (multi-matrix),
// and split one overlap's rows over several threads when there are few
// overlaps (split-row).  The same ideas, laid out for sm_103a, in three
// kernels chosen by shape:
//
//  rows  (matrices too large to keep a pair in shared memory)
//    A CTA owns Q = 4 shifts dy x 8 warps x P = 8 shifts dx of one pair.
//    The overlap rows y are the reduction: each lane of a warp sums its own
//    rows, so every lane runs the same x loop.  Rows are staged 32 at a time
//    into zero-padded shared rows (no bounds tests in the inner loop).
//  pair  (a pair fits in shared memory: one-to-many and n-to-m of medium
//    matrices) -- the whole pair is staged once; each warp then loops over
//    (4 dy x 8 dx) output blocks with the same lane scheme.
//  tiny  (H*W <= 256, many pairs) -- 32 lefts and 16 rights are staged
//    interleaved (matrix index fastest); each lane owns 4 lefts x 4 rights
//    of one shift and walks that shift's exact overlap, so no product is
//    wasted; warps pull shifts from a per-CTA list.
//
// Per lane and overlap row (rows / pair kernels): a float4 of L feeds 4 x
// steps; for each of the Q rows a float4 of R enters a 12-entry register
// ring holding R[x-dx0-p] for the P shifts, indexed at compile-time
// positions by unrolling three 4-step blocks: 5 shared loads feed
// 4*P*Q = 128 FMAs.  When the last pass has fewer rows than lanes, each row
// is split into x sub-ranges over several lanes (split-row), and a shuffle
// butterfly adds the lanes' partial sums before the stores.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.cuh"

namespace corr {
namespace {

constexpr int kP = 8;                // neighbouring shifts dx per lane
constexpr int kQ = 4;                // neighbouring shifts dy per lane
constexpr int kRing = kP + 4;        // ring of R values (multiple of 4)
constexpr int kPadL = kP;            // zero columns left of a staged row
constexpr int kWarps = 8;            // rows / pair kernels
constexpr int kThreads = 32 * kWarps;

// k-th block in order of distance from the middle of n blocks (costly
// central blocks first).
__device__ __forceinline__ int centered(int k, int n) {
  const int m = (n - 1) >> 1;
  if (k == 0) return m;
  return (k & 1) ? m + ((k + 1) >> 1) : m - (k >> 1);
}

// ---------------------------------------------------------------------------
// Per-lane ring walk over x blocks [b0, b1) of one overlap row.
//   l4:    float4 index of L[xlo] in shared memory
//   r4[q]: float4 index of R_q[u0] (u0 = xlo - dx0) in shared memory
// Block b covers x = xlo + 4b .. xlo + 4b + 3.  R_q[u0 + j] lives at ring
// position (j - 4 b0) mod 12.
// ---------------------------------------------------------------------------
extern __shared__ float4 g_smem4[];

// 16-byte shared load at byte address addr + OFF (OFF folded into the
// instruction), so a whole unrolled round of loads shares one address
// register per row.
template <int OFF>
__device__ __forceinline__ float4 lds128(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4+%5];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr), "n"(OFF));
  return v;
}

// Block J of a round: one float4 of L at la + 16 J, for each q a float4 of
// R_q at ra[q] + 16 J into ring positions 4 (J mod 3) .. +3; shift p at step
// s reads position (4 (J mod 3) + s - p) mod 12.
template <int J>
__device__ __forceinline__ void ring_block(float (&acc)[kQ][kP],
                                           float (&ring)[kQ][kRing], uint32_t la,
                                           const uint32_t (&ra)[kQ]) {
  constexpr int JR = J % 3;
  const float4 lv4 = lds128<16 * J>(la);
#pragma unroll
  for (int q = 0; q < kQ; ++q) {
    const float4 v = lds128<16 * J>(ra[q]);
    ring[q][4 * JR + 0] = v.x;
    ring[q][4 * JR + 1] = v.y;
    ring[q][4 * JR + 2] = v.z;
    ring[q][4 * JR + 3] = v.w;
  }
  const float lv[4] = {lv4.x, lv4.y, lv4.z, lv4.w};
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int p = 0; p < kP; ++p)
#pragma unroll
      for (int q = 0; q < kQ; ++q)
        acc[q][p] = fmaf(lv[s], ring[q][(4 * JR + s - p + 2 * kRing) % kRing], acc[q][p]);
}

// Per-lane ring walk over x blocks [b0, b1) of one overlap row.
//   l4:    float4 index of L[xlo] in shared memory
//   r4[q]: float4 index of R_q[u0] (u0 = xlo - dx0) in shared memory
// Block b covers x = xlo + 4b .. xlo + 4b + 3.  R_q[u0 + j] lives at ring
// position (j - 4 b0) mod 12.
__device__ __forceinline__ void lane_blocks(float (&acc)[kQ][kP], int l4,
                                            const int (&r4)[kQ], int b0, int b1) {
  static_assert(kP == 8 && kRing == 12, "ring preload assumes P = 8");
  if (b0 >= b1) return;
  const uint32_t base = uint32_t(__cvta_generic_to_shared(g_smem4));
  float ring[kQ][kRing];
  uint32_t ra[kQ];
#pragma unroll
  for (int q = 0; q < kQ; ++q) {
    // R[u0 + 4 b0 - 8 .. u0 + 4 b0 - 1] -> positions 4..11
    ra[q] = base + 16u * uint32_t(r4[q] + b0);
    const float4 a = lds128<-32>(ra[q]);
    const float4 b = lds128<-16>(ra[q]);
    ring[q][4] = a.x; ring[q][5] = a.y; ring[q][6] = a.z; ring[q][7] = a.w;
    ring[q][8] = b.x; ring[q][9] = b.y; ring[q][10] = b.z; ring[q][11] = b.w;
    ring[q][0] = ring[q][1] = ring[q][2] = ring[q][3] = 0.f;
  }
  uint32_t la = base + 16u * uint32_t(l4 + b0);
  int b = b0;
  for (; b + 6 <= b1; b += 6) {
    ring_block<0>(acc, ring, la, ra);
    ring_block<1>(acc, ring, la, ra);
    ring_block<2>(acc, ring, la, ra);
    ring_block<3>(acc, ring, la, ra);
    ring_block<4>(acc, ring, la, ra);
    ring_block<5>(acc, ring, la, ra);
    la += 96;
#pragma unroll
    for (int q = 0; q < kQ; ++q) ra[q] += 96;
  }
  // 0..5 remaining blocks, positions continue (J mod 3)
  const int rem = b1 - b;
  if (rem > 0) ring_block<0>(acc, ring, la, ra);
  if (rem > 1) ring_block<1>(acc, ring, la, ra);
  if (rem > 2) ring_block<2>(acc, ring, la, ra);
  if (rem > 3) ring_block<3>(acc, ring, la, ra);
  if (rem > 4) ring_block<4>(acc, ring, la, ra);
}

// Geometry of one output block of a warp: shifts dy0..dy0+3 x dx0..dx0+7.
struct Block {
  int dy0, dx0;
  int ylo, yhi;   // union of the overlap rows of the 4 shifts dy
  int xlo, nb;    // first x (multiple of 4) and number of 4-wide x blocks
};

__device__ __forceinline__ Block make_block(int H, int W, int dy0, int dx0) {
  Block k;
  k.dy0 = dy0;
  k.dx0 = dx0;
  k.ylo = max(0, dy0);
  k.yhi = min(H, H + dy0 + kQ - 1);
  k.xlo = max(0, dx0);
  const int xhi = min(W, W + dx0 + kP - 1);
  k.nb = xhi > k.xlo ? (xhi - k.xlo + 3) >> 2 : 0;
  return k;
}

// One pass of up to 32 overlap rows [y, y + n) of a block over the lanes of a
// warp.  lrow(y) / rrow(yr) give the float index of column 0 of a staged L
// row / R row (before the kPadL zero columns).  With n == 32 lane ph takes
// row y + ph; with fewer rows each row is split into k = 32 / n x sub-ranges
// (lanes past n*k idle).
template <typename LRow, typename RRow>
__device__ __forceinline__ void warp_pass(float (&acc)[kQ][kP], const Block &k,
                                          int y, int n, int lane, LRow lrow,
                                          RRow rrow) {
  if (n <= 0 || k.nb == 0) return;
  int row, b0, b1;
  if (n >= 32) {
    row = y + lane;
    b0 = 0;
    b1 = k.nb;
  } else {
    const int parts = 32 / n;
    const int part = lane / n;
    if (part >= parts) return;
    row = y + (lane - part * n);
    b0 = part * k.nb / parts;
    b1 = (part + 1) * k.nb / parts;
  }
  const int u0 = k.xlo - k.dx0;
  const int l4 = (lrow(row) + kPadL + k.xlo) >> 2;
  int r4[kQ];
#pragma unroll
  for (int q = 0; q < kQ; ++q) r4[q] = (rrow(row - k.dy0 - q) + kPadL + u0) >> 2;
  lane_blocks(acc, l4, r4, b0, b1);
}

// Reduce-scatter over the 32 lanes: at each step a lane keeps one half of
// its remaining partial sums and adds the partner's copy of that half, so
// after 16 + 8 + 4 + 2 + 1 shuffles lane i holds the full sum of output
// i = q * 8 + p.  Returns it and clears the accumulators.
__device__ __forceinline__ float reduce_scatter(float (&acc)[kQ][kP], int lane) {
  float v[32];
#pragma unroll
  for (int q = 0; q < kQ; ++q)
#pragma unroll
    for (int p = 0; p < kP; ++p) v[q * kP + p] = acc[q][p];
#pragma unroll
  for (int n = 16; n >= 1; n >>= 1) {
    const bool upper = (lane & n) != 0;   // keep v[n..2n) if set, else v[0..n)
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float send = upper ? v[i] : v[i + n];
      const float keep = upper ? v[i + n] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, n);
    }
  }
#pragma unroll
  for (int q = 0; q < kQ; ++q)
#pragma unroll
    for (int p = 0; p < kP; ++p) acc[q][p] = 0.f;
  return v[0];
}

// Reduce and store the block's outputs into out_pair ([2H-1][2W-1]).
__device__ __forceinline__ void reduce_store(float (&acc)[kQ][kP], const Block &k,
                                             int lane, int H, int W,
                                             float *out_pair) {
  const float v = reduce_scatter(acc, lane);
  const int dy = k.dy0 + (lane >> 3), dx = k.dx0 + (lane & 7);
  if (dy > -H && dy < H && dx > -W && dx < W)
    out_pair[size_t(dy + H - 1) * (2 * W - 1) + (dx + W - 1)] = v;
}

// Copy `rows` matrix rows (global float rows of W, src(r) = pointer or
// nullptr for a zero row) into shared rows of stride S starting at float
// `dst0`, data at column kPadL.  One warp per row.
template <typename Src>
__device__ __forceinline__ void stage_rows(float *sm, int dst0, int rows, int S, int W,
                                           bool vec4, Src src) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int r = warp; r < rows; r += nw) {
    const float *g = src(r);
    float *d = sm + dst0 + r * S + kPadL;
    if (!g) {
      for (int x = lane; x < W; x += 32) d[x] = 0.f;
    } else if (vec4) {
      const float4 *g4 = reinterpret_cast<const float4 *>(g);
      float4 *d4 = reinterpret_cast<float4 *>(d);
      for (int x = lane; x < (W >> 2); x += 32) d4[x] = __ldg(g4 + x);
    } else {
      for (int x = lane; x < W; x += 32) d[x] = __ldg(g + x);
    }
  }
}

__device__ __forceinline__ void zero_smem(float *sm, int n) {
  float4 *s4 = reinterpret_cast<float4 *>(sm);
  for (int i = threadIdx.x; i < (n >> 2); i += blockDim.x) s4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

struct XArgs {
  const float *left;
  const float *right;
  float *out;
  int nl, nr, H, W;
  int S;          // shared row stride in floats (S % 8 == 4)
  int dxbase;     // first shift of dx group 0 (multiple of 4, <= 1-W)
  int ngroups;    // dx groups of kP
  int ndyb;       // dy blocks of kQ
  int nsuper;     // rows kernel: ceil(ngroups / kWarps)
  int parts;      // pair kernel: CTAs per pair
  int vec4;       // rows can be read as float4
  int nbands;     // rows kernel: row bands of kBandRows (split-row)
  int part_row;   // rows kernel: floats per partial-sum row (8 * ngroups)
  float *part;    // rows kernel: band partial sums (nbands > 1)
};

// ---------------------------------------------------------------------------
// rows kernel: one CTA = one pair x 4 dy x 64 dx x one band of kBandRows
// overlap rows (split-row: the bands of a block are summed afterwards in a
// fixed order, so results do not depend on scheduling).  The band's rows
// are staged kChunk at a time into two shared buffers with cp.async, so the
// next chunk streams in while the current one is consumed (one barrier per
// chunk).  A chunk of 16 rows is spread over the 32 lanes by splitting each
// row's x range in two.  With a single band the CTA writes the outputs
// directly; otherwise it writes its band's partial sums to
//   part[((pair * ndyb + dyb) * nbands + band) * kQ + q][8 * group + p].
// ---------------------------------------------------------------------------
constexpr int kBandRows = 64;
constexpr int kChunk = 16;
constexpr int kChunkL = kChunk, kChunkR = kChunk + kQ - 1;
constexpr int kChunkRows = kChunkL + kChunkR;

__device__ __forceinline__ void cp_async(uint32_t dst, const float *src, bool valid,
                                         bool vec4) {
  if (vec4)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

// Issue the copies of one chunk (L rows yc .. yc+kChunkL-1 below y_end, R
// rows yr_first .. yr_first+kChunkR-1 inside [0, H); other rows zero-fill)
// into the buffer starting at float `buf`.  One warp per row.
__device__ __forceinline__ void issue_chunk(uint32_t sbase, int buf, int S, int W,
                                            bool vec4, const float *L, const float *R,
                                            int yc, int y_end, int yr_first, int H) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int step = vec4 ? 4 : 1, n = vec4 ? (W >> 2) : W;
  for (int r = warp; r < kChunkRows; r += kWarps) {
    const float *src;
    bool ok;
    if (r < kChunkL) {
      const int y = yc + r;
      ok = y < y_end;
      src = L + (ok ? size_t(y) * W : 0);
    } else {
      const int yr = yr_first + (r - kChunkL);
      ok = yr >= 0 && yr < H;
      src = R + (ok ? size_t(yr) * W : 0);
    }
    const uint32_t d = sbase + 4u * uint32_t(buf + r * S + kPadL);
    for (int c = lane; c < n; c += 32)
      cp_async(d + 4u * uint32_t(c * step), src + c * step, ok, vec4);
  }
}

__global__ void __launch_bounds__(kThreads, 2) xcorr_rows_kernel(const XArgs a) {
  float *sm = reinterpret_cast<float *>(g_smem4);
  const uint32_t sbase = uint32_t(__cvta_generic_to_shared(g_smem4));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, W = a.W, S = a.S;
  int item = blockIdx.x;
  const int band = item % a.nbands;
  item /= a.nbands;
  const int pair = item % (a.nl * a.nr);
  item /= a.nl * a.nr;
  const int dyb = centered(item % a.ndyb, a.ndyb);
  const int dxs = centered(item / a.ndyb, a.nsuper);
  const int li = pair / a.nr, ri = pair - li * a.nr;
  const size_t mat = size_t(H) * W;
  const float *L = a.left + li * mat;
  const float *R = a.right + ri * mat;

  const int group = dxs * kWarps + warp;
  const Block k = make_block(H, W, dyb * kQ - (H - 1), a.dxbase + group * kP);
  const bool active = group < a.ngroups;
  const int y_begin = max(k.ylo, band * kBandRows);
  const int y_end = min(k.yhi, (band + 1) * kBandRows);
  if (y_begin >= y_end) return;           // CTA-uniform: this band is empty

  const int buf_floats = kChunkRows * S;
  zero_smem(sm, 2 * buf_floats);          // padding columns stay zero
  __syncthreads();
  float acc[kQ][kP];
#pragma unroll
  for (int q = 0; q < kQ; ++q)
#pragma unroll
    for (int p = 0; p < kP; ++p) acc[q][p] = 0.f;

  const int nchunks = (y_end - y_begin + kChunk - 1) / kChunk;
  issue_chunk(sbase, 0, S, W, a.vec4, L, R, y_begin, y_end, y_begin - k.dy0 - (kQ - 1), H);
  cp_async_commit();
  for (int c = 0; c < nchunks; ++c) {
    const int yc = y_begin + c * kChunk;
    const int buf = (c & 1) * buf_floats;
    cp_async_wait_all();        // this thread's copies of chunk c have landed
    __syncthreads();            // ... everyone's, and chunk c-1 is consumed
    if (c + 1 < nchunks) {
      const int yn = yc + kChunk;
      issue_chunk(sbase, ((c + 1) & 1) * buf_floats, S, W, a.vec4, L, R, yn, y_end,
                  yn - k.dy0 - (kQ - 1), H);
      cp_async_commit();
    }
    const int yr_first = yc - k.dy0 - (kQ - 1);
    if (active)
      warp_pass(acc, k, yc, min(kChunk, y_end - yc), lane,
                [&](int y) { return buf + (y - yc) * S; },
                [&](int yr) { return buf + (kChunkL + yr - yr_first) * S; });
  }
  if (!active) return;
  if (a.nbands == 1) {
    reduce_store(acc, k, lane, H, W, a.out + size_t(pair) * (2 * H - 1) * (2 * W - 1));
  } else {
    const float v = reduce_scatter(acc, lane);
    const size_t slot = (size_t(pair) * a.ndyb + dyb) * a.nbands + band;
    a.part[(slot * kQ + (lane >> 3)) * a.part_row + group * kP + (lane & 7)] = v;
  }
}

// Second pass of the rows kernel: out = sum over the non-empty bands of the
// partial sums, in band order.
__global__ void xcorr_band_sum_kernel(const XArgs a) {
  const int H = a.H, W = a.W, oh = 2 * H - 1, ow = 2 * W - 1;
  const long long total = (long long)a.nl * a.nr * oh * ow;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int ox = int(i % ow);
    const long long t = i / ow;
    const int oy = int(t % oh);
    const int pair = int(t / oh);
    const int dyb = oy / kQ, q = oy - dyb * kQ;
    const int dy0 = dyb * kQ - (H - 1);
    const int ylo = max(0, dy0), yhi = min(H, H + dy0 + kQ - 1);
    const int col = (ox - (W - 1)) - a.dxbase;
    const size_t slot0 = (size_t(pair) * a.ndyb + dyb) * a.nbands;
    float sum = 0.f;
    for (int b = 0; b < a.nbands; ++b) {
      if (max(ylo, b * kBandRows) >= min(yhi, (b + 1) * kBandRows)) continue;
      sum += a.part[((slot0 + b) * kQ + q) * a.part_row + col];
    }
    a.out[i] = sum;
  }
}

// ---------------------------------------------------------------------------
// pair kernel: the CTA stages one whole pair (R with kQ-1 zero rows above and
// below), then its warps loop over output blocks of that pair.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 2) xcorr_pair_kernel(const XArgs a) {
  float *sm = reinterpret_cast<float *>(g_smem4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, W = a.W, S = a.S;
  const int pair = blockIdx.x / a.parts, part = blockIdx.x - pair * a.parts;
  const int li = pair / a.nr, ri = pair - li * a.nr;
  const size_t mat = size_t(H) * W;
  const float *L = a.left + li * mat;
  const float *R = a.right + ri * mat;
  constexpr int kPadY = kQ - 1;
  const int rrows = H + 2 * kPadY;
  zero_smem(sm, (H + rrows) * S);
  __syncthreads();
  stage_rows(sm, 0, H, S, W, a.vec4, [&](int r) -> const float * { return L + size_t(r) * W; });
  stage_rows(sm, H * S, rrows, S, W, a.vec4, [&](int r) -> const float * {
    const int yr = r - kPadY;
    return (yr >= 0 && yr < H) ? R + size_t(yr) * W : nullptr;
  });
  __syncthreads();

  float acc[kQ][kP];
#pragma unroll
  for (int q = 0; q < kQ; ++q)
#pragma unroll
    for (int p = 0; p < kP; ++p) acc[q][p] = 0.f;
  float *out_pair = a.out + size_t(pair) * (2 * H - 1) * (2 * W - 1);
  const int nitems = a.ndyb * a.ngroups;
  for (int it = part + a.parts * warp; it < nitems; it += a.parts * kWarps) {
    const int dyb = centered(it % a.ndyb, a.ndyb);
    const int g = centered(it / a.ndyb, a.ngroups);
    const Block k = make_block(H, W, dyb * kQ - (H - 1), a.dxbase + g * kP);
    for (int y = k.ylo; y < k.yhi; y += 32)
      warp_pass(acc, k, y, min(32, k.yhi - y), lane, [&](int yy) { return yy * S; },
                [&](int yr) { return (H + kPadY + yr) * S; });
    reduce_store(acc, k, lane, H, W, out_pair);
  }
}

// ---------------------------------------------------------------------------
// tiny kernel: H*W <= 256.  A CTA stages a block of 32 lefts and 16 rights
// interleaved as [y][x][matrix]; lane (lb = lane%8, rb = lane/8) owns lefts
// 4lb..4lb+3 x rights 4rb..4rb+3 of one shift and walks its exact overlap:
// per (y, x) two 16-byte loads feed 16 FMAs.  Shifts are dealt to the CTAs
// of a block pair round-robin in a centre-first order and pulled by the
// CTA's warps from a shared counter.
// ---------------------------------------------------------------------------
constexpr int kTinyL = 32, kTinyR = 16, kTinyWarps = 8;

struct TinyArgs {
  const float *left;
  const float *right;
  float *out;
  int nl, nr, H, W;
  int lblocks, rblocks;  // blocks of kTinyL lefts / kTinyR rights
  int nc;                // CTAs sharing one block pair
  int vec4;              // matrices can be read as float4 (H*W % 4 == 0, aligned)
};

__global__ void __launch_bounds__(32 * kTinyWarps) xcorr_tiny_kernel(const TinyArgs a) {
  float *Ls = reinterpret_cast<float *>(g_smem4);
  const int H = a.H, W = a.W, HW = H * W;
  float *Rs = Ls + HW * kTinyL;
  __shared__ int next_unit;
  int bid = blockIdx.x;
  const int c = bid % a.nc;
  bid /= a.nc;
  const int rbk = bid % a.rblocks, lbk = bid / a.rblocks;
  const int l_base = lbk * kTinyL, r_base = rbk * kTinyR;

  // stage: thread (m, pos4) reads 16 bytes (positions 4 pos4 .. +3) of
  // matrix m and scatters them to Ls[pos*32 + m] (lanes of a warp take 32
  // consecutive m, so each shared store touches 32 distinct banks).  H*W is
  // a multiple of 4 on this path when the rows are 16-byte aligned;
  // otherwise element loads are used.
  {
    const int hw4 = (HW + 3) >> 2;
    for (int i = threadIdx.x; i < hw4 * kTinyL; i += blockDim.x) {
      const int m = i % kTinyL, p4 = i / kTinyL;
      const int l = l_base + m;
      float e[4] = {0.f, 0.f, 0.f, 0.f};
      if (l < a.nl) {
        const float *src = a.left + size_t(l) * HW + 4 * p4;
        if (a.vec4) {
          const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
          e[0] = v.x; e[1] = v.y; e[2] = v.z; e[3] = v.w;
        } else {
#pragma unroll
          for (int t = 0; t < 4; ++t) e[t] = 4 * p4 + t < HW ? __ldg(src + t) : 0.f;
        }
      }
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (4 * p4 + t < HW) Ls[(4 * p4 + t) * kTinyL + m] = e[t];
    }
    for (int i = threadIdx.x; i < hw4 * kTinyR; i += blockDim.x) {
      const int m = i % kTinyR, p4 = i / kTinyR;
      const int r = r_base + m;
      float e[4] = {0.f, 0.f, 0.f, 0.f};
      if (r < a.nr) {
        const float *src = a.right + size_t(r) * HW + 4 * p4;
        if (a.vec4) {
          const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
          e[0] = v.x; e[1] = v.y; e[2] = v.z; e[3] = v.w;
        } else {
#pragma unroll
          for (int t = 0; t < 4; ++t) e[t] = 4 * p4 + t < HW ? __ldg(src + t) : 0.f;
        }
      }
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (4 * p4 + t < HW) Rs[(4 * p4 + t) * kTinyR + m] = e[t];
    }
  }
  if (threadIdx.x == 0) next_unit = 0;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int lb = lane & 7, rb = lane >> 3;
  const int ndy = 2 * H - 1, ndx = 2 * W - 1, nunits = ndy * ndx;
  const int mine = (nunits - c + a.nc - 1) / a.nc;   // units k = c, c+nc, ...
  for (;;) {
    int u = 0;
    if (lane == 0) u = atomicAdd(&next_unit, 1);
    u = __shfl_sync(0xffffffffu, u, 0);
    if (u >= mine) break;
    const int kk = c + u * a.nc;                     // centre-first rank
    const int dy = centered(kk % ndy, ndy) - (H - 1);
    const int dx = centered(kk / ndy, ndx) - (W - 1);
    const int ylo = max(0, dy), yhi = min(H, H + dy);
    const int xlo = max(0, dx), xhi = min(W, W + dx);
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int y = ylo; y < yhi; ++y) {
      const float4 *lp = reinterpret_cast<const float4 *>(Ls + (y * W + xlo) * kTinyL) + lb;
      const float4 *rp =
          reinterpret_cast<const float4 *>(Rs + ((y - dy) * W + (xlo - dx)) * kTinyR) + rb;
#pragma unroll 4
      for (int x = xlo; x < xhi; ++x) {
        const float4 l = *lp, r = *rp;
        const float lv[4] = {l.x, l.y, l.z, l.w}, rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(lv[i], rv[j], acc[i][j]);
        lp += kTinyL / 4;
        rp += kTinyR / 4;
      }
    }
    const size_t o = size_t(dy + H - 1) * ndx + (dx + W - 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int l = l_base + 4 * lb + i;
      if (l >= a.nl) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = r_base + 4 * rb + j;
        if (r < a.nr) a.out[(size_t(l) * a.nr + r) * nunits + o] = acc[i][j];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// General fallback for matrices too wide to stage: a warp owns one pair group
// x one shift dy x 8 shifts dx; lanes sum interleaved rows; operands are read
// through L1 with bounds predicates instead of zero-padded shared rows.
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
  int groups_x;   // dx groups per output row: ceil((2W-1) / kDirectP)
  int pair_blocks;
  long long units;
};

__global__ void __launch_bounds__(32 * kDirectWarps) xcorr_direct_kernel(const DirectArgs a) {
  constexpr int P = kDirectP;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long unit = (long long)blockIdx.x * kDirectWarps + warp;
  if (unit >= a.units) return;
  const int oh = 2 * a.H - 1, ow = 2 * a.W - 1;
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
  for (int o = 1; o < ph_count; o <<= 1) {
#pragma unroll
    for (int p = 0; p < P; ++p) acc[p] += __shfl_xor_sync(0xffffffffu, acc[p], o);
  }
  if (!pair_ok) return;
  float *orow = a.out + size_t(pair) * oh * ow + size_t(oy) * ow;
  // every lane of the slot holds the totals; lane ph stores p = ph mod 32/G
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
  xcorr_direct_kernel<<<unsigned(blocks), 32 * kDirectWarps, 0, stream>>>(a);
  return cudaGetLastError();
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return sms > 0 ? sms : 1;
}

cudaError_t launch_tiny(const float *left, int nl, const float *right, int nr, int H,
                        int W, float *out, cudaStream_t stream) {
  TinyArgs a;
  a.left = left;
  a.right = right;
  a.out = out;
  a.nl = nl;
  a.nr = nr;
  a.H = H;
  a.W = W;
  a.lblocks = (nl + kTinyL - 1) / kTinyL;
  a.rblocks = (nr + kTinyR - 1) / kTinyR;
  const long long bp = (long long)a.lblocks * a.rblocks;
  const int nunits = (2 * H - 1) * (2 * W - 1);
  a.vec4 = ((H * W) % 4 == 0 && (reinterpret_cast<uintptr_t>(left) & 15) == 0 &&
            (reinterpret_cast<uintptr_t>(right) & 15) == 0) ? 1 : 0;
  long long nc = (sm_count() + bp - 1) / bp;
  if (nc > nunits) nc = nunits;
  if (nc < 1) nc = 1;
  a.nc = int(nc);
  const long long blocks = bp * a.nc;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = size_t(H) * W * (kTinyL + kTinyR) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(xcorr_tiny_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  xcorr_tiny_kernel<<<unsigned(blocks), 32 * kTinyWarps, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

// Temporary device memory for split-row partial sums: stream-ordered
// allocations from one library-owned pool per device whose release threshold
// is unlimited, so blocks freed by one call are reused by the next without
// going back to the driver.
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxDevices] = {};

cudaError_t scratch_pool(cudaMemPool_t *pool) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  if (!g_pools[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t p;
    if ((e = cudaMemPoolCreate(&p, &props)) != cudaSuccess) return e;
    uint64_t keep = ~uint64_t(0);
    if ((e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep)) !=
        cudaSuccess) {
      cudaMemPoolDestroy(p);
      return e;
    }
    g_pools[dev] = p;
  }
  *pool = g_pools[dev];
  return cudaSuccess;
}

cudaError_t scratch_alloc(float **ptr, size_t bytes, cudaStream_t stream) {
  cudaMemPool_t pool;
  cudaError_t e = scratch_pool(&pool);
  if (e != cudaSuccess) return e;
  return cudaMallocFromPoolAsync(reinterpret_cast<void **>(ptr), bytes, pool, stream);
}

}  // namespace

// Largest shared staging area of the rows / pair kernels (two CTAs per SM).
constexpr size_t kMaxStageSmem = 110 * 1024;

namespace {

// Which kernel a shape takes, its arguments and the split-row scratch it needs.
enum class XKind { Tiny, Pair, Rows, Direct };

struct XPlan {
  XKind kind;
  XArgs a;
  size_t smem;           // dynamic shared memory of the pair / rows kernel
  long long blocks;      // grid of the pair / rows kernel
  size_t part_bytes;     // rows kernel with several bands: scratch bytes
};

XPlan make_plan(const float *left, int nl, const float *right, int nr, int H, int W,
                float *out) {
  XPlan pl;
  pl.smem = 0;
  pl.blocks = 0;
  pl.part_bytes = 0;
  const long long pairs = (long long)nl * nr;
  XArgs &a = pl.a;
  a.left = left;
  a.right = right;
  a.out = out;
  a.nl = nl;
  a.nr = nr;
  a.H = H;
  a.W = W;
  if (H * W <= 256 && pairs >= 64) {
    pl.kind = XKind::Tiny;
    return pl;
  }
  const int need = kPadL + ((W + 3) & ~3) + kP + 8;
  a.S = ((need + 7) & ~7) + 4;
  a.dxbase = -(((W - 1) + 3) & ~3);
  a.ngroups = ((W - 1) - a.dxbase) / kP + 1;
  a.ndyb = (2 * H - 1 + kQ - 1) / kQ;
  a.nsuper = (a.ngroups + kWarps - 1) / kWarps;
  a.vec4 = ((W & 3) == 0 && (reinterpret_cast<uintptr_t>(left) & 15) == 0 &&
            (reinterpret_cast<uintptr_t>(right) & 15) == 0) ? 1 : 0;
  a.parts = 1;
  a.nbands = 1;
  a.part_row = 0;
  a.part = nullptr;

  // pair kernel: the whole pair fits, and there are enough rows per lane
  const size_t pair_smem = size_t(H + H + 2 * (kQ - 1)) * a.S * sizeof(float);
  if (pair_smem <= kMaxStageSmem && H >= 24) {
    const int items = a.ndyb * a.ngroups;
    long long parts = (4LL * sm_count() + pairs - 1) / pairs;
    const long long max_parts = (items + kWarps - 1) / kWarps;
    if (parts > max_parts) parts = max_parts;
    if (parts < 1) parts = 1;
    a.parts = int(parts);
    if (pairs * a.parts <= 0x7fffffffLL) {
      pl.kind = XKind::Pair;
      pl.smem = pair_smem;
      pl.blocks = pairs * a.parts;
      return pl;
    }
  }
  const size_t rows_smem = size_t(2 * kChunkRows) * a.S * sizeof(float);
  a.nbands = (H + kBandRows - 1) / kBandRows;
  a.part_row = kP * a.ngroups;
  const long long blocks = pairs * a.ndyb * a.nsuper * a.nbands;
  if (rows_smem > kMaxStageSmem || blocks > 0x7fffffffLL || H < 24) {
    pl.kind = XKind::Direct;
    return pl;
  }
  pl.kind = XKind::Rows;
  pl.smem = rows_smem;
  pl.blocks = blocks;
  if (a.nbands > 1)
    pl.part_bytes = size_t(pairs) * a.ndyb * a.nbands * kQ * a.part_row * sizeof(float);
  return pl;
}

// Launch a plan.  Split-row scratch comes from `fixed` (at least
// pl.part_bytes long) when given, else from the library's pool.
cudaError_t run_plan(XPlan &pl, float *fixed, cudaStream_t stream) {
  XArgs &a = pl.a;
  if (pl.kind == XKind::Tiny)
    return launch_tiny(a.left, a.nl, a.right, a.nr, a.H, a.W, a.out, stream);
  if (pl.kind == XKind::Direct)
    return launch_direct(a.left, a.nl, a.right, a.nr, a.H, a.W, a.out, stream);
  if (pl.kind == XKind::Pair) {
    cudaError_t e = cudaFuncSetAttribute(
        xcorr_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem));
    if (e != cudaSuccess) return e;
    xcorr_pair_kernel<<<unsigned(pl.blocks), kThreads, pl.smem, stream>>>(a);
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(
      xcorr_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem));
  if (e != cudaSuccess) return e;
  const bool banded = a.nbands > 1;
  const bool pooled = banded && fixed == nullptr;
  a.part = banded ? fixed : nullptr;
  if (pooled && (e = scratch_alloc(&a.part, pl.part_bytes, stream)) != cudaSuccess) return e;
  xcorr_rows_kernel<<<unsigned(pl.blocks), kThreads, pl.smem, stream>>>(a);
  e = cudaGetLastError();
  if (banded && e == cudaSuccess) {
    const long long outs = (long long)a.nl * a.nr * (2LL * a.H - 1) * (2LL * a.W - 1);
    const long long sum_blocks = (outs + 255) / 256;
    xcorr_band_sum_kernel<<<unsigned(sum_blocks < 65535 * 16 ? sum_blocks : 65535 * 16), 256, 0,
                            stream>>>(a);
    e = cudaGetLastError();
  }
  if (pooled) {
    const cudaError_t f = cudaFreeAsync(a.part, stream);
    if (e == cudaSuccess) e = f;
  }
  return e;
}

}  // namespace

cudaError_t xcorr_f32_launch(const float *left, int nl, const float *right,
                             int nr, int H, int W, float *out,
                             cudaStream_t stream) {
  XPlan pl = make_plan(left, nl, right, nr, H, W, out);
  return run_plan(pl, nullptr, stream);
}

size_t xcorr_f32_scratch_bytes(const float *left, int nl, const float *right, int nr,
                               int H, int W) {
  return make_plan(left, nl, right, nr, H, W, nullptr).part_bytes;
}

cudaError_t xcorr_f32_launch_scratch(const float *left, int nl, const float *right,
                                     int nr, int H, int W, float *out, float *scratch,
                                     size_t scratch_bytes, cudaStream_t stream) {
  XPlan pl = make_plan(left, nl, right, nr, H, W, out);
  if (pl.part_bytes > scratch_bytes || (pl.part_bytes > 0 && scratch == nullptr))
    return cudaErrorInvalidValue;
  return run_plan(pl, scratch, stream);
}

}  // namespace corr
