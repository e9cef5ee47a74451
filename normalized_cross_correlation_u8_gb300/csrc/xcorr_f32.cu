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
// overlaps (split-row).  The same ideas, laid out for sm_103a, in kernels
// chosen by shape:
//
//  rows  (every shape the next two do not take)
//    A CTA owns Q = 4 shifts dy x 8 warps x P = 8 shifts dx of one pair.
//    The overlap rows y are the reduction: lane i of every warp takes row i
//    of a 32-row chunk, so every lane runs the same x loop.  Rows are staged
//    whole into zero-padded shared rows, or, when too wide, as windows of
//    the columns the CTA's shifts touch in one x segment (no bounds tests in
//    the inner loop either way).  Row bands and x segments of one output
//    block are added in a fixed order by a second pass.
//  bcast (32+ rights per left) -- rights in lanes: every lane of a warp
//    walks the same left row against its own rights, no cross-lane sums.
//  tensor cores (xcorr_tc.cu; H, W <= 16, large batches) -- the n-to-m
//    batch as a dense contraction on the tensor cores with split TF32
//    operands; taken where it measured faster than the scalar kernels.
//  tensor cores, larger matrices (xcorr_tcl.cu; large one-to-one and
//    one-to-many batches) -- the same contraction per left, K cut into
//    units whose partial sums a second kernel adds in a fixed order.
//  warp per overlap (xcorr_warp.cu; single rows of 256+ samples) -- a
//    warp sums one overlap and reduces inside the warp.
//  tiny  (H*W <= 256, many pairs) -- a block of lefts x rights (32 x 16,
//    16 x 32, 8 x 64 or 64 x 8, whichever pads the batch least) is staged
//    interleaved (matrix index fastest); each lane owns 4 lefts x 4 rights
//    of one shift and walks that shift's exact overlap, so no product is
//    wasted; warps pull shifts from a per-CTA list.
//
// Per lane and overlap row (rows / bcast kernels): a float4 of L feeds 4 x
// steps; for each of the Q rows (or rights) a float4 of R enters a 12-entry
// register ring holding R[x-dx0-p] for the P shifts, indexed at
// compile-time positions by unrolling three 4-step blocks: 5 shared loads
// feed 4*P*Q = 128 FMAs.  When a chunk has fewer rows than lanes, each row
// is split into x sub-ranges over several lanes (split-row), and a shuffle
// butterfly adds the lanes' partial sums before the stores.
#include <cuda_runtime.h>
#include <stdint.h>

#include <stdlib.h>

#include <utility>

#include "internal.cuh"

namespace corr {
namespace {

constexpr int kP = 8;                // rows / bcast kernels: shifts dx per lane
constexpr int kQ = 4;                // rows kernel: shifts dy per lane
constexpr int kPadL = kP;            // bcast kernel: zero columns left of a row
constexpr int kWarps = 8;            // rows kernel
constexpr int kThreads = 32 * kWarps;

// rows kernel: shifts dx and dy per lane.
constexpr int kRowsP = kP;
constexpr int kRowsQ = kQ;

// k-th block in order of distance from the middle of n blocks (costly
// central blocks first).
__device__ __forceinline__ int centered(int k, int n) {
  const int m = (n - 1) >> 1;
  if (k == 0) return m;
  return (k & 1) ? m + ((k + 1) >> 1) : m - (k >> 1);
}

// ---------------------------------------------------------------------------
// Per-lane ring walk.  A lane owns P neighbouring shifts dx0 .. dx0+P-1 for
// NQ right rows; for each 4-wide x block it loads one float4 of L and one
// float4 of each right row into a register ring of P + 4 entries, so that
// R[x - dx0 - p] for every shift p sits at a compile-time ring position.
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

template <int P>
struct RingGeom {
  static constexpr int kSize = P + 4;                  // ring entries per row
  static constexpr int kCycle = kSize / 4;             // blocks per ring turn
  static constexpr int kRound = kCycle >= 4 ? kCycle : 2 * kCycle;   // unrolled blocks
  static_assert(P % 4 == 0, "ring of whole float4 blocks");
};

// Block J of a round: one float4 of L at la + 16 J, for each of the NQ rows a
// float4 of R_q at ra[q] + 16 J into ring positions 4 (J mod cycle) .. +3;
// shift p at step s reads position (4 (J mod cycle) + s - p) mod (P + 4).
template <int P, int J, int NQ>
__device__ __forceinline__ void ring_block(float (&acc)[NQ][P],
                                           float (&ring)[NQ][P + 4], uint32_t la,
                                           const uint32_t (&ra)[NQ]) {
  constexpr int RS = RingGeom<P>::kSize, JR = J % RingGeom<P>::kCycle;
  const float4 lv4 = lds128<16 * J>(la);
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
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
    for (int p = 0; p < P; ++p)
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        acc[q][p] = fmaf(lv[s], ring[q][(4 * JR + s - p + 2 * RS) % RS], acc[q][p]);
}

template <int P, int NQ, int... Js>
__device__ __forceinline__ void ring_round(float (&acc)[NQ][P], float (&ring)[NQ][P + 4],
                                           uint32_t la, const uint32_t (&ra)[NQ],
                                           std::integer_sequence<int, Js...>) {
  (ring_block<P, Js, NQ>(acc, ring, la, ra), ...);
}

// The first rem (< one round) blocks of a round.
template <int P, int NQ, int... Js>
__device__ __forceinline__ void ring_tail(float (&acc)[NQ][P], float (&ring)[NQ][P + 4],
                                          uint32_t la, const uint32_t (&ra)[NQ], int rem,
                                          std::integer_sequence<int, Js...>) {
  ((rem > Js ? ring_block<P, Js, NQ>(acc, ring, la, ra) : (void)0), ...);
}

// R_q[u0 + 4 b0 - P .. u0 + 4 b0 - 1] -> ring positions 4 .. P + 3.
template <int P, int NQ, int K>
__device__ __forceinline__ void ring_load(float (&ring)[NQ][P + 4], const uint32_t (&ra)[NQ]) {
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const float4 v = lds128<-16 * (P / 4 - K)>(ra[q]);
    ring[q][4 + 4 * K + 0] = v.x;
    ring[q][4 + 4 * K + 1] = v.y;
    ring[q][4 + 4 * K + 2] = v.z;
    ring[q][4 + 4 * K + 3] = v.w;
  }
}
template <int P, int NQ, int... Ks>
__device__ __forceinline__ void ring_preload(float (&ring)[NQ][P + 4],
                                             const uint32_t (&ra)[NQ],
                                             std::integer_sequence<int, Ks...>) {
  (ring_load<P, NQ, Ks>(ring, ra), ...);
#pragma unroll
  for (int q = 0; q < NQ; ++q) ring[q][0] = ring[q][1] = ring[q][2] = ring[q][3] = 0.f;
}

// Per-lane ring walk over x blocks [b0, b1) of one overlap row.
//   l4:    float4 index of L[xlo] in shared memory
//   r4[q]: float4 index of R_q[u0] (u0 = xlo - dx0) in shared memory; at
//          least P zero (or real) values precede it
// Block b covers x = xlo + 4b .. xlo + 4b + 3.  R_q[u0 + j] lives at ring
// position (j - 4 b0) mod (P + 4).
template <int P, int NQ>
__device__ __forceinline__ void lane_blocks(float (&acc)[NQ][P], int l4,
                                            const int (&r4)[NQ], int b0, int b1) {
  using G = RingGeom<P>;
  if (b0 >= b1) return;
  const uint32_t base = uint32_t(__cvta_generic_to_shared(g_smem4));
  float ring[NQ][G::kSize];
  uint32_t ra[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) ra[q] = base + 16u * uint32_t(r4[q] + b0);
  ring_preload<P, NQ>(ring, ra, std::make_integer_sequence<int, P / 4>{});
  uint32_t la = base + 16u * uint32_t(l4 + b0);
  int b = b0;
  for (; b + G::kRound <= b1; b += G::kRound) {
    ring_round<P, NQ>(acc, ring, la, ra, std::make_integer_sequence<int, G::kRound>{});
    la += 16 * G::kRound;
#pragma unroll
    for (int q = 0; q < NQ; ++q) ra[q] += 16 * G::kRound;
  }
  // 0 .. kRound-1 remaining blocks; ring positions continue (J mod cycle)
  ring_tail<P, NQ>(acc, ring, la, ra, b1 - b,
                   std::make_integer_sequence<int, G::kRound - 1>{});
}

// Geometry of one output block of a warp: shifts dy0..dy0+Q-1 x
// dx0..dx0+P-1.
struct Block {
  int dy0, dx0;
  int ylo, yhi;   // union of the overlap rows of the Q shifts dy
  int xlo, nb;    // first x (multiple of 4) and number of 4-wide x blocks
};

template <int P, int Q>
__device__ __forceinline__ Block make_block(int H, int W, int dy0, int dx0) {
  Block k;
  k.dy0 = dy0;
  k.dx0 = dx0;
  k.ylo = max(0, dy0);
  k.yhi = min(H, H + dy0 + Q - 1);
  k.xlo = max(0, dx0);
  const int xhi = min(W, W + dx0 + P - 1);
  k.nb = xhi > k.xlo ? (xhi - k.xlo + 3) >> 2 : 0;
  return k;
}

// One pass of up to NPH overlap rows [y, y + n) of a block over NPH lanes.
// lrow(y) / rrow(yr) give the float index of column 0 of a staged L row / R
// row (after its P zero columns).  With n >= NPH lane ph takes row y + ph;
// with fewer rows each row is split into k = NPH / n x sub-ranges (lanes
// past n*k idle).
template <int P, int Q, int NPH, typename LRow, typename RRow>
__device__ __forceinline__ void warp_pass(float (&acc)[Q][P], const Block &k, int y, int n,
                                          int ph, LRow lrow, RRow rrow) {
  if (n <= 0 || k.nb == 0) return;
  int row, b0, b1;
  if (n >= NPH) {
    row = y + ph;
    b0 = 0;
    b1 = k.nb;
  } else {
    const int parts = NPH / n;
    const int part = ph / n;
    if (part >= parts) return;
    row = y + (ph - part * n);
    b0 = part * k.nb / parts;
    b1 = (part + 1) * k.nb / parts;
  }
  const int u0 = k.xlo - k.dx0;
  const int l4 = (lrow(row) + k.xlo) >> 2;
  int r4[Q];
#pragma unroll
  for (int q = 0; q < Q; ++q) r4[q] = (rrow(row - k.dy0 - q) + u0) >> 2;
  lane_blocks<P, Q>(acc, l4, r4, b0, b1);
}

// Reduce-scatter over groups of NPH lanes (lanes of a group differ in their
// low log2(NPH) bits): after log2(NPH) steps of halving, lane ph of a group
// holds the group's full sums of outputs (32/NPH) * ph + i, i < 32/NPH, in
// out[i] (output index q * P + p).  Clears the accumulators.
template <int P, int Q, int NPH>
__device__ __forceinline__ void reduce_scatter_group(float (&acc)[Q][P], int lane,
                                                     float (&out)[32 / NPH]) {
  static_assert(P * Q == 32, "32 outputs per block");
  float v[32];
#pragma unroll
  for (int q = 0; q < Q; ++q)
#pragma unroll
    for (int p = 0; p < P; ++p) v[q * P + p] = acc[q][p];
#pragma unroll
  for (int o = NPH / 2, m = 16; o >= 1; o >>= 1, m >>= 1) {
    const bool upper = (lane & o) != 0;   // keep v[m..2m) if set, else v[0..m)
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float send = upper ? v[i] : v[i + m];
      const float keep = upper ? v[i + m] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
#pragma unroll
  for (int i = 0; i < 32 / NPH; ++i) out[i] = v[i];
#pragma unroll
  for (int q = 0; q < Q; ++q)
#pragma unroll
    for (int p = 0; p < P; ++p) acc[q][p] = 0.f;
}

// Reduce-scatter over the 32 lanes: at each step a lane keeps one half of
// its remaining partial sums and adds the partner's copy of that half, so
// after 16 + 8 + 4 + 2 + 1 shuffles lane i holds the full sum of output
// i = q * P + p.  Returns it and clears the accumulators.
template <int P, int Q>
__device__ __forceinline__ float reduce_scatter(float (&acc)[Q][P], int lane) {
  float v[1];
  reduce_scatter_group<P, Q, 32>(acc, lane, v);
  return v[0];
}

// Reduce and store the block's outputs into out_pair ([2H-1][2W-1]).
template <int P, int Q>
__device__ __forceinline__ void reduce_store(float (&acc)[Q][P], const Block &k, int lane,
                                             int H, int W, float *out_pair) {
  const float v = reduce_scatter<P, Q>(acc, lane);
  const int dy = k.dy0 + lane / P, dx = k.dx0 + lane % P;
  if (dy > -H && dy < H && dx > -W && dx < W)
    out_pair[size_t(dy + H - 1) * (2 * W - 1) + (dx + W - 1)] = v;
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
  int vec4;       // rows can be read as float4
  int nbands;     // rows kernel: row bands (split-row)
  int band_rows;  // rows kernel: overlap rows per band
  int nxseg;      // rows kernel: x segments (split-row along x)
  int xseg;       // rows kernel: columns per x segment (multiple of 4)
  int SL, SR;     // rows kernel: shared L / R row strides in floats (% 8 == 4)
  long long items; // rows kernels: work items (CTAs loop over them)
  int part_row;   // rows kernel: floats per partial-sum row (P * ngroups)
  float *part;    // rows kernel: partial sums (nbands * nxseg > 1)
  int nrblk;      // bcast kernel: blocks of 32 rights
  int npairblk;   // bcast kernel: blocks of kWarps dx-group pairs
};

// ---------------------------------------------------------------------------
// rows kernel: one CTA = one pair x Q shifts dy x 8 warps' dx groups (P
// shifts each) x one band of overlap rows x one segment of x (split-row in
// both directions: the partial sums of a block are added afterwards in a
// fixed order, so results do not depend on scheduling).
//
// The CTA's groups cover shifts DX0 .. DX0 + 8P - 1; the L columns any of
// them touches inside the segment form the window [xa, xb), and the R
// columns they pair with form [xa - DX0 - 8P, xb - DX0 + 4).  Only these
// windows are staged, 32 overlap rows at a time, with cp.async into one
// shared buffer (columns outside the matrix, or past the segment for L,
// arrive as zeros, so the inner loop has no bounds tests).  Lane i of every
// warp takes overlap row i of the chunk and walks its group's whole x range
// inside the window, so a walk is long beside the per-chunk costs (staging,
// barrier, walk set-up).  Two CTAs share an SM, so one computes while the
// other waits for its chunk.  With one band and one segment the CTA writes
// the outputs directly; otherwise it writes its partial sums to
//   part[(slot * Q + q) * part_row + P * group + p],
//   slot = ((pair * ndyb + dyb) * nbands + band) * nxseg + xseg.
// ---------------------------------------------------------------------------
constexpr int kChunk = 32;
#ifndef CORR_XC_BANDROWS
#define CORR_XC_BANDROWS 128
#endif
#ifndef CORR_XC_BANDMIN
#define CORR_XC_BANDMIN 16
#endif
constexpr int kBandRows = CORR_XC_BANDROWS;   // band height when bands are needed
constexpr int kBandMinCtasPerSm = CORR_XC_BANDMIN;   // fewer unbanded CTAs per SM: bands

template <int Q, int CH = kChunk>
struct ChunkGeom {
  static_assert(CH == 16 || CH == 32, "a chunk's rows spread evenly over the lanes");
  static constexpr int kL = CH, kR = CH + Q - 1, kRows = kL + kR;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const float *src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const float *src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async(uint32_t dst, const float *src, bool valid,
                                         bool vec4) {
  if (vec4)
    cp_async16(dst, src, valid ? 16 : 0);
  else
    cp_async4(dst, src, valid);
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

// L window [xa, xb) of CTA column dxs in x segment xseg (empty if xa >= xb).
// xa is a multiple of 4.
__host__ __device__ inline void rows_window(int W, int dxbase, int P, int dxs, int xseg,
                                            int seg, int &xa, int &xb) {
  const int dx_first = dxbase + dxs * kWarps * P;
  const int dx_last = dx_first + kWarps * P - 1;
  const int xs0 = xseg * seg, xs1 = min(W, xs0 + seg);
  xa = max(xs0, max(0, dx_first));
  xb = min(xs1, W + dx_last);
}

// Copy one row window of n4 float4 slots starting at column c0 of global row
// `row` to shared byte address d; columns outside [lo, hi), and every column
// when !row_ok, arrive as zeros (their copies read nothing; `row` is still a
// valid address).  One warp.
__device__ __forceinline__ void stage_window(uint32_t d, const float *row, bool row_ok, int c0,
                                             int n4, int lo, int hi, bool vec4, int lane) {
  if (vec4) {
    // c0, lo and the row start are 16-byte aligned, hi may not be (an L
    // window ending at W + dx): a slot is whole, partial or empty
    for (int c = lane; c < n4; c += 32) {
      const int x = c0 + 4 * c;
      int bytes = 0;
      if (row_ok && x >= lo) bytes = 4 * max(0, min(4, hi - x));
      cp_async16(d + 16u * uint32_t(c), row + (bytes ? x : 0), bytes);
    }
  } else {
    for (int c = lane; c < 4 * n4; c += 32) {
      const int x = c0 + c;
      const bool ok = row_ok && x >= lo && x < hi;
      cp_async4(d + 4u * uint32_t(c), row + (ok ? x : 0), ok);
    }
  }
}

// Full-row variant for rows narrow enough that CH whole rows of L and R fit:
// rows are staged at column P of a zero-padded shared row of stride S (the
// padding is zeroed once), and every warp reads the same rows.  No x
// segments; partial sums (bands only) use the same slots with xseg = 0.
template <int Q, int CH>
__device__ __forceinline__ void issue_rows(uint32_t sbase, int S, int pad, int W, bool vec4,
                                           const float *L, const float *R, int yc, int y_end,
                                           int yr_first, int H) {
  using C = ChunkGeom<Q, CH>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int step = vec4 ? 4 : 1, n = vec4 ? (W >> 2) : W;
  for (int r = warp; r < C::kRows; r += kWarps) {
    const float *src;
    bool ok;
    if (r < C::kL) {
      const int y = yc + r;
      ok = y < y_end;
      src = L + (ok ? size_t(y) * W : 0);
    } else {
      const int yr = yr_first + (r - C::kL);
      ok = yr >= 0 && yr < H;
      src = R + (ok ? size_t(yr) * W : 0);
    }
    const uint32_t d = sbase + 4u * uint32_t(r * S + pad);
    for (int c = lane; c < n; c += 32)
      cp_async(d + 4u * uint32_t(c * step), src + c * step, ok, vec4);
  }
}

// One work item (pair, dy block, CTA column of dx groups, band) of the
// whole-row kernel.  The staging buffer's padding is zero on entry.
template <int P, int Q, int CH, typename Index>
__device__ __forceinline__ void rows_item(const XArgs &a, Index item) {
  using C = ChunkGeom<Q, CH>;
  const uint32_t sbase = uint32_t(__cvta_generic_to_shared(g_smem4));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, W = a.W, S = a.S;
  const int band = int(item % a.nbands);
  item /= a.nbands;
  const int pair = int(item % (a.nl * a.nr));
  item /= a.nl * a.nr;
  const int dyb = centered(int(item % a.ndyb), a.ndyb);
  const int dxs = centered(int(item / a.ndyb), a.nsuper);
  const int li = pair / a.nr, ri = pair - li * a.nr;
  const size_t mat = size_t(H) * W;
  const float *L = a.left + li * mat;
  const float *R = a.right + ri * mat;

  const int group = dxs * kWarps + warp;
  const bool active = group < a.ngroups;
  const int dy0 = dyb * Q - (H - 1);
  const Block k = make_block<P, Q>(H, W, dy0, a.dxbase + group * P);
  // every group of the CTA shares dy0, hence the overlap rows
  const int y_begin = max(k.ylo, band * a.band_rows);
  const int y_end = min(k.yhi, (band + 1) * a.band_rows);
  if (y_begin >= y_end) return;           // CTA-uniform: this band is empty

  float acc[Q][P];
#pragma unroll
  for (int q = 0; q < Q; ++q)
#pragma unroll
    for (int p = 0; p < P; ++p) acc[q][p] = 0.f;

  const int nchunks = (y_end - y_begin + CH - 1) / CH;
  for (int c = 0; c < nchunks; ++c) {
    const int yc = y_begin + c * CH;
    const int yr_first = yc - dy0 - (Q - 1);
    __syncthreads();            // the buffer is free (the previous chunk consumed)
    issue_rows<Q, CH>(sbase, S, P, W, a.vec4, L, R, yc, y_end, yr_first, H);
    cp_async_commit();
    cp_async_wait_all();        // this thread's copies have landed
    __syncthreads();            // ... and everyone's
    if (active)
      warp_pass<P, Q, 32>(acc, k, yc, min(CH, y_end - yc), lane,
                          [&](int y) { return (y - yc) * S + P; },
                          [&](int yr) { return (C::kL + yr - yr_first) * S + P; });
  }
  if (!active) return;
  if (a.nbands == 1) {
    reduce_store<P, Q>(acc, k, lane, H, W, a.out + size_t(pair) * (2 * H - 1) * (2 * W - 1));
  } else {
    const float v = reduce_scatter<P, Q>(acc, lane);
    const size_t slot = (size_t(pair) * a.ndyb + dyb) * a.nbands + band;
    a.part[(slot * Q + lane / P) * a.part_row + group * P + lane % P] = v;
  }
}

// LOOP = false: one item per CTA (grid = items < 2^30, 32-bit indices);
// LOOP = true: CTAs loop over more items than a grid holds.
template <int P, int Q, int CH, bool LOOP>
__global__ void __launch_bounds__(kThreads, 2) xcorr_rows_kernel(const XArgs a) {
  zero_smem(reinterpret_cast<float *>(g_smem4), ChunkGeom<Q, CH>::kRows * a.S);   // padding
  if (LOOP) {
    for (long long it = blockIdx.x; it < a.items; it += gridDim.x)
      rows_item<P, Q, CH, long long>(a, it);
  } else {
    rows_item<P, Q, CH, int>(a, int(blockIdx.x));
  }
}

// One work item (pair, dy block, CTA column of dx groups, x segment, band)
// of the windowed variant (any width).
template <int P, int Q, typename Index>
__device__ __forceinline__ void rows_win_item(const XArgs &a, Index item) {
  using C = ChunkGeom<Q>;
  const uint32_t sbase = uint32_t(__cvta_generic_to_shared(g_smem4));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, W = a.W, SL = a.SL, SR = a.SR;
  const int band = int(item % a.nbands);
  item /= a.nbands;
  const int xseg = int(item % a.nxseg);
  item /= a.nxseg;
  const int pair = int(item % (a.nl * a.nr));
  item /= a.nl * a.nr;
  const int dyb = centered(int(item % a.ndyb), a.ndyb);
  const int dxs = centered(int(item / a.ndyb), a.nsuper);
  const int li = pair / a.nr, ri = pair - li * a.nr;
  const size_t mat = size_t(H) * W;
  const float *L = a.left + li * mat;
  const float *R = a.right + ri * mat;

  const int dy0 = dyb * Q - (H - 1);
  // every group of the CTA shares dy0, hence the overlap rows
  const int y_begin = max(max(0, dy0), band * a.band_rows);
  const int y_end = min(min(H, H + dy0 + Q - 1), (band + 1) * a.band_rows);
  int xa, xb;
  rows_window(W, a.dxbase, P, dxs, xseg, a.xseg, xa, xb);
  if (y_begin >= y_end || xa >= xb) return;   // CTA-uniform: nothing to add here

  const int DX0 = a.dxbase + dxs * kWarps * P;
  const int nl4 = (xb - xa + 3) >> 2;         // L slots; block reads stay inside
  const int nr4 = nl4 + 2 * P;                // R slots from ua = xa - DX0 - 8P
  const int ua = xa - DX0 - kWarps * P;
  const int r_base = C::kL * SL;              // float index of the first R row

  const int group = dxs * kWarps + warp;
  const bool active = group < a.ngroups;
  Block k = make_block<P, Q>(H, W, dy0, a.dxbase + group * P);
  {
    // the group's x range clipped to the window
    const int xhi = min(min(W, W + k.dx0 + P - 1), xb);
    k.xlo = max(k.xlo, xa);
    k.nb = xhi > k.xlo ? (xhi - k.xlo + 3) >> 2 : 0;
  }
  float acc[Q][P];
#pragma unroll
  for (int q = 0; q < Q; ++q)
#pragma unroll
    for (int p = 0; p < P; ++p) acc[q][p] = 0.f;

  const bool vec4 = a.vec4;
  const int nchunks = (y_end - y_begin + kChunk - 1) / kChunk;
  for (int c = 0; c < nchunks; ++c) {
    const int yc = y_begin + c * kChunk;
    const int yr_first = yc - dy0 - (Q - 1);
    __syncthreads();                // the previous chunk (of this or an earlier item) is consumed
    for (int r = warp; r < C::kL + C::kR; r += kWarps) {
      if (r < C::kL) {
        const int y = yc + r;
        const bool ok = y < y_end;
        stage_window(sbase + 4u * uint32_t(r * SL), L + (ok ? size_t(y) * W : 0), ok, xa, nl4,
                     xa, xb, vec4, lane);
      } else {
        const int yr = yr_first + (r - C::kL);
        const bool ok = yr >= 0 && yr < H;
        stage_window(sbase + 4u * uint32_t(r_base + (r - C::kL) * SR),
                     R + (ok ? size_t(yr) * W : 0), ok, ua, nr4, 0, W, vec4, lane);
      }
    }
    cp_async_commit();
    cp_async_wait_all();            // this thread's copies have landed
    __syncthreads();                // ... and everyone's
    if (active)
      warp_pass<P, Q, 32>(acc, k, yc, min(kChunk, y_end - yc), lane,
                          [&](int y) { return (y - yc) * SL - xa; },
                          [&](int yr) { return r_base + (yr - yr_first) * SR - ua; });
  }
  if (!active) return;
  if (a.nbands * a.nxseg == 1) {
    reduce_store<P, Q>(acc, k, lane, H, W, a.out + size_t(pair) * (2 * H - 1) * (2 * W - 1));
  } else {
    const float v = reduce_scatter<P, Q>(acc, lane);
    const size_t slot = ((size_t(pair) * a.ndyb + dyb) * a.nbands + band) * a.nxseg + xseg;
    a.part[(slot * Q + lane / P) * a.part_row + group * P + lane % P] = v;
  }
}

template <int P, int Q, bool LOOP>
__global__ void __launch_bounds__(kThreads, 2) xcorr_rows_win_kernel(const XArgs a) {
  if (LOOP) {
    for (long long it = blockIdx.x; it < a.items; it += gridDim.x)
      rows_win_item<P, Q, long long>(a, it);
  } else {
    rows_win_item<P, Q, int>(a, int(blockIdx.x));
  }
}

// Second pass of the rows kernel: out = sum of the partial sums of the
// (band, segment) CTAs that ran, in band-then-segment order.
template <int P, int Q>
__global__ void xcorr_band_sum_kernel(const XArgs a) {
  const int H = a.H, W = a.W, oh = 2 * H - 1, ow = 2 * W - 1;
  const long long total = (long long)a.nl * a.nr * oh * ow;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int ox = int(i % ow);
    const long long t = i / ow;
    const int oy = int(t % oh);
    const int pair = int(t / oh);
    const int dyb = oy / Q, q = oy - dyb * Q;
    const int dy0 = dyb * Q - (H - 1);
    const int ylo = max(0, dy0), yhi = min(H, H + dy0 + Q - 1);
    const int col = (ox - (W - 1)) - a.dxbase;
    const int dxs = (col / P) / kWarps;
    const size_t slot0 = (size_t(pair) * a.ndyb + dyb) * a.nbands;
    float sum = 0.f;
    for (int b = 0; b < a.nbands; ++b) {
      if (max(ylo, b * a.band_rows) >= min(yhi, (b + 1) * a.band_rows)) continue;
      for (int s = 0; s < a.nxseg; ++s) {
        int xa, xb;
        rows_window(W, a.dxbase, P, dxs, s, a.xseg, xa, xb);
        if (xa >= xb) continue;
        sum += a.part[(((slot0 + b) * a.nxseg + s) * Q + q) * a.part_row + col];
      }
    }
    a.out[i] = sum;
  }
}

// ---------------------------------------------------------------------------
// bcast kernel ("rights in lanes": one-to-many and n-to-m with >= 32 rights
// per left).  A CTA owns one left, 32 rights (one per lane), one shift dy
// and kWarps pairs of dx groups.  Lane r of every warp owns right r, so all
// lanes of a warp share one left row (a broadcast load), one y range (the
// exact overlap rows of dy) and one x range: control flow is uniform and
// every lane sums all rows of its outputs itself -- no cross-lane reduction.
// Warp w takes dx groups g = w and g + ceil(G/2), whose x ranges add up to
// about W, so the warps of a CTA carry equal work between chunk barriers.  Overlap
// rows are staged kBRows at a time (left rows, then per right a slab of
// kBRows rows padded to an odd number of 16-byte units) with cp.async into
// two buffers.
// ---------------------------------------------------------------------------
#ifndef CORR_XC_BROWS
#define CORR_XC_BROWS 4
#endif
#ifndef CORR_XC_BMINB
#define CORR_XC_BMINB 1
#endif
constexpr int kBRows = CORR_XC_BROWS;     // overlap rows per chunk
static_assert(kBRows % 2 == 0, "two row halves");
#ifndef CORR_XC_BPAIRS
#define CORR_XC_BPAIRS 8
#endif
constexpr int kBWarps = 2 * kWarps;              // row parts x group pairs
constexpr int kBPairs = CORR_XC_BPAIRS;          // dx-group pairs per CTA
constexpr int kBParts = kBWarps / kBPairs;       // row parts of a chunk
static_assert(kBRows % kBParts == 0, "whole rows per row part");

// BR rights per lane (2, or 1 when that still leaves fewer CTAs than two
// per SM): 1 + 32 BR matrices staged per chunk.
__host__ __device__ inline int bcast_slab(int S) { return kBRows * S + 4; }
__host__ __device__ inline int bcast_buf(int S, int BR) {
  return kBRows * S + 32 * BR * bcast_slab(S);
}

// Issue one chunk: left rows yc .. yc+kBRows-1 (zero past yhi) and, for each
// of the CTA's 32*BR rights, rows yc-dy .. (zero past nr or past yhi).
// A row's addresses are formed once: a row of n copies goes to the smallest
// of 4, 8, 16 or 32 lanes that covers it (lanes along the row).
template <int BR>
__device__ __forceinline__ void issue_bchunk(const XArgs &a, uint32_t sbase, int buf,
                                             const float *L, int r_first, int yc,
                                             int yhi, int dy) {
  const int W = a.W, S = a.S, H = a.H;
  const bool vec4 = a.vec4;
  const int step = vec4 ? 4 : 1, n = vec4 ? (W >> 2) : W;
  const size_t mat = size_t(H) * W;
  const int slab = bcast_slab(S);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lpr = n <= 4 ? 4 : n <= 8 ? 8 : n <= 16 ? 16 : 32;   // lanes per row
  const int rpw = 32 / lpr;                     // rows per warp step
  const int sub = lane / lpr, col0 = lane % lpr;
  for (int row = warp * rpw + sub; row < (1 + 32 * BR) * kBRows; row += kBWarps * rpw) {
    const int m = row / kBRows, r = row % kBRows;
    const int y = yc + r;
    bool ok = y < yhi;
    const float *src;
    int dst;
    if (m == 0) {
      src = L + (ok ? size_t(y) * W : 0);
      dst = buf + r * S + kPadL;
    } else {
      const int ri = r_first + (m - 1);
      ok = ok && ri < a.nr;
      src = a.right + (ok ? size_t(ri) * mat + size_t(y - dy) * W : 0);
      dst = buf + kBRows * S + (m - 1) * slab + r * S + kPadL;
    }
    const uint32_t d = sbase + 4u * uint32_t(dst);
    for (int c = col0; c < n; c += lpr)
      cp_async(d + 4u * uint32_t(c * step), src + c * step, ok, vec4);
  }
}

// x geometry of one dx group: first x (multiple of 4), u0 = xlo - dx0, and
// number of 4-wide blocks of the union of its 8 shifts' overlaps.
struct XGroup {
  int dx0, xlo, u0, nb;
};

__device__ __forceinline__ XGroup make_xgroup(int W, int dx0) {
  XGroup g;
  g.dx0 = dx0;
  g.xlo = max(0, dx0);
  g.u0 = g.xlo - dx0;
  const int xhi = min(W, W + dx0 + kP - 1);
  g.nb = xhi > g.xlo ? (xhi - g.xlo + 3) >> 2 : 0;
  return g;
}


template <int BR>
__global__ void __launch_bounds__(32 * kBWarps, CORR_XC_BMINB) xcorr_bcast_kernel(const XArgs a) {
  constexpr int kBRights = BR;
  const uint32_t sbase = uint32_t(__cvta_generic_to_shared(g_smem4));
  float *sm = reinterpret_cast<float *>(g_smem4);
  const int warp_id = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int warp = warp_id % kBPairs;   // dx-group pair of this warp
  const int rh = warp_id / kBPairs;     // row part: rows rh * kBRows / kBParts .. of a chunk
  const int H = a.H, W = a.W, S = a.S;
  const int G = a.ngroups, ngp = (G + 1) / 2;
  int item = blockIdx.x;
  const int rb = item % a.nrblk;
  item /= a.nrblk;
  const int li = item % a.nl;
  item /= a.nl;
  const int pbk = item % a.npairblk;
  item /= a.npairblk;
  const int dy = centered(item, 2 * H - 1) - (H - 1);   // costly (central) dy first
  const int ylo = max(0, dy), yhi = min(H, H + dy);
  const float *L = a.left + size_t(li) * H * W;

  // groups g and g + ngp: shifts dx and dx + 8*ngp (about dx + W), whose x
  // ranges add up to about W, so every warp carries the same work
  const int gp = pbk * kBPairs + warp;
  const bool gp_ok = gp < ngp;
  const int gA = gp, gB = gp + ngp;
  const bool has_b = gp_ok && gB < G;
  const XGroup xa = make_xgroup(W, a.dxbase + gA * kP);
  const XGroup xb = make_xgroup(W, a.dxbase + gB * kP);
  const int r_first = rb * 32 * kBRights;   // lane owns rights r_first + lane + 32 j

  const int bufn = bcast_buf(S, BR), slab = bcast_slab(S);
  zero_smem(sm, 2 * bufn);
  __syncthreads();
  float accA[kBRights][kP], accB[kBRights][kP];
#pragma unroll
  for (int j = 0; j < kBRights; ++j)
#pragma unroll
    for (int p = 0; p < kP; ++p) accA[j][p] = accB[j][p] = 0.f;

  const int nchunks = (yhi - ylo + kBRows - 1) / kBRows;
  if (nchunks > 0) issue_bchunk<BR>(a, sbase, 0, L, r_first, ylo, yhi, dy);
  cp_async_commit();
  for (int c = 0; c < nchunks; ++c) {
    const int yc = ylo + c * kBRows;
    const int buf = (c & 1) * bufn;
    cp_async_wait_all();
    __syncthreads();
    if (c + 1 < nchunks) {
      issue_bchunk<BR>(a, sbase, ((c + 1) & 1) * bufn, L, r_first, yc + kBRows, yhi, dy);
      cp_async_commit();
    }
    if (!gp_ok) continue;
    const int rows = min(kBRows, yhi - yc);
    for (int k = rh * (kBRows / kBParts); k < min(rows, (rh + 1) * (kBRows / kBParts)); ++k) {
      const int lrow = buf + k * S + kPadL;
      const int rrow = buf + kBRows * S + lane * slab + k * S + kPadL;
      {
        int r4[kBRights];
#pragma unroll
        for (int j = 0; j < kBRights; ++j) r4[j] = (rrow + 32 * j * slab + xa.u0) >> 2;
        lane_blocks<kP, kBRights>(accA, (lrow + xa.xlo) >> 2, r4, 0, xa.nb);
      }
      if (has_b) {
        int r4[kBRights];
#pragma unroll
        for (int j = 0; j < kBRights; ++j) r4[j] = (rrow + 32 * j * slab + xb.u0) >> 2;
        lane_blocks<kP, kBRights>(accB, (lrow + xb.xlo) >> 2, r4, 0, xb.nb);
      }
    }
  }
  // row parts 1.. hand their partial sums to row part 0, which adds them in
  // part order (the same result on every run)
  __syncthreads();                       // chunk buffers are free again
  constexpr int kPart = 2 * kBRights * kP;   // partial sums per lane
  if (rh > 0) {
    float *part = sm + (((rh - 1) * kBPairs + warp) * kPart) * 32 + lane;
#pragma unroll
    for (int j = 0; j < kBRights; ++j)
#pragma unroll
      for (int p = 0; p < kP; ++p) {
        part[(j * kP + p) * 32] = accA[j][p];
        part[((kBRights + j) * kP + p) * 32] = accB[j][p];
      }
  }
  __syncthreads();
  if (rh > 0 || !gp_ok) return;
#pragma unroll
  for (int q = 1; q < kBParts; ++q) {
    const float *part = sm + (((q - 1) * kBPairs + warp) * kPart) * 32 + lane;
#pragma unroll
    for (int j = 0; j < kBRights; ++j)
#pragma unroll
      for (int p = 0; p < kP; ++p) {
        accA[j][p] += part[(j * kP + p) * 32];
        accB[j][p] += part[((kBRights + j) * kP + p) * 32];
      }
  }
  const int OW = 2 * W - 1;
#pragma unroll
  for (int j = 0; j < kBRights; ++j) {
    const int ri = r_first + lane + 32 * j;
    if (ri >= a.nr) continue;
    float *orow = a.out + (size_t(li) * a.nr + ri) * size_t(2 * H - 1) * OW +
                  size_t(dy + H - 1) * OW;
#pragma unroll
    for (int p = 0; p < kP; ++p) {
      const int dx = xa.dx0 + p;
      if (dx > -W && dx < W) orow[dx + W - 1] = accA[j][p];
    }
    if (has_b) {
#pragma unroll
      for (int p = 0; p < kP; ++p) {
        const int dx = xb.dx0 + p;
        if (dx > -W && dx < W) orow[dx + W - 1] = accB[j][p];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// tiny kernel: H*W <= 256.  A CTA stages a block of kTinyL lefts and kTinyR
// rights (32 x 16, 16 x 32, 8 x 64 or 64 x 8) interleaved as
// [y][x][matrix]; lane (lb = lane % (kTinyL/4), rb = lane / (kTinyL/4)) owns
// lefts 4lb..4lb+3 x rights 4rb..4rb+3 of one shift and walks its exact overlap:
// per (y, x) two 16-byte loads feed 16 FMAs.  Shifts are dealt to the CTAs
// of a block pair in snake order over a centre-first ranking and pulled by
// the CTA's warps from a shared counter.
// ---------------------------------------------------------------------------
constexpr int kTinyWarps = 16;

struct TinyArgs {
  const float *left;
  const float *right;
  float *out;
  int nl, nr, H, W;
  int lblocks, rblocks;  // blocks of kTinyL lefts / kTinyR rights
  int nc;                // CTAs sharing one block pair
  int vec4;              // matrices can be read as float4 (H*W % 4 == 0, aligned)
};

// kTinyL x kTinyR: the block of lefts x rights a CTA stages; a lane owns 4
// x 4 of them, so (kTinyL / 4) * (kTinyR / 4) = 32.
template <int kTinyL, int kTinyR>
__global__ void __launch_bounds__(32 * kTinyWarps) xcorr_tiny_kernel(const TinyArgs a) {
  static_assert((kTinyL / 4) * (kTinyR / 4) == 32, "one 4 x 4 block per lane");
  float *Ls = reinterpret_cast<float *>(g_smem4);
  const int H = a.H, W = a.W, HW = H * W;
  float *Rs = Ls + HW * kTinyL;
  __shared__ int next_unit;
  int bid = blockIdx.x;
  const int c = bid % a.nc;
  bid /= a.nc;
  const int rbk = bid % a.rblocks, lbk = bid / a.rblocks;
  const int l_base = lbk * kTinyL, r_base = rbk * kTinyR;

  // stage: item (m, p4) = 16 bytes (positions 4 p4 .. +3) of matrix m,
  // scattered to Xs[pos * NB + m]; lanes of a warp take consecutive m, so
  // each shared store hits 32 distinct banks.  Four items' loads are issued
  // before their stores so their latencies overlap.
  {
    const int hw4 = (HW + 3) >> 2;
    auto stage = [&](float *Xs, const float *src0, int base_m, int nmat, int NB) {
      const int items = hw4 * NB;
      for (int i0 = threadIdx.x; i0 < items; i0 += 4 * blockDim.x) {
        float e[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = i0 + k * blockDim.x;
          const int m = i % NB, p4 = i / NB;
          const int mm = base_m + m;
#pragma unroll
          for (int t = 0; t < 4; ++t) e[k][t] = 0.f;
          if (i < items && mm < nmat) {
            const float *src = src0 + size_t(mm) * HW + 4 * p4;
            if (a.vec4) {
              const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
              e[k][0] = v.x; e[k][1] = v.y; e[k][2] = v.z; e[k][3] = v.w;
            } else {
#pragma unroll
              for (int t = 0; t < 4; ++t) e[k][t] = 4 * p4 + t < HW ? __ldg(src + t) : 0.f;
            }
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = i0 + k * blockDim.x;
          if (i >= items) break;
          const int m = i % NB, p4 = i / NB;
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (4 * p4 + t < HW) Xs[(4 * p4 + t) * NB + m] = e[k][t];
        }
      }
    };
    stage(Ls, a.left, l_base, a.nl, kTinyL);
    stage(Rs, a.right, r_base, a.nr, kTinyR);
  }
  if (threadIdx.x == 0) next_unit = 0;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int lb = lane % (kTinyL / 4), rb = lane / (kTinyL / 4);
  const int ndy = 2 * H - 1, ndx = 2 * W - 1, nunits = ndy * ndx;
  // this CTA's units: rank j * nc + (j even ? c : nc - 1 - c) of the
  // centre-first order (snake order: every CTA gets a similar mix of costs)
  const int rounds = nunits / a.nc, rem = nunits - rounds * a.nc;
  const int mine = rounds + (((rounds & 1) ? a.nc - 1 - c : c) < rem ? 1 : 0);
  for (;;) {
    int u = 0;
    if (lane == 0) u = atomicAdd(&next_unit, 1);
    u = __shfl_sync(0xffffffffu, u, 0);
    if (u >= mine) break;
    const int kk = u * a.nc + ((u & 1) ? a.nc - 1 - c : c);   // centre-first rank
    const int dy = centered(kk % ndy, ndy) - (H - 1);
    const int dx = centered(kk / ndy, ndx) - (W - 1);
    const int ylo = max(0, dy), yhi = min(H, H + dy);
    const int xlo = max(0, dx), xhi = min(W, W + dx);
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    const int nx = xhi - xlo;
    for (int y = ylo; y < yhi; ++y) {
      const float4 *lp = reinterpret_cast<const float4 *>(Ls + (y * W + xlo) * kTinyL) + lb;
      const float4 *rp =
          reinterpret_cast<const float4 *>(Rs + ((y - dy) * W + (xlo - dx)) * kTinyR) + rb;
      // the next step's operands are loaded while this step's FMAs run
      float4 l = lp[0], r = rp[0];
      for (int t = 0; t < nx; ++t) {
        float4 ln = l, rn = r;
        if (t + 1 < nx) {
          ln = lp[(t + 1) * (kTinyL / 4)];
          rn = rp[(t + 1) * (kTinyR / 4)];
        }
        const float lv[4] = {l.x, l.y, l.z, l.w}, rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(lv[i], rv[j], acc[i][j]);
        l = ln;
        r = rn;
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

int sm_count() { return device_sm_count(); }

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
  // block shape: the one of 32 x 16, 16 x 32, 8 x 64 and 64 x 8 lefts x
  // rights that pads the batch least (32 x 16 on ties)
  static const int shapes[4][2] = {{32, 16}, {16, 32}, {8, 64}, {64, 8}};
  int best = 0;
  long long best_pad = -1;
  for (int i = 0; i < 4; ++i) {
    const long long tl = shapes[i][0], tr = shapes[i][1];
    const long long pad = ((nl + tl - 1) / tl) * tl * ((nr + tr - 1) / tr) * tr;
    if (best_pad < 0 || pad < best_pad) {
      best_pad = pad;
      best = i;
    }
  }
  const int kTinyL = shapes[best][0], kTinyR = shapes[best][1];
  a.lblocks = (nl + kTinyL - 1) / kTinyL;
  a.rblocks = (nr + kTinyR - 1) / kTinyR;
  const long long bp = (long long)a.lblocks * a.rblocks;
  const int nunits = (2 * H - 1) * (2 * W - 1);
  a.vec4 = ((H * W) % 4 == 0 && (reinterpret_cast<uintptr_t>(left) & 15) == 0 &&
            (reinterpret_cast<uintptr_t>(right) & 15) == 0) ? 1 : 0;
  // CTAs per block pair: about one CTA per SM, so a grid of bp * nc CTAs
  // runs in ceil(bp * nc / SMs) waves of CTAs that each take 1/nc of a block
  // pair: pick the nc with the fewest waves per unit of work (fewest CTAs on
  // ties)
  const long long sms = sm_count();
  long long nc = 1;
  {
    const long long cap = nunits < 4 * sms ? nunits : 4 * sms;
    double best = 1e30;
    for (long long n = 1; n <= cap; ++n) {
      const double t = double((bp * n + sms - 1) / sms) / double(n);
      if (t < best * (1.0 - 1e-9)) {
        best = t;
        nc = n;
      }
    }
  }
  a.nc = int(nc);
  const long long blocks = bp * a.nc;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = size_t(H) * W * (kTinyL + kTinyR) * sizeof(float);
  auto kern = best == 0 ? xcorr_tiny_kernel<32, 16>
            : best == 1 ? xcorr_tiny_kernel<16, 32>
            : best == 2 ? xcorr_tiny_kernel<8, 64>
                        : xcorr_tiny_kernel<64, 8>;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern));
  if (e != cudaSuccess) return e;
  kern<<<unsigned(blocks), 32 * kTinyWarps, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace


// Largest shared staging area of the rows kernels (two CTAs per SM),
// and of the bcast kernel (one CTA per SM at worst).
constexpr size_t kMaxStageSmem = 110 * 1024;
constexpr size_t kMaxBcastSmem = 200 * 1024;
constexpr long long kMaxRowsGrid = 1LL << 30;   // rows kernels loop over more items

// Grid cap of the rows kernels: kMaxRowsGrid, or the positive integer in
// the environment variable CORR_XCORR_MAX_GRID (read on every call; lets a
// test run the item loop on ordinary shapes).
long long rows_grid_cap() {
  const char *v = getenv("CORR_XCORR_MAX_GRID");
  if (v && *v) {
    char *end = nullptr;
    const long long n = strtoll(v, &end, 10);
    if (end && *end == '\0' && n > 0 && n < kMaxRowsGrid) return n;
  }
  return kMaxRowsGrid;
}

namespace {

// Which kernel a shape takes, its arguments and the split-row scratch it needs.
enum class XKind { Tiny, Bcast, Rows, Tc, Warp, Tcl };

// Largest scratch the larger-matrix tensor-core kernel may take: 512 MB of
// partial tiles and its item counter.
constexpr size_t kMaxTclScratch = (size_t(512) << 20) + 256;

// Whether a shape takes the larger-matrix tensor-core kernel (xcorr_tcl.cu):
// CORR_XCORR_TCL (read on every call) "1" / "0" forces it on / off where it
// applies; otherwise the measured policy: pairs * (H*W)^2 >= 4e8 products.
// It never takes more than max_scratch (nor 512 MB of partial tiles).
// Measured on GB300 (CUDA-graph device time, this kernel / the scalar
// one): 1 x 1 of 160^2 50 / 56 us, of 256^2 89 / 214 us, of 1024^2 10.3 /
// 43.8 ms; 1 x 32 of 64^2 39 / 74 us, 4 x 16 of 64^2 64 / 118 us, 2 x 96 of
// 48^2 96 / 102 us; below the rule 1 x 64 of 48^2 48 / 49 us, 1 x 1 of
// 128^2 32 / 31 us, 1 x 16 of 64^2 35 / 32 us, 1 x 128 of 32^2 37 / 20 us.
bool use_tcl(int nl, int nr, int H, int W, size_t max_scratch) {
  const size_t need = tcl::scratch_bytes(nl, nr, H, W);
  if (need > kMaxTclScratch || need > max_scratch) return false;
  const char *v = getenv("CORR_XCORR_TCL");
  if (v && v[0] == '0' && v[1] == '\0') return false;
  if (v && v[0] == '1' && v[1] == '\0') return true;
  const double hw = double(H) * W;
  return double(nl) * nr * hw * hw >= 4e8;
}

// CORR_XCORR_WARP (read on every call): "1" routes every shape to the
// warp-per-overlap kernel, "0" none; otherwise the measured policy: single
// rows (one-dimensional signals) of 256 or more samples, where it beat the
// rows kernel on GB300 (1 x 4096: 19.6 against 26.4 us; 1 x 16384: 207
// against 280 us; 1 x 256: 3.2 against 4.3 us), while from two rows up
// the rows kernel won (2 x 2048: 13.7 against 20.7 us).
bool use_warp(int nl, int nr, int H, int W) {
  (void)nl;
  (void)nr;
  const char *v = getenv("CORR_XCORR_WARP");
  if (v && v[0] == '0' && v[1] == '\0') return false;
  if (v && v[0] == '1' && v[1] == '\0') return true;
  return H == 1 && W >= 256;
}

// Whether a shape takes the tensor-core kernel (xcorr_tc.cu): the
// environment variable CORR_XCORR_TC (read on every call) forces it off
// ("0") or on wherever it applies ("1"); otherwise the measured policy:
// matrices of 144+ elements (up to 16 x 16) in batches of 64+ pairs.
// Measured on GB300 (CUDA-graph device time, tensor-core / scalar kernel):
// 32 x 64 of 16^2 9.8 / 20.3 us, 16 x 16 of 16^2 9.5 / 11.9 us, 8 x 8 of
// 16^2 9.7 / 11.7 us, 8 x 8 of 12^2 7.8 / 8.3 us; outside the rule the
// scalar kernels won (64 x 64 of 10^2 13.2 / 11.7 us, 4 x 8 of 16^2 9.6 /
// 4.6 us, 1 x 8 of 16^2 9.4 / 3.7 us).
bool use_tc(int nl, int nr, int H, int W) {
  if (!tc::supported(nl, nr, H, W)) return false;
  const char *v = getenv("CORR_XCORR_TC");
  if (v && v[0] == '0' && v[1] == '\0') return false;
  if (v && v[0] == '1' && v[1] == '\0') return true;
  return H * W >= 144 && double(nl) * nr >= 64;
}

struct XPlan {
  XKind kind;
  XArgs a;
  size_t smem;           // dynamic shared memory of the pair / rows kernel
  long long blocks;      // grid of the pair / rows kernel
  size_t part_bytes;     // rows kernel with several bands: scratch bytes
  int chunk;             // rows kernel: 32 / 16 (whole rows) or 0 (windows)
  int bcast_rights;      // bcast kernel: rights per lane (1 or 2)
};

XPlan make_plan(const float *left, int nl, const float *right, int nr, int H, int W,
                float *out, size_t max_scratch = ~size_t(0)) {
  XPlan pl;
  pl.smem = 0;
  pl.blocks = 0;
  pl.part_bytes = 0;
  pl.chunk = 0;
  pl.bcast_rights = 2;
  const long long pairs = (long long)nl * nr;
  XArgs &a = pl.a;
  a.left = left;
  a.right = right;
  a.out = out;
  a.nl = nl;
  a.nr = nr;
  a.H = H;
  a.W = W;
#ifndef CORR_XC_TINY
#define CORR_XC_TINY 1
#endif
  if (use_warp(nl, nr, H, W)) {
    pl.kind = XKind::Warp;
    return pl;
  }
  if (use_tc(nl, nr, H, W)) {
    pl.kind = XKind::Tc;
    return pl;
  }
  if (use_tcl(nl, nr, H, W, max_scratch)) {
    pl.kind = XKind::Tcl;
    pl.part_bytes = tcl::scratch_bytes(nl, nr, H, W);
    return pl;
  }
  if (CORR_XC_TINY && H * W <= 256 && pairs >= 64) {
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
  a.nbands = 1;
  a.band_rows = H;
  a.items = 0;
  a.nxseg = 1;
  a.xseg = 0;
  a.SL = a.SR = 0;
  a.part_row = 0;
  a.part = nullptr;
  a.nrblk = 0;
  a.npairblk = 0;

  // bcast kernel: at least 32 rights per left, rows of 8+ floats, and two
  // chunk buffers fit
  {
    // rights per lane: estimated time = max(executed work / SMs, largest
    // CTA) (work in overlap rows x rights per lane, padding rights of a
    // partial block included), one right per lane counted 1.2x slower per
    // row (two loads feed 32 FMAs instead of three feeding 64)
    int br = 2;
    {
      const int ngp0 = (a.ngroups + 1) / 2;
      const double npb = (ngp0 + kBPairs - 1) / kBPairs, sms = sm_count();
      const double rows = double(H) * H;   // sum over dy of the overlap rows
      auto est = [&](int b) {
        const double nrblk = (nr + 32 * b - 1) / (32 * b);
        const double total = double(nl) * nrblk * npb * rows * b;
        const double t = total / sms > double(H) * b ? total / sms : double(H) * b;
        return b == 1 ? 1.2 * t : t;
      };
      if (est(1) < est(2)) br = 1;
    }
    pl.bcast_rights = br;
    const size_t buf_floats = size_t(bcast_buf(a.S, br));
    const size_t bsmem = 2 * buf_floats * sizeof(float);
    const int ngp = (a.ngroups + 1) / 2;
    a.nrblk = (nr + 32 * br - 1) / (32 * br);
    a.npairblk = (ngp + kBPairs - 1) / kBPairs;
    const long long bblocks = (long long)nl * a.nrblk * a.npairblk * (2LL * H - 1);
#ifndef CORR_XC_BCAST
#define CORR_XC_BCAST 1
#endif
    if (CORR_XC_BCAST && nr >= 32 && W >= 8 && bsmem <= kMaxBcastSmem && bblocks <= 0x7fffffffLL) {
      pl.kind = XKind::Bcast;
      pl.smem = bsmem;
      pl.blocks = bblocks;
      return pl;
    }
  }
  // rows kernels (shifts per lane kRowsP x kRowsQ): whole zero-padded rows
  // in 32-row chunks, else 16-row chunks, where a chunk leaves room for two
  // CTAs per SM; else L / R windows of x segments narrow enough for that
  a.ngroups = ((W - 1) - a.dxbase) / kRowsP + 1;
  a.ndyb = (2 * H - 1 + kRowsQ - 1) / kRowsQ;
  a.nsuper = (a.ngroups + kWarps - 1) / kWarps;
  {
    const int need = kRowsP + ((W + 3) & ~3) + kRowsP + 8;
    a.S = ((need + 7) & ~7) + 4;
  }
  a.nxseg = 1;
  a.xseg = 4 * ((W + 3) / 4);
  pl.chunk = 0;
  if ((pl.smem = size_t(ChunkGeom<kRowsQ, 32>::kRows) * a.S * sizeof(float)) <= kMaxStageSmem) {
    pl.chunk = 32;
  } else if ((pl.smem = size_t(ChunkGeom<kRowsQ, 16>::kRows) * a.S * sizeof(float)) <=
             kMaxStageSmem) {
    pl.chunk = 16;
  } else {
    auto win_smem = [&](int seg) {
      const int l = 4 * ((seg + 3) / 4);
      a.SL = l | 4;                        // stride % 8 == 4: conflict-free
      a.SR = (l + 8 * kRowsP) | 4;         //   16-byte loads across rows
      return (size_t(ChunkGeom<kRowsQ>::kL) * a.SL + size_t(ChunkGeom<kRowsQ>::kR) * a.SR) *
             sizeof(float);
    };
    while (win_smem(a.xseg) > kMaxStageSmem && a.xseg > 4) {
      ++a.nxseg;
      a.xseg = 4 * (((W + a.nxseg - 1) / a.nxseg + 3) / 4);
    }
    pl.smem = win_smem(a.xseg);
  }
  // row bands only where the grid would otherwise be short of CTAs
  const long long unbanded = pairs * a.ndyb * a.nsuper * a.nxseg;
  if (unbanded >= (long long)kBandMinCtasPerSm * sm_count() || H <= kBandRows) {
    a.nbands = 1;
    a.band_rows = H;
  } else {
    a.nbands = (H + kBandRows - 1) / kBandRows;
    a.band_rows = kBandRows;
  }
  a.part_row = kRowsP * a.ngroups;
  a.items = unbanded * a.nbands;
  pl.kind = XKind::Rows;
  const long long max_grid = rows_grid_cap();
  pl.blocks = a.items < max_grid ? a.items : max_grid;
  if (a.nbands * a.nxseg > 1)
    pl.part_bytes = size_t(pairs) * a.ndyb * a.nbands * a.nxseg * kRowsQ * a.part_row *
                    sizeof(float);
  return pl;
}

// Launch a plan.  Split-row scratch comes from `fixed` (at least
// pl.part_bytes long) when given, else from the library's pool.
cudaError_t run_plan(XPlan &pl, float *fixed, cudaStream_t stream) {
  XArgs &a = pl.a;
  if (pl.kind == XKind::Tc) return tc::launch(a.left, a.nl, a.right, a.nr, a.H, a.W, a.out, stream);
  if (pl.kind == XKind::Tcl) {
    float *part = fixed;
    cudaError_t e = cudaSuccess;
    if (!part && (e = scratch_alloc(reinterpret_cast<void **>(&part), pl.part_bytes, stream)) !=
                     cudaSuccess)
      return e;
    e = tcl::launch(a.left, a.nl, a.right, a.nr, a.H, a.W, a.out, part, stream);
    if (!fixed) {
      const cudaError_t f = cudaFreeAsync(part, stream);
      if (e == cudaSuccess) e = f;
    }
    return e;
  }
  if (pl.kind == XKind::Warp)
    return warp::launch(a.left, a.nl, a.right, a.nr, a.H, a.W, a.out, stream);
  if (pl.kind == XKind::Tiny)
    return launch_tiny(a.left, a.nl, a.right, a.nr, a.H, a.W, a.out, stream);
  if (pl.kind == XKind::Bcast) {
    auto kern = pl.bcast_rights == 1 ? xcorr_bcast_kernel<1> : xcorr_bcast_kernel<2>;
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(pl.blocks), 32 * kBWarps, pl.smem, stream>>>(a);
    return cudaGetLastError();
  }
  const bool loop = a.items > pl.blocks;
  auto rows_kernel =
      loop ? (pl.chunk == 32   ? xcorr_rows_kernel<kRowsP, kRowsQ, 32, true>
              : pl.chunk == 16 ? xcorr_rows_kernel<kRowsP, kRowsQ, 16, true>
                               : xcorr_rows_win_kernel<kRowsP, kRowsQ, true>)
           : (pl.chunk == 32   ? xcorr_rows_kernel<kRowsP, kRowsQ, 32, false>
              : pl.chunk == 16 ? xcorr_rows_kernel<kRowsP, kRowsQ, 16, false>
                               : xcorr_rows_win_kernel<kRowsP, kRowsQ, false>);
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(rows_kernel));
  if (e != cudaSuccess) return e;
  const bool banded = a.nbands * a.nxseg > 1;
  const bool pooled = banded && fixed == nullptr;
  a.part = banded ? fixed : nullptr;
  if (pooled && (e = scratch_alloc(reinterpret_cast<void **>(&a.part), pl.part_bytes, stream)) != cudaSuccess) return e;
  rows_kernel<<<unsigned(pl.blocks), kThreads, pl.smem, stream>>>(a);
  e = cudaGetLastError();
  if (banded && e == cudaSuccess) {
    const long long outs = (long long)a.nl * a.nr * (2LL * a.H - 1) * (2LL * a.W - 1);
    const long long sum_blocks = (outs + 255) / 256;
    xcorr_band_sum_kernel<kRowsP, kRowsQ>
        <<<unsigned(sum_blocks < 65535 * 16 ? sum_blocks : 65535 * 16), 256, 0, stream>>>(a);
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

int xcorr_f32_kernel_kind(int nl, int nr, int H, int W) {
  const XPlan pl = make_plan(nullptr, nl, nullptr, nr, H, W, nullptr);
  switch (pl.kind) {
    case XKind::Rows: return pl.chunk ? 0 : 1;
    case XKind::Bcast: return 2;
    case XKind::Tiny: return 3;
    case XKind::Tc: return 4;
    case XKind::Tcl: return 6;
    case XKind::Warp: return 5;
  }
  return -1;
}

size_t xcorr_f32_scratch_bytes(const float *left, int nl, const float *right, int nr,
                               int H, int W, size_t max_scratch) {
  return make_plan(left, nl, right, nr, H, W, nullptr, max_scratch).part_bytes;
}

cudaError_t xcorr_f32_launch_scratch(const float *left, int nl, const float *right,
                                     int nr, int H, int W, float *out, float *scratch,
                                     size_t scratch_bytes, cudaStream_t stream) {
  XPlan pl = make_plan(left, nl, right, nr, H, W, out, scratch_bytes);
  if (pl.part_bytes > scratch_bytes || (pl.part_bytes > 0 && scratch == nullptr))
    return cudaErrorInvalidValue;
  return run_plan(pl, scratch, stream);
}


}  // namespace corr
