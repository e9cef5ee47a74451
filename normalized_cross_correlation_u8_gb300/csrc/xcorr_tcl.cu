// xcorr_tcl.cu -- float32 full 2D cross-correlation of larger matrices (one
// left against one or many rights) on the sm_103a tensor cores.
//
// Same contraction as xcorr_tc.cu ("Efficient GPU-accelerated Parallel
// Cross-correlation" artifact README, kernel overview: all overlaps of a
// left and a right matrix, one-to-one / one-to-many), with x' the column of
// the right matrix:
//
//   out[l][r][dy][dx] = sum_{y, x'} L_l[y][x' + dx] * R_r[y - dy][x'].
//
// A tile is one left's 128 shifts dx (M) by 128 (shift dy, right) slots
// (N = NDY shifts x NR rights, right fastest: 128 shifts of one right for
// one-to-one, 32 shifts x 4 rights for one-to-many).  Its K -- every row y
// and column x' that some shift of the tile reaches -- is cut into units of
// 32 rows x 32 columns.  An item is one tile's unit column and a group of G
// consecutive row units (G = 1, 2 or 4 as the items balance best, more for
// larger matrices so that the partial tiles stay within 128 MB).  The
// kernel is persistent, one CTA per SM claiming items in turn; each item's
// 128 x 128 partial sums go to scratch memory and a second kernel adds
// those of each tile in a fixed order (the result does not depend on
// scheduling).
//
// Accuracy: the tensor cores accumulate FP32 with truncation, so on inputs
// of one sign the error of a chain of accumulates grows with its length
// (measured on GB300: about 2e-8 of the sum per accumulate; 384 of them, one
// 32-row unit, reached 1.1e-5 of sum |L*R| on uniform [0, 1) inputs).  A
// chain here is at most 8 rows (96 accumulates) in one tensor-memory
// accumulator; the builder warps add each finished chain into an FP32
// running sum in registers (round to nearest).
//
// Operands: B (rows of R) is staged per unit in shared memory in the
// no-swizzle K-major layout [x'/4][row slot][right][4 floats], rows in
// reverse order, so the N rows of consecutive shifts dy are consecutive
// slots and one descriptor per (y, 8 columns) reads them; two units are
// staged at a time, by two staging warps.  A (the Toeplitz rows of L) is written per overlap row
// by sixteen builder warps straight into tensor memory (tcgen05.st); the
// rows alternate between two streams, each with two A stages, one
// accumulator and one warp issuing kind::tf32 tcgen05.mma, which reads per
// row a record (B offset, chain start / end) the builders leave beside the
// stage.  Operands are split v = tf32(v) + tf32(v - tf32(v)) and each
// product is formed as hi*hi + hi*lo + lo*hi (the three-pass TF32 scheme;
// see xcorr_tc.cu).  Every mbarrier wait is bounded (corr_device_status).
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "internal.cuh"
#include "tc_common.cuh"

namespace corr {
namespace tcl {
namespace {

using namespace tcx;

constexpr int kThreads = 512;             // builder threads (16 warps)
constexpr int kM = 128;                   // shifts dx of one left
constexpr int kN = 128;                   // (shift dy, right) slots
constexpr int kKY = 32;                   // overlap rows per unit
constexpr int kKX = 32;                   // right columns per unit
constexpr int kSteps = kKX / 8;           // 8-deep K steps per row
constexpr int kStreams = 2;               // row streams, one issuer and accumulator each
constexpr int kStagers = 2;               // warps staging the next units' operands
constexpr int kStagerThreads = 32 * kStagers;
constexpr int kAllThreads = kThreads + 32 * kStreams + kStagerThreads;
constexpr int kBlockRows = 16;            // rows per block: kBlockRows / 2 per stream's chain
constexpr int kABufs = 4;                 // A stages in tensor memory (2 per stream)
constexpr int kStageCols = kSteps * 16;   // hi + lo columns of one A stage
constexpr uint32_t kAccCols = kN;         // one FP32 accumulator
constexpr uint32_t kTmemCols = 512;       // 2 accumulators + kABufs A stages
constexpr int kLRowF = kKX + kM;          // floats of a staged left row segment
constexpr int kLBuf = kKY * kLRowF;       // floats of one unit's left rows
constexpr int kMaxSlots = kKY + kN - 1;   // right row slots (NDY = 128)
constexpr int kMaxBEntries = 8 * (kKY + 32 - 1) * 4;   // NR = 4: the largest B
constexpr int kBHalf = kMaxBEntries * 16; // bytes of the hi (or lo) parts of one B
constexpr int kBBuf = 2 * kBHalf;         // one staged B (hi, then lo)
constexpr int kTileFloats = kM * kN;      // one partial tile
constexpr size_t kTargetScratch = size_t(128) << 20;  // partial tiles, when row groups allow
constexpr uint32_t kIdesc = idesc_tf32(kM, kN);
static_assert(8 * kMaxSlots * 1 <= kMaxBEntries && 8 * (kKY + 64 - 1) * 2 <= kMaxBEntries,
              "B staging holds every right-tile shape");
static_assert(2 * kAccCols + kABufs * kStageCols == kTmemCols, "tensor memory plan");
static_assert(kKY % kBlockRows == 0, "blocks never cross a unit");
static_assert(kABufs == 2 * kStreams, "two A stages per stream");

// shared memory: two staged B (TF32 hi / lo), the raw rows of the B after
// them (as copied), two units' left rows, the row records the builders
// pass to the issuer, the mbarriers, two claimed-item slots and the
// tensor-memory address
constexpr size_t kRawOff = 2 * size_t(kBBuf);
constexpr size_t kLpOff = kRawOff + size_t(kBHalf);
constexpr size_t kInfoOff = kLpOff + 2 * size_t(kLBuf) * sizeof(float);
constexpr size_t kBarOff = kInfoOff + kABufs * sizeof(uint2);
// full, empty, chain done per stream, done, staging request, staging done
constexpr int kBars = 2 * kABufs + 5;
constexpr size_t kClaimOff = kBarOff + kBars * 8;
// two claimed-item slots, a staging request (B buffer, units u + 1, u + 2)
constexpr size_t kSmemBytes = kClaimOff + (2 + 5) * sizeof(int) + 16;

// row record flags (second word): first and last row of a chain, end of
// the stream
constexpr uint32_t kRecFirst = 1u << 9, kRecLast = 1u << 10, kRecStop = 1u << 11;

// Division of 0 <= n < 2^31 by an invariant d >= 1 as a multiply-high and
// a shift (the round-up method for unsigned division by invariant
// integers): with s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1,
// n / d = (umulhi(n, m) + n) >> s.
struct FastDiv {
  uint32_t m;
  int s, d;
};

inline FastDiv fast_div(int d) {
  FastDiv f;
  f.d = d;
  f.s = 0;
  while ((1LL << f.s) < d) ++f.s;
  f.m = uint32_t(((1ULL << 32) * ((1ULL << f.s) - uint64_t(d))) / uint64_t(d) + 1);
  return f;
}

__device__ __forceinline__ int div_of(int n, const FastDiv &f) {
  return int((__umulhi(uint32_t(n), f.m) + uint32_t(n)) >> f.s);
}

struct TclArgs {
  const float *left;
  const float *right;
  float *partial;        // [items][kN][kM]
  float *out;
  int nl, nr, H, W;
  int nr_log2;           // rights per tile NR = 1 << nr_log2 (1, 2 or 4)
  int ndy;               // shift slots per tile: kN / NR
  int ndxt, ndyt, nrt;   // tiles along dx, dy, rights
  int uy, ux;            // units along rows, columns of K
  int ug, ugn;           // row units per item, groups of them along the rows
  long long items;       // work items: tiles x ugn x ux (below 2^31 at launch)
  int *counter;          // items claimed so far (zero at launch)
  FastDiv fux, fugn, fnrt, fndyt, fndxt;   // the item index's radices
  float inv_ns;          // 1 / (kKY + ndy - 1), the right row slots of a unit
  int stall;             // test of the bounded waits: the issuers' last commit is left out
  int vec4;              // rows readable as float4
};

__device__ int g_tcl_status;   // bit 0: a bounded wait gave up

// The tile of item b (its unit column and row-unit group) and the ranges
// of the tile: rows y and columns x' that some shift of the tile reaches
// (nonempty for every tile).
struct Tile {
  int l, dxt, dyt, rt, kg, kx;
  int dx0, dy0, r0;
  int ylo, yhi, xlo, xhi;
};

__device__ __forceinline__ Tile tile_of(const TclArgs &a, int b) {
  Tile t;
  int q = div_of(b, a.fux);
  t.kx = b - q * a.ux;
  b = q;
  q = div_of(b, a.fugn);
  t.kg = b - q * a.ugn;
  b = q;
  q = div_of(b, a.fnrt);
  t.rt = b - q * a.nrt;
  b = q;
  q = div_of(b, a.fndyt);
  t.dyt = b - q * a.ndyt;
  b = q;
  q = div_of(b, a.fndxt);
  t.dxt = b - q * a.ndxt;
  t.l = q;
  t.dx0 = t.dxt * kM - (a.W - 1);
  t.dy0 = t.dyt * a.ndy - (a.H - 1);
  t.r0 = t.rt << a.nr_log2;
  t.ylo = t.dy0 > 0 ? t.dy0 : 0;
  t.yhi = a.H + t.dy0 + a.ndy - 1 < a.H ? a.H + t.dy0 + a.ndy - 1 : a.H;
  const int xl = -(t.dx0 + kM - 1);
  t.xlo = xl > 0 ? xl : 0;
  t.xhi = a.W - t.dx0 < a.W ? a.W - t.dx0 : a.W;
  return t;
}

// An item: one tile's unit column kx and its row units [ka, kb) that hold
// rows of the tile; empty when the column holds none that the tile reaches.
struct Item {
  int b;                 // -1: none
  int l, dx0, dy0, r0, ylo, yhi;
  int xa, ka, kb;
};

__device__ __forceinline__ bool item_at(const TclArgs &a, int b, Item &it) {
  const Tile tl = tile_of(a, b);
  it.b = b;
  it.l = tl.l;
  it.dx0 = tl.dx0;
  it.dy0 = tl.dy0;
  it.r0 = tl.r0;
  it.ylo = tl.ylo;
  it.yhi = tl.yhi;
  it.xa = tl.kx * kKX;
  const int x0 = it.xa > tl.xlo ? it.xa : tl.xlo;
  const int x1 = it.xa + kKX < tl.xhi ? it.xa + kKX : tl.xhi;
  const int kvlo = tl.ylo / kKY, kvhi = (tl.yhi + kKY - 1) / kKY;
  it.ka = tl.kg * a.ug > kvlo ? tl.kg * a.ug : kvlo;
  it.kb = (tl.kg + 1) * a.ug < kvhi ? (tl.kg + 1) * a.ug : kvhi;
  return it.ka < it.kb && x0 < x1;
}

// Claim the next item that holds products (one thread): items go out in
// index order from the counter; -1 once none is left.
__device__ __forceinline__ int claim_item(const TclArgs &a) {
  for (;;) {
    const int c = atomicAdd(a.counter, 1);
    if (c >= a.items) return -1;
    Item it;
    if (item_at(a, c, it)) return c;
  }
}

// Rows of unit ky of an item: [max(ky kKY, ylo), min(ky kKY + kKY, yhi)).
__device__ __forceinline__ void unit_rows(const Item &it, int ky, int &y0, int &y1) {
  const int ya = ky * kKY;
  y0 = ya > it.ylo ? ya : it.ylo;
  y1 = ya + kKY < it.yhi ? ya + kKY : it.yhi;
}

// Asynchronous copies global -> shared (cp.async); `ok` false writes zeros
// (nothing is read).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, bool ok) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "r"(ok ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Copy the right rows of unit ky of an item: raw entry e = (xc, slot, r)
// <- R[r0 + r][yr][xa + 4 xc .. + 3] with yr = ya + kKY - 1 - dy0 - slot
// (zero outside the matrix), 16 bytes each.  Thread t takes the entries
// t + k kThreads, as in convert_b.
template <int NT = kThreads>
__device__ __forceinline__ void copy_b_raw(const TclArgs &a, const Item &it, int ky,
                                           uint32_t raw, int t, int NS) {
  const int H = a.H, W = a.W, NR = 1 << a.nr_log2;
  const int nent = 8 * NS * NR;
  const int yc = ky * kKY + kKY - 1 - it.dy0;
  constexpr int kPer = (kMaxBEntries + NT - 1) / NT;
#pragma unroll 2
  for (int k = 0; k < kPer; ++k) {
    const int e = t + k * NT;
    if (e >= nent) break;
    const int r = e & (NR - 1), qq = e >> a.nr_log2;
    // qq / NS in floating point: exact for qq < 8 NS <= 2^11 (the error of
    // (qq + 1/2) / NS stays far below the 1/(2 NS) to the next integer)
    const int xc = int((float(qq) + 0.5f) * a.inv_ns), sl = qq - xc * NS;
    const int yr = yc - sl, rr = it.r0 + r, x = it.xa + 4 * xc;
    const bool row_ok = rr < a.nr && yr >= 0 && yr < H;
    const float *src = row_ok ? a.right + (size_t(rr) * H + yr) * W + x : a.right;
    const uint32_t dst = raw + uint32_t(e) * 16;
    if (a.vec4) {
      cp_async16(dst, row_ok && x < W ? src : a.right, row_ok && x < W);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const bool ok = row_ok && x + c < W;
        cp_async4(dst + 4 * c, ok ? src + c : a.right, ok);
      }
    }
  }
}

// Copy the left's rows y0 .. y1 - 1 of unit ky, columns xa + dx0 .. +
// kLRowF - 1: lpu[y - y0][p] <- L[l][y][xa + dx0 + p] (zero outside the
// matrix).
template <int NT = kThreads>
__device__ __forceinline__ void copy_lp(const TclArgs &a, const Item &it, int ky, uint32_t lpu,
                                        int t) {
  const int H = a.H, W = a.W;
  int y0, y1;
  unit_rows(it, ky, y0, y1);
  const int nl_ent = (y1 - y0) * kLRowF;
  const float *lrow = a.left + size_t(it.l) * H * W;
  const int xb = it.xa + it.dx0;
  constexpr int kPer = (kLBuf + NT - 1) / NT;
#pragma unroll 4
  for (int k = 0; k < kPer; ++k) {
    const int i = t + k * NT;
    if (i >= nl_ent) break;
    const int p = i % kLRowF, ry = i / kLRowF;
    const int x = xb + p;
    const bool ok = x >= 0 && x < W;
    cp_async4(lpu + uint32_t(i) * 4, ok ? lrow + size_t(y0 + ry) * W + x : a.left, ok);
  }
}

// B entries t + k kThreads of this thread's (landed) raw copies, split into
// TF32 hi (bb) and lo (bb + kBHalf).
template <int NT = kThreads>
__device__ __forceinline__ void convert_b(const uint8_t *raw, uint8_t *bb, int t, int nent) {
  constexpr int kPer = (kMaxBEntries + NT - 1) / NT;
#pragma unroll 4
  for (int k = 0; k < kPer; ++k) {
    const int e = t + k * NT;
    if (e >= nent) break;
    const float4 v = *reinterpret_cast<const float4 *>(raw + e * 16);
    uint4 hi, lo;
    split_tf32(v.x, hi.x, lo.x);
    split_tf32(v.y, hi.y, lo.y);
    split_tf32(v.z, hi.z, lo.z);
    split_tf32(v.w, hi.w, lo.w);
    *reinterpret_cast<uint4 *>(bb + e * 16) = hi;
    *reinterpret_cast<uint4 *>(bb + kBHalf + e * 16) = lo;
  }
  // generic-proxy stores -> the tensor cores' (async proxy) reads
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Barrier of the builder warps (named barrier 1) returning the OR of v.
__device__ __forceinline__ int builders_sync_or(int v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\t"
      "selp.s32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(v), "n"(kThreads)
      : "memory");
  return r;
}

// Persistent: each CTA claims items in turn (a counter in scratch memory)
// and runs their units' overlap rows in blocks of kBlockRows.  Within a
// block the rows alternate between two streams, each with its own issuing
// thread, two A stages and FP32 accumulator: one thread alone cannot issue
// 128 x 128 x 8 MMAs as fast as the tensor pipe runs them (about 54
// against 64 cycles each, with any per-row bookkeeping on top, and the
// pipe queues almost nothing ahead), two together can.  A stream's rows of
// one block are one accumulation chain (at most 8 rows, 96 accumulates:
// the tensor cores' FP32 accumulation truncates, so a chain stays short).
// Before a block's first rows the builders add both finished chains into
// an FP32 running sum of the item held in registers (thread: accumulator
// row 32 (warp % 4) + lane, columns 32 (warp / 4) .. + 31); at the end of
// an item the running sum goes to its partial tile.
//
// Staging runs two units ahead on two staging warps: once the builders
// have taken in unit u - 1's last chains (so its buffers are free), thread
// 0 posts a request; the stagers turn the raw rows of unit u + 1 (copied
// during unit u - 1) into its TF32 B, copy unit u + 2's raw rows and unit
// u + 1's left rows, and report, which the builders check before unit u +
// 1 starts.  (Done by the builders themselves, the staging kept both
// issuers waiting at every unit's start.)
__global__ void __launch_bounds__(kAllThreads, 1) xcorr_tcl_kernel(const TclArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *raw = smem + kRawOff;
  float *lp = reinterpret_cast<float *>(smem + kLpOff);                  // [2][kLBuf]
  uint2 *info = reinterpret_cast<uint2 *>(smem + kInfoOff);             // [kABufs]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kBarOff);        // [kABufs]
  uint64_t *empty = full + kABufs;                                       // [kABufs]
  uint64_t *chain = empty + kABufs;                                      // [kStreams]
  uint64_t *done = chain + 2;
  uint64_t *stage_go = done + 1;      // a staging request is in req
  uint64_t *stage_done = done + 2;    // the stagers finished it
  int *claimed = reinterpret_cast<int *>(smem + kClaimOff);             // [2]
  int *req = claimed + 2;             // B buffer, unit u + 1 (b, ky), unit u + 2 (b, ky)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(req + 5);

  const int NR = 1 << a.nr_log2, NS = kKY + a.ndy - 1;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int stream = warp - kThreads / 32;     // issuer warps: 0, 1; builders < 0
  const bool issuer = stream == 0 || stream == 1;
  const bool stager = stream >= kStreams;

  if (stream == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < kABufs; ++k) {
        mbar_init(smem_u32(&full[k]), kThreads / 32);
        mbar_init(smem_u32(&empty[k]), 1);
      }
      mbar_init(smem_u32(&chain[0]), 1);
      mbar_init(smem_u32(&chain[1]), 1);
      mbar_init(smem_u32(done), kStreams);
      mbar_init(smem_u32(stage_go), 1);
      mbar_init(smem_u32(stage_done), kStagers);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t a_cols = tmem + 2 * kAccCols;     // A stage s: columns + kStageCols s
  int failed = 0;

  if (issuer) {
    if (lane == 0) {
      const uint32_t lbo_b = uint32_t(NS * NR * 16);     // next 4 columns x'
      // descriptor of B at the start of shared memory; a row's descriptors
      // add their byte offset / 16 to its address field (addresses stay
      // below 2^18, so nothing carries out of it)
      const uint64_t desc0 = smem_desc(smem_u32(smem), lbo_b, 128);
      const uint64_t step_j = uint64_t((2 * lbo_b) >> 4), to_lo = uint64_t(kBHalf >> 4);
      const uint32_t d = tmem + uint32_t(stream) * kAccCols;
      int k = 0;                                   // this stream's rows so far
      for (;; ++k) {
        const int s = 2 * stream + (k & 1);
        if (!mbar_wait_bounded(smem_u32(&full[s]), uint32_t(k >> 1) & 1u)) {
          failed = 1;
          break;
        }
        fence_after_sync();
        const uint2 rec = info[s];
        if (rec.y & kRecStop) break;
        // all kSteps K steps, straight-line (a branch between tcgen05.mma
        // issues slows them well below the tensor pipe's rate): columns x'
        // no shift of the tile reaches meet left values staged as zero
        const uint32_t ab = a_cols + uint32_t(kStageCols * s);
        const uint64_t bhi = desc0 + uint64_t(rec.x >> 4);
        mma3_tf32_ta(d, ab, ab + 8, bhi, bhi + to_lo, (rec.y & kRecFirst) ? 0u : 1u, kIdesc);
#pragma unroll
        for (int j = 1; j < kSteps; ++j)
          mma3_tf32_ta(d, ab + 16 * j, ab + 16 * j + 8, bhi + j * step_j, bhi + j * step_j + to_lo,
                       1u, kIdesc);
        mma_commit(smem_u32(&empty[s]));
        if (rec.y & kRecLast) mma_commit(smem_u32(&chain[stream]));
      }
      if (!a.stall) mma_commit(smem_u32(done));
      if (!mbar_wait_bounded(smem_u32(done), 0)) failed = 1;
      // each of this stream's stages: its last release has landed (no
      // arrival on this CTA's shared memory is left pending when it exits)
      for (int b = 0; b < 2 && b < k; ++b) {
        const int uses = (k - b + 1) / 2;
        if (!mbar_wait_bounded(smem_u32(&empty[2 * stream + b]), uint32_t(uses - 1) & 1u))
          failed = 1;
      }
    }
  } else if (stager) {
    // Stagers: per request (sent once the last unit's products are done,
    // so its B and left-row buffers are free), turn unit u + 1's raw rows
    // into B, copy unit u + 2's raw rows and unit u + 1's left rows, wait
    // for the copies and report; a request for no unit ends the loop.
    const int st = t - (kThreads + 32 * kStreams);
    const int nent = 8 * NS * NR;
    const uint32_t raw_u32 = smem_u32(raw), lp_u32 = smem_u32(lp);
    for (int k = 0;; ++k) {
      if (!mbar_wait_bounded(smem_u32(stage_go), uint32_t(k) & 1u)) {
        failed = 1;
        break;
      }
      const int nb = req[0], rb1 = req[1], rky1 = req[2], rb2 = req[3], rky2 = req[4];
      if (rb1 < 0) break;
      convert_b<kStagerThreads>(raw, smem + nb * kBBuf, st, nent);
      Item it;
      if (rb2 >= 0) {
        item_at(a, rb2, it);
        copy_b_raw<kStagerThreads>(a, it, rky2, raw_u32, st, NS);
      }
      item_at(a, rb1, it);
      copy_lp<kStagerThreads>(a, it, rky1, lp_u32 + uint32_t(nb * kLBuf) * 4, st);
      cp_async_commit();
      cp_async_wait_all();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(stage_done));
    }
  } else {
    // thread: A row m = 32 q + lane (shift dx = dx0 + m) with q = warp % 4,
    // K step jh = warp / 4: the 8 values L[l][y][x' + dx], x' = xa + 8 jh ..
    // + 7, as TF32 hi and lo; accumulator columns 32 jh .. + 31 of row m
    const int q = warp & 3, jh = warp >> 2;
    const int m = 32 * q + lane;
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    const int nent = 8 * NS * NR;
    const uint32_t raw_u32 = smem_u32(raw), lp_u32 = smem_u32(lp);
    float sum[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) sum[k] = 0.f;

    // The unit ring: the current unit (item cb, row unit cky), the next
    // (b1, ky1) and the one after (b2, ky2); item -1: none.  The unit after
    // (b, ky) is (b, ky + 1) within the item, else the first unit of the
    // item thread 0 claimed into claimed[slot] before the last barrier.
    auto is_item_end = [&](int b, int ky) {
      Item it;
      item_at(a, b, it);
      return ky + 1 >= it.kb;
    };
    auto successor = [&](int b, int ky, int slot, int &ob, int &oky) {
      ob = -1;
      oky = 0;
      if (b < 0) return;
      Item it;
      item_at(a, b, it);
      if (ky + 1 < it.kb) {
        ob = b;
        oky = ky + 1;
        return;
      }
      ob = claimed[slot];
      if (ob >= 0) {
        item_at(a, ob, it);
        oky = it.ka;
      }
    };
    int cb, cky = 0, b1, ky1, b2, ky2;
    if (t == 0) claimed[0] = claim_item(a);
    failed = builders_sync_or(failed);
    cb = claimed[0];
    if (cb >= 0) {
      Item it;
      item_at(a, cb, it);
      cky = it.ka;
    }
    if (t == 0 && cb >= 0 && is_item_end(cb, cky)) claimed[1] = claim_item(a);
    failed = builders_sync_or(failed);
    successor(cb, cky, 1, b1, ky1);
    if (t == 0 && b1 >= 0 && is_item_end(b1, ky1)) claimed[0] = claim_item(a);
    failed = builders_sync_or(failed);
    successor(b1, ky1, 0, b2, ky2);
    // the first two units' B and the first unit's left rows; then the copies
    // of the third unit's raw rows and the second unit's left rows
    if (cb >= 0) {
      Item it;
      item_at(a, cb, it);
      copy_b_raw(a, it, cky, raw_u32, t, NS);
      copy_lp(a, it, cky, lp_u32, t);
      cp_async_commit();
      cp_async_wait_all();
      convert_b(raw, smem, t, nent);
      if (b1 >= 0) {
        item_at(a, b1, it);
        copy_b_raw(a, it, ky1, raw_u32, t, NS);
        cp_async_commit();
        cp_async_wait_all();
        convert_b(raw, smem + kBBuf, t, nent);
        if (b2 >= 0) {
          Item i2;
          item_at(a, b2, i2);
          copy_b_raw(a, i2, ky2, raw_u32, t, NS);
        }
        copy_lp(a, it, ky1, lp_u32 + uint32_t(kLBuf) * 4, t);
        cp_async_commit();
      }
    }
    failed = builders_sync_or(failed);

    int nreq = 0, nreq_done = 0;   // staging requests sent, and waited for
    bool stop_sent = false;

    // the chains of the last block, still to be taken in
    int pstreams = 0;         // streams that had rows in it (1 or 2; 0: none)
    int pitem = -1;           // its item, if the block ends that item
    bool punit_end = false;   // whether it ends its unit
    int nch0 = 0, nch1 = 0;   // chains taken in per stream
    int gs0 = 0, gs1 = 0, u = 0;   // rows built per stream; units begun
    uint32_t epar = 0;

    // Take in the last block's chains: wait for their products, add the
    // accumulators to the running sum; at the end of an item store the sum.
    // At the end of a unit (its products all done, its buffers free): turn
    // unit u + 1's raw rows into B and start the copies of unit u + 2's raw
    // rows and unit u + 1's left rows.
    auto take_in = [&]() {
#pragma unroll
      for (int st = 0; st < kStreams; ++st) {
        if (st >= pstreams) break;
        const int n = st == 0 ? nch0 : nch1;
        if (!failed && !mbar_wait_bounded_sleep(smem_u32(&chain[st]), uint32_t(n) & 1u))
          failed = 1;
        failed = __any_sync(~0u, failed);     // the warp's .aligned steps stay together
        fence_after_sync();
        if (!failed) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + uint32_t(st) * kAccCols + uint32_t(32 * jh), v);
#pragma unroll
          for (int k = 0; k < 32; ++k) sum[k] += __uint_as_float(v[k]);
        }
        if (st == 0) ++nch0; else ++nch1;
      }
      fence_before_sync();
      if (pitem >= 0) {
        if (!failed) {
          float *dst = a.partial + size_t(pitem) * kTileFloats + m;
#pragma unroll
          for (int k = 0; k < 32; ++k) dst[size_t(32 * jh + k) * kM] = sum[k];
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) sum[k] = 0.f;
      }
      if (punit_end && !failed && !stop_sent) {
        // the last unit's products are done: ask the stagers for the next
        // units (or, with none left, to stop)
        if (t == 0) {
          req[0] = (u + 1) & 1;
          req[1] = b1;
          req[2] = ky1;
          req[3] = b2;
          req[4] = ky2;
          mbar_arrive(smem_u32(stage_go));
        }
        if (b1 >= 0) ++nreq; else stop_sent = true;
      }
      pstreams = 0;
    };

    while (cb >= 0) {
      const int buf = u & 1;
      const float *lpu = lp + buf * kLBuf;
      Item cur;
      item_at(a, cb, cur);
      int y0, y1;
      unit_rows(cur, cky, y0, y1);
      const int ya = cky * kKY;
      const bool item_end = cky + 1 == cur.kb;
      for (int sy = y0; sy < y1; sy += kBlockRows) {
        const int sy1 = sy + kBlockRows < y1 ? sy + kBlockRows : y1;
        if (pstreams) take_in();
        for (int y = sy; y < sy1; ++y) {
          const int st = (y - sy) & 1;
          const int kr = st ? gs1 : gs0;
          const int s = 2 * st + (kr & 1);
          if (kr >= 2) {
            if (!failed && !mbar_wait_bounded_sleep(smem_u32(&empty[s]), (epar >> s) & 1u))
              failed = 1;
            failed = __any_sync(~0u, failed);
            epar ^= 1u << s;
            fence_after_sync();
          }
          if (!failed) {
            const float *ls = lpu + (y - y0) * kLRowF + m + 8 * jh;
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) split_tf32(ls[k], hi[k], lo[k]);
            const uint32_t col = a_cols + uint32_t(kStageCols * s + 16 * jh);
            tmem_st8(lane_base + col, hi);
            tmem_st8(lane_base + col + 8, lo);
          }
          if (t == 0) {
            // row n = (dyi, r) of B: right row y - dy0 - dyi at slot
            // (ya + kKY - 1 - y) + dyi, n * 16 bytes past slot ya + kKY - 1 - y
            info[s] = make_uint2(uint32_t(buf * kBBuf + (ya + kKY - 1 - y) * NR * 16),
                                 (y - sy < 2 ? kRecFirst : 0u) | (y + 2 >= sy1 ? kRecLast : 0u));
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&full[s]));
          if (st) ++gs1; else ++gs0;
        }
        pstreams = sy1 - sy >= 2 ? 2 : 1;
        const bool unit_end = sy1 == y1;
        pitem = (unit_end && item_end) ? cb : -1;
        punit_end = unit_end;
      }
      // next unit: claim the item after the ring's last unit if it needs
      // one; this thread's copies of the next unit's left rows (and the
      // raw rows after it) have landed; then everyone's have
      ++u;
      if (t == 0 && b2 >= 0 && is_item_end(b2, ky2)) claimed[u & 1] = claim_item(a);
      cp_async_wait_all();
      // the next unit's operands from the stagers
      if (nreq_done < nreq) {
        if (t == 0 && !failed &&
            !mbar_wait_bounded(smem_u32(stage_done), uint32_t(nreq_done) & 1u))
          failed = 1;
        ++nreq_done;
      }
      failed = builders_sync_or(failed);
      if (failed) break;
      cb = b1;
      cky = ky1;
      b1 = b2;
      ky1 = ky2;
      successor(b1, ky1, u & 1, b2, ky2);
    }
    if (pstreams) {
      b1 = -1;
      take_in();
    }
    if (!stop_sent && t == 0) {          // the stagers end with a request for no unit
      req[1] = -1;
      mbar_arrive(smem_u32(stage_go));
    }
    cp_async_wait_all();                 // no copy in flight when the CTA ends
    // end of both row streams
#pragma unroll
    for (int st = 0; st < kStreams; ++st) {
      const int kr = st ? gs1 : gs0;
      const int s = 2 * st + (kr & 1);
      if (kr >= 2 && !failed && !mbar_wait_bounded(smem_u32(&empty[s]), (epar >> s) & 1u))
        failed = 1;
      if (t == 0) info[s] = make_uint2(0u, kRecStop);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&full[s]));
    }
  }
  failed = __syncthreads_or(failed);
  if (failed && t == 0) atomicOr(&g_tcl_status, 1);
  fence_before_sync();
  __syncthreads();
  if (stream == 0) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// out[l][r][oy][ox] = the sum, in a fixed order (row-unit group, then unit
// column), of the partial tiles of its tile's CTAs that hold any of its
// products.  A thread takes 4 consecutive shifts dx (one 16-byte load per
// partial tile: a tile starts at a multiple of 128 shifts), loads in
// batches of 8 in flight together.
__global__ void __launch_bounds__(256) xcorr_tcl_sum_kernel(const TclArgs a) {
  const int ndy = 2 * a.H - 1, ndx = 2 * a.W - 1, nq = (ndx + 3) >> 2;
  const long long total = (long long)a.nl * a.nr * ndy * nq;
  const int NR = 1 << a.nr_log2;
  for (long long o = (long long)blockIdx.x * blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    long long rest = o;
    const int ox = 4 * int(rest % nq);
    rest /= nq;
    const int oy = int(rest % ndy);
    rest /= ndy;
    const int r = int(rest % a.nr);
    const int l = int(rest / a.nr);
    const int dxt = ox / kM, m = ox - dxt * kM;
    const int dyt = oy / a.ndy, dyi = oy - dyt * a.ndy;
    const int rt = r >> a.nr_log2, n = (dyi << a.nr_log2) + (r & (NR - 1));
    const long long b0 = ((((long long)l * a.ndxt + dxt) * a.ndyt + dyt) * a.nrt + rt) * a.ugn;
    const Tile tl = tile_of(a, int(b0 * a.ux));
    // groups holding a row unit in [ylo / kKY, ceil(yhi / kKY)), unit
    // columns in [xlo / kKX, ceil(xhi / kKX)): every such CTA wrote its tile
    const int kg0 = tl.ylo / kKY / a.ug, kg1 = ((tl.yhi + kKY - 1) / kKY - 1) / a.ug + 1;
    const int kx0 = tl.xlo / kKX, kx1 = (tl.xhi + kKX - 1) / kKX;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    const float *base = a.partial + size_t(n) * kM + m;
    for (int kg = kg0; kg < kg1; ++kg) {
      const float *row = base + ((b0 + kg) * a.ux) * size_t(kTileFloats);
      for (int kx = kx0; kx < kx1; kx += 8) {
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          v[k] = kx + k < kx1
                     ? __ldg(reinterpret_cast<const float4 *>(row + size_t(kx + k) * kTileFloats))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (kx + k < kx1) {
            s.x += v[k].x;
            s.y += v[k].y;
            s.z += v[k].z;
            s.w += v[k].w;
          }
      }
    }
    float *dst = a.out + ((size_t(l) * a.nr + r) * ndy + oy) * ndx + ox;
    dst[0] = s.x;
    if (ox + 1 < ndx) dst[1] = s.y;
    if (ox + 2 < ndx) dst[2] = s.z;
    if (ox + 3 < ndx) dst[3] = s.w;
  }
}

TclArgs make_args(const float *left, int nl, const float *right, int nr, int H, int W,
                  float *out) {
  TclArgs a;
  a.left = left;
  a.right = right;
  a.out = out;
  a.partial = nullptr;
  a.counter = nullptr;
  a.nl = nl;
  a.nr = nr;
  a.H = H;
  a.W = W;
  // rights per tile: 4 (32 shifts dy each) for four or more rights, else 1
  a.nr_log2 = nr >= 4 ? 2 : 0;
  a.ndy = kN >> a.nr_log2;
  a.ndxt = (2 * W - 1 + kM - 1) / kM;
  a.ndyt = (2 * H - 1 + a.ndy - 1) / a.ndy;
  a.nrt = (nr + (1 << a.nr_log2) - 1) >> a.nr_log2;
  a.uy = (H + kKY - 1) / kKY;
  a.ux = (W + kKX - 1) / kKX;
  // row units per item (measured on GB300): 1 while that leaves at most
  // 3 items per SM; else 4 or 2 (the largest that divides the row units
  // and leaves at least 1.5 items per SM; groups that end ragged balance
  // badly); then doubled while the partial tiles would pass kTargetScratch.
  // CORR_XCORR_TCL_GROUP=n (read on every call) sets it to n instead.
  const double tiles = double(nl) * a.ndxt * a.ndyt * a.nrt;
  auto items_of = [&](int g) { return tiles * ((a.uy + g - 1) / g) * a.ux; };
  const double sms = double(device_sm_count());
  a.ug = 1;
  if (items_of(1) > 3 * sms)
    for (int g = 4; g >= 2; g /= 2)
      if (a.uy % g == 0 && items_of(g) >= 1.5 * sms) {
        a.ug = g;
        break;
      }
  while (a.ug < a.uy && items_of(a.ug) * kTileFloats * sizeof(float) > double(kTargetScratch))
    a.ug *= 2;
  if (const char *v = getenv("CORR_XCORR_TCL_GROUP")) {
    const int n = atoi(v);
    if (n > 0) a.ug = n;
  }
  if (a.ug > a.uy) a.ug = a.uy;
  a.ugn = (a.uy + a.ug - 1) / a.ug;
  a.items = (long long)nl * a.ndxt * a.ndyt * a.nrt * a.ugn * a.ux;
  a.fux = fast_div(a.ux);
  a.fugn = fast_div(a.ugn);
  a.fnrt = fast_div(a.nrt);
  a.fndyt = fast_div(a.ndyt);
  a.fndxt = fast_div(a.ndxt);
  a.inv_ns = 1.0f / float(kKY + a.ndy - 1);
  // CORR_XCORR_TCL_STALL=1 (read on every call): a test of the failure path
  // -- the issuers' last completion barrier is never signalled, their waits
  // on it give up after about a second and corr_device_status() reports
  // CORR_ETIMEOUT (the products themselves complete)
  {
    const char *v = getenv("CORR_XCORR_TCL_STALL");
    a.stall = (v && v[0] == '1' && v[1] == '\0') ? 1 : 0;
  }
  a.vec4 = (W % 4 == 0 && (reinterpret_cast<uintptr_t>(right) & 15) == 0) ? 1 : 0;
  return a;
}

}  // namespace

size_t scratch_bytes(int nl, int nr, int H, int W) {
  const TclArgs a = make_args(nullptr, nl, nullptr, nr, H, W, nullptr);
  // partial tiles, then the item counter
  return size_t(a.items) * kTileFloats * sizeof(float) + 256;
}

cudaError_t launch(const float *left, int nl, const float *right, int nr, int H, int W,
                   float *out, float *scratch, cudaStream_t stream) {
  TclArgs a = make_args(left, nl, right, nr, H, W, out);
  a.partial = scratch;
  if (a.items > 0x7fffffffLL || scratch == nullptr) return cudaErrorInvalidValue;
  a.counter = reinterpret_cast<int *>(scratch + size_t(a.items) * kTileFloats);
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(xcorr_tcl_kernel));
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(a.counter, 0, sizeof(int), stream)) != cudaSuccess) return e;
  // persistent: one CTA per SM (its shared memory and tensor memory fill one)
  const long long ctas = a.items < device_sm_count() ? a.items : device_sm_count();
  xcorr_tcl_kernel<<<unsigned(ctas), kAllThreads, kSmemBytes, stream>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long outs = (long long)nl * nr * (2LL * H - 1) * ((2LL * W - 1 + 3) / 4);
  const long long cap = 8LL * device_sm_count() * 8;
  const long long blocks = (outs + 255) / 256 < cap ? (outs + 255) / 256 : cap;
  xcorr_tcl_sum_kernel<<<unsigned(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t take_status(int *gave_up) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tcl_status, sizeof(int));
  if (e != cudaSuccess) return e;
  *gave_up = v;
  if (v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_tcl_status, &zero, sizeof(int));
  }
  return e;
}

}  // namespace tcl
}  // namespace corr
