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
// 32 rows x 32 columns, one CTA each, so that a large pair spreads over the
// whole GPU.  A unit's partial 128 x 128 sums go to scratch memory and a
// second kernel adds the units of each tile in a fixed order (the result
// does not depend on scheduling).
//
// Operands: B (rows of R) is staged once per unit in shared memory in the
// no-swizzle K-major layout [x'/4][row slot][right][4 floats], rows in
// reverse order, so the N rows of consecutive shifts dy are consecutive
// slots and one descriptor per (y, 8 columns) reads them; A (the Toeplitz
// rows of L) is written per overlap row by eight builder warps straight
// into tensor memory (tcgen05.st), double-buffered; one warp issues
// kind::tf32 tcgen05.mma into a 128-column FP32 accumulator in tensor
// memory.  Operands are split v = tf32(v) + tf32(v - tf32(v)) and each
// product is formed as hi*hi + hi*lo + lo*hi (the three-pass TF32 scheme;
// see xcorr_tc.cu).  Every mbarrier wait is bounded (corr_device_status).
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"
#include "tc_common.cuh"

namespace corr {
namespace tcl {
namespace {

using namespace tcx;

constexpr int kThreads = 256;             // builder threads (8 warps)
constexpr int kM = 128;                   // shifts dx of one left
constexpr int kN = 128;                   // (shift dy, right) slots
constexpr int kKY = 32;                   // overlap rows per unit
constexpr int kKX = 32;                   // right columns per unit
constexpr int kSteps = kKX / 8;           // 8-deep K steps per row
constexpr int kABufs = 2;                 // A stages in tensor memory
constexpr int kStageCols = kSteps * 16;   // hi + lo columns of one A stage
constexpr uint32_t kTmemCols = 256;       // accumulator (128) + kABufs stages (64 each)
constexpr int kLRowF = kKX + kM;          // floats of a staged left row segment
constexpr int kMaxSlots = kKY + kN - 1;   // right row slots (NDY = 128)
constexpr int kMaxBEntries = 8 * (kKY + 32 - 1) * 4;   // NR = 4: the largest B
constexpr int kTileFloats = kM * kN;      // one partial tile
constexpr uint32_t kIdesc = idesc_tf32(kM, kN);
static_assert(8 * kMaxSlots * 1 <= kMaxBEntries && 8 * (kKY + 64 - 1) * 2 <= kMaxBEntries,
              "B staging holds every right-tile shape");

struct TclArgs {
  const float *left;
  const float *right;
  float *partial;        // [units][kN][kM]
  float *out;
  int nl, nr, H, W;
  int nr_log2;           // rights per tile NR = 1 << nr_log2 (1, 2 or 4)
  int ndy;               // shift slots per tile: kN / NR
  int ndxt, ndyt, nrt;   // tiles along dx, dy, rights
  int uy, ux;            // units along rows, columns of K
  int vec4;              // rows readable as float4
};

__device__ int g_tcl_status;   // bit 0: a bounded wait gave up

// The tile of unit b and its ranges: rows y and columns x' that some shift
// of the tile reaches (nonempty for every tile).
struct Tile {
  int l, dxt, dyt, rt, ky, kx;
  int dx0, dy0, r0;
  int ylo, yhi, xlo, xhi;
};

__device__ __forceinline__ Tile tile_of(const TclArgs &a, long long b) {
  Tile t;
  t.kx = int(b % a.ux);
  b /= a.ux;
  t.ky = int(b % a.uy);
  b /= a.uy;
  t.rt = int(b % a.nrt);
  b /= a.nrt;
  t.dyt = int(b % a.ndyt);
  b /= a.ndyt;
  t.dxt = int(b % a.ndxt);
  t.l = int(b / a.ndxt);
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

__global__ void __launch_bounds__(kThreads + 32, 2) xcorr_tcl_kernel(const TclArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *b_hi = smem;                                   // [8][NS][NR][4] TF32 hi
  uint8_t *b_lo = smem + kMaxBEntries * 16;               // lo parts
  float *lp = reinterpret_cast<float *>(smem + 2 * kMaxBEntries * 16);   // [kKY][kLRowF]
  uint64_t *full = reinterpret_cast<uint64_t *>(lp + kKY * kLRowF);
  uint64_t *empty = full + kABufs;
  uint64_t *done = empty + kABufs;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);

  const Tile tl = tile_of(a, blockIdx.x);
  const int ya = tl.ky * kKY, xa = tl.kx * kKX;
  const int y0 = ya > tl.ylo ? ya : tl.ylo;
  const int y1 = ya + kKY < tl.yhi ? ya + kKY : tl.yhi;
  const int x0 = xa > tl.xlo ? xa : tl.xlo;
  const int x1 = xa + kKX < tl.xhi ? xa + kKX : tl.xhi;
  if (y0 >= y1 || x0 >= x1) return;            // no product of the tile here
  const int j_lo = (x0 - xa) >> 3, j_hi = (x1 - xa + 7) >> 3;   // K steps used
  const int NR = 1 << a.nr_log2, NS = kKY + a.ndy - 1;
  const int H = a.H, W = a.W, t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const bool issuer = warp == kThreads / 32;

  if (issuer) {
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
      mbar_init(smem_u32(done), 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  } else {
    // B: entry e = (xc, slot, r) -> R[r0 + r][yr][xa + 4 xc .. + 3] with
    // yr = ya + kKY - 1 - dy0 - slot (zero outside the matrix); entries are
    // consecutive 16-byte rows, all loads of a thread in flight together
    const int nent = 8 * NS * NR;
    const int yc = ya + kKY - 1 - tl.dy0;
    constexpr int kPer = (kMaxBEntries + kThreads - 1) / kThreads;
    float4 bv[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = t + k * kThreads;
      bv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < nent) {
        const int r = e & (NR - 1), q = e >> a.nr_log2;
        const int s = q % NS, xc = q / NS;
        const int yr = yc - s, rr = tl.r0 + r, x = xa + 4 * xc;
        if (rr < a.nr && yr >= 0 && yr < H && x < W) {
          const float *src = a.right + (size_t(rr) * H + yr) * W + x;
          if (a.vec4) {
            bv[k] = __ldg(reinterpret_cast<const float4 *>(src));
          } else {
            bv[k].x = __ldg(src);
            if (x + 1 < W) bv[k].y = __ldg(src + 1);
            if (x + 2 < W) bv[k].z = __ldg(src + 2);
            if (x + 3 < W) bv[k].w = __ldg(src + 3);
          }
        }
      }
    }
    // the left's rows y0 .. y1 - 1, columns xa + dx0 .. + kLRowF - 1
    // (zero outside the matrix): lp[y - y0][p] = L[l][y][xa + dx0 + p]
    {
      const int nl_ent = (y1 - y0) * kLRowF;
      constexpr int kLPer = (kKY * kLRowF + kThreads - 1) / kThreads;
      const float *lrow = a.left + size_t(tl.l) * H * W;
      const int xb = xa + tl.dx0;
      float lv[kLPer];
#pragma unroll
      for (int k = 0; k < kLPer; ++k) {
        const int i = t + k * kThreads;
        const int p = i % kLRowF, ry = i / kLRowF;
        const int x = xb + p;
        lv[k] = 0.f;
        if (i < nl_ent && x >= 0 && x < W) lv[k] = __ldg(lrow + size_t(y0 + ry) * W + x);
      }
#pragma unroll
      for (int k = 0; k < kLPer; ++k) {
        const int i = t + k * kThreads;
        if (i < nl_ent) lp[i] = lv[k];
      }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = t + k * kThreads;
      if (e >= nent) break;
      uint4 hi, lo;
      split_tf32(bv[k].x, hi.x, lo.x);
      split_tf32(bv[k].y, hi.y, lo.y);
      split_tf32(bv[k].z, hi.z, lo.z);
      split_tf32(bv[k].w, hi.w, lo.w);
      *reinterpret_cast<uint4 *>(b_hi + e * 16) = hi;
      *reinterpret_cast<uint4 *>(b_lo + e * 16) = lo;
    }
    // generic-proxy stores -> the tensor cores' (async proxy) reads
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t a_cols = tmem + uint32_t(kN);     // A stage b: columns + kStageCols b
  const int ny = y1 - y0;
  int failed = 0;

  if (issuer) {
    if (lane == 0) {
      const uint32_t bh_base = smem_u32(b_hi), bl_base = smem_u32(b_lo);
      const uint32_t lbo_b = uint32_t(NS * NR * 16);     // next 4 columns x'
      uint32_t fpar = 0;
      int bb = 0;
      for (int i = 0; i < ny; ++i) {
        if (!mbar_wait_bounded(smem_u32(&full[bb]), (fpar >> bb) & 1u)) {
          failed = 1;
          break;
        }
        fpar ^= 1u << bb;
        fence_after_sync();
        // N row n = (dyi, r): right row y - dy0 - dyi, slot
        // (ya + kKY - 1 - y) + dyi, so row n sits n * 16 bytes past it
        const uint32_t s0off = uint32_t((ya + kKY - 1 - (y0 + i)) * NR * 16);
        const uint32_t ab = a_cols + uint32_t(kStageCols * bb);
#pragma unroll
        for (int j = 0; j < kSteps; ++j) {
          if (j < j_lo || j >= j_hi) continue;
          const uint32_t boff = s0off + uint32_t(2 * j) * lbo_b;
          const uint64_t bhi = smem_desc(bh_base + boff, lbo_b, 128);
          const uint64_t blo = smem_desc(bl_base + boff, lbo_b, 128);
          const uint32_t acc = (i > 0 || j > j_lo) ? 1u : 0u;
          mma_tf32_ta(tmem, ab + 16 * j, bhi, acc, kIdesc);
          mma_tf32_ta(tmem, ab + 16 * j, blo, 1u, kIdesc);
          mma_tf32_ta(tmem, ab + 16 * j + 8, bhi, 1u, kIdesc);
        }
        mma_commit(smem_u32(&empty[bb]));
        bb = bb + 1 == kABufs ? 0 : bb + 1;
      }
      mma_commit(smem_u32(done));
      if (!mbar_wait_bounded(smem_u32(done), 0)) failed = 1;
      for (int k = 0; k < kABufs && k < ny; ++k) {
        const int uses = (ny - k + kABufs - 1) / kABufs;
        if (!mbar_wait_bounded(smem_u32(&empty[k]), uint32_t(uses - 1) & 1u)) failed = 1;
      }
    }
  } else {
    // thread: A row m = 32 (warp % 4) + lane (shift dx = dx0 + m), K steps
    // j = warp / 4 and j + 2: the 8 values L[l][y][x' + dx], x' = xa + 8j ..
    // + 7, as TF32 hi and lo
    const int q = warp & 3, jh = warp >> 2;
    const int m = 32 * q + lane;
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    uint32_t epar = 0;
    int bb = 0;
    for (int i = 0; i < ny; ++i) {
      if (i >= kABufs) {
        if (!mbar_wait_bounded(smem_u32(&empty[bb]), (epar >> bb) & 1u)) {
          failed = 1;
          break;
        }
        epar ^= 1u << bb;
        fence_after_sync();
      }
      const float *ls = lp + i * kLRowF + m;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int j = jh + 2 * jj;
        if (j < j_lo || j >= j_hi) continue;
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) split_tf32(ls[8 * j + k], hi[k], lo[k]);
        const uint32_t col = a_cols + uint32_t(kStageCols * bb + 16 * j);
        tmem_st8(lane_base + col, hi);
        tmem_st8(lane_base + col + 8, lo);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&full[bb]));
      bb = bb + 1 == kABufs ? 0 : bb + 1;
    }
    if (!failed && !mbar_wait_bounded(smem_u32(done), 0)) failed = 1;
  }
  failed = __syncthreads_or(failed);
  fence_after_sync();

  if (!failed && !issuer) {
    // partial[unit][n][m]: warp w reads lanes 32 (w % 4) .. + 31 (rows m)
    // and columns 64 (w / 4) .. + 63 (n); for each n the lanes write 32
    // consecutive floats
    const int q = warp & 3, half = warp >> 2;
    float *dst = a.partial + size_t(blockIdx.x) * kTileFloats + 32 * q + lane;
    const uint32_t lane_base = tmem + (uint32_t(32 * q) << 16);
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {
      const int c0 = 64 * half + 32 * j;
      uint32_t v[32];
      tmem_ld32(lane_base + uint32_t(c0), v);
#pragma unroll
      for (int k = 0; k < 32; ++k) dst[size_t(c0 + k) * kM] = __uint_as_float(v[k]);
    }
  } else if (failed && t == 0) {
    atomicOr(&g_tcl_status, 1);
  }
  fence_before_sync();
  __syncthreads();
  if (issuer) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// out[l][r][oy][ox] = the sum, in unit order, of the partial tiles of the
// units of its tile that hold any of its products.
__global__ void __launch_bounds__(256) xcorr_tcl_sum_kernel(const TclArgs a) {
  const int ndy = 2 * a.H - 1, ndx = 2 * a.W - 1;
  const long long total = (long long)a.nl * a.nr * ndy * ndx;
  const int NR = 1 << a.nr_log2;
  for (long long o = (long long)blockIdx.x * blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    long long rest = o;
    const int ox = int(rest % ndx);
    rest /= ndx;
    const int oy = int(rest % ndy);
    rest /= ndy;
    const int r = int(rest % a.nr);
    const int l = int(rest / a.nr);
    const int dxt = ox / kM, m = ox - dxt * kM;
    const int dyt = oy / a.ndy, dyi = oy - dyt * a.ndy;
    const int rt = r >> a.nr_log2, n = (dyi << a.nr_log2) + (r & (NR - 1));
    const long long b0 = ((((long long)l * a.ndxt + dxt) * a.ndyt + dyt) * a.nrt + rt) * a.uy;
    const Tile tl = tile_of(a, b0 * a.ux);
    const int ky0 = tl.ylo / kKY, ky1 = (tl.yhi + kKY - 1) / kKY;
    const int kx0 = tl.xlo / kKX, kx1 = (tl.xhi + kKX - 1) / kKX;
    // units in order (ky, kx); loads in batches of 8 so that they are in
    // flight together, the adds in the same fixed order
    float s = 0.f;
    const float *base = a.partial + size_t(n) * kM + m;
    for (int ky = ky0; ky < ky1; ++ky) {
      const float *row = base + ((b0 + ky) * a.ux) * size_t(kTileFloats);
      for (int kx = kx0; kx < kx1; kx += 8) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          v[k] = kx + k < kx1 ? __ldg(row + size_t(kx + k) * kTileFloats) : 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (kx + k < kx1) s += v[k];
      }
    }
    a.out[o] = s;
  }
}

TclArgs make_args(const float *left, int nl, const float *right, int nr, int H, int W,
                  float *out) {
  TclArgs a;
  a.left = left;
  a.right = right;
  a.out = out;
  a.partial = nullptr;
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
  a.vec4 = (W % 4 == 0 && (reinterpret_cast<uintptr_t>(right) & 15) == 0) ? 1 : 0;
  return a;
}

long long units_of(const TclArgs &a) {
  return (long long)a.nl * a.ndxt * a.ndyt * a.nrt * a.uy * a.ux;
}

}  // namespace

size_t scratch_bytes(int nl, int nr, int H, int W) {
  const TclArgs a = make_args(nullptr, nl, nullptr, nr, H, W, nullptr);
  return size_t(units_of(a)) * kTileFloats * sizeof(float);
}

cudaError_t launch(const float *left, int nl, const float *right, int nr, int H, int W,
                   float *out, float *scratch, cudaStream_t stream) {
  TclArgs a = make_args(left, nl, right, nr, H, W, out);
  a.partial = scratch;
  const long long units = units_of(a);
  if (units > 0x7fffffffLL || scratch == nullptr) return cudaErrorInvalidValue;
  const size_t smem = 2 * size_t(kMaxBEntries) * 16 + size_t(kKY) * kLRowF * sizeof(float) +
                      (2 * kABufs + 2) * 8;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(xcorr_tcl_kernel));
  if (e != cudaSuccess) return e;
  xcorr_tcl_kernel<<<unsigned(units), kThreads + 32, smem, stream>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long outs = (long long)nl * nr * (2LL * H - 1) * (2LL * W - 1);
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
