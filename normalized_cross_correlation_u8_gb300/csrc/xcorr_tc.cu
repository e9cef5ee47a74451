// xcorr_tc.cu -- float32 full 2D cross-correlation of many small matrices
// (n-to-m batches, H, W <= 16) on the sm_103a tensor cores.
//
// The artifact README's n-to-m case ("Efficient GPU-accelerated Parallel
// Cross-correlation", kernel overview: multi-matrix-both, every left against
// every right) reuses each matrix against many others.  Here that reuse is
// written as a dense contraction.  With x' the column of the right matrix,
//
//   out[l][r][dy][dx] = sum_{y, x'} L_l[y][x' + dx] * R_r[y - dy][x'],
//
// (terms with an index outside a matrix are zero), so for one CTA tile
//   D[m][n] = sum_k A[m][k] * B[n][k],
//   m = (left l, shift dx)   A[m][(y, x')] = L_l[y][x' + dx]    (Toeplitz of L)
//   n = (shift dy, right r)  B[n][(y, x')] = R_r[y - dy][x']    (rows of R; r fastest)
//   k = (overlap row y, right column x').
// A CTA owns 4 lefts x R rights and every shift of those pairs: M = 4
// lefts x 32 shift slots dx, N = 32 shift slots dy x R rights, K = every
// row y and column x' (R = 4; R = 2 for batches too small to fill the GPU
// with 4 x 4 tiles, so that twice the CTAs run, two per SM).  All CTAs
// therefore do the same work, and each left's R x (2H-1)(2W-1) outputs --
// contiguous in memory -- are written by one CTA as one run in whole
// 32-byte sectors (a store that ends mid-sector costs a DRAM fill, which
// dominated earlier layouts).
//
// Operand placement.  B is read from shared memory in the tensor cores'
// no-swizzle K-major layout (8 rows x 16 bytes per core matrix, the two
// core matrices of one 8-deep K step LBO bytes apart, 8-row groups SBO
// bytes apart).  The CTA's rights are staged once as [x'/4][row slot][right]
// [4 floats] with rows in reverse order, so the N rows of consecutive
// shifts dy are consecutive slots: one descriptor per (y, K step), no
// per-row copy.  A, the Toeplitz rows of L, is written per overlap row by
// eight builder warps straight from registers into tensor memory
// (tcgen05.st) and read from there by the MMA, rotating through kABufs
// column ranges: the products are then bound by the tensor cores, not by
// shared-memory bandwidth.
//
// Precision: the tensor cores multiply TF32 operands (10 mantissa bits).
// Each operand is split v = hi + lo with hi = tf32(v) and lo = tf32(v - hi)
// (both rounded to nearest), and a product is formed as
// hi*hi + hi*lo + lo*hi, dropping lo*lo (the three-pass TF32 scheme of
// NVIDIA's CUTLASS "3xTF32" GEMMs; split-operand tensor-core products as in
// Markidis et al., "NVIDIA Tensor Core Programmability, Performance &
// Precision", 2018).  Each product is then exact to about 3 * 2^-22 of
// |l * r|, and the sums accumulate in FP32 in tensor memory: well inside
// the 1e-5 * sum |l * r| bound of the scalar kernels.
//
// Issue: one warp issues the tcgen05.mma instructions (3 per K step of 8,
// M = 128, N = 128, kind::tf32) into a 128-column FP32 accumulator in
// tensor memory and commits each row's group to an mbarrier; after the
// last row the builder warps read the accumulator back with tcgen05.ld
// (lanes = the 32 shifts dx of one left), turn each pair's block around in
// shared memory and write each left's run out row-major.  Every wait on an
// mbarrier is bounded: after about a second the CTA gives up, records it in
// a device flag that corr_device_status() reports, frees its tensor memory
// and returns.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "internal.cuh"
#include "tc_common.cuh"

namespace corr {
namespace tc {
namespace {

using namespace tcx;

constexpr int kThreads = 256;           // builder threads: 2 per A row (one K step each)
constexpr int kABufs = 4;                // A stages in flight (overlap rows)
constexpr int kLefts = 4;                 // lefts per tile (M = kLefts x kSlots)
constexpr int kSlots = 32;                // shifts dx (dy) per left (right): 2W-1 <= 31
constexpr int kM = kLefts * kSlots;       // 128
constexpr int kPadL = 15;                 // zero columns left of a staged left row
constexpr int kLRow = 64;                 // floats per staged left row
constexpr int kSlotsR = 48;               // right row slots (2H + 30 <= 47 used)
constexpr int kStreams = 2;               // row streams: an issuing warp and accumulator each

// A tile of kLefts lefts x R rights (R = 4, or 2 for batches too small to
// fill the GPU with 4 x 4 tiles: half as much work per CTA, and tensor
// memory for two CTAs per SM).
template <int R>
struct TileShape {
  static constexpr int kRights = R;
  static constexpr int kN = R * kSlots;                       // 128 or 64
  static constexpr int kBBytes = 4 * kSlotsR * R * 16;        // staged B (hi or lo): 12 / 6 KB
  static constexpr int kRunFloats = R * 31 * 31;              // one left's outputs
  // 2 accumulators + kABufs A stages (32 columns each), a power of two
  static constexpr uint32_t kTmemCols = R == 4 ? 512 : 256;
  static constexpr uint32_t kIdesc = tcx::idesc_tf32(kM, kN);
  static constexpr int kMinBlocks = R == 4 ? 1 : 2;           // CTAs per SM
  static_assert(kStreams * kN + kABufs * 32 <= int(kTmemCols), "tensor memory plan");
};

struct TcArgs {
  const float *left;
  const float *right;
  float *out;
  int nl, nr, H, W;
  int mtiles, rtiles;    // tiles of kLefts lefts x R rights
  int vec4;              // rows readable as float4
  int stall;             // test of the bounded waits: the last commit is left out
};

__device__ int g_tc_status;   // bit 0: a bounded wait gave up

// KH: 8-deep K steps per overlap row (1 for W <= 8, else 2), a template
// parameter so the row's 3 KH tensor-core instructions issue as one
// straight-line sequence.
//
// Warp roles: warps 0-7 write the A operand of one overlap row at a time
// into kABufs rotating tensor-memory stages (then, after the last row,
// read the accumulators out); warps 8 and 9 issue the tensor-core
// instructions, for the even and the odd overlap rows, each into its own
// accumulator (one thread issues a 128x128x8 MMA in about 54 cycles against
// the tensor pipe's 64, with its per-row bookkeeping on top, and the pipe
// queues almost nothing ahead; two issuers keep it busy, and each chain of
// accumulates is at most 8 rows x KH x 3 = 48 long).  Stream s owns stages
// 2s and 2s + 1; stage b is handed over through two mbarriers: full[b] (one
// arrival per builder warp once its part is in tensor memory) and empty[b]
// (a tcgen05.commit: the products that read it have completed).
template <int KH, int R>
__global__ void __launch_bounds__(kThreads + 32 * kStreams, TileShape<R>::kMinBlocks)
    xcorr_tc_kernel(const TcArgs a) {
  using TS = TileShape<R>;
  constexpr int kRights = TS::kRights, kN = TS::kN, kBBytes = TS::kBBytes;
  constexpr int kRunFloats = TS::kRunFloats;
  constexpr uint32_t kTmemCols = TS::kTmemCols, kIdesc = TS::kIdesc;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *b_hi = smem;                                   // [4][kSlotsR][kRights][4] TF32 hi
  uint8_t *b_lo = smem + kBBytes;                         // same, lo parts
  float *lp = reinterpret_cast<float *>(smem + 2 * kBBytes);   // [kLefts][16][kLRow]
  float *runs = lp + kLefts * 16 * kLRow;                 // [kLefts][kRunFloats]
  uint64_t *full = reinterpret_cast<uint64_t *>(runs + kLefts * kRunFloats);
  uint64_t *empty = full + kABufs;
  uint64_t *done = empty + kABufs;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);

  const int H = a.H, W = a.W, t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int stream = warp - kThreads / 32;      // issuer warps: 0, 1; builders < 0
  const bool issuer = stream >= 0;
  const int rt = blockIdx.x % a.rtiles, mt = blockIdx.x / a.rtiles;
  const int l0 = mt * kLefts, r0 = rt * kRights;

  if (stream == 0) {
    // tensor memory: accumulators at columns 0..127 and 128..255, A stages above
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
      mbar_init(smem_u32(done), kStreams);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  } else if (!issuer) {
    // the tile's rights as TF32 hi / lo in the B layout: entry e = (xc,
    // slot, rq) (rq fastest, so entries are consecutive 16-byte rows) holds
    // R[r0 + rq][yr][4 xc .. 4 xc + 3] with yr = 2H - 2 - slot, zero
    // outside the matrix
    constexpr int kBEntries = 4 * kSlotsR * kRights;
    constexpr int kBPer = (kBEntries + kThreads - 1) / kThreads;   // all loads in flight at once
    float4 bv[kBPer];
#pragma unroll
    for (int k = 0; k < kBPer; ++k) {
      const int e = t + k * kThreads;
      const int rq = e & (kRights - 1), q = e / kRights;
      const int slot = q % kSlotsR, xc = q / kSlotsR;
      const int yr = 2 * H - 2 - slot;
      bv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < kBEntries && r0 + rq < a.nr && yr >= 0 && yr < H && 4 * xc < W) {
        const float *src = a.right + (size_t(r0 + rq) * H + yr) * W + 4 * xc;
        if (a.vec4) {
          bv[k] = __ldg(reinterpret_cast<const float4 *>(src));
        } else {
          bv[k].x = __ldg(src);
          if (4 * xc + 1 < W) bv[k].y = __ldg(src + 1);
          if (4 * xc + 2 < W) bv[k].z = __ldg(src + 2);
          if (4 * xc + 3 < W) bv[k].w = __ldg(src + 3);
        }
      }
    }
    // zero-padded copies of the tile's lefts (a thread per row quarter):
    //   lp[lt][y][p] = L[l0+lt][y][p - kPadL]       (16 rows, H used)
    {
      const int lt = t >> 6, y = (t >> 2) & 15, q = t & 3;
      float v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int x = 16 * q + k - kPadL;
        v[k] = 0.f;
        if (y < H && l0 + lt < a.nl && x >= 0 && x < W)
          v[k] = __ldg(a.left + (size_t(l0 + lt) * H + y) * W + x);
      }
      float4 *dst = reinterpret_cast<float4 *>(lp + (lt * 16 + y) * kLRow + 16 * q);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    }
#pragma unroll
    for (int k = 0; k < kBPer; ++k) {
      const int e = t + k * kThreads;
      if (e >= kBEntries) break;
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
  const uint32_t a_cols = tmem + uint32_t(kStreams * kN);   // A stage b: columns + 32 b
  int failed = 0;

  if (issuer) {
    if (lane == 0) {
      const uint32_t bh_base = smem_u32(b_hi), bl_base = smem_u32(b_lo);
      constexpr uint32_t kLboB = kSlotsR * kRights * 16;   // next 4 columns x'
      const uint32_t d = tmem + uint32_t(stream * kN);
      const int rows = (H - stream + 1) / 2;               // rows stream, stream + 2, ...
      for (int k = 0; k < rows; ++k) {
        const int i = 2 * k + stream, bb = 2 * stream + (k & 1);
        if (!mbar_wait_bounded(smem_u32(&full[bb]), uint32_t(k >> 1) & 1u)) {
          failed = 1;
          break;
        }
        fence_after_sync();
        // N row n = (dyi, rq): right row y - dy = y + (H-1) - dyi, slot
        // H - 1 - y + dyi, so row n sits n * 16 bytes past slot H - 1 - y
        const uint32_t s0off = uint32_t((H - 1 - i) * kRights * 16);
        const uint32_t ab = a_cols + uint32_t(32 * bb);
#pragma unroll
        for (int h = 0; h < KH; ++h) {
          const uint32_t boff = s0off + uint32_t(2 * h) * kLboB;
          const uint64_t bhi = smem_desc(bh_base + boff, kLboB, 128);
          const uint64_t blo = smem_desc(bl_base + boff, kLboB, 128);
          mma3_tf32_ta(d, ab + 8 * h, ab + 16 + 8 * h, bhi, blo, (k > 0 || h > 0) ? 1u : 0u,
                       kIdesc);
        }
        mma_commit(smem_u32(&empty[bb]));
      }
      // every product issued so far, then the accumulator is final (left
      // out under the stall test: every wait on it then runs out)
      if (!a.stall) mma_commit(smem_u32(done));
      if (!mbar_wait_bounded(smem_u32(done), 0)) failed = 1;
      // and each of this stream's stages: its last release has landed (no
      // arrival on this CTA's shared memory is left pending when it exits)
      for (int b = 0; b < 2 && b < rows; ++b) {
        const int uses = (rows - b + 1) / 2;             // stream rows b, b + 2, ...
        if (!mbar_wait_bounded(smem_u32(&empty[2 * stream + b]), uint32_t(uses - 1) & 1u))
          failed = 1;
      }
    }
  } else {
    // this thread writes A row m = 32 (warp % 4) + lane (left m / 32, slot
    // n = m % 32: dx = n - (W-1)), K step h = warp / 4: the 8 values
    // L[l0+lt][y][x' + dx], x' = 8h .. 8h + 7, as TF32 hi and lo
    const int lt = warp & 3, h = warp >> 2, n = lane;
    const bool active = h < KH;
    const float *lsrc = lp + lt * 16 * kLRow + n + kPadL - (W - 1) + 8 * h;
    const uint32_t lane_base = uint32_t(32 * lt) << 16;
    uint32_t epar = 0;        // bit k: parity of empty[k]'s next completion
    for (int i = 0; i < H; ++i) {
      // row i: stream i % 2, its row k = i / 2, stage 2 (i % 2) + k % 2; the
      // products that read the stage two rows of the stream ago are done
      const int bb = 2 * (i & 1) + ((i >> 1) & 1);
      if (i >= kABufs) {
        if (!mbar_wait_bounded(smem_u32(&empty[bb]), (epar >> bb) & 1u)) {
          failed = 1;
          break;
        }
        epar ^= 1u << bb;
        fence_after_sync();
      }
      if (active) {
        const float *ls = lsrc + i * kLRow;
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) split_tf32(ls[k], hi[k], lo[k]);
        const uint32_t col = a_cols + uint32_t(32 * bb + 8 * h);
        tmem_st8(lane_base + col, hi);
        tmem_st8(lane_base + col + 16, lo);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&full[bb]));
    }
    if (!failed && !mbar_wait_bounded(smem_u32(done), 0)) failed = 1;
  }
  failed = __syncthreads_or(failed);
  fence_after_sync();

  if (!failed && !issuer) {
    // epilogue: warp w reads lanes 32 (w % 4) .. + 31 (left l0 + w % 4,
    // shift slots dx) and columns kN / 2 (w / 4) .. + kN / 2 - 1 (shift
    // slots dy 16 (w / 4) .. + 15 of all R rights) of both accumulators
    // into the left's output run, laid out as in memory: [right][dy][dx]
    const int lt = warp & 3, half = warp >> 2;
    const int ndy = 2 * H - 1, ndx = 2 * W - 1, per_pair = ndy * ndx;
    float *lrun = runs + lt * kRunFloats;
    const uint32_t lane_base = tmem + (uint32_t(32 * lt) << 16);
#pragma unroll 1
    for (int j = 0; j < kN / 64; ++j) {
      const int c0 = (kN / 2) * half + 32 * j;
      uint32_t v[32], w[32];
      tmem_ld32(lane_base + uint32_t(c0), v);           // even rows' accumulator
      tmem_ld32(lane_base + uint32_t(kN + c0), w);      // odd rows' (none when H = 1)
      if (H == 1) {
#pragma unroll
        for (int k = 0; k < 32; ++k) w[k] = 0u;
      }
      if (lane < ndx) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int c = c0 + k, dyi = c / kRights;     // c = dyi * kRights + rq
          if (dyi < ndy)
            lrun[(c % kRights) * per_pair + dyi * ndx + lane] =
                __uint_as_float(v[k]) + __uint_as_float(w[k]);
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");   // builder warps only
    // left l0 + lt: its pairs with rights r0 .. r0 + nrr - 1 are one
    // contiguous run; warps w and w + 4 store alternate 32-float chunks of
    // it at 128-byte-aligned addresses (whole sectors but at the run's ends)
    const int l = l0 + lt;
    const int nrr = a.nr - r0 < kRights ? a.nr - r0 : kRights;
    if (l < a.nl) {
      float *run = a.out + (size_t(l) * a.nr + r0) * per_pair;
      const int len = nrr * per_pair;
      const int off = int((reinterpret_cast<uintptr_t>(run) >> 2) & 31);   // floats past 128 B
#pragma unroll 4
      for (int f = 32 * half + lane - off; f < len; f += 64)
        if (f >= 0) run[f] = lrun[f];
    }
  } else if (failed && t == 0) {
    atomicOr(&g_tc_status, 1);
  }
  fence_before_sync();
  __syncthreads();
  if (stream == 0) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

bool supported(int nl, int nr, int H, int W) {
  (void)nl;
  (void)nr;
  return H >= 1 && H <= 16 && W >= 1 && W <= 16;
}

cudaError_t launch(const float *left, int nl, const float *right, int nr, int H, int W,
                   float *out, cudaStream_t stream) {
  if (!supported(nl, nr, H, W)) return cudaErrorInvalidValue;
  TcArgs a;
  a.left = left;
  a.right = right;
  a.out = out;
  a.nl = nl;
  a.nr = nr;
  a.H = H;
  a.W = W;
  a.mtiles = (nl + kLefts - 1) / kLefts;
  // 4 rights per tile once that gives 100+ tiles (measured on GB300: 32 x
  // 64 of 16^2 9.8 us with 4 against 10.4 with 2), else 2 (16 x 16 of 16^2
  // 8.1 against 9.5 us; 8 x 8 of 12^2 6.7 against 7.8 us)
  const int R = (long long)a.mtiles * ((nr + 3) / 4) >= 100 ? 4 : 2;
  a.rtiles = (nr + R - 1) / R;
  a.vec4 = (W % 4 == 0 && (reinterpret_cast<uintptr_t>(right) & 15) == 0) ? 1 : 0;
  // CORR_XCORR_TC_STALL=1 (read on every call): a test of the failure path
  // -- the kernel's last completion barrier is never signalled, each wait
  // on it gives up after about a second, the outputs stay unwritten and
  // corr_device_status() reports CORR_ETIMEOUT
  {
    const char *v = getenv("CORR_XCORR_TC_STALL");
    a.stall = (v && v[0] == '1' && v[1] == '\0') ? 1 : 0;
  }
  const long long blocks = (long long)a.mtiles * a.rtiles;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t bbytes = size_t(4) * kSlotsR * R * 16, run = size_t(R) * 31 * 31;
  const size_t smem = 2 * bbytes + size_t(kLefts) * 16 * kLRow * sizeof(float) +
                      size_t(kLefts) * run * sizeof(float) + (2 * kABufs + 2) * 8;
  auto kern = R == 4 ? (W > 8 ? xcorr_tc_kernel<2, 4> : xcorr_tc_kernel<1, 4>)
                     : (W > 8 ? xcorr_tc_kernel<2, 2> : xcorr_tc_kernel<1, 2>);
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern));
  if (e != cudaSuccess) return e;
  kern<<<unsigned(blocks), kThreads + 32 * kStreams, smem, stream>>>(a);
  return cudaGetLastError();
}

// Reads and clears the device flag of bounded waits that gave up.
cudaError_t take_status(int *gave_up) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(int));
  if (e != cudaSuccess) return e;
  *gave_up = v;
  if (v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int));
  }
  return e;
}

}  // namespace tc
}  // namespace corr
