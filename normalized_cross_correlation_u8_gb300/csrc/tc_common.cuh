// tc_common.cuh -- device helpers shared by the tensor-core kernels of
// libcorr.so (xcorr_tc.cu, xcorr_tcl.cu): shared-memory matrix descriptors,
// TF32 operand splitting, mbarrier waits with a bound, and the tcgen05
// instructions the kernels issue, as inline PTX for sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace corr {
namespace tcx {

constexpr long long kWaitCycles = 1LL << 31;   // ~1 s at 2 GHz

// Instruction descriptor of tcgen05.mma kind::tf32 with an M x N FP32
// accumulator: D = F32 (bits 4-5 = 1), A = B = TF32 (bits 7-9, 10-12 = 2),
// both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(N >> 3) << 17) |
         (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor (tcgen05): start address, leading (K)
// and stride (M / N) byte offsets, each >> 4 in 14 bits; descriptor version
// 1 at bit 46; base offset 0, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t((lbo & 0x3FFFFu) >> 4) << 16) |
         (uint64_t((sbo & 0x3FFFFu) >> 4) << 32) | (uint64_t(1) << 46);
}

// v rounded to TF32 (10 explicit mantissa bits), to nearest with ties away
// from zero, as an FP32 bit pattern with the low 13 bits clear: adding half
// of the dropped unit (bit 12) to the sign-magnitude pattern carries into
// the kept bits exactly when the dropped part is at least half, and a
// carry out of the mantissa moves to the next binade (or to infinity) as
// rounding does.  Integer ALU work only; the same bits as cvt.rna.tf32.f32
// for every finite v and for infinities.
__device__ __forceinline__ uint32_t tf32_rna(float v) {
  return (__float_as_uint(v) + 0x1000u) & 0xFFFFE000u;
}

// v = hi + lo (+ a remainder below 2^-22 |v|), hi and lo TF32 bit patterns.
__device__ __forceinline__ void split_tf32(float v, uint32_t &hi, uint32_t &lo) {
  hi = tf32_rna(v);
  lo = tf32_rna(v - __uint_as_float(hi));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, letting the hardware suspend the thread for up to
// `ns` nanoseconds while the phase is incomplete (it resumes as soon as the
// phase completes), so that a waiting warp takes no issue slots from the
// warps that share its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of the barrier to complete; false after about a
// second without it.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitCycles) return false;
  return true;
}

// mbar_wait_bounded for threads whose waits should leave the scheduler to
// others: each try suspends the thread for up to 20 us.
__device__ __forceinline__ bool mbar_wait_bounded_sleep(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, 20000u))
    if (clock64() - t0 > kWaitCycles) return false;
  return true;
}

// Three tcgen05.mma kind::tf32 with A in tensor memory into one FP32
// accumulator: A a0 x B b0 (accumulating unless first == 0), A a0 x B b1,
// A a1 x B b0 -- hi*hi, hi*lo and lo*hi of one K step.
__device__ __forceinline__ void mma3_tf32_ta(uint32_t d, uint32_t a0, uint32_t a1, uint64_t b0,
                                             uint64_t b1, uint32_t first, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "setp.eq.b32 q, %5, %5;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %3, %5, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %4, %5, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%2], %3, %5, q;\n\t}"
      ::"r"(d), "r"(a0), "r"(a1), "l"(b0), "l"(b1), "r"(idesc), "r"(first)
      : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on the barrier once every tcgen05.mma this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive FP32 columns of this warp's 32 accumulator lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 8 consecutive 32-bit columns of this warp's 32 accumulator lanes.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

}  // namespace tcx
}  // namespace corr
