// ncc_u8_wide.cu -- the fast 8-bit NCC kernel for templates of 17 .. 32
// words (68 .. 128 pixels wide), in a translation unit of its own so that it
// compiles beside ncc_u8.cu (kernels: ncc_u8_kernels.cuh).
#include "ncc_u8_kernels.cuh"

namespace corr {

cudaError_t ncc_u8_launch_fixed_wide(const ncc::NccArgs &a, size_t smem, int vb,
                                     cudaStream_t stream) {
  using namespace ncc;
  constexpr int R = CORR_NCC_ROWS;
  constexpr int kWide = kMaxFixedWords - kNarrowWords;
  static constexpr auto table =
      fixed_launchers<R, false, kNarrowWords + 1>(std::make_integer_sequence<int, kWide>{});
  if (a.wtw <= kNarrowWords || a.wtw > kMaxFixedWords) return cudaErrorInvalidValue;
  return table[a.wtw - kNarrowWords - 1](a, smem, vb, stream);
}

}  // namespace corr
