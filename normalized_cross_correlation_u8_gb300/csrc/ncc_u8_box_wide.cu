// ncc_u8_box_wide.cu -- the box form of the fast kernel (ncc_u8_box.cu) for
// templates of 17 .. 32 words, in a translation unit of its own so that it
// compiles beside the others (kernels: ncc_u8_kernels.cuh).
#include "ncc_u8_kernels.cuh"

namespace corr {

cudaError_t ncc_u8_launch_fixed_box_wide(const ncc::NccArgs &a, size_t smem, int vb,
                                         cudaStream_t stream) {
  using namespace ncc;
  constexpr int R = kBoxRows;
  constexpr int kWide = kMaxFixedWords - kNarrowWords;
  static constexpr auto table =
      fixed_launchers<R, true, kNarrowWords + 1>(std::make_integer_sequence<int, kWide>{});
  if (a.wtw <= kNarrowWords || a.wtw > kMaxFixedWords || a.rows != R)
    return cudaErrorInvalidValue;
  return table[a.wtw - kNarrowWords - 1](a, smem, vb, stream);
}

}  // namespace corr
