// ncc_u8_box.cu -- the box-sum form of the 8-bit NCC fast kernel for
// templates of 1 .. 16 words (kernels: ncc_u8_kernels.cuh).
//
// SumI and SumISq depend on the template's size only: they are box filters
// of I and I^2.  A box filter separates into a column step (each column of
// the tile: windows of ht pixels, sliding down by one row) and a row step
// (each output row: windows of wt column sums, sliding right by one column),
// both in unsigned 32-bit arithmetic that is exact here (every partial sum
// is below 2^32), so the sums equal the direct ones bit for bit.  The tiled
// kernel forms them from the tile it already holds in shared memory, and
// its dp4a loop accumulates SumIT alone: one unsigned dp4a per 4 pixels
// instead of the three of The CUDA Handbook ch. 15, section 15.5.  This
// reformulation is not on the pages.
#include "ncc_u8_kernels.cuh"

static_assert(corr::ncc::kBoxNarrowWords >= 0 &&
                  corr::ncc::kBoxNarrowWords < corr::ncc::kNarrowWords,
              "narrow box widths must be a strict subset of ncc_u8_box.cu's table");

namespace corr {

cudaError_t ncc_u8_launch_box(const ncc::NccArgs &a, size_t smem, int vb,
                              cudaStream_t stream) {
  using namespace ncc;
  if (a.wtw < 1 || a.wtw > kMaxFixedWords) return cudaErrorInvalidValue;
  if (a.wtw > kNarrowWords) return ncc_u8_launch_fixed_box_wide(a, smem, vb, stream);
  // a.rows output rows per half-warp: kBoxRows, or 1 for narrow templates
  // (the launch geometry in a.units was computed for it)
  static constexpr auto narrow = fixed_launchers<1, true, 1>(
      std::make_integer_sequence<int, kBoxNarrowWords>{});
  static constexpr auto table = fixed_launchers<kBoxRows, true, 1>(
      std::make_integer_sequence<int, kNarrowWords>{});
  if (a.rows == kBoxRows) return table[a.wtw - 1](a, smem, vb, stream);
  if (a.rows == 1 && a.wtw <= kBoxNarrowWords) return narrow[a.wtw - 1](a, smem, vb, stream);
  return cudaErrorInvalidValue;
}

}  // namespace corr
