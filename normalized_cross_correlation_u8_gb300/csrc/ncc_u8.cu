// ncc_u8.cu -- 8-bit normalized cross-correlation on sm_103a: the entry
// point, the general kernel's instantiation and the fast kernel for
// templates of 1 .. 16 words (method and kernels: ncc_u8_kernels.cuh).
#include "ncc_u8_kernels.cuh"

namespace corr {

using namespace ncc;

cudaError_t ncc_u8_launch(const uint8_t *image, int w, int h, size_t pitch,
                          const uint8_t *tmpl, int wt, int ht,
                          uint32_t *sums_out, float *coef_out, int method,
                          cudaStream_t stream) {
  constexpr int R = CORR_NCC_ROWS;
  NccArgs a;
  a.image = image;
  a.tmpl = tmpl;
  a.sums = sums_out;
  a.coef = coef_out;
  a.w = w;
  a.pitch = pitch;
  a.h = h;
  a.wt = wt;
  a.ht = ht;
  a.wtw = (wt + 3) / 4;
  a.tail = wt % 4;
  a.tail_ones = a.tail ? 0x01010101u >> (8 * (4 - a.tail)) : 0x01010101u;
  a.tail_mask = a.tail ? 0xffffffffu >> (8 * (4 - a.tail)) : 0xffffffffu;
  a.wtp = (a.wtw + 3) & ~3;
  a.ow = w - wt + 1;
  a.oh = h - ht + 1;
  a.plane = size_t(a.ow) * a.oh;
  a.rows = R;
  a.staged = 0;

  // whole-vector staging needs every row start and width on the vector size
  const bool aligned8 =
      (reinterpret_cast<uintptr_t>(image) & 7) == 0 && (w & 7) == 0 && (pitch & 7) == 0;
  const bool aligned16 =
      (reinterpret_cast<uintptr_t>(image) & 15) == 0 && (w & 15) == 0 && (pitch & 15) == 0;
  if (a.wtw >= 1 && a.wtw <= kMaxFixedWords) {
    const bool box = method == kMethodBox;
    const int warps = box ? kBoxWarps : kWarpsPerCta;   // row groups per tile
    auto tiles_for = [&](int rows) {
      return (long long)((a.ow + kHalfUnitCols - 1) / kHalfUnitCols) *
             ((a.oh + 2 * rows * warps - 1) / (2 * rows * warps));
    };
    int rows = box ? kBoxRows : R;
    if (box && kBoxRows != 1 && a.wtw <= kBoxNarrowWords &&
        tiles_for(kBoxRows) < (long long)CORR_NCC_BOX_NARROW_TILES_PER_SM * device_sm_count())
      rows = 1;
    a.rows = rows;
    a.staged = !box || (long long)a.wtw * ht <= CORR_NCC_STAGED_BOX_WORDS;
    const int ty = 2 * rows * warps;
    const size_t ts = fixed_tile_layout(ht, a.wtw, a.wtp, rows, warps,
                                        box ? kBoxSplit : kSplit, box ? 1 : 3, box, wt).total;
    if (ts > 200 * 1024) goto general;   // very tall template: general path
    a.tiles_x = (a.ow + kHalfUnitCols - 1) / kHalfUnitCols;
    const long long tiles = (long long)a.tiles_x * ((a.oh + ty - 1) / ty);
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    a.units = int(tiles);
    const int vb = aligned16 ? 16 : aligned8 ? 8 : 1;
    if (box) return ncc_u8_launch_box(a, ts, vb, stream);
    if (a.wtw > kNarrowWords) return ncc_u8_launch_fixed_wide(a, ts, vb, stream);
    static constexpr auto table =
        fixed_launchers<R, false, 1>(std::make_integer_sequence<int, kNarrowWords>{});
    return table[a.wtw - 1](a, ts, vb, stream);
  }
general:
  // the general kernel walks template words one at a time: rows packed at
  // their own word count, not padded to whole 16-byte vectors
  a.wtp = a.wtw;
  const size_t smem = size_t(ht) * a.wtp * 4;
  a.tiles_x = (a.ow + kUnitCols - 1) / kUnitCols;
  const long long units = (long long)a.tiles_x * ((a.oh + R - 1) / R);
  if (units > 0x7fffffffLL - kWarpsPerCta) return cudaErrorInvalidConfiguration;
  a.units = int(units);
  return launch(ncc_u8_general_kernel<R>, a, smem, stream);
}

}  // namespace corr
