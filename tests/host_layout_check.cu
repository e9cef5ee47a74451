// Host-only check of the u8 fast kernel's shared-memory layout (no kernel is
// launched and no GPU is needed): for every template width the fast path
// instantiates and every height up to the pixel limit, in both methods and
// both row counts, the regions fixed_tile_layout places are 16-byte aligned,
// disjoint, and as large as what the kernel later writes over them.
#include <stdio.h>

#include "../normalized_cross_correlation_u8_gb300/csrc/ncc_u8_kernels.cuh"

using namespace corr::ncc;

static int fails = 0;
#define CHECK(c, ...)                        \
  do {                                       \
    if (!(c)) {                              \
      if (fails < 20) printf(__VA_ARGS__);   \
      ++fails;                               \
    }                                        \
  } while (0)

int main() {
  long cases = 0;
  // finished sums: the chunks 2k (and 2k + 1) of 8 consecutive k fill all
  // 32 banks
  for (int g = 0; g < 4; ++g)
    for (int odd = 0; odd < 2; ++odd) {
      unsigned banks = 0;
      for (int k = 8 * (g % 2); k < 8 * (g % 2) + 8; ++k)
        for (int w = 0; w < 4; ++w) banks |= 1u << ((4 * box_s_chunk(2 * k + odd + 32 * (g / 2)) + w) & 31);
      CHECK(banks == 0xffffffffu, "finished-sum chunks of group %d conflict\n", g);
    }
  for (int wt = 1; wt <= 4 * kMaxFixedWords; ++wt) {
    const int wtw = (wt + 3) / 4, wtp = (wtw + 3) & ~3;
    // column sums: stride 16 mod 32, room for the last skewed column, and
    // the row pass's reads (columns 8 k + j of two rows) on 32 distinct banks
    const int vs = box_v_stride(wt);
    const int nv = kHalfUnitCols + wt - 1;
    CHECK(vs % 32 == 16, "wt %d: v stride %d not 16 mod 32\n", wt, vs);
    CHECK(box_v_col(nv - 1) < vs, "wt %d: v stride %d too small\n", wt, vs);
    for (int x0 = 0; x0 + 8 * 15 + 7 < nv; x0 += 1) {
      unsigned banks = 0;
      for (int row = 0; row < 2; ++row)
        for (int k = 0; k < 16; ++k)
          banks |= 1u << ((row * vs + box_v_col(x0 + 8 * k)) & 31);
      CHECK(banks == 0xffffffffu, "wt %d x0 %d: row-pass reads conflict\n", wt, x0);
    }
    for (int ht = 1; ht * wt <= 66051; ++ht) {
      for (int box = 0; box < 2; ++box) {
        for (int rows = 1; rows <= 2; ++rows) {
          const int warps = box ? kBoxWarps : kWarpsPerCta;
          const int groups = box ? kBoxSplit : kSplit, ns = box ? 1 : 3;
          const TileLayout l = fixed_tile_layout(ht, wtw, wtp, rows, warps, groups, ns,
                                                 box != 0, wt);
          ++cases;
          const int ty = 2 * rows * warps;
          const size_t rb = (kHalfUnitCols + 4 * wtw + 8 + 15) & ~15;
          const size_t tile = size_t(ty + ht - 1) * rb;
          const size_t part = size_t(groups - 1) * warps * 32 * ns * rows * kCols * 4;
          const size_t tmpl = size_t(ht) * wtp * 4;
          CHECK(l.tile % 16 == 0 && l.part % 16 == 0 && l.tmpl % 16 == 0,
                "wt %d ht %d box %d: unaligned region\n", wt, ht, box);
          // a tile row must hold 128 columns plus the windows' reach
          CHECK(rb >= size_t(kHalfUnitCols + 4 * wtw + 8), "wt %d: tile row too short\n", wt);
          if (!box) {
            CHECK(l.tmpl == 0 && l.tile >= tmpl && l.part >= l.tile + tile &&
                      l.total >= l.part + part,
                  "wt %d ht %d: dp4a regions overlap\n", wt, ht);
          } else {
            const size_t s = size_t(2) * ty * kHalfUnitCols * 4;
            const size_t v = size_t(2) * ty * vs * 4;
            CHECK(l.tile == 0 && l.part >= tile && l.part >= s,
                  "wt %d ht %d: tile / box-sum region too small\n", wt, ht);
            CHECK(l.tmpl >= l.part + part, "wt %d ht %d: exchange overlaps\n", wt, ht);
            CHECK(l.total >= l.tmpl + tmpl && l.total >= l.tmpl + v,
                  "wt %d ht %d: template / column-sum region too small\n", wt, ht);
          }
          // the warp-private staging area of the coalesced stores
          CHECK(size_t(ns) * rows * kCols * 32 >= size_t(2) * rows * kHalfUnitCols,
                "rows %d ns %d: staging area too small\n", rows, ns);
        }
      }
    }
  }
  printf("%ld layouts checked, %d failures\n", cases, fails);
  return fails ? 1 : 0;
}
