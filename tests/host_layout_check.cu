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
  for (int wt = 1; wt <= 4 * kMaxFixedWords; ++wt) {
    const int wtw = (wt + 3) / 4, wtp = (wtw + 3) & ~3;
    // column sums: stride = 16 mod 32 and room for the last skewed column
    const int vs = box_v_stride(wt);
    const int nv = kHalfUnitCols + wt - 1;
    CHECK(vs % 32 == 16, "wt %d: v stride %d not 16 mod 32\n", wt, vs);
    CHECK((nv - 1) + ((nv - 1) >> 3) < vs, "wt %d: v stride %d too small\n", wt, vs);
    for (int ht = 1; ht * wt <= 66052; ++ht) {
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
