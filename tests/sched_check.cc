// Host-side check of the unit decode that every tensor-core kernel uses to
// walk its tiles (decode_unit in csrc/kernels.h), compiled by
// tests/test_schedule.py with the host compiler. Exit code 0: every check
// passed; otherwise the first failure is printed.
//
// - Bijection: units 0 .. n_blocks * num_panels - 1 map one to one onto
//   (panel, block) pairs, for every group size (the last group may be
//   smaller, and a group larger than n_blocks is one group).
// - Order: a group of 1 is block after block, panels fastest (the plain
//   GEMM's row-after-row order); within a group, blocks run fastest.
// - Locality: with the chunked projection's grouping (16 row tiles, 128
//   column tiles), the first wave of 76 pairs covers all 16 row tiles and
//   only the first 5 column tiles.
// - The plain GEMM's packed (row tile << 8 | split) argument round-trips.
#include <cstdio>
#include <vector>

#include "kernels.h"

using flce::decode_unit;

static int fail(const char* what, int a, int b, int c, int d) {
  std::printf("FAIL %s (%d, %d, %d, %d)\n", what, a, b, c, d);
  return 1;
}

int main() {
  for (int n_blocks = 1; n_blocks <= 40; ++n_blocks) {
    for (int group = 1; group <= n_blocks + 2; ++group) {
      for (int panels = 1; panels <= 12; ++panels) {
        std::vector<int> seen(static_cast<size_t>(n_blocks) * panels, 0);
        int prev_g_block = -1, prev_panel = -1;
        for (int u = 0; u < n_blocks * panels; ++u) {
          int panel = -1, nb = -1;
          decode_unit(u, n_blocks, group, panels, panel, nb);
          if (panel < 0 || panel >= panels || nb < 0 || nb >= n_blocks)
            return fail("out of range", n_blocks, group, panels, u);
          if (seen[static_cast<size_t>(nb) * panels + panel]++)
            return fail("tile visited twice", n_blocks, group, panels, u);
          if (group == 1 && (nb != u / panels || panel != u % panels))
            return fail("group 1 is not row after row", n_blocks, group, panels, u);
          // within a group, consecutive units of one panel take the next block
          const int g = nb / group;
          if (g == prev_g_block && panel == prev_panel && group > 1) {
            int p2 = -1, nb2 = -1;
            decode_unit(u - 1, n_blocks, group, panels, p2, nb2);
            if (nb2 != nb - 1) return fail("blocks not fastest in a group", n_blocks, group, panels, u);
          }
          prev_g_block = g;
          prev_panel = panel;
        }
      }
    }
  }
  // the chunked projection: 16 row tiles in one group, 128 column tiles
  {
    bool rows[16] = {};
    int max_col = 0;
    for (int u = 0; u < 76; ++u) {
      int nt = -1, mt = -1;
      decode_unit(u, 16, 16, 128, nt, mt);
      rows[mt] = true;
      if (nt > max_col) max_col = nt;
    }
    for (int m = 0; m < 16; ++m)
      if (!rows[m]) return fail("first wave misses a row tile", m, 0, 0, 0);
    if (max_col != 4) return fail("first wave spans too many column tiles", max_col, 0, 0, 0);
  }
  // (row tile << 8 | split) as the plain GEMM packs it
  const int mts[] = {0, 1, 255, 256, 4095, (1 << 22) - 1};
  for (int mt : mts)
    for (int sp = 0; sp < 256; sp += 17) {
      const int ta = (mt << 8) | sp;
      if ((ta & 255) != sp || (ta >> 8) != mt) return fail("packed unit", mt, sp, ta, 0);
    }
  std::printf("ok\n");
  return 0;
}
