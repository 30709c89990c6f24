// Host check of the walks' closed-form totals: for many mesh geometries,
// KvWalk::total() and QWalk::total() equal the number of tiles the walk
// actually visits (stepping it to the end) and the copy-walking count().
// Compiled by tests/test_walk_totals.py with the host compiler.
#include <cstdio>

#define __host__
#define __device__
#include "ring.cuh"

using namespace loong;

int main() {
  // cp = inner * outer, zigzag, causal, tokens per block
  const int geoms[][5] = {{1, 1, 1, 1, 384}, {4, 2, 1, 1, 200}, {8, 4, 1, 1, 512}, {16, 8, 1, 1, 4096},
                          {6, 3, 0, 1, 250}, {4, 4, 1, 0, 300}, {8, 2, 0, 0, 128}, {2, 1, 1, 1, 16}};
  int bad = 0, checked = 0;
  for (const auto& q : geoms) {
    RingGeom g;
    g.cp = q[0];
    g.inner = q[1];
    g.outer = q[0] / q[1];
    g.zigzag = q[2];
    g.causal = q[3];
    g.blk = q[4];
    g.nblocks = g.zigzag ? 2 * g.cp : g.cp;
    g.ntile = (g.blk + kTile - 1) / kTile;
    const int nsteps = g.inner * g.outer;
    // the whole ring, then every single step, then a partial range
    for (int r = 0; r < nsteps + 2; ++r) {
      const int t0 = r == 0 ? 0 : (r <= nsteps ? r - 1 : 1);
      const int t1 = r == 0 ? nsteps : (r <= nsteps ? r : nsteps);
      if (t0 >= t1) continue;
      for (int b = 0; b < g.nblocks; ++b)
        for (int tile = 0; tile < g.ntile; ++tile) {
          KvWalk kw;
          kw.init(g, b, tile, t0, t1);
          int steps = 0;
          for (KvWalk w = kw; !w.done(); w.advance()) ++steps;
          for (int G = 1; G <= 3; ++G) {
            QWalk qw;
            qw.init(g, G, b, tile, t0, t1);
            int qsteps = 0;
            for (QWalk w = qw; !w.done(); w.advance()) ++qsteps;
            if (qw.total() != qsteps || qw.count() != qsteps) {
              if (bad++ < 10)
                std::printf("QWalk cp=%d blk=%d zz=%d causal=%d t=[%d,%d) bk=%d kt=%d G=%d: total %d count %d walked %d\n",
                            g.cp, g.blk, g.zigzag, g.causal, t0, t1, b, tile, G, qw.total(), qw.count(), qsteps);
            }
            ++checked;
          }
          if (kw.total() != steps || kw.count() != steps) {
            if (bad++ < 10)
              std::printf("KvWalk cp=%d blk=%d zz=%d causal=%d t=[%d,%d) bq=%d qi=%d: total %d count %d walked %d\n",
                          g.cp, g.blk, g.zigzag, g.causal, t0, t1, b, tile, kw.total(), kw.count(), steps);
          }
          ++checked;
        }
    }
  }
  std::printf("%d walks checked, %d mismatches\n", checked, bad);
  return bad ? 1 : 0;
}
