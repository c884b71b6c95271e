// Host-only check of the decode kernels' shared-memory layouts: every
// (engine variant, element size, head_dim, rows, pipeline depth, batch,
// cluster receive slots) a plan can pick must pass layout_check (alignment,
// extent and order of every region), and every (depth, batch) of the tcgen05
// kernel tc_layout_check.  Prints one line per failure and "ok <count>" at the end.
#include <cstdio>

#include "decode_tc.cuh"

int main() {
  using namespace da;
  int bad = 0, count = 0;
  int batches[80];
  int nb = 0;
  for (int b = 1; b <= 64; ++b) batches[nb++] = b;
  for (int b : {65, 100, 127, 128, 129, 255, 256, 257, 511, 512, 513, 1000, 1023, 1024})
    batches[nb++] = b;
  struct V { int variant, es; int rks[4]; int nrk; };
  const V vs[] = {{kVariantCore, 2, {1, 2, 4, 8}, 4}, {kVariantCore, 4, {1, 2, 4, 8}, 4},
                  {kVariantMma, 2, {8, 16, 32, 0}, 3}};
  for (const V& v : vs)
    for (int d : {64, 128})
      for (int i = 0; i < v.nrk; ++i)
        for (int stages = 2; stages <= 8; ++stages)
          for (int j = 0; j < nb; ++j)
            // 0: the flat partition; otherwise the cluster partition with that
            // many receive slots in rank 0
            for (int recv : {0, 1, 2, 4, 8, 10, 16}) {
              const int rk = v.rks[i], batch = batches[j];
              const Layout L = make_layout(v.variant, v.es, d, rk, stages, batch, recv);
              const int rc = layout_check(L, v.variant, v.es, d, rk, stages, batch, recv);
              ++count;
              if (rc != 0) {
                ++bad;
                if (bad < 20)
                  std::printf("bad layout: variant %d es %d d %d rk %d stages %d batch %d recv %d: "
                              "check %d\n", v.variant, v.es, d, rk, stages, batch, recv, rc);
              }
            }
  // the tcgen05 kernel's own layout
  for (int stages = 2; stages <= kTcMaxStages; ++stages)
    for (int j = 0; j < nb; ++j) {
      const TcLayout L = make_tc_layout(stages, batches[j]);
      const int rc = tc_layout_check(L, stages, batches[j]);
      ++count;
      if (rc != 0) {
        ++bad;
        if (bad < 20) std::printf("bad tcgen05 layout: stages %d batch %d: check %d\n", stages, batches[j], rc);
      }
    }
  if (bad) {
    std::printf("failed %d of %d\n", bad, count);
    return 1;
  }
  std::printf("ok %d\n", count);
  return 0;
}
