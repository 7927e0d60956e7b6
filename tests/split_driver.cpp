// Prints the create-time work splits of mla_split.cpp for test_splits.py:
// one line per (split, heads, CTAs), all integers.
//   abs  H C  task[0..C] rope[0..C]
//   pair H C ok  head[0..C/2] rope[0..C]      (heads spread evenly)
//   pairf H C ok  head[0..C/2] rope[0..C]     (heads first)
//   pairmax H C most                        (most loaded CTA, heads first)
//   fmafirst H most_fma most_pair fma         (152 SMs; at most 76, 36 and 15
//                                              clusters of 2, 4 and 8, as on GB300)
//   wide H C ok ndouble  head[0..C/2] dbl[0..C/2] sgl[0..C/2]
//   small H C K ok most  head[0..C/K] rope[0..C]  (clusters of K CTAs)
//   choose H S ctas K most  (the cluster size chosen for S SMs)
#include <cstdio>

#include "mla_internal.h"
#include "mla_query.h"

int main() {
  const int ctas_list[] = {2, 4, 6, 20, 132, 148, 150, 152, 256};
  for (int ctas : ctas_list) {
    const int pairs = ctas / 2;
    for (int h = 1; h <= MLA_MAX_HEADS; ++h) {
      static mla::AbsSplit as;
      mla::make_abs_split(h, ctas, &as);
      std::printf("abs %d %d", h, ctas);
      for (int i = 0; i <= ctas; ++i) std::printf(" %d", as.task[i]);
      for (int i = 0; i <= ctas; ++i) std::printf(" %d", as.rope[i]);
      std::printf("\n");
      for (int first = 0; first < 2; ++first) {
        static mla::PairSplit ps;
        const bool pok = mla::make_pair_split(h, ctas, first != 0, &ps);
        std::printf("%s %d %d %d", first ? "pairf" : "pair", h, ctas, pok ? 1 : 0);
        for (int c = 0; c <= pairs; ++c) std::printf(" %d", pok ? ps.head[c] : 0);
        for (int i = 0; i <= ctas; ++i) std::printf(" %d", pok ? ps.rope[i] : 0);
        std::printf("\n");
        if (first && pok)
          std::printf("pairmax %d %d %lld\n", h, ctas, (long long)mla::pair_split_max_bytes(ctas, ps));
        if (first && pok && ctas == 152) {
          static mla::SmallSplit fs;
          const int gb300[3] = {76, 36, 15};
          const int fc = mla::choose_small_split(h, 152, gb300, &fs);
          const long long fm = fc ? (long long)mla::small_split_max_bytes(h, fc, fs) : 0;
          const long long pm = (long long)mla::pair_split_max_bytes(ctas, ps);
          std::printf("fmafirst %d %d %lld %lld %d\n", h, ctas, fm, pm, fc > 0 && 5 * fm <= 4 * pm);
        }
      }
      static mla::WideSplit ws;
      const bool wok = mla::make_wide_split(h, ctas, &ws);
      std::printf("wide %d %d %d %d", h, ctas, wok ? 1 : 0, wok ? ws.ndouble : 0);
      for (int c = 0; c <= pairs; ++c) std::printf(" %d", wok ? ws.head[c] : 0);
      for (int c = 0; c <= pairs; ++c) std::printf(" %d", wok ? ws.dbl[c] : 0);
      for (int c = 0; c <= pairs; ++c) std::printf(" %d", wok ? ws.sgl[c] : 0);
      std::printf("\n");
      for (int k = 2; k <= 8; k *= 2) {
        static mla::SmallSplit ss;
        const int sc = (ctas / k) * k;
        const bool sok = sc >= k && mla::make_small_split(h, sc, k, &ss);
        std::printf("small %d %d %d %d %lld", h, sc, k, sok ? 1 : 0,
                    sok ? (long long)mla::small_split_max_bytes(h, sc, ss) : 0LL);
        for (int g = 0; g <= sc / k; ++g) std::printf(" %d", sok ? ss.head[g] : 0);
        for (int i = 0; i <= sc; ++i) std::printf(" %d", sok ? ss.rope[i] : 0);
        std::printf("\n");
      }
      static mla::SmallSplit cs;
      const int cc = mla::choose_small_split(h, ctas, nullptr, &cs);
      std::printf("choose %d %d %d %d %lld\n", h, ctas, cc, cc ? cs.cluster : 0,
                  cc ? (long long)mla::small_split_max_bytes(h, cc, cs) : 0LL);
    }
  }
  return 0;
}
