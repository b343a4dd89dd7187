// Host-side check of the backward's work-split policy (the number of CTAs that
// share one (page, KV head)): on the workload shapes of the benchmark it must pick
// the counts that measured fastest on GB300 (152 SMs):
//   window of 32 pages over 4K chunks (64 slots)        -> 3
//   top-64 + sink + 32 own pages, 4K chunks (97 slots)  -> 2
//   top-128 + sink + 64 own pages, 8K chunks (193 slots) -> 2
//   dense 32K, last 4K chunk (256 slots)                 -> 2
// and never fewer than two.  Exit status 0 = all hold.
#include <cstdio>

namespace oomb {
int bwd_split(int max_sel, int n_own, int n_tiles, int G, int Hkv, int n_sm);
}

int main() {
  struct Case {
    const char* name;
    int max_sel, n_own, n_tiles, want;
  } cases[] = {{"window128k", 64, 32, 32, 3},
               {"sparse128k", 97, 32, 32, 2},
               {"sparse1m", 193, 64, 64, 2},
               {"dense32k chunk 7", 256, 32, 32, 2}};
  int bad = 0;
  for (const Case& c : cases) {
    const int got = oomb::bwd_split(c.max_sel, c.n_own, c.n_tiles, 7, 4, 152);
    std::printf("%-18s %d (want %d)\n", c.name, got, c.want);
    bad += got != c.want;
  }
  for (int ms = 1; ms <= 300; ms += 7)
    for (int own = 1; own <= 64 && own <= ms; own += 9) {
      const int got = oomb::bwd_split(ms, own, own, 7, 4, 152);
      if (got < 2 || got > 4) {
        std::printf("max_sel %d own %d: %d outside [2, 4]\n", ms, own, got);
        ++bad;
      }
    }
  return bad;
}
