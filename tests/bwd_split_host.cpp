// Host-side check of the backward's work-split policy (the number of CTAs, one
// thread-block cluster, that share one (page, KV head)).  The policy replays a
// greedy schedule of clusters onto the device's cluster slots; with the cluster
// occupancy of a GB300 (152 SMs) it must pick, on the workload shapes of the
// benchmark:
//   window of 32 pages over 4K chunks (64 slots)        -> 2
//   top-64 + sink + 32 own pages, 4K chunks (97 slots)  -> 2
//   top-128 + sink + 64 own pages, 8K chunks (193 slots) -> 2
//   dense 32K, last 4K chunk (256 slots)                 -> 2
// and never fewer than two or more than four.  Exit status 0 = all hold.
#include <cstdio>

namespace oomb {
int bwd_split(int max_sel, int n_own, int n_tiles, int G, int Hkv, const int* cluster_slots);
}

int main() {
  // clusters of 1..4 CTAs (448 threads, ~200 KB shared memory each) resident at once
  // on a GB300, as cudaOccupancyMaxActiveClusters reported them (GPCs whose SM count
  // is not a multiple of the cluster size leave SMs idle: 138 and 144 CTAs for 3 and 4)
  const int gb300_slots[5] = {0, 152, 76, 46, 36};
  struct Case {
    const char* name;
    int max_sel, n_own, n_tiles, want;
  } cases[] = {{"window128k", 64, 32, 32, 2},
               {"sparse128k", 97, 32, 32, 2},
               {"sparse1m", 193, 64, 64, 2},
               {"dense32k chunk 7", 256, 32, 32, 2}};
  int bad = 0;
  for (const Case& c : cases) {
    const int got = oomb::bwd_split(c.max_sel, c.n_own, c.n_tiles, 7, 4, gb300_slots);
    std::printf("%-18s %d (want %d)\n", c.name, got, c.want);
    bad += got != c.want;
  }
  for (int ms = 1; ms <= 300; ms += 7)
    for (int own = 1; own <= 64 && own <= ms; own += 9) {
      const int got = oomb::bwd_split(ms, own, own, 7, 4, gb300_slots);
      if (got < 2 || got > 4) {
        std::printf("max_sel %d own %d: %d outside [2, 4]\n", ms, own, got);
        ++bad;
      }
    }
  return bad;
}
