// Host-only check of the work-item order of the attention kernels without materialised scores
// (item_of, heads_per_group): over nheads heads and nb blocks per head, item t = 0 .. nheads nb - 1 maps
// to every (rank, head) exactly once; heads come in groups of `group` consecutive heads (the last group
// ragged) that are walked one after the other; inside a group the rank never decreases with t, so the
// blocks of one rank (the forward's query blocks from the last, the backward's key blocks from the
// first: the heaviest items) are fetched before lighter ones.  Prints "ok <cases>" and exits 0, or the
// first mismatch and exits 1.
#include <cstdio>
#include <vector>

#include "../../rank_bottleneck_block_gb300/csrc/attn_flash.cuh"

using lr::flash::heads_per_group;
using lr::flash::item_of;

int main() {
  int cases = 0;
  const int heads_list[] = {1, 2, 3, 7, 32, 256, 300};
  const int nb_list[] = {1, 2, 16, 18};
  const long long bytes_list[] = {1LL << 10, 1LL << 20, 1LL << 22, 1LL << 26};
  for (int nheads : heads_list)
    for (int nb : nb_list)
      for (long long bytes : bytes_list) {
        const int group = heads_per_group(nheads, bytes);
        if (group < 1 || group > nheads) {
          printf("bad group %d for %d heads, %lld bytes\n", group, nheads, bytes);
          return 1;
        }
        std::vector<int> seen(static_cast<size_t>(nheads) * nb, 0);
        int prev_gi = 0, prev_rank = -1;
        for (int t = 0; t < nheads * nb; ++t) {
          int rank = -1, n = -1;
          item_of(t, nheads, nb, group, rank, n);
          if (rank < 0 || rank >= nb || n < 0 || n >= nheads) {
            printf("item %d out of range: rank %d head %d (heads %d, nb %d, group %d)\n", t, rank, n, nheads, nb, group);
            return 1;
          }
          const int gi = n / group;
          if (gi < prev_gi) {
            printf("group order broken at item %d (heads %d, nb %d, group %d)\n", t, nheads, nb, group);
            return 1;
          }
          if (gi != prev_gi) prev_rank = -1;
          if (rank < prev_rank) {
            printf("rank decreases at item %d (heads %d, nb %d, group %d)\n", t, nheads, nb, group);
            return 1;
          }
          prev_gi = gi;
          prev_rank = rank;
          ++seen[static_cast<size_t>(n) * nb + rank];
        }
        for (size_t i = 0; i < seen.size(); ++i)
          if (seen[i] != 1) {
            printf("item (head %zu, rank %zu) seen %d times (heads %d, nb %d, group %d)\n", i / nb, i % nb, seen[i],
                   nheads, nb, group);
            return 1;
          }
        ++cases;
      }
  printf("ok %d\n", cases);
  return 0;
}
