// Host-only check of the tcgen05 GEMM's static tile schedule (decode_tile, batch_tiles): every pair
// tile a launch must compute is visited exactly once, and no other.  Plain cases: all
// batches x m-pairs x n-tiles.  Causal mode 1 (row-batched attention scores, M = N): only the tiles
// on or below the diagonal (pair p takes key tiles 0 .. (p + 1) 256 / BN - 1).  Grouped: each batch
// its own M, N.  Both tile orders (forward and reversed) and both CTAs of a pair.
// Prints "ok <cases>" and exits 0, or the first mismatch and exits 1.
#include <cstdio>
#include <cstring>
#include <vector>

#include "../../rank_bottleneck_block_gb300/csrc/umma_gemm.cuh"

using lr::umma::Shape;
using lr::umma::decode_tile;
using lr::umma::batch_tiles;

namespace {

int g_cases = 0;

template <bool RB>
bool check(const Shape& sh, const std::vector<int>& want_tiles_per_batch_pair, int BN) {
  const long long per_split = sh.grouped ? sh.g_tiles : 1LL * sh.batches * batch_tiles<RB>(sh);
  const long long total = sh.ksplit * per_split;
  // seen[split][batch][mb pair][nb]
  const int maxp = 64, maxn = 128;
  std::vector<int> seen(static_cast<size_t>(sh.ksplit) * sh.batches * maxp * maxn, 0);
  for (long long t = 0; t < total; ++t) {
    int s0 = -1, b0 = -1, p0 = -1, n0 = -1;
    for (int rank = 0; rank < 2; ++rank) {
      int split, batch, mb, nb;
      decode_tile<RB>(sh, static_cast<int>(t), rank, split, batch, mb, nb);
      if ((mb & 1) != rank || split < 0 || split >= sh.ksplit || batch < 0 || batch >= sh.batches || nb < 0 ||
          nb >= maxn || (mb >> 1) >= maxp) {
        std::printf("tile %lld rank %d decodes out of range: split %d batch %d mb %d nb %d\n", t, rank, split,
                    batch, mb, nb);
        return false;
      }
      if (rank == 0) {
        s0 = split, b0 = batch, p0 = mb >> 1, n0 = nb;
      } else if (split != s0 || batch != b0 || (mb >> 1) != p0 || nb != n0) {
        std::printf("tile %lld: the two CTAs of the pair disagree\n", t);
        return false;
      }
    }
    ++seen[((static_cast<size_t>(s0) * sh.batches + b0) * maxp + p0) * maxn + n0];
  }
  for (int sp = 0; sp < sh.ksplit; ++sp)
    for (int b = 0; b < sh.batches; ++b)
      for (int p = 0; p < maxp; ++p)
        for (int n = 0; n < maxn; ++n) {
          int want = 0;
          const int m_pairs = sh.grouped ? want_tiles_per_batch_pair[2 * b] : sh.m_pairs;
          const int n_tiles = sh.grouped ? want_tiles_per_batch_pair[2 * b + 1] : sh.n_tiles;
          if (p < m_pairs && n < n_tiles) want = (RB && sh.causal == 1) ? (n < (p + 1) * (256 / BN)) : 1;
          if (seen[((static_cast<size_t>(sp) * sh.batches + b) * maxp + p) * maxn + n] != want) {
            std::printf("split %d batch %d pair %d n-tile %d visited %d times, want %d\n", sp, b, p, n,
                        seen[((static_cast<size_t>(sp) * sh.batches + b) * maxp + p) * maxn + n], want);
            return false;
          }
        }
  ++g_cases;
  return true;
}

Shape plain(int M, int N, int BN, int batches, int ksplit, int reverse) {
  Shape sh;
  std::memset(&sh, 0, sizeof(sh));
  sh.M = M, sh.N = N, sh.K = 64, sh.batches = batches, sh.ksplit = ksplit, sh.reverse = reverse;
  sh.m_tiles = (M + 127) / 128, sh.n_tiles = (N + BN - 1) / BN, sh.m_pairs = (sh.m_tiles + 1) / 2;
  return sh;
}

}  // namespace

int main() {
  for (int BN : {128, 256})
    for (int rev : {0, 1}) {
      // plain (including ragged M, N and split-K)
      for (int M : {128, 256, 300, 1024, 4096})
        for (int N : {128, 200, 1024, 5632})
          for (int batches : {1, 2, 4})
            for (int ks : {1, 3})
              if (!check<false>(plain(M, N, BN, batches, ks, rev), {}, BN)) return 1;
      // causal mode 1, row-batched over heads: s x s scores
      for (int s = 256; s <= 8192; s += 256)
        for (int heads : {1, 3, 32}) {
          if (heads == 32 && s > 2048) continue;
          Shape sh = plain(s, s, BN, heads, 1, rev);
          sh.rowbatch = 1, sh.bh = heads, sh.causal = 1;
          if (!check<true>(sh, {}, BN)) return 1;
          // causal modes 2 and 3 narrow K only: every tile of the [s, dh] output is scheduled
          Shape sk = plain(s, 128, BN, heads, 1, rev);
          sk.rowbatch = 1, sk.bh = heads, sk.causal = 2;
          if (!check<true>(sk, {}, BN)) return 1;
          sk.causal = 3;
          if (!check<true>(sk, {}, BN)) return 1;
        }
      // grouped batches of their own shapes
      const int gm[4] = {2048, 512, 300, 4096}, gn[4] = {512, 2048, 1000, 128};
      for (int nb = 1; nb <= 4; ++nb) {
        Shape sh = plain(0, 0, BN, nb, 1, rev);
        sh.grouped = 1;
        std::vector<int> want;
        int t = 0;
        for (int b = 0; b < lr::kMaxBatch; ++b) {
          sh.g_n_tiles[b] = b < nb ? (gn[b] + BN - 1) / BN : 1;
          sh.g_tile0[b] = t;
          if (b < nb) {
            const int mp = (gm[b] + 255) / 256;
            t += mp * sh.g_n_tiles[b];
            want.push_back(mp);
            want.push_back(sh.g_n_tiles[b]);
          }
        }
        sh.g_tiles = t;
        if (!check<false>(sh, want, BN)) return 1;
      }
    }
  std::printf("ok %d\n", g_cases);
  return 0;
}
