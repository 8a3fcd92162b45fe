// Host-side check of the 2-CTA weight-row tile order (pair_tiles.cuh): the
// incremental TileIter each role of the kernel walks must give, at every
// tile a CTA pair visits, exactly what decode() gives from scratch.  Random
// expert loads (many empty and single-tile experts, a few with many token
// tiles), weight-tile counts and pair counts.  Prints "ok" and exits 0, or
// reports the first mismatch and exits 1.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "pair_tiles.cuh"

using moe::pair::Sched;
using moe::pair::Tile;

static unsigned long long rng_state = 0x9E3779B97F4A7C15ull;
static unsigned rnd() {  // SplitMix64
  unsigned long long z = (rng_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return static_cast<unsigned>((z ^ (z >> 31)) >> 32);
}

int main() {
  const int kTok = moe::pair::kNmax;
  for (int trial = 0; trial < 400; ++trial) {
    const int E = 1 + rnd() % 300;
    const int w_tiles = 1 + rnd() % 40;
    std::vector<int32_t> ntk(E), hp(E + 1), cp(E + 1);
    for (int e = 0; e < E; ++e) {
      const unsigned u = rnd() % 100;
      const int rows = u < 30 ? 0 : u < 80 ? 1 + rnd() % kTok : u < 95 ? 1 + rnd() % (4 * kTok)
                                                                     : 1 + rnd() % (40 * kTok);
      ntk[e] = rows ? (rows + kTok - 1) / kTok : 0;
    }
    int h = 0, c = 0;
    for (int e = 0; e < E; ++e) {  // the prefixes build_sched writes
      hp[e] = h;
      cp[e] = c;
      if (ntk[e] > 1) h += ntk[e] * w_tiles; else c += ntk[e] * w_tiles;
    }
    hp[E] = h;
    cp[E] = c;
    const Sched s{hp.data(), cp.data(), ntk.data(), E, w_tiles, h, c};
    const int pairs_choices[4] = {1, 7, 76, 1 + static_cast<int>(rnd() % 200)};
    for (int pc : pairs_choices) {
      for (int first = 0; first < pc && first < s.total(); first += (pc > 16 ? 5 : 1)) {
        moe::pair::TileIter it;
        it.init(first, pc, s);
        for (int tile = first; tile < s.total(); tile += pc, it.next()) {
          const Tile a = moe::pair::decode(tile, s);
          const Tile b = it.get(s);
          if (it.tile != tile || a.e != b.e || a.m != b.m || a.n != b.n || a.hot != b.hot) {
            std::printf("mismatch: trial %d E %d w_tiles %d pairs %d first %d tile %d: decode "
                        "(%d,%d,%d,%d) iter (%d,%d,%d,%d)\n",
                        trial, E, w_tiles, pc, first, tile, a.e, a.m, a.n, a.hot, b.e, b.m, b.n,
                        b.hot);
            return 1;
          }
        }
      }
    }
  }
  std::printf("ok\n");
  return 0;
}
