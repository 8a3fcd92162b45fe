// Weight-row tiles on 2-CTA clusters: the tile schedule and the cluster-scope
// PTX both pair kernels share (bf16 weights in grouped_gemm_swap2.cu, NVFP4
// weights in grouped_gemm_fp4_pair.cu).
//
// A pair tile is 256 weight rows (M; 128 per CTA) x N token rows of one
// expert, N = 2 * half, half = ceil(rows / 2) rounded up to 16, N <= 256.
// Each CTA loads its 128 weight rows and its half of the token rows; the
// leader CTA issues tcgen05.mma.cta_group::2 with M = 256 that reads both
// CTAs' shared memory, and each CTA's TMEM receives its 128 weight rows x N.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace moe {
namespace pair {

constexpr int kNmax = 256;  // token rows per pair tile
constexpr int kM = 128;     // weight rows per CTA

struct Tile {
  int e, m, n;  // expert, weight pair tile, token tile
  bool hot;
};

// Token tiles of a hot expert are visited in groups of kGroup: all weight
// tiles for one group, the token tile innermost.  A weight tile is then read
// by the group's tiles at about the same time (one HBM read), and a token
// tile comes back after one sweep of the group (it stays in L2) instead of
// after a sweep over all of the expert's rows.
#ifndef MOE_PAIR_GROUP
#define MOE_PAIR_GROUP 8
#endif
constexpr int kGroup = MOE_PAIR_GROUP;

// Tile order.  Experts with more than one token tile ("hot": their weight
// tiles are reused from L2 and the MMAs bound them) and experts with one
// ("cold": every tile streams fresh weights from HBM) form two lists, each
// expert-major.  The lists are merged in proportion -- position t is hot iff
// floor((t+1) nh / N) > floor(t nh / N) -- so that every wave of CTA pairs
// mixes compute-bound and HBM-bound tiles and the weight stream overlaps the
// tensor-core work instead of alternating with it.
struct Sched {
  const int32_t* hot_prefix;   // [E+1] tiles of hot experts before e
  const int32_t* cold_prefix;  // [E+1] tiles of cold experts before e
  const int32_t* ntk;          // [E] token tiles of e
  int E, w_tiles, nh, nc;
  __host__ __device__ __forceinline__ int total() const { return nh + nc; }
};

// (m, n) of the tile at position `local` inside expert e's list.
__host__ __device__ __forceinline__ Tile tile_in_expert(int e, bool hot, int local, int nt,
                                                       int w_tiles) {
  const int per_group = kGroup * w_tiles;
  const int g = local / per_group;
  const int within = local - g * per_group;
  const int left = nt - g * kGroup;
  const int gsz = left < kGroup ? left : kGroup;
  Tile t;
  t.e = e;
  t.hot = hot;
  t.m = within / gsz;
  t.n = g * kGroup + (within - t.m * gsz);
  return t;
}

// The tile at position `tile` of the merged order, from scratch (two 64-bit
// divisions and a binary search over the experts).
__host__ __device__ __forceinline__ Tile decode(int tile, const Sched& s) {
  const long long n = static_cast<long long>(s.nh) + s.nc;
  const int hb = static_cast<int>(static_cast<long long>(tile) * s.nh / n);
  const int ha = static_cast<int>(static_cast<long long>(tile + 1) * s.nh / n);
  const bool hot = ha > hb;
  const int idx = hot ? hb : tile - hb;
  const int32_t* pf = hot ? s.hot_prefix : s.cold_prefix;
  int lo = 0, hi = s.E - 1;  // the last expert whose first tile is <= idx
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pf[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  return tile_in_expert(lo, hot, idx - pf[lo], s.ntk[lo], s.w_tiles);
}

// The tiles one CTA pair visits -- first, first + stride, first + 2 stride,
// ... -- each exactly as decode() gives it, but in O(1) amortised per tile,
// which matters because the producer, the MMA issuer and the epilogue each
// walk the sequence between their K steps.  The merge position is kept as a
// running quotient hb = floor(tile nh / N) and remainder r = tile nh mod N
// (tile is hot iff r + nh >= N), and each list's expert by a forward scan: a
// list's index never decreases along the sequence (hb grows by
// floor(stride nh / N) or one more, the cold index tile - hb by the rest).
struct TileIter {
  int tile, stride;
  long long n;        // nh + nc
  int nh, hb, q_s;    // floor(stride nh / N)
  long long r, r_s;   // tile nh mod N, stride nh mod N
  int e_hot, e_cold;  // expert cursors of the two lists

  __host__ __device__ __forceinline__ void init(int first, int step, const Sched& s) {
    tile = first;
    stride = step;
    nh = s.nh;
    n = static_cast<long long>(s.nh) + s.nc;
    e_hot = 0;
    e_cold = 0;
    if (n == 0) {
      hb = q_s = 0;
      r = r_s = 0;
      return;
    }
    const long long a = static_cast<long long>(first) * s.nh;
    const long long b = static_cast<long long>(step) * s.nh;
    hb = static_cast<int>(a / n);
    r = a - static_cast<long long>(hb) * n;
    q_s = static_cast<int>(b / n);
    r_s = b - static_cast<long long>(q_s) * n;
  }

  __host__ __device__ __forceinline__ Tile get(const Sched& s) {
    const bool hot = r + nh >= n;
    const int idx = hot ? hb : tile - hb;
    const int32_t* pf = hot ? s.hot_prefix : s.cold_prefix;
    int e = hot ? e_hot : e_cold;
    while (e + 1 < s.E && pf[e + 1] <= idx) ++e;
    if (hot) e_hot = e; else e_cold = e;
    return tile_in_expert(e, hot, idx - pf[e], s.ntk[e], s.w_tiles);
  }

  __host__ __device__ __forceinline__ void next() {
    tile += stride;
    hb += q_s;
    r += r_s;
    if (r >= n) {
      r -= n;
      ++hb;
    }
  }
};

// Fills ntk[E], hot_prefix[E+1], cold_prefix[E+1] (shared memory) from the
// expert offsets off[E+1] (shared memory); every thread of the block calls it.
// Expert e owns w_tiles * ceil(rows_e / kTok) tiles (kTok token rows per tile).
template <int kThreads, int kTok = kNmax>
__device__ __forceinline__ Sched build_sched(const int32_t* off, int E, int w_tiles, int32_t* ntk,
                                             int32_t* hp, int32_t* cp) {
  __shared__ int s_part[2][kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = (E + kThreads - 1) / kThreads;
  const int e0 = min(E, static_cast<int>(threadIdx.x) * per), e1 = min(E, e0 + per);
  int run_h = 0, run_c = 0;
  for (int e = e0; e < e1; ++e) {
    const int rows = off[e + 1] - off[e];
    const int nt = rows > 0 ? (rows + kTok - 1) / kTok : 0;
    ntk[e] = nt;
    if (nt > 1) run_h += nt * w_tiles; else run_c += nt * w_tiles;
  }
  int inc_h = run_h, inc_c = run_c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int yh = __shfl_up_sync(0xffffffffu, inc_h, o);
    const int yc = __shfl_up_sync(0xffffffffu, inc_c, o);
    if (lane >= o) { inc_h += yh; inc_c += yc; }
  }
  if (lane == 31) { s_part[0][warp] = inc_h; s_part[1][warp] = inc_c; }
  __syncthreads();
  int acc_h = inc_h - run_h, acc_c = inc_c - run_c;
  for (int w = 0; w < warp; ++w) { acc_h += s_part[0][w]; acc_c += s_part[1][w]; }
  for (int e = e0; e < e1; ++e) {
    hp[e] = acc_h;
    cp[e] = acc_c;
    const int nt = ntk[e];
    if (nt > 1) acc_h += nt * w_tiles; else acc_c += nt * w_tiles;
  }
  int th = 0, tc = 0;
  for (int w = 0; w < kThreads / 32; ++w) { th += s_part[0][w]; tc += s_part[1][w]; }
  if (threadIdx.x == kThreads - 1) {
    hp[E] = th;
    cp[E] = tc;
  }
  __syncthreads();
  return Sched{hp, cp, ntk, E, w_tiles, th, tc};
}

// Token rows this CTA loads for a tile of nval tokens: half = ceil(nval / 2)
// rounded up to 16, and the smallest box of 16/32/64/128 rows that holds it.
__device__ __forceinline__ int half_rows(int nval) { return ((nval + 1) / 2 + 15) & ~15; }
__device__ __forceinline__ int box_index(int half) {
  return half <= 16 ? 0 : half <= 32 ? 1 : half <= 64 ? 2 : 3;
}

// Token-row tensor maps with boxes of 16, 32, ..., 128 rows: a tile loads
// exactly its half (a multiple of 16 rows) with map m[half / 16 - 1].
constexpr int kTokenBoxes = kNmax / 2 / 16;
struct TokenMaps {
  CUtensorMap m[kTokenBoxes];
};
__device__ __forceinline__ int token_box(int half) { return half / 16 - 1; }

// ------------------------------------------------------------------ byte ring
// A ring of `cap` bytes holding blocks of varying size in issue order, each
// contiguous (a block that does not fit before the end starts at 0), with
// kSlots barrier pairs (block j uses slot j % kSlots).  Producer and consumer
// replay the same placement, so both know every block's offset.
__device__ __forceinline__ uint32_t ring_place(uint32_t& pos, uint32_t bytes, uint32_t cap) {
  const uint32_t start = pos + bytes > cap ? 0u : pos;
  pos = start + bytes;
  return start;
}

// The producer's record of the blocks in flight, by slot, held in registers
// (every index below is a compile-time constant after unrolling).
template <int kSlots>
struct RingQueue {
  int32_t lo[kSlots], hi[kSlots];
};

template <int kSlots>
__device__ __forceinline__ void ring_record(RingQueue<kSlots>& q, int slot, uint32_t start,
                                            uint32_t bytes) {
#pragma unroll
  for (int i = 0; i < kSlots; ++i) {
    if (i == slot) {
      q.lo[i] = static_cast<int32_t>(start);
      q.hi[i] = static_cast<int32_t>(start + bytes);
    }
  }
}

// Producer: before block `head` is written at [start, start + bytes), wait
// (in issue order) until no block still in flight overlaps it and a barrier
// slot is free; tail is the oldest block not yet known to be consumed.
// False on a timed-out wait.
template <int kSlots>
__device__ __forceinline__ bool ring_make_room(uint32_t start, uint32_t bytes, int& tail,
                                               int head, const RingQueue<kSlots>& q,
                                               uint64_t* empty, uint32_t* status) {
  const int lo = static_cast<int>(start), hi = static_cast<int>(start + bytes);
  while (tail < head) {
    const int n = head - tail;
    const int t0 = tail % kSlots;
    bool overlap = false;
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      const int age = (i - t0 + kSlots) % kSlots;  // 0: the oldest in flight
      overlap |= age < n && lo < q.hi[i] && q.lo[i] < hi;
    }
    if (!overlap && n < kSlots) return true;
    if (!mbar_wait(&empty[t0], static_cast<uint32_t>(tail / kSlots) & 1u, status)) return false;
    ++tail;
  }
  return true;
}

// Weight rows of this CTA's two 64-row boxes inside one expert.  GEMM1: the
// 64 gate rows and the matching 64 up rows of outputs f0 .. f0 + 63,
// f0 = 128 m + 64 rank, for the GLU interleave I (0: [gate F | up F]; else
// blocks of I gate rows then I up rows).  GEMM2: features 256 m + 128 rank ..
// + 127.
__device__ __forceinline__ void weight_rows(bool glu, int m, uint32_t rank, int F, int interleave,
                                            int& r0, int& r1) {
  if (glu) {
    const int f0 = m * kM + static_cast<int>(rank) * 64;
    if (interleave == 32) {
      r0 = 2 * f0;
      r1 = 2 * f0 + 64;
    } else if (interleave == 0) {
      r0 = f0;
      r1 = F + f0;
    } else {  // 64 or a multiple of 128
      r0 = (f0 / interleave) * 2 * interleave + f0 % interleave;
      r1 = r0 + interleave;
    }
  } else {
    r0 = m * (2 * kM) + static_cast<int>(rank) * kM;
    r1 = r0 + 64;
  }
}

// ------------------------------------------------------------------ cluster-scope PTX

__device__ __forceinline__ uint32_t mapa(uint32_t smem_addr, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(cta));
  return r;
}

// 2D tile load into this CTA's shared memory whose completion is counted on
// an mbarrier of the pair (a shared::cluster address, normally the leader's).
__device__ __forceinline__ void tma_load(void* smem_dst, const CUtensorMap* map, int32_t c0,
                                         int32_t c1, uint32_t bar_cluster, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster), "l"(policy)
      : "memory");
}

// 3-D and 4-D forms of the same load (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, int32_t c2, uint32_t bar_cluster,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes.L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cluster),
      "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3,
                                            uint32_t bar_cluster, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes.L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(bar_cluster), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// mbarrier wait with cluster-scope acquire: data written by the other CTA of
// the pair before its release-arrive is visible afterwards.  Bounded like
// mbar_wait.
__device__ __forceinline__ bool wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* status) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_status(status, kStatusTimeout);
      return false;
    }
  }
}

// Hand-off of this CTA's shared-memory writes to a thread of the other CTA:
// a release fence restricted to shared::cta at cluster scope, then a relaxed
// arrive on the (remote) mbarrier.  Lighter than a cluster-wide release.
__device__ __forceinline__ void arrive_remote_smem(uint32_t bar_cluster) {
  asm volatile(
      "fence.release.sync_restrict::shared::cta.cluster;\n\t"
      "mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
      : "memory");
}

// The matching side: relaxed wait on a local mbarrier, then an acquire fence
// restricted to shared::cluster at cluster scope.  Bounded like mbar_wait.
__device__ __forceinline__ bool wait_cluster_smem(uint64_t* bar, uint32_t parity,
                                                  uint32_t* status) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.relaxed.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) {
      asm volatile("fence.acquire.sync_restrict::shared::cluster.cluster;" ::: "memory");
      return true;
    }
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_status(status, kStatusTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                    uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at this offset in both CTAs when the MMAs
// issued so far have completed.
__device__ __forceinline__ void commit_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(static_cast<uint16_t>(0x3))
      : "memory");
}

__device__ __forceinline__ void commit_local(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

template <uint32_t kCols>
__device__ __forceinline__ void tmem_alloc2(uint32_t* slot) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "n"(kCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <uint32_t kCols>
__device__ __forceinline__ void tmem_dealloc2(uint32_t base) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(base), "n"(kCols)
               : "memory");
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr_cluster, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr_cluster), "f"(v) : "memory");
}

}  // namespace pair
}  // namespace moe
