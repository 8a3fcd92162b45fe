// Grouped GEMM on CTA pairs: tcgen05.mma.cta_group::2, one 256 x 256 x 16
// MMA per instruction across two SMs.
//
// A 2-CTA cluster takes two m-tiles of one (expert, n-tile): CTA r holds the
// 128 token rows of m-tile 2*mp + r (the A half) and the 128 weight rows
// 128*r .. 128*r+127 of the 256-row weight tile (the B half), both loaded by
// its own producer into its own shared memory.  The leader CTA (rank 0)
// issues every MMA for the pair; the hardware reads each CTA's A half and
// both B halves and writes each CTA's 128 x 256 fp32 accumulator into that
// CTA's TMEM.  Compared with one CTA per 128 x 256 tile this halves the
// operand bytes each SM loads per FLOP and the MMA instructions issued.
//
// Synchronisation (all waits bounded):
//   full[s]   leader's barrier; both CTAs' TMA loads complete their bytes on
//             it (.cta_group::2 lets a load signal the peer's barrier), the
//             leader's producer arms it with the pair's byte count
//   empty[s]  each CTA's own; the leader's MMA commit arrives on both
//   tfull[b]  each CTA's own; the leader's commit after a tile arrives on both
//   tempty[b] leader's; all 256 epilogue threads of the pair arrive
// Epilogues as in grouped_gemm.cu (SwiGLU for GEMM1, plain bf16 for GEMM2).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

bool make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);  // grouped_gemm.cu

namespace {

constexpr int kStages2 = 6;
constexpr int kThreads2 = 192;
constexpr uint32_t kAHalf = kBM * kBK * 2;          // 16 KB: this CTA's 128 token rows
constexpr uint32_t kBHalf = (kBN / 2) * kBK * 2;    // 16 KB: this CTA's 128 weight rows
constexpr uint32_t kStage2 = kAHalf + kBHalf;       // 32 KB per CTA
constexpr uint32_t kPairTx = 2 * kStage2;           // bytes landing per stage, both CTAs
constexpr uint32_t kTmemCols2 = 2 * kBN;            // two 256-column accumulators
constexpr uint32_t kIdesc2 = idesc_bf16_f32(2 * kBM, kBN);  // M = 256 across the pair
constexpr int kMaxE2 = 1024;
static_assert((2 * kStages2 + 5) * 8 + 8 <= 256, "barrier area");
constexpr size_t kSmem2 = 1024 + kStages2 * kStage2 + 256 + 3 * (kMaxE2 + 1) * sizeof(int32_t);
static_assert(kSmem2 <= 232448, "shared memory budget");

struct P2 {
  const int32_t* expert_offsets;
  const int32_t* mtile_prefix;
  uint4* out;
  int E, K, n_tiles, b_rows_per_expert, ldo_vec, out_rows, F, interleave, ieff;
  float clamp;
  uint32_t* status;
};

struct Tile2 {
  int e, m, n;
};

__device__ __forceinline__ Tile2 decode_tile2(int tile, const int32_t* ptp, int E, int n_tiles,
                                              uint32_t rank) {
  const int q = tile / n_tiles;
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ptp[mid] <= q) lo = mid; else hi = mid - 1;
  }
  Tile2 t;
  t.e = lo;
  const int mp = ptp[lo + 1] - ptp[lo];
  const int local = tile - ptp[lo] * n_tiles;
  t.n = local / mp;
  t.m = 2 * (local - t.n * mp) + static_cast<int>(rank);
  return t;
}

__device__ __forceinline__ uint32_t mapa_u32(uint32_t smem_addr, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(cta));
  return r;
}

// 2-D tile load into this CTA's shared memory whose completion is counted on
// an mbarrier given by its cluster address (here: the leader's).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map,
                                                 int32_t c0, int32_t c1, uint32_t bar_cluster,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ void mma2_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the barrier at this offset in both CTAs of the pair once every
// MMA the leader issued so far has completed.
__device__ __forceinline__ void mma2_commit_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(static_cast<uint16_t>(0x3))
      : "memory");
}

__device__ __forceinline__ float silu2(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <Epi kEpi>
__global__ void __launch_bounds__(kThreads2, 1)
grouped_gemm_2cta_kernel(const __grid_constant__ CUtensorMap map_a,
                         const __grid_constant__ CUtensorMap map_b, const P2 p) {
  pdl_enter();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages2 * kAHalf;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages2 * kStage2);
  uint64_t* empty = full + kStages2;
  uint64_t* tfull = empty + kStages2;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + kStages2 * kStage2 + 256);
  int32_t* s_mtp = s_off + (p.E + 1);
  int32_t* s_ptp = s_mtp + (p.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  for (int i = threadIdx.x; i <= p.E; i += kThreads2) {
    s_off[i] = p.expert_offsets[i];
    s_mtp[i] = p.mtile_prefix[i];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages2; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
  }
  if (warp == 1) {  // one warp of each CTA allocates the pair's columns together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "n"(kTmemCols2)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  __syncthreads();
  {  // prefix of ceil(m-tiles / 2) per expert
    __shared__ int s_part[kThreads2 / 32];
    const int per = (p.E + kThreads2 - 1) / kThreads2;
    const int e0 = min(p.E, static_cast<int>(threadIdx.x) * per), e1 = min(p.E, e0 + per);
    int run = 0;
    for (int e = e0; e < e1; ++e) run += (s_mtp[e + 1] - s_mtp[e] + 1) >> 1;
    int incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) s_part[warp] = incl;
    __syncthreads();
    int acc = incl - run;
    for (int w = 0; w < warp; ++w) acc += s_part[w];
    for (int e = e0; e < e1; ++e) {
      s_ptp[e] = acc;
      acc += (s_mtp[e + 1] - s_mtp[e] + 1) >> 1;
    }
    if (threadIdx.x == kThreads2 - 1) {
      int total = 0;
      for (int w = 0; w < kThreads2 / 32; ++w) total += s_part[w];
      s_ptp[p.E] = total;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before anything signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = s_ptp[p.E] * p.n_tiles;
  const int tile0 = static_cast<int>(blockIdx.x >> 1);
  const int tstride = static_cast<int>(gridDim.x >> 1);
  const int num_kb = p.K / kBK;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_b = policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      for (int tile = tile0; tile < total_tiles && !*abort_flag; tile += tstride) {
        const Tile2 t = decode_tile2(tile, s_ptp, p.E, p.n_tiles, rank);
        const int a_row = s_off[t.e] + t.m * kBM;
        int b_row;
        if (kEpi == Epi::kSwiGLU) {
          const int f0 = t.n * (kBN / 2);
          int r0, r1;
          if (p.interleave == 0) {
            r0 = f0;
            r1 = p.F + f0;
          } else if (p.ieff == 128) {
            r0 = (f0 / p.interleave) * 2 * p.interleave + f0 % p.interleave;
            r1 = r0 + p.interleave;
          } else {
            r0 = 2 * f0;
            r1 = 2 * f0 + 128;
          }
          b_row = rank ? r1 : r0;
        } else {
          b_row = t.n * kBN + static_cast<int>(rank) * 128;
        }
        b_row += t.e * p.b_rows_per_expert;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.status)) { *abort_flag = 1; break; }
          if (leader) mbar_arrive_expect_tx(&full[stage], kPairTx);
          const uint32_t bar = mapa_u32(smem_u32(&full[stage]), 0);
          const int kx = kb * kBK;
          tma_load_2d_pair(sA + stage * kAHalf, &map_a, kx, a_row, bar, pol_a);
          tma_load_2d_pair(sB + stage * kBHalf, &map_b, kx, b_row, bar, pol_b);
          ++issued;
          if (++stage == kStages2) { stage = 0; phase ^= 1; }
        }
      }
      // leader: its loads and the peer's complete on full[]; wait for the last ones
      if (leader) {
        for (int i = 1; i <= kStages2 && i <= issued; ++i) {
          int s = stage - i;
          uint32_t ph = phase;
          if (s < 0) { s += kStages2; ph ^= 1; }
          mbar_wait(&full[s], ph, p.status);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA (leader only)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int tile = tile0; tile < total_tiles && !*abort_flag; tile += tstride, ++local) {
        const int buf = local & 1;
        const uint32_t tph = (local >> 1) & 1;
        if (!mbar_wait(&tempty[buf], tph ^ 1, p.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kBN;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint64_t a_desc = sw128_kmajor_desc(smem_u32(sA + stage * kAHalf));
          const uint64_t b_desc = sw128_kmajor_desc(smem_u32(sB + stage * kBHalf));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma2_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, kIdesc2, (kb | kk) != 0);
          mma2_commit_both(&empty[stage]);
          if (++stage == kStages2) { stage = 0; phase ^= 1; }
        }
        if (!ok) { *abort_flag = 1; break; }
        mma2_commit_both(&tfull[buf]);
      }
      asm volatile(
          "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              smem_u32(drain))
          : "memory");
      mbar_wait(drain, 0, p.status);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    int local = 0;
    for (int tile = tile0; tile < total_tiles && !*abort_flag; tile += tstride, ++local) {
      const int buf = local & 1;
      const uint32_t tph = (local >> 1) & 1;
      if (!mbar_wait(&tfull[buf], tph, p.status)) { *abort_flag = 1; break; }
      tc_fence_after();
      const Tile2 t = decode_tile2(tile, s_ptp, p.E, p.n_tiles, rank);
      const int seg_rows = s_off[t.e + 1] - s_off[t.e];
      const bool row_ok = t.m * kBM + row_in_tile < seg_rows;
      const long out_row = static_cast<long>(s_off[t.e]) + t.m * kBM + row_in_tile;
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * kBN;
      if (kEpi == Epi::kSwiGLU) {
        uint4* dst = p.out + out_row * p.ldo_vec + (t.n * (kBN / 2)) / 8;
        const bool clamp = p.clamp > 0.f && isfinite(p.clamp);
#pragma unroll 1
        for (int c = 0; c < (kBN / 2) / 32; ++c) {
          const int i0 = c * 32;
          const int gcol = (i0 / p.ieff) * 2 * p.ieff + i0 % p.ieff;
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(t_lane + gcol, g);
          tmem_ld_32x32b_x32(t_lane + gcol + p.ieff, u);
          tmem_ld_wait();
          if (row_ok) {
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float g0 = __uint_as_float(g[i]), g1 = __uint_as_float(g[i + 1]);
              float u0 = __uint_as_float(u[i]), u1 = __uint_as_float(u[i + 1]);
              if (clamp) {
                g0 = fminf(g0, p.clamp);
                g1 = fminf(g1, p.clamp);
                u0 = fminf(fmaxf(u0, -p.clamp), p.clamp);
                u1 = fminf(fmaxf(u1, -p.clamp), p.clamp);
              }
              packed[i / 2] = pack2(silu2(g0) * u0, silu2(g1) * u1);
            }
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c * 4 + v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                          packed[4 * v + 3]);
          }
        }
      } else {
        uint4* dst = p.out + out_row * p.ldo_vec + (t.n * kBN) / 8;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t a[32];
          tmem_ld_32x32b_x32(t_lane + c * 32, a);
          tmem_ld_wait();
          if (row_ok) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c * 4 + v] = make_uint4(
                  pack2(__uint_as_float(a[8 * v + 0]), __uint_as_float(a[8 * v + 1])),
                  pack2(__uint_as_float(a[8 * v + 2]), __uint_as_float(a[8 * v + 3])),
                  pack2(__uint_as_float(a[8 * v + 4]), __uint_as_float(a[8 * v + 5])),
                  pack2(__uint_as_float(a[8 * v + 6]), __uint_as_float(a[8 * v + 7])));
          }
        }
      }
      tc_fence_before();
      mbar_arrive_cluster(mapa_u32(smem_u32(&tempty[buf]), 0));  // the leader's barrier
    }
    // Rows past the last expert's segment (masked routes) are zero outputs.
    if (kEpi == Epi::kPlain) {
      const long first = s_off[p.E];
      const long nvec = (static_cast<long>(p.out_rows) - first) * p.ldo_vec;
      const int et = threadIdx.x - 64;
      for (long v = static_cast<long>(blockIdx.x) * 128 + et; v < nvec;
           v += static_cast<long>(gridDim.x) * 128)
        p.out[first * p.ldo_vec + v] = make_uint4(0, 0, 0, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA frees TMEM or exits while the pair still works
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "n"(kTmemCols2)
                 : "memory");
  }
}

template <Epi kEpi>
cudaError_t launch_2cta_impl(const CUtensorMap& ma, const CUtensorMap& mb, const P2& pp,
                             int grid, cudaStream_t s) {
  auto kern = grouped_gemm_2cta_kernel<kEpi>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmem2));
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads2), kSmem2, s, 2,
                       ma, mb, pp);
}

}  // namespace

cudaError_t launch_grouped_gemm_2cta(const GroupedGemmArgs& g, cudaStream_t s) {
  if (g.a_rows == 0) return cudaSuccess;
  if (g.E > kMaxE2) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  if (!make_map_2d(&ma, g.a, static_cast<uint64_t>(g.a_rows), static_cast<uint64_t>(g.K), kBM))
    return cudaErrorInvalidValue;
  if (!make_map_2d(&mb, g.b, static_cast<uint64_t>(g.E) * g.b_rows_per_expert,
                   static_cast<uint64_t>(g.K), 128))
    return cudaErrorInvalidValue;
  P2 pp;
  pp.expert_offsets = g.expert_offsets;
  pp.mtile_prefix = g.mtile_prefix;
  pp.out = static_cast<uint4*>(g.out);
  pp.E = g.E;
  pp.K = g.K;
  pp.n_tiles = g.n_tiles;
  pp.b_rows_per_expert = g.b_rows_per_expert;
  pp.ldo_vec = g.ldo / 8;
  pp.out_rows = g.out_rows;
  pp.F = g.F;
  pp.interleave = g.interleave;
  pp.ieff = (g.interleave == 0 || g.interleave % 128 == 0) ? 128 : g.interleave;
  pp.clamp = g.clamp;
  pp.status = g.status;
  const long max_pair_tiles =
      (static_cast<long>(ceil_div(g.a_rows, 2 * kBM)) + std::min(g.E, g.a_rows)) * g.n_tiles;
  const long want = std::min<long>(num_sms() & ~1, 2 * max_pair_tiles);
  const int grid = static_cast<int>(std::max(2L, want & ~1L));
  if (g.epi == Epi::kSwiGLU) return launch_2cta_impl<Epi::kSwiGLU>(ma, mb, pp, grid, s);
  if (g.epi == Epi::kPlain) return launch_2cta_impl<Epi::kPlain>(ma, mb, pp, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
