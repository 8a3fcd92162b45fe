// Weight-row tiles on CTA pairs: tcgen05.mma.cta_group::2 with the weight
// rows on M (256 per pair) and the expert's tokens on N (fitted per tile).
//
// Ragged experts of a few hundred rows waste up to a whole 256-row tile when
// tokens are on M; with tokens on N a tile pads at most 31 rows.  A pair tile
// is 256 weight rows x N token rows (N <= 256, a multiple of 32):
//   CTA r loads 128 weight rows (GEMM1: 64 gate + the matching 64 up rows of
//   output columns f0 + 64 r .. f0 + 64 r + 63; GEMM2: output features
//   128 r .. 128 r + 127 of the 256) and token rows r*N/2 .. (r+1)*N/2 - 1;
//   the leader issues M=256 MMAs that read both CTAs' halves; each CTA's TMEM
//   receives its 128 weight rows x N tokens.
// So each CTA's epilogue is the 1-CTA weight-row epilogue (GEMM1 exchanges
// gate and up rows through shared memory, 32 tokens at a time).  Tile order
// and the cluster-scope helpers are in pair_tiles.cuh; every role walks the
// order with its own incremental iterator (no per-tile division or search
// between K steps).
//
// Operands move in stages of two 64-deep K steps (three stages of 32 KB of
// weights + up to 32 KB of tokens per CTA): one 4-D bulk-tensor copy brings a
// CTA's 128 weight rows (two 64-row blocks a fixed gap apart) for both K
// steps and one 3-D copy its token rows, each row a 256-byte segment of
// global memory.  A TMA unit keeps a bounded number of row requests in
// flight, so 256-byte rows stream about twice as fast per SM as the 128-byte
// rows of a 64-column box, and the producer issues a third of the copies.
//
// Synchronisation: both CTAs' copies complete on the leader's full barrier
// (the leader's producer expects both CTAs' bytes); the leader's MMA commits
// release the stage on both CTAs' empty barriers and the accumulator on both
// CTAs' tfull barriers; every epilogue thread of both CTAs arrives on the
// leader's tempty barrier.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "pair_tiles.cuh"
#include "ptx.cuh"

namespace moe {

bool make_map_kplanes(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows);  // grouped_gemm.cu
bool make_map_kplanes_pair(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint64_t gap);  // grouped_gemm.cu

namespace {

constexpr int kThreadsP = 192;
constexpr int kMP = pair::kM;                  // weight rows per CTA
constexpr int kNmaxP = pair::kNmax;            // token rows per pair tile
// A stage is two 64-deep K steps: every weight and token row of it is one
// 256-byte segment of global memory, so one bulk-tensor copy moves twice the
// bytes of a 64-column box for the same number of row requests.
constexpr int kBKS = 2 * kBK;
constexpr int kStagesP = 3;
constexpr uint32_t kWBytesP = kMP * kBKS * 2;   // 32 KB
constexpr uint32_t kXBytesP = (kNmaxP / 2) * kBKS * 2;  // 32 KB: this CTA's token half
constexpr uint32_t kStageP = kWBytesP + kXBytesP;
constexpr uint32_t kTmemColsP = 2 * kNmaxP;
constexpr int kMaxEP = 1024;
constexpr int kDPitchP = 33;
constexpr uint32_t kBarBytesP = 256;
static_assert((2 * kStagesP + 5) * 8 + 8 <= kBarBytesP, "barrier area");
constexpr size_t kSmemP = 1024 + kStagesP * kStageP + kBarBytesP +
                          4 * (kMaxEP + 1) * sizeof(int32_t) + kMP * kDPitchP * sizeof(float);
static_assert(kSmemP + 1024 <= 232448, "shared memory budget (dynamic + the 1024-aligned static part)");

struct PParams {
  const int32_t* expert_offsets;
  uint16_t* out;  // bf16 [rows, ldo]
  int E, K, w_tiles, w_rows_per_expert, ldo, F, interleave, out_rows;
  float clamp;
  uint32_t* status;
};

__device__ __forceinline__ float silu_p(float z) { return z / (1.0f + expf(-z)); }

template <Epi kEpi>
__global__ void __launch_bounds__(kThreadsP, 1)
grouped_gemm_swap2_kernel(const __grid_constant__ CUtensorMap map_w,
                          const __grid_constant__ CUtensorMap map_x16,
                          const __grid_constant__ CUtensorMap map_x32,
                          const __grid_constant__ CUtensorMap map_x64,
                          const __grid_constant__ CUtensorMap map_x128, const PParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sW = smem;
  uint8_t* sX = smem + kStagesP * kWBytesP;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStagesP * kStageP);
  uint64_t* empty = full + kStagesP;
  uint64_t* tfull = empty + kStagesP;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + kStagesP * kStageP + kBarBytesP);
  int32_t* s_hp = s_off + (kMaxEP + 1);
  int32_t* s_cp = s_hp + (kMaxEP + 1);
  int32_t* s_ntk = s_cp + (kMaxEP + 1);
  float* sD = reinterpret_cast<float*>(s_ntk + (kMaxEP + 1));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesP; ++s) {
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
    prefetch_tensormap(&map_w);
    prefetch_tensormap(&map_x16);
    prefetch_tensormap(&map_x32);
    prefetch_tensormap(&map_x64);
    prefetch_tensormap(&map_x128);
  }
  if (warp == 1) {  // one warp of each CTA allocates the pair's columns together
    pair::tmem_alloc2<kTmemColsP>(tmem_slot);
  }
  // Everything above touches only this CTA's shared memory and tensor memory
  // and the kernel parameters: it overlaps the previous kernel's tail.
  pdl_enter();
  for (int i = threadIdx.x; i <= p.E; i += kThreadsP) s_off[i] = p.expert_offsets[i];
  __syncthreads();
  const pair::Sched sched =
      pair::build_sched<kThreadsP>(s_off, p.E, p.w_tiles, s_ntk, s_hp, s_cp);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before anything signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = sched.total();
  const int tile0 = static_cast<int>(blockIdx.x >> 1);
  const int tstride = static_cast<int>(gridDim.x >> 1);
  const int num_kb = p.K / kBKS;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_normal();
      const uint64_t pol_w_once = policy_evict_first();  // a cold expert's tile: read once
      const uint64_t pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      pair::TileIter it;
      it.init(tile0, tstride, sched);
      for (int tile = tile0; tile < total_tiles && !*abort_flag; tile += tstride, it.next()) {
        const pair::Tile t = it.get(sched);
        const int tok0 = t.n * kNmaxP;
        const int nval = min(kNmaxP, s_off[t.e + 1] - s_off[t.e] - tok0);
        const int half = pair::half_rows(nval);
        const int bi = pair::box_index(half);
        const int box = 16 << bi;
        const CUtensorMap* mx = bi == 0 ? &map_x16 : bi == 1 ? &map_x32 : bi == 2 ? &map_x64
                                                                                  : &map_x128;
        const int x_row = s_off[t.e] + tok0 + static_cast<int>(rank) * half;
        int w_row0, w_row1;  // the second block is the map's fixed gap further
        pair::weight_rows(kEpi == Epi::kSwiGLU, t.m, rank, p.F, p.interleave, w_row0, w_row1);
        w_row0 += t.e * p.w_rows_per_expert;
        const uint32_t bytes = kWBytesP + static_cast<uint32_t>(box) * kBKS * 2;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.status)) { *abort_flag = 1; break; }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * bytes);
          const uint32_t bar = pair::mapa(smem_u32(&full[stage]), 0);
          const int plane = 2 * kb;
          const uint64_t pw = t.hot ? pol_w : pol_w_once;
          pair::tma_load_4d(sW + stage * kWBytesP, &map_w, 0, w_row0, 0, plane, bar, pw);
          pair::tma_load_3d(sX + stage * kXBytesP, mx, 0, x_row, plane, bar, pol_x);
          ++issued;
          if (++stage == kStagesP) { stage = 0; phase ^= 1; }
        }
      }
      if (leader) {
        for (int i = 1; i <= kStagesP && i <= issued; ++i) {
          int s = stage - i;
          uint32_t ph = phase;
          if (s < 0) { s += kStagesP; ph ^= 1; }
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
      pair::TileIter it;
      it.init(tile0, tstride, sched);
      for (int tile = tile0; tile < total_tiles && !*abort_flag;
           tile += tstride, ++local, it.next()) {
        const int buf = local & 1;
        const uint32_t tph = (local >> 1) & 1;
        const pair::Tile t = it.get(sched);
        const int nval = min(kNmaxP, s_off[t.e + 1] - s_off[t.e] - t.n * kNmaxP);
        const int half = pair::half_rows(nval);
        const uint32_t nmma = static_cast<uint32_t>(2 * half);
        const uint32_t idesc = idesc_bf16_f32(2 * kMP, nmma);
        // the token box's second plane follows its first (box rows x 128 B)
        const uint32_t x_plane = (16u << pair::box_index(half)) * kBK * 2;
        if (!mbar_wait(&tempty[buf], tph ^ 1, p.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kNmaxP;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.status)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int pl = 0; pl < 2; ++pl) {
            const uint64_t w_desc =
                sw128_kmajor_desc(smem_u32(sW + stage * kWBytesP + pl * (kWBytesP / 2)));
            const uint64_t x_desc =
                sw128_kmajor_desc(smem_u32(sX + stage * kXBytesP + pl * x_plane));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              pair::mma(d_tmem, w_desc + 2 * kk, x_desc + 2 * kk, idesc, (kb | pl | kk) != 0);
          }
          pair::commit_both(&empty[stage]);
          if (++stage == kStagesP) { stage = 0; phase ^= 1; }
        }
        if (!ok) { *abort_flag = 1; break; }
        pair::commit_both(&tfull[buf]);
      }
      pair::commit_local(drain);
      mbar_wait(drain, 0, p.status);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int quad = warp & 3;
    const int et = threadIdx.x - 64;
    const int wrow = quad * 32 + lane;  // weight row inside this CTA's 128
    const int ie = (p.interleave == 32) ? 32 : 64;
    const int fl = et & 63;
    const int grow = (fl / ie) * 2 * ie + fl % ie;
    const int urow = grow + ie;
    const bool clamp = p.clamp > 0.f && isfinite(p.clamp);
    const uint32_t tempty_leader0 = pair::mapa(smem_u32(&tempty[0]), 0);
    const uint32_t tempty_leader1 = pair::mapa(smem_u32(&tempty[1]), 0);
    int local = 0;
    pair::TileIter it;
    it.init(tile0, tstride, sched);
    for (int tile = tile0; tile < total_tiles; tile += tstride, ++local, it.next()) {
      const int buf = local & 1;
      const uint32_t tph = (local >> 1) & 1;
      const bool ok = mbar_wait(&tfull[buf], tph, p.status);
      if (bar_red_or(1, 128, !ok || *abort_flag != 0)) {  // leave together
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const pair::Tile t = it.get(sched);
      const int tok0 = t.n * kNmaxP;
      const int nval = min(kNmaxP, s_off[t.e + 1] - s_off[t.e] - tok0);
      const int nchunk = (nval + 31) / 32;
      const long row0 = static_cast<long>(s_off[t.e]) + tok0;
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * kNmaxP;
      for (int c = 0; c < nchunk; ++c) {
        uint32_t a[32];
        tmem_ld_32x32b_x32(t_lane + c * 32, a);
        tmem_ld_wait();
        if (c == nchunk - 1) {  // the accumulator is no longer needed
          tc_fence_before();
          pair::arrive_remote(buf ? tempty_leader1 : tempty_leader0);
        }
        const int n0 = c * 32;
        if (kEpi == Epi::kPlain) {
          const int feat = t.m * (2 * kMP) + static_cast<int>(rank) * kMP + wrow;
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            if (n0 + n < nval) {
              const __nv_bfloat16 v = __float2bfloat16_rn(__uint_as_float(a[n]));
              p.out[(row0 + n0 + n) * p.ldo + feat] = *reinterpret_cast<const uint16_t*>(&v);
            }
          }
        } else {
          if (c > 0) bar_sync_named(1, 128);
#pragma unroll
          for (int n = 0; n < 32; ++n) sD[wrow * kDPitchP + n] = __uint_as_float(a[n]);
          bar_sync_named(1, 128);
          const int f = t.m * kMP + static_cast<int>(rank) * 64 + fl;
#pragma unroll 4
          for (int n = et >> 6; n < 32; n += 2) {
            if (n0 + n < nval) {
              float g = sD[grow * kDPitchP + n], u = sD[urow * kDPitchP + n];
              if (clamp) {
                g = fminf(g, p.clamp);
                u = fminf(fmaxf(u, -p.clamp), p.clamp);
              }
              const __nv_bfloat16 v = __float2bfloat16_rn(silu_p(g) * u);
              p.out[(row0 + n0 + n) * p.ldo + f] = *reinterpret_cast<const uint16_t*>(&v);
            }
          }
        }
      }
    }
    if (kEpi == Epi::kPlain) {  // rows past the last expert's segment are zero
      const long first = s_off[p.E];
      const long n = (static_cast<long>(p.out_rows) - first) * p.ldo;
      for (long i = static_cast<long>(blockIdx.x) * 128 + et; i < n;
           i += static_cast<long>(gridDim.x) * 128)
        p.out[first * p.ldo + i] = 0;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    pair::tmem_dealloc2<kTmemColsP>(tmem_base);
  }
}

template <Epi kEpi>
cudaError_t launch_swap2_impl(const CUtensorMap* maps, const PParams& pp, int grid,
                              cudaStream_t s) {
  auto kern = grouped_gemm_swap2_kernel<kEpi>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemP));
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreadsP), kSmemP, s, 2,
                       maps[0], maps[1], maps[2], maps[3], maps[4], pp);
}

}  // namespace

cudaError_t launch_grouped_gemm_swap2(const GroupedGemmArgs& g, cudaStream_t s) {
  if (g.a_rows == 0) return cudaSuccess;
  if (g.E > kMaxEP || g.K % kBKS != 0) return cudaErrorInvalidValue;
  // rows between a CTA's two 64-row weight blocks (pair::weight_rows)
  uint64_t gap = 64;
  if (g.epi == Epi::kSwiGLU && g.interleave == 0) gap = static_cast<uint64_t>(g.F);
  else if (g.epi == Epi::kSwiGLU && g.interleave > 64) gap = static_cast<uint64_t>(g.interleave);
  CUtensorMap maps[5];
  if (!make_map_kplanes_pair(&maps[0], g.b, static_cast<uint64_t>(g.E) * g.b_rows_per_expert,
                             static_cast<uint64_t>(g.K), gap))
    return cudaErrorInvalidValue;
  const uint32_t boxes[4] = {16, 32, 64, 128};
  for (int i = 0; i < 4; ++i)
    if (!make_map_kplanes(&maps[1 + i], g.a, static_cast<uint64_t>(g.a_rows),
                          static_cast<uint64_t>(g.K), boxes[i]))
      return cudaErrorInvalidValue;
  PParams pp;
  pp.expert_offsets = g.expert_offsets;
  pp.out = static_cast<uint16_t*>(g.out);
  pp.E = g.E;
  pp.K = g.K;
  pp.w_rows_per_expert = g.b_rows_per_expert;
  pp.ldo = g.ldo;
  pp.out_rows = g.out_rows;
  pp.F = g.F;
  pp.interleave = g.interleave;
  pp.clamp = g.clamp;
  pp.status = g.status;
  // pair tiles along the weights: GEMM1 covers 128 output columns, GEMM2 256 features
  pp.w_tiles = (g.epi == Epi::kSwiGLU) ? g.F / kMP : g.ldo / (2 * kMP);
  const long max_tiles =
      (static_cast<long>(ceil_div(g.a_rows, kNmaxP)) + std::min(g.E, g.a_rows)) * pp.w_tiles;
  const long want = std::min<long>(num_sms() & ~1, 2 * max_tiles);
  const int grid = static_cast<int>(std::max(2L, want & ~1L));
  if (g.epi == Epi::kSwiGLU) return launch_swap2_impl<Epi::kSwiGLU>(maps, pp, grid, s);
  if (g.epi == Epi::kPlain) return launch_swap2_impl<Epi::kPlain>(maps, pp, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
