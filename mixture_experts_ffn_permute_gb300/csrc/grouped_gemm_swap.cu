// Decode-sized grouped GEMMs: the weight rows are the MMA's M side and the
// few tokens of each expert its N side ("swap-AB").
//
// A tile is 128 weight rows x up to kNmax = 32 token rows of one expert:
//   D[128 x N] = W[128 weight rows of e, K] * X[N token rows of e, K]^T
// with N = the expert's remaining rows rounded up to 16, set per tile in the
// instruction descriptor.  At decode sizes an expert sees a handful of
// tokens: a K step moves 16 KB of weights and 4 KB of activations, so the
// weights stream once at HBM speed.  One ring of four stages of two 64-deep
// K steps holds both: one 4-D copy brings the tile's weight rows for both K
// steps (each row a 256-byte segment: the copy path counts row requests) and
// one 3-D copy its 32 token rows; the MMA issuer releases a stage with one
// commit (at this N a tcgen05.commit costs about as much as a K step's four
// MMAs).  The tile count is (expert, weight-row tile, token tile), token
// tiles fastest so that CTAs sharing a weight tile run together and the
// second read hits L2.
//
// Epilogues:
//   GEMM1 (kSwiGLU): the 128 weight rows are 64 gate rows and the matching
//     64 up rows; the accumulator goes through shared memory so one thread
//     sees both halves, and h[token row][f] is stored as bf16.
//   GEMM2 (kPlain):  y[token row][feature] bf16, 32 consecutive features per
//     warp store.
// Pipeline, TMEM double buffering and bounded waits are as in
// grouped_gemm.cu; the per-expert tile prefix is computed by every CTA from
// expert_offsets at start-up.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

bool make_map_kplanes(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows);  // grouped_gemm.cu
bool make_map_kplanes_pair(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint64_t gap);  // grouped_gemm.cu

namespace {

constexpr int kM = 128;                                // weight rows per tile
constexpr int kXBox = 32;                              // token rows per TMA box
constexpr int kThreadsS = 192;
constexpr uint32_t kWBytes = 2 * kM * kBK * 2;         // 32 KB: two K steps
constexpr int kMaxES = 1024;
constexpr int kDPitch = 33;                            // padded fp32 row of the exchange chunk
constexpr int kNmaxS = 32;                             // token rows per tile
constexpr int kStagesS = 4;                            // x 2 K steps

template <int kNmax, int kStages>
struct SwapCfg {
  static constexpr uint32_t kXPlane = kNmax * kBK * 2;  // one K step of token rows
  static constexpr uint32_t kXBytes = 2 * kXPlane;
  static constexpr uint32_t kRingBytes = kStages * (kWBytes + kXBytes);
  static constexpr uint32_t kTmemCols = 2 * kNmax;     // two accumulators
  // mbarriers (full/empty per stage, 2 + 2 accumulator, drain) plus the TMEM
  // address word and the abort flag
  static constexpr uint32_t kBarBytes = 512;
  static_assert((2 * kStages + 5) * 8 + 8 <= kBarBytes, "barrier area");
  static constexpr size_t kSmem = 1024 + kRingBytes + kBarBytes +
                                  3 * (kMaxES + 1) * sizeof(int32_t) +
                                  kM * kDPitch * sizeof(float);
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kTmemCols >= 32 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation");
};

struct SParams {
  const int32_t* expert_offsets;
  uint16_t* out;               // bf16 [rows, ldo]
  int E, K, w_tiles, w_rows_per_expert, ldo, F, interleave, out_rows;
  float clamp;
  uint32_t* status;
};

struct STile {
  int e, m, n;  // expert, weight-row tile, token tile
};

__device__ __forceinline__ STile decode_stile(int tile, const int32_t* tp, const int32_t* ntk,
                                              int E, int w_tiles) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tp[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  STile t;
  t.e = lo;
  const int local = tile - tp[lo];
  const int nt = ntk[lo];
  t.m = local / nt;
  t.n = local - t.m * nt;
  return t;
}

__device__ __forceinline__ float silu_s(float z) { return z / (1.0f + expf(-z)); }

template <Epi kEpi, int kNmax, int kStages>
__global__ void __launch_bounds__(kThreadsS, 1)
grouped_gemm_swap_kernel(const __grid_constant__ CUtensorMap map_w,
                         const __grid_constant__ CUtensorMap map_x, const SParams p) {
  using Cfg = SwapCfg<kNmax, kStages>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, kept as a shared-array pointer so that accesses
  // compile to shared-memory instructions
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sW = smem;
  uint8_t* sX = smem + kStages * kWBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kRingBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + Cfg::kRingBytes + Cfg::kBarBytes);
  int32_t* s_tp = s_off + (kMaxES + 1);   // tile prefix per expert
  int32_t* s_ntk = s_tp + (kMaxES + 1);   // token tiles per expert
  float* sD = reinterpret_cast<float*>(s_ntk + (kMaxES + 1));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&map_w);
    prefetch_tensormap(&map_x);
  }
  if (warp == 1) tmem_alloc<Cfg::kTmemCols>(tmem_slot);
  // Everything above touches only this CTA's shared memory and tensor memory
  // and the kernel parameters: it overlaps the previous kernel's tail.
  pdl_enter();
  for (int i = threadIdx.x; i <= p.E; i += kThreadsS) s_off[i] = p.expert_offsets[i];
  __syncthreads();
  // tile prefix: expert e owns w_tiles * ceil(rows_e / kNmax) tiles.  Thread
  // i scans a run of at most ceil(E / 192) experts; runs are then offset by a
  // scan over the threads.
  {
    __shared__ int s_part[kThreadsS / 32];
    const int per = (p.E + kThreadsS - 1) / kThreadsS;
    const int e0 = min(p.E, threadIdx.x * per), e1 = min(p.E, e0 + per);
    int run = 0;
    for (int e = e0; e < e1; ++e) {
      const int rows = s_off[e + 1] - s_off[e];
      const int nt = rows > 0 ? (rows + kNmax - 1) / kNmax : 0;
      s_ntk[e] = nt;
      run += nt * p.w_tiles;
    }
    int incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) s_part[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_part[w];
    int acc = base + incl - run;
    for (int e = e0; e < e1; ++e) {
      s_tp[e] = acc;
      acc += s_ntk[e] * p.w_tiles;
    }
    if (threadIdx.x == kThreadsS - 1) {
      int total = 0;
      for (int w = 0; w < kThreadsS / 32; ++w) total += s_part[w];
      s_tp[p.E] = total;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = s_tp[p.E];
  const int num_kb = p.K / kBK;  // even: stages hold two K steps

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_normal();
      const uint64_t pol_x = policy_evict_last();
      int st = 0;
      uint32_t ph = 0;
      long issued = 0;
      for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
        const STile t = decode_stile(tile, s_tp, s_ntk, p.E, p.w_tiles);
        const int tok0 = t.n * kNmax;
        const int nval = min(kNmax, s_off[t.e + 1] - s_off[t.e] - tok0);
        static_assert(kNmax == kXBox, "one token box per tile");
        (void)nval;
        const int x_row = s_off[t.e] + tok0;
        int w_row0, w_row1;
        if (kEpi == Epi::kSwiGLU) {
          const int f0 = t.m * (kM / 2);
          if (p.interleave == 32) {
            w_row0 = 2 * f0;
            w_row1 = 2 * f0 + kM / 2;
          } else if (p.interleave == 0) {
            w_row0 = f0;
            w_row1 = p.F + f0;
          } else {  // 64 or a multiple of 128: 64 whole gate rows, then 64 up rows
            w_row0 = (f0 / p.interleave) * 2 * p.interleave + f0 % p.interleave;
            w_row1 = w_row0 + p.interleave;
          }
        } else {
          w_row0 = t.m * kM;
          w_row1 = w_row0 + kM / 2;
        }
        w_row0 += t.e * p.w_rows_per_expert;
        (void)w_row1;  // the weight map's second block is its fixed gap further
        for (int kb = 0; kb < num_kb; kb += 2) {
          if (!mbar_wait(&empty[st], ph ^ 1, p.status)) { *abort_flag = 1; break; }
          mbar_arrive_expect_tx(&full[st], kWBytes + Cfg::kXBytes);
          tma_load_4d(sW + st * kWBytes, &map_w, 0, w_row0, 0, kb, &full[st], pol_w);
          tma_load_3d(sX + st * Cfg::kXBytes, &map_x, 0, x_row, kb, &full[st], pol_x);
          ++issued;
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
      }
      for (int i = 1; i <= kStages && i <= issued; ++i) {
        int s = st - i;
        uint32_t q = ph;
        if (s < 0) { s += kStages; q ^= 1; }
        mbar_wait(&full[s], q, p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      int local = 0;
      for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t tph = (local >> 1) & 1;
        const STile t = decode_stile(tile, s_tp, s_ntk, p.E, p.w_tiles);
        const int nval = min(kNmax, s_off[t.e + 1] - s_off[t.e] - t.n * kNmax);
        const uint32_t nmma = static_cast<uint32_t>((nval + 15) & ~15);  // MMA N: multiple of 16
        const uint32_t idesc = idesc_bf16_f32(kM, nmma);
        if (!mbar_wait(&tempty[buf], tph ^ 1, p.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kNmax;
        bool ok = true;
        for (int kb = 0; kb < num_kb; kb += 2) {
          if (!mbar_wait(&full[st], ph, p.status)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int pl = 0; pl < 2; ++pl) {
            const uint64_t w_desc =
                sw128_kmajor_desc(smem_u32(sW + st * kWBytes + pl * (kWBytes / 2)));
            const uint64_t x_desc =
                sw128_kmajor_desc(smem_u32(sX + st * Cfg::kXBytes + pl * Cfg::kXPlane));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_bf16_ss(d_tmem, w_desc + 2 * kk, x_desc + 2 * kk, idesc, (kb | pl | kk) != 0);
          }
          mma_commit(&empty[st]);  // one commit releases the stage
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
        if (!ok) { *abort_flag = 1; break; }
        mma_commit(&tfull[buf]);
      }
      mma_commit(drain);
      mbar_wait(drain, 0, p.status);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quad = warp & 3;
    const int et = threadIdx.x - 64;  // 0..127
    const int wrow = quad * 32 + lane;  // weight row inside the tile
    const int ie = (p.interleave == 32) ? 32 : 64;
    const int fl = et & 63;  // SwiGLU output column inside the tile
    const int grow = (fl / ie) * 2 * ie + fl % ie;
    const int urow = grow + ie;
    const bool clamp = p.clamp > 0.f && isfinite(p.clamp);
    int local = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++local) {
      const int buf = local & 1;
      const uint32_t tph = (local >> 1) & 1;
      const bool ok = mbar_wait(&tfull[buf], tph, p.status);
      // All four epilogue warps leave together (they share named barrier 1);
      // the vote is also the barrier that frees sD of the previous tile.
      if (bar_red_or(1, 128, !ok || *abort_flag != 0)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const STile t = decode_stile(tile, s_tp, s_ntk, p.E, p.w_tiles);
      const int tok0 = t.n * kNmax;  // first token row of the tile inside the expert
      const int nval = min(kNmax, s_off[t.e + 1] - s_off[t.e] - tok0);
      const int nchunk = (nval + 31) / 32;
      const long row0 = static_cast<long>(s_off[t.e]) + tok0;
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * kNmax;
      for (int c = 0; c < nchunk; ++c) {
        uint32_t a[32];
        tmem_ld_32x32b_x32(t_lane + c * 32, a);
        tmem_ld_wait();
        if (c == nchunk - 1) {  // the accumulator is no longer needed
          tc_fence_before();
          mbar_arrive(&tempty[buf]);
        }
        const int n0 = c * 32;
        if (kEpi == Epi::kPlain) {
          const int feat = t.m * kM + wrow;
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            if (n0 + n < nval) {
              const __nv_bfloat16 v = __float2bfloat16_rn(__uint_as_float(a[n]));
              p.out[(row0 + n0 + n) * p.ldo + feat] = *reinterpret_cast<const uint16_t*>(&v);
            }
          }
        } else {
          // exchange: gate and up rows of one output column live in different warps
          if (c > 0) bar_sync_named(1, 128);  // previous chunk's readers are done
#pragma unroll
          for (int n = 0; n < 32; ++n) sD[wrow * kDPitch + n] = __uint_as_float(a[n]);
          bar_sync_named(1, 128);
          const int f = t.m * (kM / 2) + fl;
#pragma unroll 4
          for (int n = et >> 6; n < 32; n += 2) {
            if (n0 + n < nval) {
              float g = sD[grow * kDPitch + n], u = sD[urow * kDPitch + n];
              if (clamp) {
                g = fminf(g, p.clamp);
                u = fminf(fmaxf(u, -p.clamp), p.clamp);
              }
              const __nv_bfloat16 v = __float2bfloat16_rn(silu_s(g) * u);
              p.out[(row0 + n0 + n) * p.ldo + f] = *reinterpret_cast<const uint16_t*>(&v);
            }
          }
        }
      }
    }
    // Rows past the last expert's segment (masked routes) are zero outputs.
    if (kEpi == Epi::kPlain) {
      const long first = s_off[p.E];
      const long n = (static_cast<long>(p.out_rows) - first) * p.ldo;
      for (long i = static_cast<long>(blockIdx.x) * 128 + et; i < n;
           i += static_cast<long>(gridDim.x) * 128)
        p.out[first * p.ldo + i] = 0;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<Cfg::kTmemCols>(tmem_base);
  }
}

template <Epi kEpi, int kNmax, int kStages>
cudaError_t launch_swap_impl(const CUtensorMap& mw, const CUtensorMap& mx, const SParams& sp,
                             int grid, cudaStream_t s) {
  using Cfg = SwapCfg<kNmax, kStages>;
  auto kern = grouped_gemm_swap_kernel<kEpi, kNmax, kStages>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::kSmem));
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreadsS), Cfg::kSmem, s, 1,
                       mw, mx, sp);
}

}  // namespace

cudaError_t launch_grouped_gemm_swap(const GroupedGemmArgs& g, cudaStream_t s) {
  if (g.a_rows == 0) return cudaSuccess;
  if (g.E > kMaxES || g.K % (2 * kBK) != 0) return cudaErrorInvalidValue;
  // rows between a tile's two 64-row weight blocks (the producer's w_row1 - w_row0)
  uint64_t gap = kM / 2;
  if (g.epi == Epi::kSwiGLU && g.interleave == 0) gap = static_cast<uint64_t>(g.F);
  else if (g.epi == Epi::kSwiGLU && g.interleave != 32) gap = static_cast<uint64_t>(g.interleave);
  CUtensorMap mw, mx;
  // weights: two 64-row blocks x two planes; tokens: 32-row boxes x two planes
  if (!make_map_kplanes_pair(&mw, g.b, static_cast<uint64_t>(g.E) * g.b_rows_per_expert,
                             static_cast<uint64_t>(g.K), gap))
    return cudaErrorInvalidValue;
  if (!make_map_kplanes(&mx, g.a, static_cast<uint64_t>(g.a_rows), static_cast<uint64_t>(g.K),
                        kXBox))
    return cudaErrorInvalidValue;
  SParams sp;
  sp.expert_offsets = g.expert_offsets;
  sp.out = static_cast<uint16_t*>(g.out);
  sp.E = g.E;
  sp.K = g.K;
  sp.w_rows_per_expert = g.b_rows_per_expert;
  sp.ldo = g.ldo;
  sp.out_rows = g.out_rows;
  sp.F = g.F;
  sp.interleave = g.interleave;
  sp.clamp = g.clamp;
  sp.status = g.status;
  sp.w_tiles = (g.epi == Epi::kSwiGLU) ? g.F / (kM / 2) : g.ldo / kM;
  // every expert may add one ragged token tile
  const long max_tiles =
      (static_cast<long>(ceil_div(g.a_rows, kNmaxS)) + std::min(g.E, g.a_rows)) * sp.w_tiles;
  const int grid = static_cast<int>(std::max(1L, std::min<long>(num_sms(), max_tiles)));
  if (g.epi == Epi::kSwiGLU)
    return launch_swap_impl<Epi::kSwiGLU, kNmaxS, kStagesS>(mw, mx, sp, grid, s);
  if (g.epi == Epi::kPlain)
    return launch_swap_impl<Epi::kPlain, kNmaxS, kStagesS>(mw, mx, sp, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
