// Persistent grouped GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One launch covers every expert: output tiles (expert, n-tile, m-tile) are
// enumerated from the device-side m-tile prefix, so ragged and empty experts
// need no host round trip and no padding of the permuted rows.  Per tile
//   D[128 x 256] = A[rows of expert e, K] * B[256 weight rows of e, K]^T
// accumulates in fp32 in TMEM; the epilogue applies either SwiGLU (GEMM1:
// gate and up halves of the tile -> 128 outputs, "Support GEMM + Swiglu fused
// MLP") or a plain bf16 store (GEMM2; the weighted top-k reduction of the
// "[SM90] Add W4A8 MegaMoE support" description runs in the combine step).
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: A tile 128x64 and two B boxes 128x64 per stage
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//   warps 2..5  epilogue: tcgen05.ld -> math -> global stores
// A 4-stage smem ring (full/empty mbarriers) feeds the MMA; two TMEM
// accumulators (2 x 256 columns) let the epilogue of tile i overlap the
// mainloop of tile i+1.  Every wait is bounded (ptx.cuh).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kABytes = kBM * kBK * 2;          // 16 KB
constexpr uint32_t kBBoxRows = 128;
constexpr uint32_t kBBytes = kBN * kBK * 2;          // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;  // 48 KB
constexpr uint32_t kTmemCols = 2 * kBN;              // two accumulators
constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN);
constexpr int kMaxE = 1024;
constexpr size_t kSmemBytes =
    1024 /*alignment slack*/ + kStages * kStageBytes + 256 /*barriers*/ +
    2 * (kMaxE + 1) * sizeof(int32_t) /*offsets + m-tile prefix*/;

struct KParams {
  const int32_t* expert_offsets;
  const int32_t* mtile_prefix;
  uint4* out;
  int E, K, n_tiles, b_rows_per_expert, ldo_vec, out_rows, F, interleave, ieff;
  float clamp;
  uint32_t* status;
};

struct Tile {
  int e, m, n;
};

// Largest expert e with mtp[e] <= q (the owner of global m-tile q).
__device__ __forceinline__ int find_expert(const int32_t* mtp, int E, int q) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mtp[mid] <= q) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ Tile decode_tile(int tile, const int32_t* mtp, int E, int n_tiles) {
  const int q = tile / n_tiles;
  Tile t;
  t.e = find_expert(mtp, E, q);
  const int mt = mtp[t.e + 1] - mtp[t.e];
  const int local = tile - mtp[t.e] * n_tiles;
  t.n = local / mt;  // m-tiles of one n-tile are adjacent: the weight tile is reused from L2
  t.m = local - t.n * mt;
  return t;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <Epi kEpi>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b, const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + kStages * kStageBytes + 256);
  int32_t* s_mtp = s_off + (p.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i <= p.E; i += kThreads) {
    s_off[i] = p.expert_offsets[i];
    s_mtp[i] = p.mtile_prefix[i];
  }
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
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
  }
  if (warp == 1) tmem_alloc<kTmemCols>(tmem_slot);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total_tiles = s_mtp[p.E] * p.n_tiles;
  const int num_kb = p.K / kBK;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_b = policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
        const Tile t = decode_tile(tile, s_mtp, p.E, p.n_tiles);
        const int a_row = s_off[t.e] + t.m * kBM;
        int b_row0, b_row1;
        const int b_base = t.e * p.b_rows_per_expert;
        if (kEpi == Epi::kSwiGLU) {
          const int f0 = t.n * (kBN / 2);
          if (p.interleave == 0) {
            b_row0 = f0;
            b_row1 = p.F + f0;
          } else if (p.ieff == 128) {  // interleave a multiple of 128
            b_row0 = (f0 / p.interleave) * 2 * p.interleave + f0 % p.interleave;
            b_row1 = b_row0 + p.interleave;
          } else {  // interleave 32 or 64: the 256 rows from 2*f0 hold 128 gate/up pairs
            b_row0 = 2 * f0;
            b_row1 = 2 * f0 + static_cast<int>(kBBoxRows);
          }
        } else {
          b_row0 = t.n * kBN;
          b_row1 = b_row0 + static_cast<int>(kBBoxRows);
        }
        b_row0 += b_base;
        b_row1 += b_base;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.status)) { *abort_flag = 1; break; }
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          const int kx = kb * kBK;
          tma_load_2d(sA + stage * kABytes, &map_a, kx, a_row, &full[stage], pol_a);
          uint8_t* b_dst = sB + stage * kBBytes;
          tma_load_2d(b_dst, &map_b, kx, b_row0, &full[stage], pol_b);
          tma_load_2d(b_dst + kBBytes / 2, &map_b, kx, b_row1, &full[stage], pol_b);
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      // Leave no bulk copy in flight: wait for the last fill of every stage.
      for (int i = 1; i <= kStages && i <= issued; ++i) {
        int s = stage - i;
        uint32_t ph = phase;
        if (s < 0) { s += kStages; ph ^= 1; }
        mbar_wait(&full[s], ph, p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t tph = (local >> 1) & 1;
        if (!mbar_wait(&tempty[buf], tph ^ 1, p.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kBN;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint64_t a_desc = sw128_kmajor_desc(smem_u32(sA + stage * kABytes));
          const uint64_t b_desc = sw128_kmajor_desc(smem_u32(sB + stage * kBBytes));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // +32 bytes along K inside the 128-byte swizzle atom = +2 in the
            // descriptor's 16-byte address units
            mma_bf16_ss(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, kIdesc, (kb | kk) != 0);
          }
          mma_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) { *abort_flag = 1; break; }
        mma_commit(&tfull[buf]);
      }
      // All MMAs of this CTA done before TMEM is released.
      mma_commit(drain);
      mbar_wait(drain, 0, p.status);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lanes this warp may access
    const int row_in_tile = quad * 32 + lane;
    int local = 0;
    for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x, ++local) {
      const int buf = local & 1;
      const uint32_t tph = (local >> 1) & 1;
      if (!mbar_wait(&tfull[buf], tph, p.status)) { *abort_flag = 1; break; }
      tc_fence_after();
      const Tile t = decode_tile(tile, s_mtp, p.E, p.n_tiles);
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
              packed[i / 2] = pack_bf16(silu_f(g0) * u0, silu_f(g1) * u1);
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
                  pack_bf16(__uint_as_float(a[8 * v + 0]), __uint_as_float(a[8 * v + 1])),
                  pack_bf16(__uint_as_float(a[8 * v + 2]), __uint_as_float(a[8 * v + 3])),
                  pack_bf16(__uint_as_float(a[8 * v + 4]), __uint_as_float(a[8 * v + 5])),
                  pack_bf16(__uint_as_float(a[8 * v + 6]), __uint_as_float(a[8 * v + 7])));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
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
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem_base);
  }
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2-D bf16 map over a row-major [rows, cols] matrix; box = 64 cols x box_rows
// rows with the 128-byte swizzle the MMA descriptors expect.
bool make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <Epi kEpi>
cudaError_t launch_impl(const GroupedGemmArgs& g, const CUtensorMap& ma, const CUtensorMap& mb,
                        const KParams& kp, int grid, cudaStream_t s) {
  (void)g;
  cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<kEpi>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
  if (err != cudaSuccess) return err;
  grouped_gemm_kernel<kEpi><<<grid, kThreads, kSmemBytes, s>>>(ma, mb, kp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm(const GroupedGemmArgs& g, cudaStream_t s) {
  if (g.a_rows == 0) return cudaSuccess;
  CUtensorMap ma, mb;
  if (!make_map_2d(&ma, g.a, static_cast<uint64_t>(g.a_rows), static_cast<uint64_t>(g.K), kBM))
    return cudaErrorInvalidValue;
  if (!make_map_2d(&mb, g.b, static_cast<uint64_t>(g.E) * g.b_rows_per_expert,
                   static_cast<uint64_t>(g.K), kBBoxRows))
    return cudaErrorInvalidValue;
  KParams kp;
  kp.expert_offsets = g.expert_offsets;
  kp.mtile_prefix = g.mtile_prefix;
  kp.out = static_cast<uint4*>(g.out);
  kp.E = g.E;
  kp.K = g.K;
  kp.n_tiles = g.n_tiles;
  kp.b_rows_per_expert = g.b_rows_per_expert;
  kp.ldo_vec = g.ldo / 8;
  kp.out_rows = g.out_rows;
  kp.F = g.F;
  kp.interleave = g.interleave;
  kp.ieff = (g.interleave == 0 || g.interleave % 128 == 0) ? 128 : g.interleave;
  kp.clamp = g.clamp;
  kp.status = g.status;
  // Upper bound on tiles: every expert may add one ragged m-tile.
  const long max_mtiles = ceil_div(g.a_rows, kBM) + std::min(g.E, g.a_rows);
  const long max_tiles = max_mtiles * g.n_tiles;
  const int grid = static_cast<int>(std::max(1L, std::min<long>(num_sms(), max_tiles)));
  if (g.epi == Epi::kSwiGLU) return launch_impl<Epi::kSwiGLU>(g, ma, mb, kp, grid, s);
  return launch_impl<Epi::kPlain>(g, ma, mb, kp, grid, s);
}

}  // namespace moe
