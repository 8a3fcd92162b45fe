// Persistent grouped GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One launch covers every expert: output tiles (expert, n-tile, m-tile) are
// enumerated from the device-side m-tile prefix, so ragged and empty experts
// need no host round trip and no padding of the permuted rows.  Per tile
//   D[128 x 256] = A[rows of expert e, K] * B[256 weight rows of e, K]^T
// accumulates in fp32 in TMEM.  Epilogues:
//   kSwiGLU   GEMM1: gate and up halves of the tile -> 128 SwiGLU outputs
//             ("Support GEMM + Swiglu fused MLP")
//   kPlain    GEMM2: unweighted bf16 rows y (the stand-alone MLP entry point)
//   kCombine  GEMM2 fused with the weighted top-k reduction of the
//             "[SM90] Add W4A8 MegaMoE support" description: each row's
//             w * y goes to a bf16 partial buffer, a per-(token, n-tile)
//             counter counts arrivals, and the last arriving route sums the
//             token's partials in slot order j = 0..k-1 (fixed order, so the
//             result does not depend on which route finished last).
// With kGatherA the A rows are gathered straight from the token matrix x by
// permuted_token with TMA tile::gather4 (4 rows per copy), so the permuted
// copy of x never exists in HBM.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: A tile 128x64 (one 128-row box, or 32 four-row
//               gathers issued by the 32 lanes) and two B boxes 128x64 per stage
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
// mbarriers: full/empty per stage, 2 + 2 accumulator, drain; then the TMEM
// address word and the abort flag
static_assert((2 * kStages + 5) * 8 + 8 <= 256, "barrier area");
constexpr size_t kSmemBytes =
    1024 /*alignment slack*/ + kStages * kStageBytes + 256 /*barriers*/ +
    2 * (kMaxE + 1) * sizeof(int32_t) /*offsets, m-tile prefix*/;

struct KParams {
  const int32_t* expert_offsets;
  const int32_t* mtile_prefix;
  uint4* out;
  int E, K, n_tiles, b_rows_per_expert, ldo_vec, out_rows, F, interleave, ieff;
  float clamp;
  uint32_t* status;
  // gathered A rows / fused combine
  const int32_t* permuted_token;  // [R] token of each permuted row
  const int32_t* row_id_map;      // [T, k]
  const float* topk_w;            // [T, k]
  int32_t* counters;              // [T, n_tiles], zero at launch
  uint4* partials;                // [R, ldo] bf16 weighted rows
  int k;
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

static_assert(kBN / 8 == 32, "the combine reduction maps one 16-byte vector to each lane");

__device__ __forceinline__ void add_bf16x8(const uint4& v, float (&acc)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] += f.x;
    acc[2 * i + 1] += f.y;
  }
}

template <Epi kEpi, bool kGatherA>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b, const KParams p) {
  pdl_enter();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, kept as a shared-array pointer so that accesses
  // compile to shared-memory instructions
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
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

  // tile list: (expert, n-tile, m-tile)
  const int total_tiles = s_mtp[p.E] * p.n_tiles;
  const int tile0 = static_cast<int>(blockIdx.x);
  const int tstride = static_cast<int>(gridDim.x);
  auto tile_at = [&](int tile) { return decode_tile(tile, s_mtp, p.E, p.n_tiles); };
  const int num_kb = p.K / kBK;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // Lane 0 drives the ring (waits, expect-tx, B boxes, plain A box); with a
    // gathered A every lane also issues one 4-row gather per stage: rows
    // 4*lane .. 4*lane+3 of the tile.
    const uint64_t pol_a = policy_evict_last();
    const uint64_t pol_b = policy_evict_normal();
    int stage = 0;
    uint32_t phase = 0;
    long issued = 0;
    bool go = true;
    for (int tile = tile0; tile < total_tiles && go; tile += tstride) {
      go = __shfl_sync(0xffffffffu, lane == 0 ? (*abort_flag == 0) : 0, 0) != 0;
      if (!go) break;
      const Tile t = tile_at(tile);
      const int seg_start = s_off[t.e];
      const int seg_rows = s_off[t.e + 1] - seg_start;
      const int a_row = seg_start + t.m * kBM;
      int g0 = 0, g1 = 0, g2 = 0, g3 = 0;
      if (kGatherA) {
        // token rows of this lane's four tile rows; rows past the segment
        // read token 0 (their results are never stored)
        const int base = t.m * kBM + 4 * lane;
        int tk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = base + i;
          const int v = rr < seg_rows ? __ldg(p.permuted_token + seg_start + rr) : 0;
          tk[i] = v < 0 ? 0 : v;
        }
        g0 = tk[0]; g1 = tk[1]; g2 = tk[2]; g3 = tk[3];
      }
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
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(&empty[stage], phase ^ 1, p.status) ? 1 : 0;
          if (ok) mbar_arrive_expect_tx(&full[stage], kStageBytes);
          else *abort_flag = 1;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) { go = false; break; }
        const int kx = kb * kBK;
        if (kGatherA)
          tma_gather4(sA + stage * kABytes + lane * 512, &map_a, kx, g0, g1, g2, g3, &full[stage],
                      pol_a);
        if (lane == 0) {
          if (!kGatherA) tma_load_2d(sA + stage * kABytes, &map_a, kx, a_row, &full[stage], pol_a);
          uint8_t* b_dst = sB + stage * kBBytes;
          tma_load_2d(b_dst, &map_b, kx, b_row0, &full[stage], pol_b);
          tma_load_2d(b_dst + kBBytes / 2, &map_b, kx, b_row1, &full[stage], pol_b);
        }
        ++issued;
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
    }
    // Leave no bulk copy in flight: wait for the last fill of every stage.
    if (lane == 0) {
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
    for (int tile = tile0; tile < total_tiles && !*abort_flag; tile += tstride, ++local) {
      const int buf = local & 1;
      const uint32_t tph = (local >> 1) & 1;
      if (!mbar_wait(&tfull[buf], tph, p.status)) { *abort_flag = 1; break; }
      tc_fence_after();
      const Tile t = tile_at(tile);
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
      } else if (kEpi == Epi::kPlain) {
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
      } else {
        // kCombine: partial = w * y (bf16) for this route; last arrival sums.
        int tok = 0, nvalid = 0;
        float w = 0.f;
        if (row_ok) {
          tok = __ldg(p.permuted_token + out_row);
          const int32_t* rm = p.row_id_map + static_cast<long>(tok) * p.k;
          int j = 0;
          for (int jj = 0; jj < p.k; ++jj) {
            const int v = __ldg(rm + jj);
            nvalid += v >= 0;
            if (v == out_row) j = jj;
          }
          w = __ldg(p.topk_w + static_cast<long>(tok) * p.k + j);
        }
        const int col_vec = (t.n * kBN) / 8;
        uint4* dst = (nvalid == 1 ? p.out + static_cast<long>(tok) * p.ldo_vec
                                  : p.partials + out_row * p.ldo_vec) + col_vec;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t a[32];
          tmem_ld_32x32b_x32(t_lane + c * 32, a);
          tmem_ld_wait();
          if (row_ok) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c * 4 + v] = make_uint4(
                  pack_bf16(w * __uint_as_float(a[8 * v + 0]), w * __uint_as_float(a[8 * v + 1])),
                  pack_bf16(w * __uint_as_float(a[8 * v + 2]), w * __uint_as_float(a[8 * v + 3])),
                  pack_bf16(w * __uint_as_float(a[8 * v + 4]), w * __uint_as_float(a[8 * v + 5])),
                  pack_bf16(w * __uint_as_float(a[8 * v + 6]), w * __uint_as_float(a[8 * v + 7])));
          }
        }
        // The accumulator is no longer needed: release it before the reduction.
        tc_fence_before();
        mbar_arrive(&tempty[buf]);
        // Arrival count per (token, n-tile); the last arriving route's warp
        // reduces that token's partials, one 16-byte column vector per lane.
        bool last = false;
        if (row_ok && nvalid > 1) {
          __threadfence();
          const int prev = atomicAdd(p.counters + static_cast<long>(tok) * p.n_tiles + t.n, 1);
          last = prev == nvalid - 1;
        }
        __threadfence();
        uint32_t todo = __ballot_sync(0xffffffffu, last);
        __syncwarp();
        while (todo) {
          const int src = __ffs(todo) - 1;
          todo &= todo - 1;
          const int tk = __shfl_sync(0xffffffffu, tok, src);
          const int32_t* rm = p.row_id_map + static_cast<long>(tk) * p.k;
          float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          for (int jj = 0; jj < p.k; ++jj) {  // slot order: deterministic
            const int r = __ldg(rm + jj);
            if (r < 0) continue;
            add_bf16x8(__ldcg(p.partials + static_cast<long>(r) * p.ldo_vec + col_vec + lane), acc);
          }
          p.out[static_cast<long>(tk) * p.ldo_vec + col_vec + lane] =
              make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]),
                         pack_bf16(acc[4], acc[5]), pack_bf16(acc[6], acc[7]));
        }
        continue;  // tempty already released
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

template <Epi kEpi, bool kGatherA>
cudaError_t launch_impl(const CUtensorMap& ma, const CUtensorMap& mb, const KParams& kp,
                        int grid, cudaStream_t s) {
  auto kern = grouped_gemm_kernel<kEpi, kGatherA>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemBytes, s,
                       1, ma, mb, kp);
}

}  // namespace

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
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


// bf16 [rows, cols] viewed as 64-column planes {64, rows, cols / 64}: a box
// of box_rows rows x 2 planes (two 64-deep K steps) lands as two consecutive
// 128-byte-swizzled K-major tiles, and every row of it is one 256-byte
// segment of global memory.
bool make_map_kplanes(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc || cols % 128 != 0) return false;
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same planes for two 64-row blocks `gap` rows apart (a GLU's gate and up
// rows): {64, rows - gap, 2, cols / 64} with boxes of 64 rows x both blocks
// x 2 planes, so each plane holds the 64 + 64 rows as one 128-row tile.
bool make_map_kplanes_pair(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint64_t gap) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc || cols % 128 != 0 || gap == 0 || gap >= rows) return false;
  cuuint64_t dims[4] = {64, rows - gap, 2, cols / 64};
  cuuint64_t strides[3] = {cols * 2, gap * cols * 2, 128};
  cuuint32_t box[4] = {64, 64, 2, 2};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [rows, cols] map with box_cols x box_rows boxes and no swizzle (tiles
// staged row-major in shared memory, e.g. for bulk-tensor stores).
bool make_map_2d_plain(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows, cols] map with 32-column x box_rows boxes (128 bytes wide) and
// the 128-byte swizzle (fp32 tiles staged in shared memory for bulk stores).
bool make_map_2d_f32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {32u, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// uint8 [rows, cols] map with 32-byte x 128-row boxes and no swizzle (packed
// E2M1 weight codes, two per byte).
bool make_map_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_grouped_gemm(const GroupedGemmArgs& g, cudaStream_t s) {
  if (g.a_rows == 0) return cudaSuccess;
  CUtensorMap ma, mb;
  const bool gather = g.permuted_token != nullptr && g.epi == Epi::kSwiGLU;
  // gathered A: a map over the token matrix x [x_rows, K] with one-row boxes
  if (!make_map_2d(&ma, g.a, static_cast<uint64_t>(gather ? g.x_rows : g.a_rows),
                   static_cast<uint64_t>(g.K), gather ? 1u : static_cast<uint32_t>(kBM)))
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
  kp.permuted_token = g.permuted_token;
  kp.row_id_map = g.row_id_map;
  kp.topk_w = g.topk_w;
  kp.counters = g.counters;
  kp.partials = static_cast<uint4*>(g.partials);
  kp.k = g.k;
  // Upper bound on tiles: every expert may add one ragged m-tile.
  const long max_mtiles = ceil_div(g.a_rows, kBM) + std::min(g.E, g.a_rows);
  const long max_tiles = max_mtiles * g.n_tiles;
  const int grid = static_cast<int>(std::max(1L, std::min<long>(num_sms(), max_tiles)));
  switch (g.epi) {
    case Epi::kSwiGLU:
      return gather ? launch_impl<Epi::kSwiGLU, true>(ma, mb, kp, grid, s)
                    : launch_impl<Epi::kSwiGLU, false>(ma, mb, kp, grid, s);
    case Epi::kPlain:
      return launch_impl<Epi::kPlain, false>(ma, mb, kp, grid, s);
    case Epi::kCombine:
      return launch_impl<Epi::kCombine, false>(ma, mb, kp, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
