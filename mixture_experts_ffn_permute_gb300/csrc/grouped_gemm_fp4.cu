// Grouped GEMMs with NVFP4 weights (E2M1 codes + E4M3 scales per 16 values +
// an fp32 scale per expert tensor) and f16 activations, the low-precision
// form of the layer ("[SM90] Add W4A8 MegaMoE support", Usage: FP8
// activations with FP32 scales per 128 channels, weight scales E4M3 per 16).
//
// The weights stay 4-bit in HBM.  Per 64-deep K step a CTA loads, for its 256
// weight rows, 8 KB of packed codes (TMA) and 1 KB of scales (bulk copy from
// the layout moe_prepare_weights writes); eight transform warps turn them into
// f16 in the 128-byte-swizzled layout the MMA reads (E2M1 pair -> f16x2 with
// one cvt, times the E4M3 scale with one f16x2 multiply; both exact), and
// tcgen05.mma kind::f16 multiplies them with the f16 activation tile.  The
// expert's fp32 tensor scale is applied to the fp32 accumulator.
//
// Activations: the permute gather dequantises FP8 rows to f16 (x_perm);
// GEMM1's epilogue computes SwiGLU, re-quantises every 128-wide row block of
// h to E4M3 with scale amax/448 (as the split GEMM1 of the MegaMoE page does
// before GEMM2), and stores the dequantised values as f16 for GEMM2.
//
// Warp roles (448 threads, one CTA per SM):
//   warp 0       TMA producer (A tile, two packed-code boxes, two scale runs)
//   warp 1       TMEM allocator + single-thread MMA issuer
//   warps 2..5   epilogue
//   warps 6..13  transform (one weight row each per stage)
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "lowprec.cuh"
#include "ptx.cuh"

namespace moe {

bool make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);  // grouped_gemm.cu (2-byte elements, 128-byte swizzle)
bool make_map_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);  // grouped_gemm.cu (32-byte wide boxes, no swizzle)

namespace {

// Three rings: activations (TMA), packed weight codes + scales (TMA + bulk
// copy; deep, so HBM latency is covered), and the expanded f16 weight tiles
// the MMA reads (written by the transform warps).
constexpr int kStagesA = 4;
constexpr int kStagesR = 6;
constexpr int kStagesB = 3;
constexpr int kThreadsF = 448;
constexpr int kTransformThreads = 256;
constexpr uint32_t kABytesF = kBM * kBK * 2;       // 16 KB f16
constexpr uint32_t kB16Bytes = kBN * kBK * 2;      // 32 KB f16
constexpr uint32_t kRawBytes = kBN * kBK / 2;      // 8 KB packed E2M1
constexpr uint32_t kScBytes = kBN * kBK / 16;      // 1 KB E4M3 scales
constexpr uint32_t kTxRaw = kRawBytes + kScBytes;
constexpr uint32_t kTmemColsF = 2 * kBN;
// kind::f16 with f16 A and B (format 0), fp32 accumulator
constexpr uint32_t kIdescF16 = (1u << 4) | ((kBN >> 3) << 17) | ((kBM >> 4) << 24);
constexpr int kMaxEF = 1024;
constexpr size_t kRingBytes = kStagesA * kABytesF + kStagesB * kB16Bytes +
                              kStagesR * (kRawBytes + kScBytes);
// mbarriers of the three rings, 2 + 2 accumulator, drain; then the TMEM
// address word and the abort flag
static_assert((2 * (kStagesA + kStagesR + kStagesB) + 5) * 8 + 8 <= 256, "barrier area");
constexpr size_t kSmemBytesF = 1024 + kRingBytes + 256 + 2 * (kMaxEF + 1) * sizeof(int32_t);
static_assert(kSmemBytesF <= 232448, "shared memory budget");

struct FParams {
  const int32_t* expert_offsets;
  const int32_t* mtile_prefix;
  const uint8_t* scales;       // prepared: [E][N/128][K/64][128][4]
  const float* gscale;         // [E] fp32 tensor scale
  uint4* out;                  // f16 h (SwiGLU) or bf16 y (plain), rows of ldo elements
  int E, K, n_tiles, rows_per_expert, ldo_vec, F, interleave, ieff;
  float clamp;
  uint32_t* status;
};

struct FTile {
  int e, m, n;
};

__device__ __forceinline__ FTile decode_ftile(int tile, const int32_t* mtp, int E, int n_tiles) {
  const int q = tile / n_tiles;
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mtp[mid] <= q) lo = mid; else hi = mid - 1;
  }
  FTile t;
  t.e = lo;
  const int mt = mtp[lo + 1] - mtp[lo];
  const int local = tile - mtp[lo] * n_tiles;
  t.n = local / mt;
  t.m = local - t.n * mt;
  return t;
}

__device__ __forceinline__ float silu_f4(float z) { return z / (1.0f + expf(-z)); }

template <Epi kEpi>
__global__ void __launch_bounds__(kThreadsF, 1)
grouped_gemm_fp4_kernel(const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_q, const FParams p) {
  pdl_enter();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, kept as a shared-array pointer so that accesses
  // compile to shared-memory instructions
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = sA + kStagesA * kABytesF;
  uint8_t* sRaw = sB + kStagesB * kB16Bytes;
  uint8_t* sSc = sRaw + kStagesR * kRawBytes;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + kRingBytes);
  uint64_t* a_empty = a_full + kStagesA;
  uint64_t* r_full = a_empty + kStagesA;
  uint64_t* r_empty = r_full + kStagesR;
  uint64_t* b_full = r_empty + kStagesR;
  uint64_t* b_empty = b_full + kStagesB;
  uint64_t* afull = b_empty + kStagesB;  // accumulator ready
  uint64_t* aempty = afull + 2;          // accumulator drained
  uint64_t* drain = aempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + kRingBytes + 256);
  int32_t* s_mtp = s_off + (p.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i <= p.E; i += kThreadsF) {
    s_off[i] = p.expert_offsets[i];
    s_mtp[i] = p.mtile_prefix[i];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < kStagesR; ++s) {
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], kTransformThreads);
    }
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(&b_full[s], kTransformThreads);
      mbar_init(&b_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_q);
  }
  if (warp == 1) tmem_alloc<kTmemColsF>(tmem_slot);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = s_mtp[p.E] * p.n_tiles;
  const int num_kb = p.K / kBK;
  const int kblocks = p.K / kBK;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_b = policy_evict_normal();
      int sa = 0, sr = 0;
      uint32_t pa = 0, pr = 0;
      long issued = 0;
      for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
        const FTile t = decode_ftile(tile, s_mtp, p.E, p.n_tiles);
        const int a_row = s_off[t.e] + t.m * kBM;
        int r0, r1;  // first weight row of each 128-row half of the B tile
        if (kEpi == Epi::kSwiGLU) {
          const int f0 = t.n * (kBN / 2);
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
        } else {
          r0 = t.n * kBN;
          r1 = r0 + 128;
        }
        const long rb_base = static_cast<long>(t.e) * (p.rows_per_expert / 128);
        const int qrow0 = t.e * p.rows_per_expert + r0, qrow1 = t.e * p.rows_per_expert + r1;
        const uint8_t* sc0 = p.scales + ((rb_base + r0 / 128) * kblocks) * 512;
        const uint8_t* sc1 = p.scales + ((rb_base + r1 / 128) * kblocks) * 512;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&a_empty[sa], pa ^ 1, p.status)) { *abort_flag = 1; break; }
          mbar_arrive_expect_tx(&a_full[sa], kABytesF);
          tma_load_2d(sA + sa * kABytesF, &map_a, kb * kBK, a_row, &a_full[sa], pol_a);
          if (!mbar_wait(&r_empty[sr], pr ^ 1, p.status)) { *abort_flag = 1; break; }
          mbar_arrive_expect_tx(&r_full[sr], kTxRaw);
          uint8_t* raw = sRaw + sr * kRawBytes;
          tma_load_2d(raw, &map_q, kb * (kBK / 2), qrow0, &r_full[sr], pol_b);
          tma_load_2d(raw + kRawBytes / 2, &map_q, kb * (kBK / 2), qrow1, &r_full[sr], pol_b);
          uint8_t* sc = sSc + sr * kScBytes;
          bulk_load(sc, sc0 + static_cast<long>(kb) * 512, 512, &r_full[sr]);
          bulk_load(sc + 512, sc1 + static_cast<long>(kb) * 512, 512, &r_full[sr]);
          ++issued;
          if (++sa == kStagesA) { sa = 0; pa ^= 1; }
          if (++sr == kStagesR) { sr = 0; pr ^= 1; }
        }
      }
      // Leave no bulk copy in flight.
      for (int i = 1; i <= kStagesA && i <= issued; ++i) {
        int s = sa - i;
        uint32_t ph = pa;
        if (s < 0) { s += kStagesA; ph ^= 1; }
        mbar_wait(&a_full[s], ph, p.status);
      }
      for (int i = 1; i <= kStagesR && i <= issued; ++i) {
        int s = sr - i;
        uint32_t ph = pr;
        if (s < 0) { s += kStagesR; ph ^= 1; }
        mbar_wait(&r_full[s], ph, p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int sa = 0, sb = 0;
      uint32_t pa = 0, pb = 0;
      int local = 0;
      for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t tph = (local >> 1) & 1;
        if (!mbar_wait(&aempty[buf], tph ^ 1, p.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kBN;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&a_full[sa], pa, p.status) || !mbar_wait(&b_full[sb], pb, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = sw128_kmajor_desc(smem_u32(sA + sa * kABytesF));
          const uint64_t b_desc = sw128_kmajor_desc(smem_u32(sB + sb * kB16Bytes));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16_ss(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, kIdescF16, (kb | kk) != 0);
          mma_commit(&a_empty[sa]);
          mma_commit(&b_empty[sb]);
          if (++sa == kStagesA) { sa = 0; pa ^= 1; }
          if (++sb == kStagesB) { sb = 0; pb ^= 1; }
        }
        if (!ok) { *abort_flag = 1; break; }
        mma_commit(&afull[buf]);
      }
      mma_commit(drain);
      mbar_wait(drain, 0, p.status);
    }
  } else if (warp >= 6) {
    // ---------------------------------------------------------------- transform
    const int row = threadIdx.x - 6 * 32;  // weight row of the B tile, 0..255
    int sr = 0, sb = 0;
    uint32_t pr = 0, pb = 0;
    for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(&r_full[sr], pr, p.status) || !mbar_wait(&b_empty[sb], pb ^ 1, p.status)) {
          ok = false;
          break;
        }
        // The row's 32 code bytes as two 16-byte loads; rows with bit 2 set
        // take the halves in the other order, so the eight threads of each
        // load phase cover all 32 banks (rows 32 bytes apart otherwise put
        // threads t and t+4 on the same banks).
        const uint8_t* raw = sRaw + sr * kRawBytes + row * 32;
        const int h0 = (row & 4) ? 16 : 0;
        const uint4 qa = *reinterpret_cast<const uint4*>(raw + h0);
        const uint4 qb = *reinterpret_cast<const uint4*>(raw + (h0 ^ 16));
        const uint4 q0 = h0 ? qb : qa;
        const uint4 q1 = h0 ? qa : qb;
        const uint32_t sw = *reinterpret_cast<const uint32_t*>(sSc + sr * kScBytes + row * 4);
        mbar_arrive(&r_empty[sr]);  // codes and scales are in registers now
        const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        uint8_t* dst = sB + sb * kB16Bytes + row * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // 16 values per E4M3 scale
          const uint32_t sbyte = (sw >> (8 * j)) & 0xFFu;
          const uint32_t s2 = e4m3x2_to_f16x2(sbyte | (sbyte << 8));
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {  // two 16-byte chunks of 8 values
            const uint32_t w = qw[2 * j + h2];
            uint4 v;
            v.x = hmul2_u32(e2m1x2_to_f16x2(w & 0xFFu), s2);
            v.y = hmul2_u32(e2m1x2_to_f16x2((w >> 8) & 0xFFu), s2);
            v.z = hmul2_u32(e2m1x2_to_f16x2((w >> 16) & 0xFFu), s2);
            v.w = hmul2_u32(e2m1x2_to_f16x2(w >> 24), s2);
            const int c = 2 * j + h2;
            *reinterpret_cast<uint4*>(dst + ((c ^ (row & 7)) << 4)) = v;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&b_full[sb]);
        if (++sr == kStagesR) { sr = 0; pr ^= 1; }
        if (++sb == kStagesB) { sb = 0; pb ^= 1; }
      }
      if (!ok) { *abort_flag = 1; break; }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    int local = 0;
    for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x, ++local) {
      const int buf = local & 1;
      const uint32_t tph = (local >> 1) & 1;
      if (!mbar_wait(&afull[buf], tph, p.status)) { *abort_flag = 1; break; }
      tc_fence_after();
      const FTile t = decode_ftile(tile, s_mtp, p.E, p.n_tiles);
      const int seg_rows = s_off[t.e + 1] - s_off[t.e];
      const bool row_ok = t.m * kBM + row_in_tile < seg_rows;
      const long out_row = static_cast<long>(s_off[t.e]) + t.m * kBM + row_in_tile;
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * kBN;
      const float gs = __ldg(p.gscale + t.e);
      if (kEpi == Epi::kSwiGLU) {
        const bool clamp = p.clamp > 0.f && isfinite(p.clamp);
        // pass 1: amax of this row's 128 SwiGLU outputs
        float amax = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const int i0 = c * 32;
          const int gcol = (i0 / p.ieff) * 2 * p.ieff + i0 % p.ieff;
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(t_lane + gcol, g);
          tmem_ld_32x32b_x32(t_lane + gcol + p.ieff, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float gv = __uint_as_float(g[i]) * gs, uv = __uint_as_float(u[i]) * gs;
            if (clamp) {
              gv = fminf(gv, p.clamp);
              uv = fminf(fmaxf(uv, -p.clamp), p.clamp);
            }
            amax = fmaxf(amax, fabsf(silu_f4(gv) * uv));
          }
        }
        const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
        // pass 2: E4M3 code of h / sc, stored dequantised (code * sc) as f16
        uint4* dst = p.out + out_row * p.ldo_vec + (t.n * (kBN / 2)) / 8;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
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
              float hv[2];
#pragma unroll
              for (int d = 0; d < 2; ++d) {
                float gv = __uint_as_float(g[i + d]) * gs, uv = __uint_as_float(u[i + d]) * gs;
                if (clamp) {
                  gv = fminf(gv, p.clamp);
                  uv = fminf(fmaxf(uv, -p.clamp), p.clamp);
                }
                hv[d] = silu_f4(gv) * uv;
              }
              const uint32_t q2 = f32x2_to_e4m3x2(hv[0] / sc, hv[1] / sc);
              const uint32_t f2 = e4m3x2_to_f16x2(q2);
              const float2 qf = __half22float2(*reinterpret_cast<const __half2*>(&f2));
              const __half2 o = __floats2half2_rn(qf.x * sc, qf.y * sc);
              packed[i / 2] = *reinterpret_cast<const uint32_t*>(&o);
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
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(a[i]) * gs,
                                                             __uint_as_float(a[i + 1]) * gs);
              packed[i / 2] = *reinterpret_cast<const uint32_t*>(&b);
            }
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c * 4 + v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                          packed[4 * v + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&aempty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kTmemColsF>(tmem_base);
  }
}

template <Epi kEpi>
cudaError_t launch_fp4_impl(const CUtensorMap& ma, const CUtensorMap& mq, const FParams& fp,
                            int grid, cudaStream_t s) {
  cudaError_t err = cudaFuncSetAttribute(grouped_gemm_fp4_kernel<kEpi>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytesF));
  if (err != cudaSuccess) return err;
  return launch_kernel(grouped_gemm_fp4_kernel<kEpi>, dim3(static_cast<unsigned>(grid)),
                       dim3(kThreadsF), kSmemBytesF, s, 1, ma, mq, fp);
}

// scales [E][N][K/16] -> [E][N/128][K/64][128][4]
__global__ void __launch_bounds__(256)
prepare_scales_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int E, int N,
                      int K) {
  pdl_enter();
  const long groups = static_cast<long>(E) * N * (K / 64);
  const int kblocks = K / 64;
  for (long g = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
       g += static_cast<long>(gridDim.x) * blockDim.x) {
    const int kb = static_cast<int>(g % kblocks);
    const long er = g / kblocks;           // e * N + n
    const int n = static_cast<int>(er % N);
    const long e = er / N;
    const uint32_t v = *reinterpret_cast<const uint32_t*>(src + er * (K / 16) + kb * 4);
    const long rb = e * (N / 128) + n / 128;
    *reinterpret_cast<uint32_t*>(dst + ((rb * kblocks + kb) * 128 + (n % 128)) * 4) = v;
  }
}

// MXFP4 scales -> the prepared E4M3 layout above, exactly: one CTA per (expert,
// tensor).  With e_max the largest E8M0 byte of the expert's tensor, the
// expert scale is g = 2^k, k = (e_max - 127) - 8, and each block's scale
// 2^(e - 127) becomes the E4M3 power of two 2^(e - 127 - k) in [2^-9, 2^8]
// (every power of two there is an E4M3 code), written for both 16-value
// halves of its 32-value block.  A block more than 17 binades below e_max
// gets scale 0 (its values are below 2^-17 of the expert's largest block).
// The byte 255 (not a number) is out of contract and treated as 0.
__device__ __forceinline__ uint32_t e4m3_power_of_two(int j) {  // j in [-9, 8]
  return j >= -6 ? static_cast<uint32_t>(j + 7) << 3 : 1u << (j + 9);
}

__global__ void __launch_bounds__(512)
prepare_mxfp4_scales_kernel(const uint8_t* __restrict__ s1, const uint8_t* __restrict__ s2,
                            uint8_t* __restrict__ dst1, uint8_t* __restrict__ dst2, int F, int H,
                            float* __restrict__ g1, float* __restrict__ g2) {
  pdl_enter();
  __shared__ int s_max[16];
  const int e = blockIdx.x;
  const bool second = blockIdx.y == 1;
  const int N = second ? H : 2 * F, K = second ? F : H;
  const uint8_t* src = (second ? s2 : s1) + static_cast<long>(e) * N * (K / 32);
  uint8_t* dst = second ? dst2 : dst1;
  const long nbytes = static_cast<long>(N) * (K / 32);
  int m = 0;
  for (long i = threadIdx.x; i < nbytes; i += blockDim.x) {
    const int b = src[i];
    if (b != 255) m = max(m, b);
  }
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
  __syncthreads();
  int emax = 0;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) emax = max(emax, s_max[w]);
  const int k = min(127, max(-126, emax - 127 - 8));
  if (threadIdx.x == 0) (second ? g2 : g1)[e] = ldexpf(1.0f, k);
  const int kblocks = K / 64;
  for (long i = threadIdx.x; i < static_cast<long>(N) * kblocks; i += blockDim.x) {
    const int n = static_cast<int>(i / kblocks), kb = static_cast<int>(i % kblocks);
    uint32_t word = 0;
    for (int h = 0; h < 2; ++h) {
      const int b = src[static_cast<long>(n) * (K / 32) + 2 * kb + h];
      const int j = b - 127 - k;
      const uint32_t c = (b == 255 || j < -9) ? 0u : e4m3_power_of_two(j);
      word |= (c | (c << 8)) << (16 * h);
    }
    const long rb = static_cast<long>(e) * (N / 128) + n / 128;
    *reinterpret_cast<uint32_t*>(dst + ((rb * kblocks + kb) * 128 + (n % 128)) * 4) = word;
  }
}

// x_perm[r][c] = f16(E4M3(xq[t][c]) * xs[t][c / 128]), t = permuted_token[r]
// (zero rows for -1); 8 values per thread.
__global__ void __launch_bounds__(256)
gather_dequant_fp8_kernel(const uint8_t* __restrict__ xq, const float* __restrict__ xs,
                          const int32_t* __restrict__ permuted_token, int R, int H,
                          uint4* __restrict__ x_perm) {
  pdl_enter();
  const int vecs = H / 8;
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const int t = permuted_token ? permuted_token[r] : r;
    uint4* dst = x_perm + static_cast<size_t>(r) * vecs;
    for (int v = threadIdx.x; v < vecs; v += blockDim.x) {
      if (t < 0) {
        dst[v] = make_uint4(0, 0, 0, 0);
        continue;
      }
      const uint2 q = __ldg(reinterpret_cast<const uint2*>(xq + static_cast<size_t>(t) * H) + v);
      const float s = __ldg(xs + static_cast<size_t>(t) * (H / 128) + (v * 8) / 128);
      const uint32_t w[4] = {q.x & 0xFFFFu, q.x >> 16, q.y & 0xFFFFu, q.y >> 16};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t f2 = e4m3x2_to_f16x2(w[i]);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&f2));
        const __half2 hv = __floats2half2_rn(f.x * s, f.y * s);
        o[i] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

cudaError_t launch_grouped_gemm_fp4(const GroupedGemmArgs& g, const uint8_t* scales,
                                    const float* gscale, cudaStream_t s) {
  if (g.a_rows == 0) return cudaSuccess;
  if (g.E > kMaxEF) return cudaErrorInvalidValue;
  CUtensorMap ma, mq;
  if (!make_map_2d(&ma, g.a, static_cast<uint64_t>(g.a_rows), static_cast<uint64_t>(g.K), kBM))
    return cudaErrorInvalidValue;
  if (!make_map_u8(&mq, g.b, static_cast<uint64_t>(g.E) * g.b_rows_per_expert,
                   static_cast<uint64_t>(g.K) / 2, 128))
    return cudaErrorInvalidValue;
  FParams fp;
  fp.expert_offsets = g.expert_offsets;
  fp.mtile_prefix = g.mtile_prefix;
  fp.scales = scales;
  fp.gscale = gscale;
  fp.out = static_cast<uint4*>(g.out);
  fp.E = g.E;
  fp.K = g.K;
  fp.n_tiles = g.n_tiles;
  fp.rows_per_expert = g.b_rows_per_expert;
  fp.ldo_vec = g.ldo / 8;
  fp.F = g.F;
  fp.interleave = g.interleave;
  fp.ieff = (g.interleave == 0 || g.interleave % 128 == 0) ? 128 : g.interleave;
  fp.clamp = g.clamp;
  fp.status = g.status;
  const long max_mtiles = ceil_div(g.a_rows, kBM) + std::min(g.E, g.a_rows);
  const long max_tiles = max_mtiles * g.n_tiles;
  const int grid = static_cast<int>(std::max(1L, std::min<long>(num_sms(), max_tiles)));
  if (g.epi == Epi::kSwiGLU) return launch_fp4_impl<Epi::kSwiGLU>(ma, mq, fp, grid, s);
  if (g.epi == Epi::kPlain) return launch_fp4_impl<Epi::kPlain>(ma, mq, fp, grid, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prepare_scales(const uint8_t* src, uint8_t* dst, int E, int N, int K,
                                  cudaStream_t s) {
  const long groups = static_cast<long>(E) * N * (K / 64);
  if (groups == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<long>((groups + 255) / 256, num_sms() * 16L));
  return launch_kernel(prepare_scales_kernel, dim3(blocks), dim3(256), 0, s, 1, src, dst, E, N, K);
}

cudaError_t launch_prepare_mxfp4_scales(const uint8_t* s1, const uint8_t* s2, uint8_t* dst1,
                                        uint8_t* dst2, int E, int F, int H, float* g1, float* g2,
                                        cudaStream_t s) {
  if (E == 0) return cudaSuccess;
  return launch_kernel(prepare_mxfp4_scales_kernel, dim3(E, 2), dim3(512), 0, s, 1, s1, s2, dst1,
                       dst2, F, H, g1, g2);
}

cudaError_t launch_gather_dequant_fp8(const uint8_t* xq, const float* xs,
                                      const int32_t* permuted_token, int R, int H, void* x_perm,
                                      cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const int blocks = std::min(R, num_sms() * 8);
  return launch_kernel(gather_dequant_fp8_kernel, dim3(blocks), dim3(256), 0, s, 1, xq, xs,
                       permuted_token, R, H, static_cast<uint4*>(x_perm));
}

}  // namespace moe
