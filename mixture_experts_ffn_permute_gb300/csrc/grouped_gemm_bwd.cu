// Grouped GEMMs of the layer's backward on the sm_103a tensor cores (tcgen05
// + TMEM + TMA).  The backward needs every operand in the layout the forward
// stored it in, so the tiles are read as the MMA wants them instead of being
// transposed in memory first:
//
//   recomputed forward (ragged M)
//     a   = Xp W1_e^T A = Xp [R, H], B = W1_e [2F, H], both K-major; the
//                     pre-activations are kept in fp32
//   data gradients (ragged M: the permuted rows of each expert)
//     dH  = dY W2_e   A = dY [R, H] K-major; B = W2_e [H, F] read MN-major
//                     epilogue: SwiGLU backward -- reads the fp32
//                     pre-activations, writes dA (bf16), h_w = w h, and the
//                     per-route partial <dh, h> of the router gradient
//     dXp = dA W1_e   A = dA [R, 2F] K-major; B = W1_e [2F, H] read MN-major
//   weight gradients (ragged K: the contraction runs over an expert's rows)
//     dW2_e = dY_e^T h_w_e   A = dY [R, H], B = h_w [R, F], both read MN-major
//     dW1_e = dA_e^T Xp_e    A = dA [R, 2F], B = Xp [R, H], both read MN-major
//
// An MN-major operand tile comes from a row-major [K rows, MN cols] matrix as
// TMA boxes of 64 columns x 64 rows with the 128-byte swizzle: 128-byte rows
// hold 64 consecutive MN elements of one k, 8-row groups are 1024 bytes apart
// (the descriptor's stride offset) and the next 64 MN columns sit one box
// (8 KB) further (its leading offset).  One K=16 MMA step is 16 rows = 2 KB.
//
// Warp roles (192 threads, one CTA per SM, persistent over the tile list):
//   warp 0      TMA producer.  1-CTA tiles (weight gradients): a ring of 48 KB
//               stages (A 16 KB + B 32 KB), 4 deep, 3 for the weight gradients
//               of small experts; 2-CTA pairs (data gradients): 6 stages of
//               32 KB per CTA (A 16 KB + half of B)
//   warp 1      TMEM allocation + MMA issue (lane 0; the leader's for a pair);
//               in the weight-gradient kernel the whole warp first zeroes the
//               rows of a ragged last K step that belong to the next expert
//   warps 2..5  epilogue (TMEM lanes 32*(warp%4) ..), two 256-column
//               accumulators so a tile's epilogue overlaps the next mainloop;
//               weight gradients and fp32 pre-activations leave through
//               swizzled shared-memory staging and bulk-tensor stores
// Every wait is bounded (ptx.cuh).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>

#include "../../include/moe_ffn.h"
#include "internal.h"
#include "pair_tiles.cuh"
#include "ptx.cuh"

namespace moe {

// 2-D bf16 tensor map, boxes of 64 columns x box_rows rows, 128-byte swizzle
// (grouped_gemm.cu).
bool make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);
bool make_map_2d_f32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows);

namespace {

// pipeline depth: 2-CTA pairs (32 KB per CTA and stage) keep 6 stages; 1-CTA
// tiles (48 KB) 4, the weight gradients of small experts trade one for output
// staging
template <int kMode, bool kPair>
__host__ __device__ constexpr int stages_of() { return kPair ? 6 : (kMode == 2 ? 3 : 4); }
// threads: producer warp, MMA warp, then the epilogue warps -- one per TMEM
// lane quadrant, kBwdSwiGLUSplit per quadrant for the SwiGLU backward
template <int kMode>
__host__ __device__ constexpr int epi_warps_of() { return kMode == 1 ? 4 * kBwdSwiGLUSplit : 4; }
template <int kMode>
__host__ __device__ constexpr int threads_of() { return 64 + 32 * epi_warps_of<kMode>(); }
constexpr uint32_t kABytesB = kBM * kBK * 2;             // 16 KB
constexpr uint32_t kBBytesB = kBN * kBK * 2;             // 32 KB
// B bytes per stage in one CTA: the whole 256-column tile, or a pair's half
__host__ __device__ constexpr uint32_t b_stage_bytes(bool pair) {
  return pair ? kBBytesB / 2 : kBBytesB;
}
constexpr uint32_t kBoxBytes = 64 * 64 * 2;              // one MN-major box, 8 KB
constexpr uint32_t kStepBytesMN = 16 * 128;              // one K=16 step of an MN-major tile
constexpr uint32_t kTmemColsB = 2 * kBN;
constexpr int kMaxEB = MOE_MAX_EXPERTS;
// weight-gradient output staging, in 64-column x 32-row boxes with the
// 128-byte swizzle: experts with few rows (short K loops, mode 2) stage 128
// columns per step in two buffers per epilogue warp (64 KB, 3 pipeline
// stages); experts with many rows (mode 4) keep 4 pipeline stages and stage 64
// columns per step in one buffer per warp (16 KB)
constexpr uint32_t kOutBoxBytes = 32 * 128;  // 32 rows x 64 bf16
template <int kMode>
__host__ __device__ constexpr int out_step_cols() { return kMode == 2 ? 128 : 64; }
template <int kMode>
__host__ __device__ constexpr int out_buffers() { return kMode == 2 ? 2 : 1; }
template <int kMode>
__host__ __device__ constexpr uint32_t out_stage_bytes() {
  return (kMode == 2 || kMode == 4)
             ? 4 * out_buffers<kMode>() * (out_step_cols<kMode>() / 64) * kOutBoxBytes
         : kMode == 3 ? 4 * kOutBoxBytes  // fp32 pre-activations: 32 x 32 per warp
                      : 0;
}
template <int kMode, bool kPair>
constexpr size_t smem_bytes_of() {
  return 1024 + stages_of<kMode, kPair>() * (kABytesB + b_stage_bytes(kPair)) +
         out_stage_bytes<kMode>() + 256 + 3 * (kMaxEB + 1) * sizeof(int32_t);
}
static_assert((2 * 6 + 5) * 8 + 8 <= 256, "barrier area");
static_assert(smem_bytes_of<0, false>() <= 232448 && smem_bytes_of<2, false>() <= 232448 &&
                  smem_bytes_of<3, false>() <= 232448 && smem_bytes_of<4, false>() <= 232448 &&
                  smem_bytes_of<0, true>() <= 232448 && smem_bytes_of<1, true>() <= 232448 &&
                  smem_bytes_of<3, true>() <= 232448,
              "shared memory budget");

enum class BwdMode : int {
  kDataPlain = 0,
  kDataSwiGLU = 1,
  kWeight = 2,      // weight gradients, experts with few rows
  kPreact = 3,
  kWeightLong = 4   // weight gradients, experts with many rows
};

struct BwdParams {
  const int32_t* expert_offsets;  // [E + 1]
  const int32_t* mtile_prefix;    // [E + 1] (data gradients)
  int E;
  int K;        // data gradients: contraction length (rows of B per expert)
  int N;        // output columns
  int n_tiles;  // ceil(N / 256)
  int M;        // weight gradients: output rows per expert
  int m_tiles;  // M / 128
  int m_outer;  // weight gradients: 1 = the n-tiles of one m-tile adjacent
  uint4* out;   // data: [R, N] bf16; weight: [E, M, N] bf16; pre-activations [R, N] fp32
  int ldo_vec;  // N / 8 (bf16) or N / 4 (fp32)
  // SwiGLU backward
  const float4* act;     // [R, 2F] fp32 pre-activations
  int act_vec;           // 2F / 4
  uint4* dact;           // [R, 2F] bf16 out: dA
  int dact_vec;          // 2F / 8
  uint4* hw;             // [R, F] bf16: w * h
  float* dw_part;        // [R, n_tiles]: partial <dh, h>
  const float* w_perm;   // [R] routing weight of each permuted row
  int F, interleave;
  float clamp;           // > 0: clamp value, else none
  uint32_t* status;
};

struct BTile {
  int e, m, n;
};

__device__ __forceinline__ int find_expert_b(const int32_t* mtp, int E, int q) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mtp[mid] <= q) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <BwdMode kMode>
__device__ __forceinline__ BTile decode_btile(int tile, const int32_t* mtp, const BwdParams& p) {
  BTile t;
  if (kMode == BwdMode::kWeight || kMode == BwdMode::kWeightLong) {
    const int per = p.m_tiles * p.n_tiles;
    t.e = tile / per;
    const int local = tile - t.e * per;
    // the larger operand's column blocks outermost, so each is streamed once
    // while the smaller one stays in L2
    if (p.m_outer) {
      t.m = local / p.n_tiles;
      t.n = local - t.m * p.n_tiles;
    } else {
      t.n = local / p.m_tiles;
      t.m = local - t.n * p.m_tiles;
    }
  } else {
    const int q = tile / p.n_tiles;
    t.e = find_expert_b(mtp, p.E, q);
    const int mt = mtp[t.e + 1] - mtp[t.e];
    const int local = tile - mtp[t.e] * p.n_tiles;
    t.n = local / mt;  // m-tiles of one n-tile adjacent: the weight tile is reused from L2
    t.m = local - t.n * mt;
  }
  return t;
}

// Shared-memory descriptor of an MN-major tile stored as 64-column boxes with
// the 128-byte swizzle (see the file comment): leading offset = one box,
// stride offset = 8 rows of 128 bytes.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(kBoxBytes >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor with the MN-major (transposed) operand bits.
__host__ __device__ constexpr uint32_t idesc_bwd(bool a_mn, bool b_mn) {
  return idesc_bf16_f32(kBM, kBN) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16);
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Column of W1 (and of the pre-activation row) holding gate (resp. up) output
// f: interleave 0 -> [gate | up] halves; I -> blocks of I gate then I up.
__device__ __forceinline__ int gate_col(int f, int F, int I) {
  return I == 0 ? f : (f / I) * 2 * I + f % I;
}
__device__ __forceinline__ int up_col(int f, int F, int I) {
  return I == 0 ? F + f : (f / I) * 2 * I + f % I + I;
}

// kPair (data gradients only): 2-CTA clusters.  CTA r of a pair holds the 128
// token rows of m-tile 2*mp + r and the 128 columns 128*r .. 128*r+127 of the
// 256-column B tile; both load into their own shared memory and complete on
// the leader's full barrier (.cta_group::2 loads); the leader (rank 0) issues
// tcgen05.mma.cta_group::2 (M = 256 across the pair) and its commits arrive
// on both CTAs' empty / TMEM-full barriers; every epilogue thread of the pair
// arrives on the leader's TMEM-empty barrier.  Each SM then loads half the B
// bytes per 256 x 256 MMA, which shared-memory bandwidth rewards.
template <BwdMode kMode, bool kPair>
__global__ void __launch_bounds__(threads_of<static_cast<int>(kMode)>(), 1)
grouped_gemm_bwd_kernel(const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_b,
                        const __grid_constant__ CUtensorMap map_out, const BwdParams p) {
  pdl_enter();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  constexpr int kStagesB = stages_of<static_cast<int>(kMode), kPair>();
  constexpr uint32_t kOutStageBytes = out_stage_bytes<static_cast<int>(kMode)>();
  constexpr uint32_t kBStage = b_stage_bytes(kPair);     // B bytes per stage, this CTA
  constexpr uint32_t kStageBytes = kABytesB + kBStage;   // bytes per stage, this CTA
  uint8_t* sB = smem + kStagesB * kABytesB;
  uint8_t* s_out = sB + kStagesB * kBStage;  // output staging (1024-aligned)
  uint64_t* full = reinterpret_cast<uint64_t*>(s_out + kOutStageBytes);
  uint64_t* empty = full + kStagesB;
  uint64_t* tfull = empty + kStagesB;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_off =
      reinterpret_cast<int32_t*>(smem + kStagesB * kStageBytes + kOutStageBytes + 256);
  int32_t* s_mtp = s_off + (p.E + 1);
  int32_t* s_ptp = s_mtp + (p.E + 1);  // kPair: prefix of ceil(m-tiles / 2)

  constexpr bool kWeightGrad = kMode == BwdMode::kWeight || kMode == BwdMode::kWeightLong;
  constexpr bool kBKMajor = kMode == BwdMode::kPreact;  // B = weight rows, K-major
  static_assert(!(kPair && kWeightGrad), "pairs serve the data gradients");
  constexpr uint32_t kIdescB =
      kPair ? idesc_bf16_f32(2 * kBM, kBN) | (static_cast<uint32_t>(!kBKMajor) << 16)
            : idesc_bwd(kWeightGrad, !kBKMajor);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0;
  const bool leader = rank == 0;
  constexpr int kThreadsB = threads_of<static_cast<int>(kMode)>();
  constexpr int kEpiWarps = epi_warps_of<static_cast<int>(kMode)>();
  for (int i = threadIdx.x; i <= p.E; i += kThreadsB) {
    s_off[i] = p.expert_offsets[i];
    s_mtp[i] = kWeightGrad ? 0 : p.mtile_prefix[i];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], (kPair ? 2 : 1) * 32 * kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
    if (kWeightGrad || kMode == BwdMode::kPreact) prefetch_tensormap(&map_out);
  }
  if (warp == 1) {
    if (kPair) pair::tmem_alloc2<kTmemColsB>(tmem_slot);  // the pair's columns together
    else tmem_alloc<kTmemColsB>(tmem_slot);
  }
  __syncthreads();
  if (kPair) {  // prefix of ceil(m-tiles / 2) per expert
    __shared__ int s_part[kThreadsB / 32];
    const int per = (p.E + kThreadsB - 1) / kThreadsB;
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
    if (threadIdx.x == kThreadsB - 1) {
      int total = 0;
      for (int w = 0; w < kThreadsB / 32; ++w) total += s_part[w];
      s_ptp[p.E] = total;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();  // both CTAs' barriers exist before anything signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total_tiles = kWeightGrad ? p.E * p.m_tiles * p.n_tiles
                          : kPair     ? s_ptp[p.E] * p.n_tiles
                                      : s_mtp[p.E] * p.n_tiles;
  const int tile0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tstride = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  auto tile_at = [&](int tile) {
    if (!kPair) return decode_btile<kMode>(tile, s_mtp, p);
    BTile t = decode_btile<kMode>(tile, s_ptp, p);  // m = the pair index
    t.m = 2 * t.m + static_cast<int>(rank);
    return t;
  };
  auto rows_of = [&](int e) { return s_off[e + 1] - s_off[e]; };
  auto ksteps = [&](const BTile& t) {
    return kWeightGrad ? (rows_of(t.e) + kBK - 1) / kBK : p.K / kBK;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      // a pair's loads complete on the leader's barrier (its cluster address)
      auto load = [&](void* dst, const CUtensorMap* map, int c0, int c1, int st) {
        if (kPair) pair::tma_load(dst, map, c0, c1, pair::mapa(smem_u32(&full[st]), 0), pol);
        else tma_load_2d(dst, map, c0, c1, &full[st], pol);
      };
      for (int tile = tile0; tile < total_tiles; tile += tstride) {
        if (*abort_flag) break;
        const BTile t = tile_at(tile);
        const int nk = ksteps(t);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.status)) { ok = false; break; }
          if (leader) mbar_arrive_expect_tx(&full[stage], (kPair ? 2 : 1) * kStageBytes);
          uint8_t* a_dst = sA + stage * kABytesB;
          uint8_t* b_dst = sB + stage * kBStage;
          int brow;
          if (kWeightGrad) {
            brow = s_off[t.e] + kb * kBK;  // the expert's rows are the contraction
            load(a_dst, &map_a, t.m * kBM, brow, stage);
            load(a_dst + kBoxBytes, &map_a, t.m * kBM + 64, brow, stage);
          } else {
            load(a_dst, &map_a, kb * kBK, s_off[t.e] + t.m * kBM, stage);
            brow = t.e * p.K + kb * kBK;  // rows of the expert's weight matrix
          }
          // this CTA's B columns: all 256, or a pair member's 128
          const int bcol0 = t.n * kBN + (kPair ? static_cast<int>(rank) * (kBN / 2) : 0);
          if (kBKMajor) {  // weight rows x 64 K in one box
            load(b_dst, &map_b, kb * kBK, t.e * p.N + bcol0, stage);
          } else {
#pragma unroll
            for (int i = 0; i < static_cast<int>(kBStage / kBoxBytes); ++i)
              load(b_dst + i * kBoxBytes, &map_b, bcol0 + 64 * i, brow, stage);
          }
          ++issued;
          if (++stage == kStagesB) { stage = 0; phase ^= 1; }
        }
        if (!ok) { *abort_flag = 1; break; }
      }
      // Leave no bulk copy in flight: wait for the last fill of every stage
      // (a pair's copies all complete on the leader's barriers; the peer's
      // shared memory outlives them through the final cluster barrier).
      for (int i = 1; leader && i <= kStagesB && i <= issued; ++i) {
        int s = stage - i;
        uint32_t ph = phase;
        if (s < 0) { s += kStagesB; ph ^= 1; }
        mbar_wait(&full[s], ph, p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // (only the leader's for a pair: one cta_group::2 MMA covers both CTAs)
    if (leader) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int tile = tile0; tile < total_tiles; tile += tstride, ++local) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        const int buf = local & 1;
        const uint32_t tph = (local >> 1) & 1;
        const BTile t = tile_at(tile);
        const int nk = ksteps(t);
        int ok = lane == 0 ? (mbar_wait(&tempty[buf], tph ^ 1, p.status) ? 1 : 0) : 1;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kBN;
        for (int kb = 0; kb < nk; ++kb) {
          ok = lane == 0 ? (mbar_wait(&full[stage], phase, p.status) ? 1 : 0) : 1;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          int nkk = kBK / 16;  // K=16 MMA steps of this stage
          if (kWeightGrad) {
            const int valid = rows_of(t.e) - kb * kBK;
            if (valid < kBK) {
              // the MMAs read rows 0 .. 16*nkk-1; rows valid .. 16*nkk-1 of each
              // of the six boxes are the next expert's (or past the matrix):
              // zero them, then hand the writes to the async proxy the MMA reads
              nkk = (valid + 15) / 16;
              const int zrows = 16 * nkk - valid;
              if (zrows > 0) {
                __syncwarp();
                const int per_box = zrows * 8;  // 16-byte vectors per box
                for (int i = lane; i < 6 * per_box; i += 32) {
                  const int b = i / per_box, v = i - b * per_box;
                  uint8_t* box = b < 2 ? sA + stage * kABytesB + b * kBoxBytes
                                       : sB + stage * kBStage + (b - 2) * kBoxBytes;
                  reinterpret_cast<uint4*>(box + valid * 128)[v] = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_shared();
              }
            }
            __syncwarp();
          }
          if (lane == 0) {
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sA + stage * kABytesB);
            const uint32_t b_addr = smem_u32(sB + stage * kBStage);
  #pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              if (kk >= nkk) break;
              const uint64_t a_desc = kWeightGrad
                                          ? sw128_mnmajor_desc(a_addr + kk * kStepBytesMN)
                                          : sw128_kmajor_desc(a_addr) + 2 * kk;
              const uint64_t b_desc = kBKMajor ? sw128_kmajor_desc(b_addr) + 2 * kk
                                               : sw128_mnmajor_desc(b_addr + kk * kStepBytesMN);
              if (kPair) pair::mma(d_tmem, a_desc, b_desc, kIdescB, (kb | kk) != 0);
              else mma_bf16_ss(d_tmem, a_desc, b_desc, kIdescB, (kb | kk) != 0);
            }
            if (kPair) pair::commit_both(&empty[stage]);  // both CTAs' copies of the stage
            else mma_commit(&empty[stage]);
          }
          __syncwarp();
          if (++stage == kStagesB) { stage = 0; phase ^= 1; }
        }
        if (!ok) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        // an expert without rows commits no MMA: the epilogue writes zeros
        if (lane == 0) {
          if (kPair) pair::commit_both(&tfull[buf]);
          else mma_commit(&tfull[buf]);
        }
        __syncwarp();
      }
      if (lane == 0) {
        // All MMAs of this CTA (or pair) done before TMEM is released.
        if (kPair) pair::commit_local(drain);
        else mma_commit(drain);
        mbar_wait(drain, 0, p.status);
      }
      __syncwarp();
    }  // leader
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lanes this warp may access
    const int row_in_tile = quad * 32 + lane;
    int local = 0;
    int n_stores = 0;  // bulk-tensor stores this warp issued (kWeight)
    for (int tile = tile0; tile < total_tiles; tile += tstride, ++local) {
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const int buf = local & 1;
      const uint32_t tph = (local >> 1) & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[buf], tph, p.status));
      if (!ok) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const BTile t = tile_at(tile);
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * kBN;
      const int col0 = t.n * kBN;
      // chunks of 32 columns, read from TMEM two at a time (one wait per pair)
      const int nch = min(kBN / 32, (p.N - col0) / 32);
      auto chunk_pairs = [&](bool zeros, auto&& handle) {
#pragma unroll 1
        for (int c = 0; c < nch; c += 2) {
          uint32_t a0[32], a1[32];
          const bool two = c + 1 < nch;
          if (zeros) {
#pragma unroll
            for (int i = 0; i < 32; ++i) a0[i] = a1[i] = 0u;
          } else {
            tmem_ld_32x32b_x32(t_lane + c * 32, a0);
            if (two) tmem_ld_32x32b_x32(t_lane + (c + 1) * 32, a1);
            tmem_ld_wait();
          }
          handle(c, a0);
          if (two) handle(c + 1, a1);
        }
      };
      if (kWeightGrad) {
        // each warp's 32 rows x kStep columns staged in shared memory as
        // 64-column boxes with the 128-byte swizzle (lane r puts 16-byte
        // chunk j of its row at slot j ^ (r % 8): no bank conflicts), then
        // bulk-tensor stores; kNB buffers per warp alternate
        constexpr int kStep = out_step_cols<static_cast<int>(kMode)>();
        constexpr int kNB = out_buffers<static_cast<int>(kMode)>();
        constexpr uint32_t kBufBytes = (kStep / 64) * kOutBoxBytes;
        const int orow0 = t.e * p.M + t.m * kBM + quad * 32;
        const bool none = rows_of(t.e) == 0;
        uint8_t* stg = s_out + (warp - 2) * kNB * kBufBytes;
        const int rsw = lane & 7;
#pragma unroll 1
        for (int h = 0; h < kBN / kStep; ++h) {
          const int c0 = col0 + h * kStep;
          if (c0 >= p.N) break;
          const int nq = min(kStep / 32, (p.N - c0) / 32);
          uint8_t* buf = stg + (n_stores % kNB) * kBufBytes;
          if (lane == 0) bulk_wait_group_read<kNB - 1>();  // the buffer's last stores read it
          __syncwarp();
#pragma unroll
          for (int qp = 0; qp < kStep / 32; qp += 2) {  // two 32-column chunks per TMEM wait
            if (qp >= nq) break;
            uint32_t a[2][32];
            if (none) {
#pragma unroll
              for (int i2 = 0; i2 < 32; ++i2) a[0][i2] = a[1][i2] = 0u;
            } else {
              tmem_ld_32x32b_x32(t_lane + h * kStep + qp * 32, a[0]);
              if (qp + 1 < nq) tmem_ld_32x32b_x32(t_lane + h * kStep + (qp + 1) * 32, a[1]);
              tmem_ld_wait();
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int q = qp + u;
              if (q < nq) {
                uint8_t* row = buf + (q >> 1) * kOutBoxBytes + lane * 128;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  const int jj = (q & 1) * 4 + v;
                  *reinterpret_cast<uint4*>(row + ((jj ^ rsw) << 4)) = make_uint4(
                      pack2_bf16(__uint_as_float(a[u][8 * v + 0]), __uint_as_float(a[u][8 * v + 1])),
                      pack2_bf16(__uint_as_float(a[u][8 * v + 2]), __uint_as_float(a[u][8 * v + 3])),
                      pack2_bf16(__uint_as_float(a[u][8 * v + 4]), __uint_as_float(a[u][8 * v + 5])),
                      pack2_bf16(__uint_as_float(a[u][8 * v + 6]), __uint_as_float(a[u][8 * v + 7])));
                }
              }
            }
          }
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int b = 0; b < kStep / 64; ++b)
              if (c0 + 64 * b < p.N) tma_store_2d(&map_out, buf + b * kOutBoxBytes, c0 + 64 * b, orow0);
            bulk_commit_group();
          }
          ++n_stores;
        }
      } else {
        const bool row_ok = t.m * kBM + row_in_tile < rows_of(t.e);
        const long out_row = static_cast<long>(s_off[t.e]) + t.m * kBM + row_in_tile;
        if (kMode == BwdMode::kPreact) {
          // a warp whose 32 rows all belong to the expert stages each 32 x 32
          // fp32 chunk (128-byte swizzle) and bulk-stores it; a ragged warp
          // stores its valid rows directly
          const bool warp_full = t.m * kBM + quad * 32 + 32 <= rows_of(t.e);
          uint8_t* stg = s_out + (warp - 2) * kOutBoxBytes;
          const int rsw = lane & 7;
          const long orow0 = static_cast<long>(s_off[t.e]) + t.m * kBM + quad * 32;
          float4* dst = reinterpret_cast<float4*>(p.out) + out_row * p.ldo_vec + col0 / 4;
          chunk_pairs(false, [&](int c, const uint32_t(&a)[32]) {
            if (warp_full) {
              if (lane == 0) bulk_wait_group_read<0>();  // the buffer's last store read it
              __syncwarp();
              uint8_t* row = stg + lane * 128;
#pragma unroll
              for (int v = 0; v < 8; ++v)
                *reinterpret_cast<uint4*>(row + ((v ^ rsw) << 4)) =
                    make_uint4(a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]);
              fence_proxy_async_shared();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&map_out, stg, col0 + c * 32, static_cast<int>(orow0));
                bulk_commit_group();
              }
            } else if (row_ok) {
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[c * 8 + v] = make_float4(__uint_as_float(a[4 * v]), __uint_as_float(a[4 * v + 1]),
                                             __uint_as_float(a[4 * v + 2]),
                                             __uint_as_float(a[4 * v + 3]));
            }
          });
        } else if (kMode == BwdMode::kDataPlain) {
          uint4* dst = p.out + out_row * p.ldo_vec + col0 / 8;
          chunk_pairs(false, [&](int c, const uint32_t(&a)[32]) {
            if (!row_ok) return;
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c * 4 + v] = make_uint4(
                  pack2_bf16(__uint_as_float(a[8 * v + 0]), __uint_as_float(a[8 * v + 1])),
                  pack2_bf16(__uint_as_float(a[8 * v + 2]), __uint_as_float(a[8 * v + 3])),
                  pack2_bf16(__uint_as_float(a[8 * v + 4]), __uint_as_float(a[8 * v + 5])),
                  pack2_bf16(__uint_as_float(a[8 * v + 6]), __uint_as_float(a[8 * v + 7])));
          });
        } else {
          // SwiGLU backward of 32 columns f at a time: dh (unweighted) from
          // TMEM, g and u from the fp32 pre-activations (the clamp decisions
          // are taken on exactly these values)
          const float w = row_ok ? __ldg(p.w_perm + out_row) : 0.f;
          const bool clamped = p.clamp > 0.f;
          const float cl = p.clamp;
          const float4* arow = p.act + out_row * p.act_vec;
          uint4* drow = p.dact + out_row * p.dact_vec;
          uint4* hrow = p.hw + out_row * (p.F / 8);
          float dw_acc = 0.f;
          // the two warps of a quadrant take alternate chunks
          const int half = (warp - 2) / 4;
#pragma unroll 1
          for (int c = half; c < kBN / 32 && col0 + c * 32 < p.N; c += kEpiWarps / 4) {
            const int f0 = col0 + c * 32;
            const int gc0 = gate_col(f0, p.F, p.interleave);
            const int uc0 = up_col(f0, p.F, p.interleave);
            // all 64 pre-activations of the chunk in flight before the TMEM
            // load: one memory round trip per chunk
            float4 ga[8], ua[8];
            if (row_ok) {
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                ga[q4] = __ldg(arow + gc0 / 4 + q4);
                ua[q4] = __ldg(arow + uc0 / 4 + q4);
              }
            }
            uint32_t d[32];
            tmem_ld_32x32b_x32(t_lane + c * 32, d);
            tmem_ld_wait();
            if (!row_ok) continue;
            uint32_t dgp[16], dup[16], hp[16];
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {  // 4 columns per step
              const float4 g4 = ga[q4];
              const float4 u4 = ua[q4];
              const float gs[4] = {g4.x, g4.y, g4.z, g4.w};
              const float us[4] = {u4.x, u4.y, u4.z, u4.w};
              float dg[4], du[4], hh[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float g = gs[q], u = us[q];
                const float dh = __uint_as_float(d[4 * q4 + q]);
                float gc = g, uc = u, mg = 1.f, mu = 1.f;
                if (clamped) {
                  mg = g <= cl ? 1.f : 0.f;
                  mu = (u >= -cl && u <= cl) ? 1.f : 0.f;
                  gc = fminf(g, cl);
                  uc = fminf(fmaxf(u, -cl), cl);
                }
                const float sg = 1.f / (1.f + expf(-gc));
                const float si = gc * sg;
                const float h = si * uc;
                const float dhw = w * dh;
                dg[q] = mg * dhw * uc * (sg * (1.f + gc * (1.f - sg)));
                du[q] = mu * dhw * si;
                hh[q] = w * h;
                dw_acc = fmaf(dh, h, dw_acc);
              }
              dgp[2 * q4] = pack2_bf16(dg[0], dg[1]);
              dgp[2 * q4 + 1] = pack2_bf16(dg[2], dg[3]);
              dup[2 * q4] = pack2_bf16(du[0], du[1]);
              dup[2 * q4 + 1] = pack2_bf16(du[2], du[3]);
              hp[2 * q4] = pack2_bf16(hh[0], hh[1]);
              hp[2 * q4 + 1] = pack2_bf16(hh[2], hh[3]);
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              drow[gc0 / 8 + v] = make_uint4(dgp[4 * v], dgp[4 * v + 1], dgp[4 * v + 2], dgp[4 * v + 3]);
              drow[uc0 / 8 + v] = make_uint4(dup[4 * v], dup[4 * v + 1], dup[4 * v + 2], dup[4 * v + 3]);
              hrow[f0 / 8 + v] = make_uint4(hp[4 * v], hp[4 * v + 1], hp[4 * v + 2], hp[4 * v + 3]);
            }
          }
          if (row_ok) p.dw_part[(out_row * p.n_tiles + t.n) * (kEpiWarps / 4) + half] = dw_acc;
        }
      }
      tc_fence_before();
      if (kPair) pair::arrive_remote(pair::mapa(smem_u32(&tempty[buf]), 0));  // the leader's
      else mbar_arrive(&tempty[buf]);
    }
    // the staged outputs must be written before the CTA's shared memory goes
    if ((kWeightGrad || kMode == BwdMode::kPreact) && lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA of a pair frees TMEM or exits while the other may still signal
  // its barriers or the leader's MMAs may still write its TMEM
  if (kPair) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if (kPair) pair::tmem_dealloc2<kTmemColsB>(tmem_base);
    else tmem_dealloc<kTmemColsB>(tmem_base);
  }
}

template <BwdMode kMode, bool kPair>
cudaError_t launch_bwd_impl(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                            const BwdParams& kp, int grid, cudaStream_t s) {
  auto kern = grouped_gemm_bwd_kernel<kMode, kPair>;
  constexpr size_t smem = smem_bytes_of<static_cast<int>(kMode), kPair>();
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)),
                       dim3(threads_of<static_cast<int>(kMode)>()), smem, s, kPair ? 2 : 1, ma,
                       mb, mo, kp);
}

// The data gradients run on 2-CTA pairs; building with -DMOE_BWD_1CTA keeps
// the 1-CTA tiles instead (for comparison timings only).
constexpr bool bwd_pairs() {
#ifdef MOE_BWD_1CTA
  return false;
#else
  return true;
#endif
}

}  // namespace

cudaError_t launch_grouped_gemm_bwd(const BwdGemmArgs& g, cudaStream_t s) {
  if (g.R == 0 || g.E == 0) return cudaSuccess;
  if (g.N % 32 != 0 || g.E > kMaxEB) return cudaErrorInvalidValue;
  const bool weight = g.mode == kBwdWeight;
  if (weight && g.M % kBM != 0) return cudaErrorInvalidValue;
  if (!weight && g.K % kBK != 0) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  // A: data gradients [R, K] in 128-row K-major boxes; weight gradients
  // [R, M] in 64-row MN-major boxes.  B: 64-row MN-major boxes over the
  // stacked weights [E * K, N] or the activations [R, N].
  if (!make_map_2d(&ma, g.a, static_cast<uint64_t>(g.R),
                   static_cast<uint64_t>(weight ? g.M : g.K), weight ? 64u : static_cast<uint32_t>(kBM)))
    return cudaErrorInvalidValue;
  const bool preact = g.mode == kBwdPreact;
  const bool pair = !weight && bwd_pairs();
  if (preact) {  // the stacked weight rows [E * N, K], K-major boxes of a CTA's rows
    if (g.N % kBN != 0 ||
        !make_map_2d(&mb, g.b, static_cast<uint64_t>(g.E) * static_cast<uint64_t>(g.N),
                     static_cast<uint64_t>(g.K), static_cast<uint32_t>(pair ? kBN / 2 : kBN)))
      return cudaErrorInvalidValue;
  } else if (!make_map_2d(&mb, g.b,
                          weight ? static_cast<uint64_t>(g.R)
                                 : static_cast<uint64_t>(g.E) * static_cast<uint64_t>(g.K),
                          static_cast<uint64_t>(g.N), 64u)) {
    return cudaErrorInvalidValue;
  }
  // weight gradients: the output [E * M, N] in 64-column x 32-row boxes
  // (128-byte swizzle) for the bulk-tensor stores; unused by other modes
  CUtensorMap mo = ma;
  if (weight && !make_map_2d(&mo, g.out, static_cast<uint64_t>(g.E) * static_cast<uint64_t>(g.M),
                             static_cast<uint64_t>(g.N), 32u))
    return cudaErrorInvalidValue;
  // pre-activations: the fp32 output [R, N] in 32 x 32 boxes (128-byte swizzle)
  if (preact && !make_map_2d_f32(&mo, g.out, static_cast<uint64_t>(g.R),
                                 static_cast<uint64_t>(g.N), 32u))
    return cudaErrorInvalidValue;
  BwdParams kp{};
  kp.expert_offsets = g.expert_offsets;
  kp.mtile_prefix = g.mtile_prefix;
  kp.E = g.E;
  kp.K = g.K;
  kp.N = g.N;
  kp.n_tiles = ceil_div(g.N, kBN);
  kp.M = g.M;
  kp.m_tiles = weight ? g.M / kBM : 0;
  kp.m_outer = weight && g.M >= g.N ? 1 : 0;
  kp.out = static_cast<uint4*>(g.out);
  kp.ldo_vec = preact ? g.N / 4 : g.N / 8;
  kp.act = static_cast<const float4*>(g.act);
  kp.act_vec = g.F * 2 / 4;
  kp.dact = static_cast<uint4*>(g.dact);
  kp.dact_vec = g.F * 2 / 8;
  kp.hw = static_cast<uint4*>(g.hw);
  kp.dw_part = g.dw_part;
  kp.w_perm = g.w_perm;
  kp.F = g.F;
  kp.interleave = g.interleave;
  kp.clamp = g.clamp;
  kp.status = g.status;
  long max_tiles;
  if (weight) {
    max_tiles = static_cast<long>(g.E) * kp.m_tiles * kp.n_tiles;
  } else {
    max_tiles = (ceil_div(g.R, kBM) + std::min(g.E, g.R)) * static_cast<long>(kp.n_tiles);
  }
  if (pair) {  // clusters of two CTAs: an even grid, at most one CTA per SM
    const long pairs = (ceil_div(g.R, 2 * kBM) + std::min(g.E, g.R)) * static_cast<long>(kp.n_tiles);
    const int grid = static_cast<int>(2 * std::max(1L, std::min<long>(num_sms() / 2, pairs)));
    switch (g.mode) {
      case kBwdDataPlain: return launch_bwd_impl<BwdMode::kDataPlain, true>(ma, mb, mo, kp, grid, s);
      case kBwdDataSwiGLU:
        return launch_bwd_impl<BwdMode::kDataSwiGLU, true>(ma, mb, mo, kp, grid, s);
      case kBwdPreact: return launch_bwd_impl<BwdMode::kPreact, true>(ma, mb, mo, kp, grid, s);
    }
    return cudaErrorInvalidValue;
  }
  const int grid = static_cast<int>(std::max(1L, std::min<long>(num_sms(), max_tiles)));
  switch (g.mode) {
    case kBwdDataPlain: return launch_bwd_impl<BwdMode::kDataPlain, false>(ma, mb, mo, kp, grid, s);
    case kBwdDataSwiGLU:
      return launch_bwd_impl<BwdMode::kDataSwiGLU, false>(ma, mb, mo, kp, grid, s);
    case kBwdWeight:
      // experts averaging 512 rows or more: K loops long enough to want the
      // fourth pipeline stage more than the wider output staging
      return static_cast<long>(g.R) >= 512L * g.E
                 ? launch_bwd_impl<BwdMode::kWeightLong, false>(ma, mb, mo, kp, grid, s)
                 : launch_bwd_impl<BwdMode::kWeight, false>(ma, mb, mo, kp, grid, s);
    case kBwdPreact: return launch_bwd_impl<BwdMode::kPreact, false>(ma, mb, mo, kp, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
