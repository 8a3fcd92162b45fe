// Grouped GEMMs with NVFP4 weights expanded into tensor memory: the
// low-precision form of the layer ("[SM90] Add W4A8 MegaMoE support", Usage:
// FP8 activations with FP32 scales per 128 channels, NVFP4 weights with E4M3
// scales per 16 values and an FP32 scale per tensor), weight rows on M.
//
// Each CTA computes 128 weight rows (M) x N token rows of one expert with
// 1-CTA tcgen05.mma kind::f16, which runs at full rate for every N >= 128 on
// GB300 (N is fitted to the expert's rows, at most 192).  The weights stay
// 4-bit in HBM; per 64-deep K step two transform warpgroups (alternate steps)
// expand a CTA's 128 rows of codes x E4M3 scales to f16 (both exact) and store
// them with tcgen05.st straight into a tensor-memory A stage -- one weight row
// per TMEM lane -- so the expanded weights never pass through shared memory;
// the MMA reads A from tensor memory and the f16 token rows (B) from shared
// memory.  The expert's fp32 tensor scale multiplies the accumulator.
//
// CTA pairs (clusters of two) take the two 128-row halves of a 256-row weight
// tile and the same token rows: each CTA loads half of the rows and multicasts
// them to both, and a token block is reused only after both CTAs' MMAs have
// read it.  GEMM1's epilogue re-quantises h per 1 x 128 block (E4M3, scale
// amax/448, stored dequantised as f16); the block is the pair's 128 outputs,
// so the epilogue makes two passes over the accumulator and swaps per-token
// partial maxima with the other CTA through distributed shared memory.
//
// Warp roles (480 threads, one CTA per SM):
//   warp 0       weight producer: codes (TMA) + scales (bulk copies), local ring
//   warp 1       TMEM allocation and the single-thread MMA issuer
//   warps 2..5   epilogue (one TMEM lane quadrant each)
//   warps 6..13  transform: two warpgroups on alternate K steps, each warp
//                writing its own lane quadrant
//   warp 14      token producer (byte ring of exact-size blocks, multicast)
// Every wait is bounded (2 s); on expiry the kernel records the timeout in
// the status word and leaves its loops together with the other roles.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "lowprec.cuh"
#include "pair_tiles.cuh"
#include "ptx.cuh"

namespace moe {

bool make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);  // grouped_gemm.cu (2-byte elements, 128-byte swizzle)
bool make_map_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);  // grouped_gemm.cu (32-byte wide boxes, no swizzle)

namespace {

constexpr int kThreadsT = 480;
constexpr int kNmaxT = 192;                          // token rows per tile
constexpr int kHalfMaxT = kNmaxT / 2;                // rows each CTA of a pair loads
constexpr int kStagesA = 4;                          // tensor-memory A stages (even)
constexpr int kStagesRT = 8;                         // packed codes + scales (even)
static_assert(kStagesA % 2 == 0 && kStagesRT % 2 == 0, "a stage belongs to one warpgroup");
static_assert((kStagesA & (kStagesA - 1)) == 0, "A stage index by mask");
constexpr uint32_t kColsA = kBK / 2;                 // 64 f16 per row = 32 columns
constexpr uint32_t kAccCols = kNmaxT;                // one accumulator
constexpr uint32_t kACol0 = 2 * kAccCols;            // A stages after two accumulators
static_assert(kACol0 + kStagesA * kColsA <= 512, "tensor memory budget");
constexpr uint32_t kCodeBytesT = pair::kM * kBK / 2;   // 4 KB
constexpr uint32_t kScBytesT = pair::kM * kBK / 16;    // 512 B
constexpr uint32_t kXBlockMax = kNmaxT * kBK * 2;      // 24 KB
#ifndef MOE_FP4T_XRING
#define MOE_FP4T_XRING 6
#endif
constexpr uint32_t kXRingBytesT = MOE_FP4T_XRING * kXBlockMax;  // 144 KB
// K steps in flight at most.  One pair of barriers per step: full (this CTA's
// token block and expanded weights are in place) and done (the MMAs of both
// CTAs that read the block have completed; the A stage too, locally).
constexpr int kXSlotsT = 8;
static_assert((kXSlotsT & (kXSlotsT - 1)) == 0 && kXSlotsT >= kStagesA, "step slots");
constexpr int kMaxET = 1024;
constexpr int kDPitchT = 33;
constexpr uint32_t kBarBytesT = 512;
constexpr int kNumBarsT = 2 * kXSlotsT + 2 * kStagesRT + 2 + 2 + 2 + 1;
static_assert(kNumBarsT * 8 + 8 <= kBarBytesT, "barrier area");
constexpr size_t kRingBytesT = kXRingBytesT + kStagesRT * (kCodeBytesT + kScBytesT);
constexpr size_t kSmemT = 1024 + kRingBytesT + kBarBytesT + 4 * (kMaxET + 1) * sizeof(int32_t) +
                          pair::kM * kDPitchT * sizeof(float) +     // gate/up exchange
                          (4 + 2 + 1) * kNmaxT * sizeof(float);     // amax partials, peer, scale
static_assert(kSmemT + 1024 <= 232448, "shared memory budget (dynamic + the 1024-aligned static part)");

struct TParams {
  const int32_t* expert_offsets;
  const uint8_t* scales;  // prepared: [E][rows/128][K/64][128][4]
  const float* gscale;    // [E] fp32 tensor scale
  uint16_t* out;          // f16 h (GEMM1) or bf16 y (GEMM2), rows of ldo elements
  int E, K, w_tiles, rows_per_expert, ldo, F, interleave, out_rows;
  float clamp;
  uint32_t* status;
};

// kind::f16 with f16 A and B (format 0), fp32 accumulator, M x N.
__host__ __device__ constexpr uint32_t idesc_f16_t(uint32_t m, uint32_t n) {
  return (1u << 4) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ float silu_t(float z) { return z / (1.0f + expf(-z)); }

// 1-CTA MMA with A in tensor memory and B described in shared memory.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 columns of this warp's quadrant from 32 registers per thread.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <Epi kEpi>
__global__ void __launch_bounds__(kThreadsT, 1)
grouped_gemm_fp4_tmem_kernel(const __grid_constant__ CUtensorMap map_q,
                             const __grid_constant__ CUtensorMap map_q128,
                             const __grid_constant__ pair::TokenMaps map_x, const TParams p) {
  pdl_enter();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sX = smem;
  uint8_t* sCode = sX + kXRingBytesT;
  uint8_t* sSc = sCode + kStagesRT * kCodeBytesT;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRingBytesT);  // step's operands ready
  uint64_t* done = full + kXSlotsT;        // step's MMAs completed in both CTAs
  uint64_t* r_full = done + kXSlotsT;
  uint64_t* r_empty = r_full + kStagesRT;
  uint64_t* tfull = r_empty + kStagesRT;
  uint64_t* tempty = tfull + 2;
  uint64_t* amax_bar = tempty + 2;         // the other CTA's partial maxima have arrived
  uint64_t* drain = amax_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + kRingBytesT + kBarBytesT);
  int32_t* s_hp = s_off + (kMaxET + 1);
  int32_t* s_cp = s_hp + (kMaxET + 1);
  int32_t* s_ntk = s_cp + (kMaxET + 1);
  float* sD = reinterpret_cast<float*>(s_ntk + (kMaxET + 1));
  float* s_pam = sD + pair::kM * kDPitchT;   // [4][kNmaxT] per-warp partial maxima
  float* s_peer = s_pam + 4 * kNmaxT;        // [2][kNmaxT] the other CTA's maxima
  float* s_scale = s_peer + 2 * kNmaxT;      // [kNmaxT] this tile's per-token scales

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  for (int i = threadIdx.x; i <= p.E; i += kThreadsT) s_off[i] = p.expert_offsets[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kXSlotsT; ++s) {
      // own token producer's arm (+ the bytes of both halves) and the four
      // transform warps of the step's warpgroup
      mbar_init(&full[s], 1 + 4);
      mbar_init(&done[s], 2);  // one commit from each CTA's MMA issuer
    }
    for (int s = 0; s < kStagesRT; ++s) {
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], 4);  // the four warps of the stage's warpgroup
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
      mbar_init(&amax_bar[b], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&map_q);
    prefetch_tensormap(&map_q128);
    for (int i = 0; i < pair::kTokenBoxes; ++i) prefetch_tensormap(&map_x.m[i]);
  }
  if (warp == 1) tmem_alloc<512>(tmem_slot);
  __syncthreads();
  const pair::Sched sched =
      pair::build_sched<kThreadsT, kNmaxT>(s_off, p.E, p.w_tiles, s_ntk, s_hp, s_cp);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before anything signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = sched.total();
  const int tile0 = static_cast<int>(blockIdx.x >> 1);
  const int tstride = static_cast<int>(gridDim.x >> 1);
  const int num_kb = p.K / kBK;
  const bool glu = kEpi == Epi::kSwiGLU;

  if (warp == 0) {
    // ---------------------------------------------------------- weight producer (local ring)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_normal();
      const uint64_t pol_w_once = policy_evict_first();  // a cold expert's tile: read once
      int sr = 0;
      uint32_t pr = 0;
      long issued = 0;
      for (int tile = tile0; tile < total_tiles && !*abort_flag; tile += tstride) {
        const pair::Tile t = pair::decode(tile, sched);
        int r0, r1;
        pair::weight_rows(glu, t.m, rank, p.F, p.interleave, r0, r1);
        const int q0 = t.e * p.rows_per_expert + r0, q1 = t.e * p.rows_per_expert + r1;
        const long rb = static_cast<long>(t.e) * (p.rows_per_expert / 128);
        const uint8_t* sc0 = p.scales + ((rb + r0 / 128) * num_kb) * 512 + (r0 % 128) * 4;
        const uint8_t* sc1 = p.scales + ((rb + r1 / 128) * num_kb) * 512 + (r1 % 128) * 4;
        const uint64_t pw = t.hot ? pol_w : pol_w_once;
        // the 128 rows in one piece (GEMM2; GEMM1 with interleave 32): one copy each
        const bool whole = r1 == r0 + 64 && r0 % 128 == 0;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&r_empty[sr], pr ^ 1, p.status)) { *abort_flag = 1; break; }
          mbar_arrive_expect_tx(&r_full[sr], kCodeBytesT + kScBytesT);
          uint8_t* code = sCode + sr * kCodeBytesT;
          uint8_t* sc = sSc + sr * kScBytesT;
          if (whole) {
            tma_load_2d(code, &map_q128, kb * (kBK / 2), q0, &r_full[sr], pw);
            bulk_load(sc, sc0 + static_cast<long>(kb) * 512, 512, &r_full[sr]);
          } else {
            tma_load_2d(code, &map_q, kb * (kBK / 2), q0, &r_full[sr], pw);
            tma_load_2d(code + kCodeBytesT / 2, &map_q, kb * (kBK / 2), q1, &r_full[sr], pw);
            bulk_load(sc, sc0 + static_cast<long>(kb) * 512, 256, &r_full[sr]);
            bulk_load(sc + 256, sc1 + static_cast<long>(kb) * 512, 256, &r_full[sr]);
          }
          ++issued;
          if (++sr == kStagesRT) { sr = 0; pr ^= 1; }
        }
      }
      for (int i = 1; i <= kStagesRT && i <= issued; ++i) {  // leave no copy in flight
        int s = sr - i;
        uint32_t ph = pr;
        if (s < 0) { s += kStagesRT; ph ^= 1; }
        if (!mbar_wait(&r_full[s], ph, p.status)) break;
      }
    }
  } else if (warp == 14) {
    // ---------------------------------------------------------- token producer (byte ring)
    // A tile's N = 2 * half token rows form one block per K step; each CTA loads
    // its half and multicasts it into both CTAs at the same offset, so both
    // place blocks identically and a block's space is reused only when both
    // MMA issuers have committed it.
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_last();
      pair::RingQueue<kXSlotsT> xq;
      uint32_t xpos = 0;
      int head = 0, tail = 0;
      for (int tile = tile0; tile < total_tiles && !*abort_flag; tile += tstride) {
        const pair::Tile t = pair::decode(tile, sched);
        const int tok0 = t.n * kNmaxT;
        const int nval = min(kNmaxT, s_off[t.e + 1] - s_off[t.e] - tok0);
        const int half = pair::half_rows(nval);
        const CUtensorMap* mx = &map_x.m[pair::token_box(half)];
        const int x_row = s_off[t.e] + tok0 + static_cast<int>(rank) * half;
        const uint32_t bytes = static_cast<uint32_t>(2 * half) * kBK * 2;
        const uint32_t my_off = rank * static_cast<uint32_t>(half) * kBK * 2;
        for (int kb = 0; kb < num_kb; ++kb) {
          const uint32_t start = pair::ring_place(xpos, bytes, kXRingBytesT);
          if (!pair::ring_make_room<kXSlotsT>(start, bytes, tail, head, xq, done, p.status)) {
            *abort_flag = 1;
            break;
          }
          const int slot = head % kXSlotsT;
          pair::ring_record(xq, slot, start, bytes);
          mbar_arrive_expect_tx(&full[slot], bytes);  // both halves land here
          tma_load_2d_multicast(sX + start + my_off, mx, kb * kBK, x_row, &full[slot], 0x3,
                                pol_x);
          ++head;
        }
      }
      // Leave no copy in flight (after a timed-out wait the copies have long landed).
      for (int j = tail > head - kXSlotsT ? tail : head - kXSlotsT; j < head; ++j)
        if (!mbar_wait(&done[j % kXSlotsT], static_cast<uint32_t>(j / kXSlotsT) & 1u, p.status))
          break;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer (each CTA)
    if (lane == 0) {
      const uint32_t x_base = smem_u32(sX);
      uint32_t xpos = 0;  // the token producer's placement, replayed
      uint32_t step = 0;  // K steps issued
      int local = 0;
      for (int tile = tile0; tile < total_tiles && !*abort_flag; tile += tstride, ++local) {
        const int buf = local & 1;
        const uint32_t tph = (local >> 1) & 1;
        const pair::Tile t = pair::decode(tile, sched);
        const int nval = min(kNmaxT, s_off[t.e + 1] - s_off[t.e] - t.n * kNmaxT);
        const int half = pair::half_rows(nval);
        const uint32_t xbytes = static_cast<uint32_t>(2 * half) * kBK * 2;
        const uint32_t idesc = idesc_f16_t(pair::kM, static_cast<uint32_t>(2 * half));
        if (!mbar_wait(&tempty[buf], tph ^ 1, p.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kAccCols;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb, ++step) {
          const uint32_t xstart = pair::ring_place(xpos, xbytes, kXRingBytesT);
          const uint32_t slot = step & (kXSlotsT - 1);
          if (!mbar_wait(&full[slot], (step / kXSlotsT) & 1u, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem_base + kACol0 + (step & (kStagesA - 1)) * kColsA;
          const uint64_t x_desc = sw128_kmajor_desc(x_base + xstart);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_ts(d_tmem, a_tmem + kk * 8, x_desc + 2 * kk, idesc, (kb | kk) != 0);
          mma_commit_multicast(&done[slot], 0x3);  // both CTAs: token block and A stage free
        }
        if (!ok) { *abort_flag = 1; break; }
        mma_commit(&tfull[buf]);
      }
      mma_commit(drain);
      mbar_wait(drain, 0, p.status);
    }
  } else if (warp >= 6) {
    // ---------------------------------------------------------- transform (each CTA)
    // Warpgroup g expands K steps g, g + 2, ...; thread (quadrant q, lane) owns
    // weight row 32 q + lane = its TMEM lane.  Before it overwrites an A stage
    // the MMAs that read it must be done.
    const int grp = (warp - 6) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + kACol0;
    const int my_tiles = tile0 < total_tiles ? (total_tiles - tile0 + tstride - 1) / tstride : 0;
    const int steps = my_tiles * num_kb;
    // Leave decisions are warp votes: the warp stays converged for the .sync.aligned ops.
    for (int i = grp; i < steps; i += 2) {
      const int sr = i % kStagesRT, sa = i % kStagesA;
      const uint32_t pr = static_cast<uint32_t>(i / kStagesRT) & 1u;
      const int prev = i - kStagesA;  // the K step that last used this A stage
      const bool got =
          *abort_flag == 0 && mbar_wait(&r_full[sr], pr, p.status) &&
          (prev < 0 || mbar_wait(&done[prev & (kXSlotsT - 1)],
                                 static_cast<uint32_t>(prev / kXSlotsT) & 1u, p.status));
      if (!__all_sync(0xffffffffu, got)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint8_t* code = sCode + sr * kCodeBytesT + row * 32;
      const uint4 q0 = *reinterpret_cast<const uint4*>(code);
      const uint4 q1 = *reinterpret_cast<const uint4*>(code + 16);
      const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(sSc + sr * kScBytesT + row * 4);
      __syncwarp();
      if (lane == 0) mbar_arrive(&r_empty[sr]);  // this warp's codes are in registers
      const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
      uint32_t v[32];  // f16 pairs in K order: word j holds k = 2j (low half) and 2j + 1
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // 16 values per E4M3 scale
        const uint32_t sbyte = (sc4 >> (8 * j)) & 0xFFu;
        const uint32_t s2 = e4m3x2_to_f16x2(sbyte | (sbyte << 8));
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const uint32_t w = qw[2 * j + h2];
#pragma unroll
          for (int b = 0; b < 4; ++b)
            v[8 * j + 4 * h2 + b] = hmul2_u32(e2m1x2_to_f16x2((w >> (8 * b)) & 0xFFu), s2);
        }
      }
      tmem_st_32x32b_x32(lane_base + sa * kColsA, v);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[i & (kXSlotsT - 1)]);
    }
  } else {
    // ---------------------------------------------------------- epilogue (warps 2..5)
    const int quad = warp & 3;            // TMEM lane quadrant of this warp
    const int et = threadIdx.x - 64;      // 0..127
    const int wrow = quad * 32 + lane;    // weight row inside this CTA's 128
    const int ie = (p.interleave == 32) ? 32 : 64;
    const bool clamp = p.clamp > 0.f && isfinite(p.clamp);
    const uint32_t peer = rank ^ 1u;
    const uint32_t amax_peer0 = pair::mapa(smem_u32(&amax_bar[0]), peer);
    const uint32_t s_peer_remote = pair::mapa(smem_u32(s_peer), peer);
    int local = 0;
    for (int tile = tile0; tile < total_tiles; tile += tstride, ++local) {
      const int buf = local & 1;
      const uint32_t tph = (local >> 1) & 1;
      const bool ok = mbar_wait(&tfull[buf], tph, p.status);
      if (bar_red_or(1, 128, !ok || *abort_flag != 0)) {  // leave together
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const pair::Tile t = pair::decode(tile, sched);
      const int tok0 = t.n * kNmaxT;
      const int nval = min(kNmaxT, s_off[t.e + 1] - s_off[t.e] - tok0);
      const int nchunk = (nval + 31) / 32;
      const long row0 = static_cast<long>(s_off[t.e]) + tok0;
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * kAccCols;
      const float gs = __ldg(p.gscale + t.e);
      if (kEpi == Epi::kPlain) {
        const int feat = t.m * (2 * pair::kM) + static_cast<int>(rank) * pair::kM + wrow;
        for (int c = 0; c < nchunk; ++c) {
          uint32_t a[32];
          tmem_ld_32x32b_x32(t_lane + c * 32, a);
          tmem_ld_wait();
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            if (c * 32 + n < nval) {
              const __nv_bfloat16 v = __float2bfloat16_rn(__uint_as_float(a[n]) * gs);
              p.out[(row0 + c * 32 + n) * p.ldo + feat] = *reinterpret_cast<const uint16_t*>(&v);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[buf]);
      } else {
        // Token `lane` of each 32-token chunk; this warp's 16 outputs q*16 .. q*16+15.
        const int q = quad;
        bool leave = false;  // set only from a bar_red_or result: the same in all 128 threads
        for (int pass = 0; pass < 2; ++pass) {
          for (int c = 0; c < nchunk; ++c) {
            uint32_t a[32];
            tmem_ld_32x32b_x32(t_lane + c * 32, a);
            tmem_ld_wait();
            if (pass == 1 && c == nchunk - 1) {  // the accumulator is no longer needed
              tc_fence_before();
              mbar_arrive(&tempty[buf]);
            }
            if (c > 0) bar_sync_named(1, 128);
#pragma unroll
            for (int n = 0; n < 32; ++n) sD[wrow * kDPitchT + n] = __uint_as_float(a[n]);
            bar_sync_named(1, 128);
            const int tok = c * 32 + lane;
            const bool live = tok < nval;
            const float sc = pass == 1 && live ? s_scale[tok] : 1.f;
            float hv[16];
            float am = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int fl = q * 16 + i;
              const int grow = (fl / ie) * 2 * ie + fl % ie;
              float g = sD[grow * kDPitchT + lane] * gs, u = sD[(grow + ie) * kDPitchT + lane] * gs;
              if (clamp) {
                g = fminf(g, p.clamp);
                u = fminf(fmaxf(u, -p.clamp), p.clamp);
              }
              hv[i] = silu_t(g) * u;
              am = fmaxf(am, fabsf(hv[i]));
            }
            if (pass == 0) {
              s_pam[q * kNmaxT + tok] = live ? am : 0.f;
            } else if (live) {
              uint32_t packed[8];
#pragma unroll
              for (int i = 0; i < 16; i += 2) {
                const uint32_t q2 = f32x2_to_e4m3x2(hv[i] / sc, hv[i + 1] / sc);
                const uint32_t f2 = e4m3x2_to_f16x2(q2);
                const float2 qf = __half22float2(*reinterpret_cast<const __half2*>(&f2));
                const __half2 o = __floats2half2_rn(qf.x * sc, qf.y * sc);
                packed[i / 2] = *reinterpret_cast<const uint32_t*>(&o);
              }
              uint4* dst = reinterpret_cast<uint4*>(
                  p.out + (row0 + tok) * p.ldo + t.m * pair::kM + static_cast<int>(rank) * 64 + q * 16);
              dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
              dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            }
          }
          if (pass == 0) {
            // this CTA's maximum per token over its 64 outputs, swapped with the other CTA
            bar_sync_named(1, 128);
            for (int tk = et; tk < kNmaxT; tk += 128) {
              float m = 0.f;
#pragma unroll
              for (int w = 0; w < 4; ++w) m = fmaxf(m, s_pam[w * kNmaxT + tk]);
              s_scale[tk] = m;
              pair::st_cluster_f32(s_peer_remote + (buf * kNmaxT + tk) * 4, m);
            }
            pair::arrive_remote(amax_peer0 + buf * 8);
            const bool got = pair::wait_cluster(&amax_bar[buf], tph, p.status);
            if (bar_red_or(1, 128, !got)) {
              *abort_flag = 1;
              leave = true;
              break;
            }
            for (int tk = et; tk < kNmaxT; tk += 128) {
              const float m = fmaxf(s_scale[tk], s_peer[buf * kNmaxT + tk]);
              s_scale[tk] = m > 0.f ? m / 448.0f : 1.0f;
            }
            bar_sync_named(1, 128);
          }
        }
        if (leave) break;
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
    tmem_dealloc<512>(tmem_base);
  }
}

template <Epi kEpi>
cudaError_t launch_fp4_tmem_impl(const CUtensorMap& map_q, const CUtensorMap& map_q128,
                                 const pair::TokenMaps& map_x, const TParams& tp, int grid,
                                 cudaStream_t s) {
  auto kern = grouped_gemm_fp4_tmem_kernel<kEpi>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemT));
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreadsT), kSmemT, s, 2,
                       map_q, map_q128, map_x, tp);
}

}  // namespace

cudaError_t launch_grouped_gemm_fp4_tmem(const GroupedGemmArgs& g, const uint8_t* scales,
                                         const float* gscale, cudaStream_t s) {
  if (g.a_rows == 0) return cudaSuccess;
  if (g.E > kMaxET || g.b_rows_per_expert % 128 != 0 || g.K % kBK != 0)
    return cudaErrorInvalidValue;
  CUtensorMap map_q, map_q128;
  pair::TokenMaps map_x;
  // packed codes: [E * rows, K/2] bytes, 32-byte wide boxes of 64 or 128 rows
  if (!make_map_u8(&map_q, g.b, static_cast<uint64_t>(g.E) * g.b_rows_per_expert,
                   static_cast<uint64_t>(g.K) / 2, 64) ||
      !make_map_u8(&map_q128, g.b, static_cast<uint64_t>(g.E) * g.b_rows_per_expert,
                   static_cast<uint64_t>(g.K) / 2, 128))
    return cudaErrorInvalidValue;
  for (int i = 0; i < pair::kTokenBoxes; ++i)
    if (!make_map_2d(&map_x.m[i], g.a, static_cast<uint64_t>(g.a_rows),
                     static_cast<uint64_t>(g.K), static_cast<uint32_t>(16 * (i + 1))))
      return cudaErrorInvalidValue;
  TParams tp;
  tp.expert_offsets = g.expert_offsets;
  tp.scales = scales;
  tp.gscale = gscale;
  tp.out = static_cast<uint16_t*>(g.out);
  tp.E = g.E;
  tp.K = g.K;
  tp.rows_per_expert = g.b_rows_per_expert;
  tp.ldo = g.ldo;
  tp.F = g.F;
  tp.interleave = g.interleave;
  tp.out_rows = g.out_rows;
  tp.clamp = g.clamp;
  tp.status = g.status;
  // pair tiles along the weights: GEMM1 covers 128 output columns, GEMM2 256 features
  tp.w_tiles = (g.epi == Epi::kSwiGLU) ? g.F / pair::kM : g.ldo / (2 * pair::kM);
  const long max_tiles =
      (static_cast<long>(ceil_div(g.a_rows, kNmaxT)) + std::min(g.E, g.a_rows)) * tp.w_tiles;
  const long want = std::min<long>(num_sms() & ~1, 2 * max_tiles);
  const int grid = static_cast<int>(std::max(2L, want & ~1L));
  if (g.epi == Epi::kSwiGLU)
    return launch_fp4_tmem_impl<Epi::kSwiGLU>(map_q, map_q128, map_x, tp, grid, s);
  if (g.epi == Epi::kPlain)
    return launch_fp4_tmem_impl<Epi::kPlain>(map_q, map_q128, map_x, tp, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
