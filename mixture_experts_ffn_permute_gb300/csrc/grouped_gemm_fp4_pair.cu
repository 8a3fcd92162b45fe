// Grouped GEMMs with NVFP4 weights on 2-CTA clusters, weight rows on M: the
// low-precision form of the layer ("[SM90] Add W4A8 MegaMoE support", Usage:
// FP8 activations with FP32 scales per 128 channels, NVFP4 weights with E4M3
// scales per 16 values and an FP32 scale per tensor) with the tiling of
// grouped_gemm_swap2.cu (pair_tiles.cuh: 256 weight rows x N <= 256 token
// rows fitted per expert, hot/cold tile interleave).
//
// The weights stay 4-bit in HBM.  Per 64-deep K step each CTA of a pair
// streams the packed codes (4 KB) and E4M3 scales (512 B) of its 128 weight
// rows into a deep ring; eight transform warps expand them to f16 in the
// 128-byte-swizzled K-major layout (cvt.rn.f16x2.e2m1x2, then an f16x2
// multiply by the scale: both exact) and signal the leader, whose M = 256
// tcgen05.mma kind::f16 reads both CTAs' expanded weights and both halves of
// the f16 token tile.  The expert's fp32 tensor scale multiplies the
// accumulator.  Splitting the 256 weight rows over two SMs halves each SM's
// transform work and shared-memory traffic per MMA.
//
// GEMM1's epilogue re-quantises h per 1 x 128 block (E4M3, scale amax/448,
// stored dequantised as f16).  A pair tile holds exactly one such block per
// token -- 64 outputs in each CTA -- so the epilogue makes two passes over the
// accumulator: pass 1 reduces each token's |h| over this CTA's 64 outputs and
// swaps the partial maxima with the other CTA through distributed shared
// memory; pass 2 recomputes h and stores the quantised values.
//
// Warp roles (one CTA per SM, both CTAs of a pair alike):
//   warp 0       weight producer: codes (TMA) + scales (bulk copies), local ring
//   warp 1       TMEM allocation; in the leader one lane issues the MMAs
//   warps 2..5   epilogue (TMEM lanes = this CTA's 128 weight rows)
//   warps 6..    transform, one warp per expanded-weight stage
//   last warp    token producer: this CTA's half of the token rows (TMA, counted
//                on the leader's barrier)
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

#ifndef MOE_FP4P_XSTAGES
#define MOE_FP4P_XSTAGES 4
#endif
#ifndef MOE_FP4P_WSTAGES
#define MOE_FP4P_WSTAGES 5
#endif
constexpr int kStagesX = MOE_FP4P_XSTAGES;  // token ring capacity in 16 KB units (128 rows x 64)
constexpr int kStagesW = MOE_FP4P_WSTAGES;  // expanded f16 weights: 128 rows x 64
constexpr int kStagesR = 8;                 // packed codes + scales
constexpr int kFirstTransformWarp = 6;      // one transform warp per expanded-weight stage
constexpr int kTokenWarp = kFirstTransformWarp + kStagesW;
constexpr int kThreadsQ = 32 * (kTokenWarp + 1);
constexpr uint32_t kXBytesQ = (pair::kNmax / 2) * kBK * 2;  // 16 KB
constexpr uint32_t kWBytesQ = pair::kM * kBK * 2;           // 16 KB
constexpr uint32_t kCodeBytesQ = pair::kM * kBK / 2;        // 4 KB
constexpr uint32_t kScBytesQ = pair::kM * kBK / 16;         // 512 B
constexpr uint32_t kTmemColsQ = 2 * pair::kNmax;
constexpr int kMaxEQ = 1024;
constexpr int kDPitchQ = 33;
constexpr uint32_t kXRingBytes = kStagesX * kXBytesQ;
// K steps in flight at most: one token block and one expanded-weight stage
// each, tracked by one pair of barriers (full: both operands ready in both
// CTAs; done: the MMAs that read them have completed).
constexpr int kXSlots = 8;
static_assert(kXSlots >= kStagesW, "a K step's barriers outlive its weight stage");
constexpr uint32_t kBarBytesQ = 512;
constexpr int kNumBars = 2 * kXSlots + 2 * kStagesR + 2 + 2 + 2 + 1;
static_assert(kNumBars * 8 + 8 <= kBarBytesQ, "barrier area");
constexpr size_t kRingBytesQ = kStagesX * kXBytesQ + kStagesW * kWBytesQ +
                               kStagesR * (kCodeBytesQ + kScBytesQ);
constexpr size_t kSmemQ = 1024 + kRingBytesQ + kBarBytesQ + 4 * (kMaxEQ + 1) * sizeof(int32_t) +
                          pair::kM * kDPitchQ * sizeof(float) +  // gate/up exchange
                          (4 + 2 + 1) * pair::kNmax * sizeof(float);  // amax partials, peer, scale
static_assert(kSmemQ + 1024 <= 232448, "shared memory budget (dynamic + the 1024-aligned static part)");

struct QParams {
  const int32_t* expert_offsets;
  const uint8_t* scales;  // prepared: [E][rows/128][K/64][128][4]
  const float* gscale;    // [E] fp32 tensor scale
  uint16_t* out;          // f16 h (GEMM1) or bf16 y (GEMM2), rows of ldo elements
  int E, K, w_tiles, rows_per_expert, ldo, F, interleave, out_rows;
  float clamp;
  uint32_t* status;
};

// kind::f16 with f16 A and B (format 0), fp32 accumulator, M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t m, uint32_t n) {
  return (1u << 4) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ float silu_q(float z) { return z / (1.0f + expf(-z)); }

template <Epi kEpi>
__global__ void __launch_bounds__(kThreadsQ, 1)
grouped_gemm_fp4_pair_kernel(const __grid_constant__ CUtensorMap map_q,
                             const __grid_constant__ CUtensorMap map_q128,
                             const __grid_constant__ pair::TokenMaps map_x, const QParams p) {
  pdl_enter();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sX = smem;
  uint8_t* sW = sX + kStagesX * kXBytesQ;
  uint8_t* sCode = sW + kStagesW * kWBytesQ;
  uint8_t* sSc = sCode + kStagesR * kCodeBytesQ;
  // leader: the K step's token halves (TMA bytes, armed by the token producer)
  // and expanded weights (one arrival per CTA) are in place
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRingBytesQ);
  uint64_t* done = full + kXSlots;        // both CTAs: the K step's MMAs completed
  uint64_t* r_full = done + kXSlots;
  uint64_t* r_empty = r_full + kStagesR;
  uint64_t* tfull = r_empty + kStagesR;
  uint64_t* tempty = tfull + 2;            // leader: both epilogues drained the accumulator
  uint64_t* amax_bar = tempty + 2;         // the other CTA's partial maxima have arrived
  uint64_t* drain = amax_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + kRingBytesQ + kBarBytesQ);
  int32_t* s_hp = s_off + (kMaxEQ + 1);
  int32_t* s_cp = s_hp + (kMaxEQ + 1);
  int32_t* s_ntk = s_cp + (kMaxEQ + 1);
  float* sD = reinterpret_cast<float*>(s_ntk + (kMaxEQ + 1));
  float* s_pam = sD + pair::kM * kDPitchQ;       // [4][256] per-warp partial maxima
  float* s_peer = s_pam + 4 * pair::kNmax;       // [2][256] the other CTA's maxima
  float* s_scale = s_peer + 2 * pair::kNmax;     // [256] this tile's per-token scales

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  for (int i = threadIdx.x; i <= p.E; i += kThreadsQ) s_off[i] = p.expert_offsets[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kXSlots; ++s) {
      mbar_init(&full[s], 3);  // token producer's arm + the transform warp of each CTA
      mbar_init(&done[s], 1);
    }
    for (int s = 0; s < kStagesR; ++s) {
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], 1);  // the transform warp that took the stage
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * 128);
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
  if (warp == 1) pair::tmem_alloc2<kTmemColsQ>(tmem_slot);
  __syncthreads();
  const pair::Sched sched =
      pair::build_sched<kThreadsQ>(s_off, p.E, p.w_tiles, s_ntk, s_hp, s_cp);
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
      const int kblocks = num_kb;
      int sr = 0;
      uint32_t pr = 0;
      long issued = 0;
      for (int tile = tile0; tile < total_tiles && !*abort_flag; tile += tstride) {
        const pair::Tile t = pair::decode(tile, sched);
        int r0, r1;
        pair::weight_rows(glu, t.m, rank, p.F, p.interleave, r0, r1);
        const int q0 = t.e * p.rows_per_expert + r0, q1 = t.e * p.rows_per_expert + r1;
        const long rb = static_cast<long>(t.e) * (p.rows_per_expert / 128);
        const uint8_t* sc0 = p.scales + ((rb + r0 / 128) * kblocks) * 512 + (r0 % 128) * 4;
        const uint8_t* sc1 = p.scales + ((rb + r1 / 128) * kblocks) * 512 + (r1 % 128) * 4;
        const uint64_t pw = t.hot ? pol_w : pol_w_once;
        // the 128 rows in one piece (GEMM2; GEMM1 with interleave 32): one copy each
        const bool whole = r1 == r0 + 64 && r0 % 128 == 0;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&r_empty[sr], pr ^ 1, p.status)) { *abort_flag = 1; break; }
          mbar_arrive_expect_tx(&r_full[sr], kCodeBytesQ + kScBytesQ);
          uint8_t* code = sCode + sr * kCodeBytesQ;
          uint8_t* sc = sSc + sr * kScBytesQ;
          if (whole) {
            tma_load_2d(code, &map_q128, kb * (kBK / 2), q0, &r_full[sr], pw);
            bulk_load(sc, sc0 + static_cast<long>(kb) * 512, 512, &r_full[sr]);
          } else {
            tma_load_2d(code, &map_q, kb * (kBK / 2), q0, &r_full[sr], pw);
            tma_load_2d(code + kCodeBytesQ / 2, &map_q, kb * (kBK / 2), q1, &r_full[sr], pw);
            bulk_load(sc, sc0 + static_cast<long>(kb) * 512, 256, &r_full[sr]);
            bulk_load(sc + 256, sc1 + static_cast<long>(kb) * 512, 256, &r_full[sr]);
          }
          ++issued;
          if (++sr == kStagesR) { sr = 0; pr ^= 1; }
        }
      }
      for (int i = 1; i <= kStagesR && i <= issued; ++i) {  // leave no copy in flight
        int s = sr - i;
        uint32_t ph = pr;
        if (s < 0) { s += kStagesR; ph ^= 1; }
        mbar_wait(&r_full[s], ph, p.status);
      }
    }
  } else if (warp == kTokenWarp) {
    // ---------------------------------------------------------- token producer (pair ring)
    // Blocks of exactly this tile's token half go into a byte ring; both CTAs
    // place them identically, so the leader's descriptors address both.
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_last();
      pair::RingQueue<kXSlots> xq;
      uint32_t xpos = 0;
      int head = 0, tail = 0;
      for (int tile = tile0; tile < total_tiles && !*abort_flag; tile += tstride) {
        const pair::Tile t = pair::decode(tile, sched);
        const int tok0 = t.n * pair::kNmax;
        const int nval = min(pair::kNmax, s_off[t.e + 1] - s_off[t.e] - tok0);
        const int half = pair::half_rows(nval);
        const CUtensorMap* mx = &map_x.m[pair::token_box(half)];
        const int x_row = s_off[t.e] + tok0 + static_cast<int>(rank) * half;
        const uint32_t bytes = static_cast<uint32_t>(half) * kBK * 2;
        for (int kb = 0; kb < num_kb; ++kb) {
          const uint32_t start = pair::ring_place(xpos, bytes, kXRingBytes);
          if (!pair::ring_make_room<kXSlots>(start, bytes, tail, head, xq, done, p.status)) {
            *abort_flag = 1;
            break;
          }
          const int slot = head % kXSlots;
          pair::ring_record(xq, slot, start, bytes);
          if (leader) mbar_arrive_expect_tx(&full[slot], 2 * bytes);
          pair::tma_load(sX + start, mx, kb * kBK, x_row, pair::mapa(smem_u32(&full[slot]), 0),
                         pol_x);
          ++head;
        }
      }
      // Leave no copy in flight: every issued block's K step has completed.
      // (After a timed-out wait the copies have long landed: stop there.)
      for (int j = tail > head - kXSlots ? tail : head - kXSlots; j < head; ++j)
        if (!mbar_wait(&done[j % kXSlots], static_cast<uint32_t>(j / kXSlots) & 1u, p.status))
          break;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer (leader only)
    if (lane == 0 && leader) {
      const uint32_t w_base = smem_u32(sW), x_base = smem_u32(sX);
      uint32_t sw_off = 0;   // expanded-weight stage of this K step, bytes
      uint32_t xpos = 0;     // the token producer's placement, replayed
      uint32_t step = 0;     // K steps issued
      int local = 0;
      for (int tile = tile0; tile < total_tiles && !*abort_flag; tile += tstride, ++local) {
        const int buf = local & 1;
        const uint32_t tph = (local >> 1) & 1;
        const pair::Tile t = pair::decode(tile, sched);
        const int nval = min(pair::kNmax, s_off[t.e + 1] - s_off[t.e] - t.n * pair::kNmax);
        const int half = pair::half_rows(nval);
        const uint32_t xbytes = static_cast<uint32_t>(half) * kBK * 2;
        const uint32_t idesc = idesc_f16_f32(2 * pair::kM, static_cast<uint32_t>(2 * half));
        if (!mbar_wait(&tempty[buf], tph ^ 1, p.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * pair::kNmax;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb, ++step) {
          const uint32_t xstart = pair::ring_place(xpos, xbytes, kXRingBytes);
          const uint32_t slot = step % kXSlots;
          if (!pair::wait_cluster_smem(&full[slot], (step / kXSlots) & 1u, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t w_desc = sw128_kmajor_desc(w_base + sw_off);
          const uint64_t x_desc = sw128_kmajor_desc(x_base + xstart);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            pair::mma(d_tmem, w_desc + 2 * kk, x_desc + 2 * kk, idesc, (kb | kk) != 0);
          pair::commit_both(&done[slot]);
          sw_off = sw_off + kWBytesQ == kStagesW * kWBytesQ ? 0u : sw_off + kWBytesQ;
        }
        if (!ok) { *abort_flag = 1; break; }
        pair::commit_both(&tfull[buf]);
      }
      pair::commit_local(drain);
      mbar_wait(drain, 0, p.status);
    }
  } else if (warp >= kFirstTransformWarp) {
    // ---------------------------------------------------------- transform (both CTAs)
    // Transform warp w owns expanded-weight stage w: it expands K steps
    // w, w + kStagesW, ... of this CTA's sequence, all 128 weight rows (four
    // per lane), then signals the step's full barrier in the leader (a
    // shared-memory release at cluster scope).  Before it overwrites the
    // stage, the K step that last read it must be done.
    const int tw = warp - kFirstTransformWarp;  // == its stage in the ring
    const uint32_t full_leader0 = pair::mapa(smem_u32(&full[0]), 0);
    const int my_tiles = tile0 < total_tiles ? (total_tiles - tile0 + tstride - 1) / tstride : 0;
    const long steps = static_cast<long>(my_tiles) * num_kb;
    uint8_t* wst = sW + tw * kWBytesQ;
    // Leave decisions are warp votes: the warp stays converged for __syncwarp.
    for (long i = tw; i < steps; i += kStagesW) {
      const int sr = static_cast<int>(i % kStagesR);
      const uint32_t pr = static_cast<uint32_t>(i / kStagesR) & 1u;
      const long prev = i - kStagesW;  // the K step that last used this stage
      const bool got =
          *abort_flag == 0 && mbar_wait(&r_full[sr], pr, p.status) &&
          (prev < 0 || mbar_wait(&done[prev % kXSlots],
                                 static_cast<uint32_t>(prev / kXSlots) & 1u, p.status));
      if (!__all_sync(0xffffffffu, got)) {
        *abort_flag = 1;
        break;
      }
      uint4 q[4][2];
      uint32_t sc4[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = r * 32 + lane;
        // the row's 32 code bytes as two 16-byte loads; rows with bit 2 set
        // take the halves in the other order, so the eight lanes of each
        // load phase cover all 32 banks (rows 32 bytes apart would otherwise
        // put lanes t and t+4 on the same banks)
        const uint8_t* code = sCode + sr * kCodeBytesQ + row * 32;
        const int h0 = (row & 4) ? 16 : 0;
        const uint4 qa = *reinterpret_cast<const uint4*>(code + h0);
        const uint4 qb = *reinterpret_cast<const uint4*>(code + (h0 ^ 16));
        q[r][0] = h0 ? qb : qa;
        q[r][1] = h0 ? qa : qb;
        sc4[r] = *reinterpret_cast<const uint32_t*>(sSc + sr * kScBytesQ + row * 4);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&r_empty[sr]);  // the codes are in registers
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = r * 32 + lane;
        const uint32_t qw[8] = {q[r][0].x, q[r][0].y, q[r][0].z, q[r][0].w,
                                q[r][1].x, q[r][1].y, q[r][1].z, q[r][1].w};
        uint8_t* dst = wst + row * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // 16 values per E4M3 scale
          const uint32_t sbyte = (sc4[r] >> (8 * j)) & 0xFFu;
          const uint32_t s2 = e4m3x2_to_f16x2(sbyte | (sbyte << 8));
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {  // 8 values per 16-byte chunk
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
      }
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
      __syncwarp();
      if (lane == 0)  // shared-memory release at cluster scope
        pair::arrive_remote_smem(full_leader0 + static_cast<uint32_t>(i % kXSlots) * 8);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---------------------------------------------------------- epilogue (both CTAs)
    const int quad = warp & 3;            // TMEM lane quadrant of this warp
    const int et = threadIdx.x - 64;      // 0..127
    const int wrow = quad * 32 + lane;    // weight row inside this CTA's 128
    const int ie = (p.interleave == 32) ? 32 : 64;
    const bool clamp = p.clamp > 0.f && isfinite(p.clamp);
    const uint32_t peer = rank ^ 1u;
    const uint32_t tempty_leader0 = pair::mapa(smem_u32(&tempty[0]), 0);
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
      const int tok0 = t.n * pair::kNmax;
      const int nval = min(pair::kNmax, s_off[t.e + 1] - s_off[t.e] - tok0);
      const int nchunk = (nval + 31) / 32;
      const long row0 = static_cast<long>(s_off[t.e]) + tok0;
      const uint32_t t_lane =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * pair::kNmax;
      const float gs = __ldg(p.gscale + t.e);
      if (kEpi == Epi::kPlain) {
        const int feat = t.m * (2 * pair::kM) + static_cast<int>(rank) * pair::kM + wrow;
        for (int c = 0; c < nchunk; ++c) {
          uint32_t a[32];
          tmem_ld_32x32b_x32(t_lane + c * 32, a);
          tmem_ld_wait();
          if (c == nchunk - 1) {
            tc_fence_before();
            pair::arrive_remote(tempty_leader0 + buf * 8);
          }
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            if (c * 32 + n < nval) {
              const __nv_bfloat16 v = __float2bfloat16_rn(__uint_as_float(a[n]) * gs);
              p.out[(row0 + c * 32 + n) * p.ldo + feat] = *reinterpret_cast<const uint16_t*>(&v);
            }
          }
        }
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
              pair::arrive_remote(tempty_leader0 + buf * 8);
            }
            if (c > 0) bar_sync_named(1, 128);
#pragma unroll
            for (int n = 0; n < 32; ++n) sD[wrow * kDPitchQ + n] = __uint_as_float(a[n]);
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
              float g = sD[grow * kDPitchQ + lane] * gs, u = sD[(grow + ie) * kDPitchQ + lane] * gs;
              if (clamp) {
                g = fminf(g, p.clamp);
                u = fminf(fmaxf(u, -p.clamp), p.clamp);
              }
              hv[i] = silu_q(g) * u;
              am = fmaxf(am, fabsf(hv[i]));
            }
            if (pass == 0) {
              s_pam[q * pair::kNmax + tok] = live ? am : 0.f;
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
            for (int tk = et; tk < pair::kNmax; tk += 128) {
              float m = 0.f;
#pragma unroll
              for (int w = 0; w < 4; ++w) m = fmaxf(m, s_pam[w * pair::kNmax + tk]);
              s_scale[tk] = m;
              pair::st_cluster_f32(s_peer_remote + (buf * pair::kNmax + tk) * 4, m);
            }
            pair::arrive_remote(amax_peer0 + buf * 8);
            const bool got = pair::wait_cluster(&amax_bar[buf], tph, p.status);
            if (bar_red_or(1, 128, !got)) {
              *abort_flag = 1;
              leave = true;
              break;
            }
            for (int tk = et; tk < pair::kNmax; tk += 128) {
              const float m = fmaxf(s_scale[tk], s_peer[buf * pair::kNmax + tk]);
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
    pair::tmem_dealloc2<kTmemColsQ>(tmem_base);
  }
}

template <Epi kEpi>
cudaError_t launch_fp4_pair_impl(const CUtensorMap& map_q, const CUtensorMap& map_q128,
                                 const pair::TokenMaps& map_x,
                                 const QParams& qp, int grid, cudaStream_t s) {
  auto kern = grouped_gemm_fp4_pair_kernel<kEpi>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemQ));
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreadsQ), kSmemQ, s, 2,
                       map_q, map_q128, map_x, qp);
}

}  // namespace

cudaError_t launch_grouped_gemm_fp4_pair(const GroupedGemmArgs& g, const uint8_t* scales,
                                         const float* gscale, cudaStream_t s) {
  if (g.a_rows == 0) return cudaSuccess;
  if (g.E > kMaxEQ || g.b_rows_per_expert % 128 != 0 || g.K % kBK != 0)
    return cudaErrorInvalidValue;
  CUtensorMap map_q, map_q128;
  pair::TokenMaps map_x;
  // packed codes: [E * rows, K/2] bytes, two 64-row boxes of 32 bytes per K step
  if (!make_map_u8(&map_q, g.b, static_cast<uint64_t>(g.E) * g.b_rows_per_expert,
                   static_cast<uint64_t>(g.K) / 2, 64))
    return cudaErrorInvalidValue;
  if (!make_map_u8(&map_q128, g.b, static_cast<uint64_t>(g.E) * g.b_rows_per_expert,
                   static_cast<uint64_t>(g.K) / 2, 128))
    return cudaErrorInvalidValue;
  for (int i = 0; i < pair::kTokenBoxes; ++i)
    if (!make_map_2d(&map_x.m[i], g.a, static_cast<uint64_t>(g.a_rows),
                     static_cast<uint64_t>(g.K), static_cast<uint32_t>(16 * (i + 1))))
      return cudaErrorInvalidValue;
  QParams qp;
  qp.expert_offsets = g.expert_offsets;
  qp.scales = scales;
  qp.gscale = gscale;
  qp.out = static_cast<uint16_t*>(g.out);
  qp.E = g.E;
  qp.K = g.K;
  qp.rows_per_expert = g.b_rows_per_expert;
  qp.ldo = g.ldo;
  qp.F = g.F;
  qp.interleave = g.interleave;
  qp.out_rows = g.out_rows;
  qp.clamp = g.clamp;
  qp.status = g.status;
  // pair tiles along the weights: GEMM1 covers 128 output columns, GEMM2 256 features
  qp.w_tiles = (g.epi == Epi::kSwiGLU) ? g.F / pair::kM : g.ldo / (2 * pair::kM);
  const long max_tiles =
      (static_cast<long>(ceil_div(g.a_rows, pair::kNmax)) + std::min(g.E, g.a_rows)) * qp.w_tiles;
  const long want = std::min<long>(num_sms() & ~1, 2 * max_tiles);
  const int grid = static_cast<int>(std::max(2L, want & ~1L));
  if (g.epi == Epi::kSwiGLU)
    return launch_fp4_pair_impl<Epi::kSwiGLU>(map_q, map_q128, map_x, qp, grid, s);
  if (g.epi == Epi::kPlain)
    return launch_fp4_pair_impl<Epi::kPlain>(map_q, map_q128, map_x, qp, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
