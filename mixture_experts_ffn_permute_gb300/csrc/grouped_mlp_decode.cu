// Decode-sized expert MLP in ONE launch: the GEMM1 (+SwiGLU) tiles, the GEMM2
// tiles and the weighted top-k combine of every expert with tokens, run by one
// persistent kernel.
//
// At decode sizes the layer streams the weights of the selected experts once
// (W1 2F x H and W2 H x F per expert) against a handful of token rows; the
// time goes to HBM streaming, to launch boundaries and to the last wave of
// each GEMM, where most SMs sit idle.  Here both GEMMs are one tile list:
//
//   tiles [0, n1)        GEMM1: 64 gate + 64 up weight rows x <= 32 tokens of
//                        expert e, K = H; SwiGLU epilogue -> h (bf16)
//   tiles [n1, n1 + n2)  GEMM2: 128 W2 rows (output features) x <= 32 tokens,
//                        K = F; epilogue -> y (bf16), then the combine
//
// (expert-major, token tiles fastest), claimed one at a time from a global
// counter, so a CTA that runs out of GEMM1 tiles starts streaming GEMM2
// weights at once.  A GEMM2 tile of expert e needs every h row of e: the
// GEMM1 epilogue of each tile of e adds one to done[e] (release, after its h
// stores), and the thread that loads the GEMM2 tile's h rows waits until
// done[e] counts all of e's GEMM1 tiles (acquire, then a proxy fence before
// the bulk-tensor loads).  The weight loads of that tile do not wait, so the
// wait overlaps its weight streaming.  Tiles are claimed in index order by
// CTAs that are running (each holds at most one claimed tile beyond the one
// it is loading, and a GEMM1 tile held back is only ever behind another GEMM1
// tile), and a GEMM1 tile waits on nothing, so every wait is on work already
// claimed by a running CTA that will finish it: the kernel needs no
// co-residency guarantee.  Every wait is still bounded (2 s) and reported on
// expiry.
//
// Combine (the "top-k reduction" of the "[SM90] Add W4A8 MegaMoE support"
// description): after storing its y rows, a GEMM2 tile adds one to the
// arrival counter of each (token, 128-feature block) it covers; the tile that
// brings a counter to k (the token's routes; every route of moe_forward's own
// routing is valid) sums the token's k rows of y for that block in slot order
// j = 0..k-1 in fp32 (fmaf, w * y) and rounds once to bf16 -- the same
// arithmetic, in the same order, as the separate combine kernel, so the
// output is bit-identical to it and independent of which tile came last.
//
// The counters (next tile, GEMM1 tiles finished, done[E], arrivals[T][H/128])
// are zeroed by the routing/permutation kernel of the same call.
//
// Warp roles (224 threads, one CTA per SM):
//   warp 0      tile claims (a 4-deep tile queue in shared memory) and the
//               weight TMA loads: one 4-D copy per stage of the tile's two
//               64-row blocks for both K steps (32 KB), each row a 256-byte
//               segment, so the SM's copy path -- which counts row requests --
//               streams twice the bytes of 64-column boxes
//   warp 1      TMEM allocation + single-thread tcgen05.mma issue, one commit
//               per stage
//   warps 2..5  epilogue (tcgen05.ld -> SwiGLU / bf16 -> global stores)
//   warp 6      token-row TMA loads (8 KB per stage): GEMM1 gathers its
//               rows straight from x by permuted_token (tile::gather4, four
//               rows per copy, only as many copies as the tile has rows), so
//               no permuted copy of x is made; GEMM2 loads 32-row boxes of h
//               after waiting on done[e]
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

bool make_map_kplanes_pair(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint64_t gap);  // grouped_gemm.cu
bool make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);  // grouped_gemm.cu

namespace {

constexpr int kM = 128;              // weight rows per tile
constexpr int kN = 32;               // token rows per tile (max)
constexpr int kThreadsD = 224;
// One ring of stages of two 64-deep K steps: weights and token rows land on
// their own full barriers and the MMA releases both with one commit (a
// tcgen05.commit costs about as much as the four MMAs of a small-N K step).
constexpr int kStagesD = 4;
constexpr int kQueue = 4;
constexpr int kClaimLead = 2;        // stages before a tile's last load that the next is claimed
constexpr uint32_t kWBytesD = 2 * kM * kBK * 2;   // 32 KB: two K steps
constexpr uint32_t kXPlaneD = kN * kBK * 2;       // 4 KB: one K step of token rows
constexpr uint32_t kXBytesD = 2 * kXPlaneD;        // 8 KB: two K steps
constexpr uint32_t kRingBytesD = kStagesD * (kWBytesD + kXBytesD);
constexpr uint32_t kTmemColsD = 2 * kN;
constexpr int kMaxED = 1024;
constexpr int kDPitchD = 33;
// arrivals on a tile-queue slot: token producer, MMA issuer, 4 epilogue warps
constexpr uint32_t kQueueConsumers = 6;
// mbarriers: full/empty per ring stage, 2 + 2 accumulator, drain, queue
// full/empty; then the queue slots, the TMEM address word and the abort flag
constexpr uint32_t kBarBytesD = 512;
static_assert((3 * kStagesD + 5 + 2 * kQueue) * 8 + (kQueue + 2) * 4 <=
                  kBarBytesD,
              "barrier area");
constexpr size_t kSmemD = 1024 + kRingBytesD + kBarBytesD +
                          3 * (kMaxED + 1) * sizeof(int32_t) +
                          kM * kDPitchD * sizeof(float) + kN * sizeof(int32_t);
static_assert(kSmemD <= 232448, "shared memory budget");

struct DParams {
  const int32_t* expert_offsets;  // [E + 1]
  uint16_t* h;                    // bf16 [R, F]
  uint16_t* y;                    // bf16 [R, H]
  uint16_t* out;                  // bf16 [T, H]; NULL: no combine, y is the output
  const int32_t* permuted_token;  // [R]
  const int32_t* row_id_map;      // [T, k]
  const float* topk_w;            // [T, k]
  int32_t* ctr;                   // [2 + E + T * (H / 128)], zero at launch
  int E, H, F, k, R, T, interleave, w1t, w2t;
  float clamp;
  uint32_t* status;
};

struct DTile {
  int gemm, e, m, n;  // GEMM (0: GEMM1, 1: GEMM2), expert, weight tile, token tile
};

// ntp: prefix over experts of their token tiles; ntk: token tiles per expert.
__device__ __forceinline__ DTile decode_dtile(int tile, const int32_t* ntp, const int32_t* ntk,
                                              int E, int w1t, int w2t) {
  DTile t;
  const int n1 = ntp[E] * w1t;
  t.gemm = tile >= n1 ? 1 : 0;
  const int wt = t.gemm ? w2t : w1t;
  const int local_all = t.gemm ? tile - n1 : tile;
  // largest e with ntp[e] * wt <= local_all, i.e. ntp[e] <= local_all / wt
  const int v = local_all / wt;
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ntp[mid] <= v) lo = mid; else hi = mid - 1;
  }
  t.e = lo;
  const int local = local_all - ntp[lo] * wt;
  t.m = local / ntk[lo];
  t.n = local - t.m * ntk[lo];
  return t;
}

__device__ __forceinline__ float silu_d(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}


// Orders this thread's generic-proxy global accesses with its later (or the
// earlier ones with others') bulk-tensor accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__global__ void __launch_bounds__(kThreadsD, 1)
grouped_mlp_decode_kernel(const __grid_constant__ CUtensorMap map_w1,
                          const __grid_constant__ CUtensorMap map_x,
                          const __grid_constant__ CUtensorMap map_w2,
                          const __grid_constant__ CUtensorMap map_h, const DParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sW = smem;
  uint8_t* sX = smem + kStagesD * kWBytesD;
  uint64_t* w_full = reinterpret_cast<uint64_t*>(smem + kRingBytesD);
  uint64_t* x_full = w_full + kStagesD;
  uint64_t* empty = x_full + kStagesD;  // stage consumed: weights and token rows
  uint64_t* tfull = empty + kStagesD;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* q_full = drain + 1;
  uint64_t* q_empty = q_full + kQueue;
  volatile int32_t* q_tile = reinterpret_cast<volatile int32_t*>(q_empty + kQueue);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int32_t*>(q_tile) + kQueue);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + kRingBytesD + kBarBytesD);
  int32_t* s_ntp = s_off + (kMaxED + 1);
  int32_t* s_ntk = s_ntp + (kMaxED + 1);
  float* sD = reinterpret_cast<float*>(s_ntk + (kMaxED + 1));
  int32_t* s_last = reinterpret_cast<int32_t*>(sD + kM * kDPitchD);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesD; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kStagesD; ++s) {
      mbar_init(&x_full[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < kQueue; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], kQueueConsumers);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&map_w1);
    prefetch_tensormap(&map_w2);
  }
  if (warp == 6 && lane == 0) {
    prefetch_tensormap(&map_x);
    prefetch_tensormap(&map_h);
  }
  if (warp == 1) tmem_alloc<kTmemColsD>(tmem_slot);
  // Only this CTA's shared and tensor memory so far: overlaps the previous
  // kernel's tail.
  pdl_enter();
  for (int i = threadIdx.x; i <= p.E; i += kThreadsD) s_off[i] = p.expert_offsets[i];
  __syncthreads();
  {
    // token-tile prefix over the experts: thread i scans a run of at most
    // ceil(E / 224) experts; the runs are offset by a scan over the threads
    __shared__ int s_part[kThreadsD / 32];
    const int per = (p.E + kThreadsD - 1) / kThreadsD;
    const int e0 = min(p.E, static_cast<int>(threadIdx.x) * per), e1 = min(p.E, e0 + per);
    int run = 0;
    for (int e = e0; e < e1; ++e) {
      const int rows = s_off[e + 1] - s_off[e];
      const int nt = rows > 0 ? (rows + kN - 1) / kN : 0;
      s_ntk[e] = nt;
      run += nt;
    }
    int incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) s_part[warp] = incl;
    __syncthreads();
    int acc = incl - run;
    for (int w = 0; w < warp; ++w) acc += s_part[w];
    for (int e = e0; e < e1; ++e) {
      s_ntp[e] = acc;
      acc += s_ntk[e];
    }
    if (threadIdx.x == kThreadsD - 1) s_ntp[p.E] = acc;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_ntp[p.E] * (p.w1t + p.w2t);
  int32_t* next_tile = p.ctr;
  int32_t* gemm1_finished = p.ctr + 1;
  int32_t* done = p.ctr + 2;
  int32_t* arrivals = p.ctr + 2 + p.E;

  if (warp == 0) {
    // ------------------------------------------------- tile claims + weights
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_normal();
      int qs = 0, sw = 0;
      uint32_t qp = 0, pw = 0;
      long issued = 0;
      // The next tile is claimed kClaimLead stages before this tile's last
      // load, and never before the ring has made this tile wait for a stage
      // the MMA consumed (stage >= ring depth): the atomic's round trip
      // overlaps loads still in flight, yet a CTA whose tile cannot start
      // (a GEMM2 tile waiting for h) holds no second tile that an idle CTA
      // could take.
      int claimed = atomicAdd(next_tile, 1);
      while (true) {
        const int tile = claimed;
        const bool stop = tile >= total || *abort_flag != 0;
        if (!mbar_wait(&q_empty[qs], qp ^ 1, p.status)) { *abort_flag = 1; break; }
        q_tile[qs] = stop ? -1 : tile;
        mbar_arrive(&q_full[qs]);
        if (++qs == kQueue) { qs = 0; qp ^= 1; }
        if (stop) break;
        const DTile t = decode_dtile(tile, s_ntp, s_ntk, p.E, p.w1t, p.w2t);
        const CUtensorMap* mw = t.gemm ? &map_w2 : &map_w1;
        const int num_kb = (t.gemm ? p.F : p.H) / kBK;
        int w_row0, w_row1;
        if (t.gemm == 0) {
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
          w_row0 += t.e * 2 * p.F;
          w_row1 += t.e * 2 * p.F;
        } else {
          w_row0 = t.e * p.H + t.m * kM;
          w_row1 = w_row0 + kM / 2;
        }
        (void)w_row1;  // the map's second block is its fixed gap further
        const int num_ks = num_kb / 2;  // stages of two K steps
        const int claim_at = max(num_ks - kClaimLead, kStagesD);
        bool ok = true;
        for (int ks = 0; ks < num_ks; ++ks) {
          if (!mbar_wait(&empty[sw], pw ^ 1, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&w_full[sw], kWBytesD);
          tma_load_4d(sW + sw * kWBytesD, mw, 0, w_row0, 0, 2 * ks, &w_full[sw], pol_w);
          ++issued;
          if (++sw == kStagesD) { sw = 0; pw ^= 1; }
          if (ks == claim_at) claimed = atomicAdd(next_tile, 1);
        }
        if (ok && claim_at >= num_ks) claimed = atomicAdd(next_tile, 1);
        if (!ok) { *abort_flag = 1; break; }
      }
      // no bulk copy may still be writing this CTA's shared memory at exit
      for (int i = 1; i <= kStagesD && i <= issued; ++i) {
        int s = sw - i;
        uint32_t ph = pw;
        if (s < 0) { s += kStagesD; ph ^= 1; }
        mbar_wait(&w_full[s], ph, p.status);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------- token rows (x or h)
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_last();
      int qs = 0, sx = 0;
      uint32_t qp = 0, px = 0;
      long issued = 0;
      const int n1 = s_ntp[p.E] * p.w1t;
      bool all_h = false;  // every GEMM1 tile has published its h rows
      while (true) {
        if (!mbar_wait(&q_full[qs], qp, p.status)) { *abort_flag = 1; break; }
        const int tile = q_tile[qs];
        mbar_arrive(&q_empty[qs]);
        if (++qs == kQueue) { qs = 0; qp ^= 1; }
        if (tile < 0) break;
        const DTile t = decode_dtile(tile, s_ntp, s_ntk, p.E, p.w1t, p.w2t);
        const int x_row = s_off[t.e] + t.n * kN;
        const int nval = min(kN, s_off[t.e + 1] - x_row);
        const int ng = (nval + 3) >> 2;  // GEMM1: four-row gathers
        int tk[kN];  // GEMM1: token of each tile row (rows past nval read token 0)
#pragma unroll
        for (int i = 0; i < kN; ++i) {
          const int v = (t.gemm == 0 && i < nval) ? __ldg(p.permuted_token + x_row + i) : 0;
          tk[i] = min(max(v, 0), p.T - 1);
        }
        if (t.gemm == 1 && !all_h) {
          // every GEMM1 tile of expert e has stored its h rows (once all
          // GEMM1 tiles have, no later tile needs to ask)
          const int need = p.w1t * s_ntk[t.e];
          all_h = ld_acquire_gpu(gemm1_finished) >= n1;
          bool ok = all_h || ld_acquire_gpu(done + t.e) >= need;
          if (!ok) {
            const uint64_t t0 = globaltimer_ns();
            while (!(ok = ld_acquire_gpu(done + t.e) >= need)) {
              if (*abort_flag != 0) break;
              if (globaltimer_ns() - t0 > kWaitLimitNs) {
                record_status(p.status, kStatusTimeout);
                break;
              }
              __nanosleep(64);
            }
          }
          if (!ok) { *abort_flag = 1; break; }
          fence_proxy_async_global();
        }
        const int num_kb = (t.gemm ? p.F : p.H) / kBK;
        // rows of the stage past those loaded keep older data: they only
        // feed accumulator columns that are never stored
        const uint32_t bytes = 2 * (t.gemm ? kXPlaneD : static_cast<uint32_t>(ng) * 512u);
        bool ok = true;
        for (int kb = 0; kb < num_kb; kb += 2) {  // stages of two K steps
          if (!mbar_wait(&empty[sx], px ^ 1, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&x_full[sx], bytes);
#pragma unroll
          for (int pl = 0; pl < 2; ++pl) {
            uint8_t* dst = sX + sx * kXBytesD + pl * kXPlaneD;
            if (t.gemm) {
              tma_load_2d(dst, &map_h, (kb + pl) * kBK, x_row, &x_full[sx], pol_x);
            } else {
#pragma unroll
              for (int g = 0; g < kN / 4; ++g)
                if (g < ng)
                  tma_gather4(dst + g * 512, &map_x, (kb + pl) * kBK, tk[4 * g], tk[4 * g + 1],
                              tk[4 * g + 2], tk[4 * g + 3], &x_full[sx], pol_x);
            }
          }
          ++issued;
          if (++sx == kStagesD) { sx = 0; px ^= 1; }
        }
        if (!ok) { *abort_flag = 1; break; }
      }
      for (int i = 1; i <= kStagesD && i <= issued; ++i) {
        int s = sx - i;
        uint32_t ph = px;
        if (s < 0) { s += kStagesD; ph ^= 1; }
        mbar_wait(&x_full[s], ph, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer
    if (lane == 0) {
      int qs = 0, sw = 0;
      uint32_t qp = 0, pw = 0;
      int local = 0;
      while (true) {
        if (!mbar_wait(&q_full[qs], qp, p.status)) { *abort_flag = 1; break; }
        const int tile = q_tile[qs];
        mbar_arrive(&q_empty[qs]);
        if (++qs == kQueue) { qs = 0; qp ^= 1; }
        if (tile < 0 || *abort_flag != 0) break;
        const DTile t = decode_dtile(tile, s_ntp, s_ntk, p.E, p.w1t, p.w2t);
        const int nval = min(kN, s_off[t.e + 1] - s_off[t.e] - t.n * kN);
        const uint32_t idesc = idesc_bf16_f32(kM, static_cast<uint32_t>((nval + 15) & ~15));
        const int num_kb = (t.gemm ? p.F : p.H) / kBK;
        const int buf = local & 1;
        const uint32_t tph = (local >> 1) & 1;
        ++local;
        if (!mbar_wait(&tempty[buf], tph ^ 1, p.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kN;
        bool ok = true;
        for (int kb = 0; kb < num_kb; kb += 2) {  // stages of two K steps
          if (!mbar_wait(&w_full[sw], pw, p.status) || !mbar_wait(&x_full[sw], pw, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int pl = 0; pl < 2; ++pl) {
            const uint64_t w_desc =
                sw128_kmajor_desc(smem_u32(sW + sw * kWBytesD + pl * (kWBytesD / 2)));
            const uint64_t x_desc = sw128_kmajor_desc(smem_u32(sX + sw * kXBytesD + pl * kXPlaneD));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_bf16_ss(d_tmem, w_desc + 2 * kk, x_desc + 2 * kk, idesc, (kb | pl | kk) != 0);
          }
          mma_commit(&empty[sw]);  // releases the stage's weights and token rows
          if (++sw == kStagesD) { sw = 0; pw ^= 1; }
        }
        if (!ok) { *abort_flag = 1; break; }
        mma_commit(&tfull[buf]);
      }
      mma_commit(drain);
      mbar_wait(drain, 0, p.status);
    }
  } else {
    // ------------------------------------------------- epilogue (warps 2..5)
    const int quad = warp & 3;
    const int et = threadIdx.x - 64;    // 0..127
    const int wrow = quad * 32 + lane;  // weight row inside the tile
    const int ie = (p.interleave == 32) ? 32 : 64;
    const int fl = et & 63;             // SwiGLU output column inside the tile
    const int grow = (fl / ie) * 2 * ie + fl % ie;
    const int urow = grow + ie;
    const bool clamp = p.clamp > 0.f && isfinite(p.clamp);
    int qs = 0;
    uint32_t qp = 0;
    int local = 0;
    while (true) {
      const bool got = mbar_wait(&q_full[qs], qp, p.status);
      const int tile = got ? q_tile[qs] : -1;
      __syncwarp();
      if (lane == 0 && got) mbar_arrive(&q_empty[qs]);
      if (++qs == kQueue) { qs = 0; qp ^= 1; }
      const int buf = local & 1;
      const uint32_t tph = (local >> 1) & 1;
      ++local;
      const bool ok = tile >= 0 && mbar_wait(&tfull[buf], tph, p.status);
      // The four warps leave together (they share named barrier 1); the vote
      // is also the barrier that frees sD and s_last of the previous tile.
      if (bar_red_or(1, 128, !ok || *abort_flag != 0)) {
        if (!got || (tile >= 0 && !ok)) *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const DTile t = decode_dtile(tile, s_ntp, s_ntk, p.E, p.w1t, p.w2t);
      const int nval = min(kN, s_off[t.e + 1] - s_off[t.e] - t.n * kN);
      const long row0 = static_cast<long>(s_off[t.e]) + t.n * kN;
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * kN;
      uint32_t a[32];
      tmem_ld_32x32b_x32(t_lane, a);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&tempty[buf]);  // the accumulator is free for the next tile
      if (t.gemm == 0) {
        // gate and up rows of one output column live in different warps
#pragma unroll
        for (int n = 0; n < 32; ++n) sD[wrow * kDPitchD + n] = __uint_as_float(a[n]);
        bar_sync_named(1, 128);
        const int f = t.m * (kM / 2) + fl;
#pragma unroll 4
        for (int n = et >> 6; n < 32; n += 2) {
          if (n < nval) {
            float g = sD[grow * kDPitchD + n], u = sD[urow * kDPitchD + n];
            if (clamp) {
              g = fminf(g, p.clamp);
              u = fminf(fmaxf(u, -p.clamp), p.clamp);
            }
            const __nv_bfloat16 v = __float2bfloat16_rn(silu_d(g) * u);
            p.h[(row0 + n) * p.F + f] = *reinterpret_cast<const uint16_t*>(&v);
          }
        }
        // publish: h rows of this tile are stored (generic proxy) before the
        // counts that let another CTA's bulk-tensor loads read them; the
        // barrier orders every epilogue thread's stores before the release
        fence_proxy_async_global();
        bar_sync_named(1, 128);
        if (et == 0) {
          red_release_gpu_add(done + t.e, 1);
          red_release_gpu_add(gemm1_finished, 1);
        }
      } else {
        const int feat = t.m * kM + wrow;
#pragma unroll
        for (int n = 0; n < 32; ++n) {
          if (n < nval) {
            const __nv_bfloat16 v = __float2bfloat16_rn(__uint_as_float(a[n]));
            p.y[(row0 + n) * p.H + feat] = *reinterpret_cast<const uint16_t*>(&v);
          }
        }
        if (p.out != nullptr) {
          // arrivals per (token, 128-feature block); the tile completing a
          // token's k routes sums them in slot order.  The barrier orders all
          // threads' y stores before each row's release, and the acquiring
          // thread's barrier orders the other tiles' y rows before the reads.
          bar_sync_named(1, 128);
          if (et < kN) {
            int tok = -1;
            if (et < nval) {
              const int tk = __ldg(p.permuted_token + row0 + et);
              const int prev =
                  atom_add_acq_rel_gpu(arrivals + static_cast<long>(tk) * p.w2t + t.m, 1);
              if (prev == p.k - 1) tok = tk;
            }
            s_last[et] = tok;
          }
          bar_sync_named(1, 128);
          const int col = t.m * kM + et;
          for (int i = 0; i < nval; ++i) {
            const int tok = s_last[i];
            if (tok < 0) continue;
            const int32_t* rm = p.row_id_map + static_cast<long>(tok) * p.k;
            const float* wk = p.topk_w + static_cast<long>(tok) * p.k;
            float acc = 0.f;
            // eight slots' loads in flight at a time, summed in slot order
            for (int j0 = 0; j0 < p.k; j0 += 8) {
              float yv[8], wv[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int j = j0 + u;
                const int r = j < p.k ? __ldg(rm + j) : -1;
                wv[u] = r >= 0 ? __ldg(wk + j) : 0.f;
                const unsigned short yb =
                    r >= 0 ? __ldcg(reinterpret_cast<const unsigned short*>(p.y) +
                                    static_cast<long>(r) * p.H + col)
                           : static_cast<unsigned short>(0);
                yv[u] = r >= 0 ? __uint_as_float(static_cast<uint32_t>(yb) << 16) : 0.f;
              }
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int j = j0 + u;
                if (j < p.k && __ldg(rm + j) >= 0) acc = fmaf(wv[u], yv[u], acc);
              }
            }
            const __nv_bfloat16 v = __float2bfloat16_rn(acc);
            p.out[static_cast<long>(tok) * p.H + col] = *reinterpret_cast<const uint16_t*>(&v);
          }
        }
      }
    }
    // Without the combine, y is the output: rows past the last expert's
    // segment (masked routes) are zero.
    if (p.out == nullptr) {
      const long first = s_off[p.E];
      const long n = (static_cast<long>(p.R) - first) * p.H;
      for (long i = static_cast<long>(blockIdx.x) * 128 + et; i < n;
           i += static_cast<long>(gridDim.x) * 128)
        p.y[first * p.H + i] = 0;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kTmemColsD>(tmem_base);
  }
}

}  // namespace

int decode_mlp_counters(int T, int E, int H) { return 2 + E + T * (H / kM); }

cudaError_t launch_grouped_mlp_decode(const DecodeMlpArgs& g, cudaStream_t s) {
  if (g.R == 0) return cudaSuccess;
  // weight stages hold two 64-deep K steps: H and F are multiples of 128
  if (g.E > kMaxED || g.H % kM != 0 || g.F % kM != 0) return cudaErrorInvalidValue;
  // rows between a GEMM1 tile's 64 gate and 64 up rows (the producer's w_row1 - w_row0)
  uint64_t gap1 = kM / 2;
  if (g.interleave == 0) gap1 = static_cast<uint64_t>(g.F);
  else if (g.interleave != 32) gap1 = static_cast<uint64_t>(g.interleave);
  CUtensorMap mw1, mx, mw2, mh;
  if (!make_map_kplanes_pair(&mw1, g.w1, static_cast<uint64_t>(g.E) * 2 * g.F,
                             static_cast<uint64_t>(g.H), gap1) ||
      !make_map_2d(&mx, g.x, static_cast<uint64_t>(g.T), static_cast<uint64_t>(g.H), 1) ||
      !make_map_kplanes_pair(&mw2, g.w2, static_cast<uint64_t>(g.E) * g.H,
                             static_cast<uint64_t>(g.F), kM / 2) ||
      !make_map_2d(&mh, g.h, static_cast<uint64_t>(g.R), static_cast<uint64_t>(g.F), kN))
    return cudaErrorInvalidValue;
  DParams p;
  p.expert_offsets = g.expert_offsets;
  p.h = static_cast<uint16_t*>(g.h);
  p.y = static_cast<uint16_t*>(g.y);
  p.out = static_cast<uint16_t*>(g.out);
  p.permuted_token = g.permuted_token;
  p.row_id_map = g.row_id_map;
  p.topk_w = g.topk_w;
  p.ctr = g.counters;
  p.E = g.E;
  p.H = g.H;
  p.F = g.F;
  p.k = g.k;
  p.R = g.R;
  p.T = g.T;
  p.interleave = g.interleave;
  p.w1t = g.F / (kM / 2);
  p.w2t = g.H / kM;
  p.clamp = g.clamp;
  p.status = g.status;
  // at most min(E, R) experts with tokens, plus one ragged token tile each
  const long max_tiles = (static_cast<long>(ceil_div(g.R, kN)) + std::min(g.E, g.R)) *
                         (p.w1t + p.w2t);
  const int grid = static_cast<int>(std::max(1L, std::min<long>(num_sms(), max_tiles)));
  cudaError_t err = cudaFuncSetAttribute(grouped_mlp_decode_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemD));
  if (err != cudaSuccess) return err;
  return launch_kernel(grouped_mlp_decode_kernel, dim3(static_cast<unsigned>(grid)),
                       dim3(kThreadsD), kSmemD, s, 1, mw1, mx, mw2, mh, p);
}

}  // namespace moe
