// Routing, permute bookkeeping, row gather and the weighted combine.
//
// Routing ("[SM90] Add W4A8 MegaMoE support", Usage: integer expert indices
// and fp32 weights per route) runs one warp per token.  The permute ("add
// permute fusion into hybrid ep", PR description: rows reordered into
// expert-contiguous order) is a three-kernel histogram / scan / scatter
// whose scatter is stable in token order, so row assignment is deterministic
// and matches a sequential walk over (expert, token).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "../../include/moe_ffn.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kRouteWarps = 8;

// Selection key of expert e with logit v: larger logit first, ties to the
// lower id.  The high word is the logit's bits mapped to an unsigned order
// (-0 counted as +0, so the two compare equal); the low word is ~e.  Two warp
// max-reductions (high word, then low word among the lanes holding that
// high word) find the best key of the warp.  NaN logits are not supported.
__device__ __forceinline__ uint32_t order_bits(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Routes one token with one warp: its logits are staged in `row` (shared
// memory) and each lane owns experts lane, lane+32, ... (at most 32 of them).
// Writes the k expert ids (ties to the lowest id) and their weights, then the
// S shared experts (ids E .. E+S-1, weight 1), and the ids to s_idx too when
// it is given.
__device__ __forceinline__ void route_token(const float* __restrict__ src, float* row, int E,
                                            int k, int S, int renormalize, int lane,
                                            int32_t* __restrict__ idx_out,
                                            float* __restrict__ w_out, int32_t* s_idx) {
  const int per_lane = (E + 31) >> 5;
  // stage the logits: eight independent loads per lane before any store, so
  // a token costs one memory round trip per 256 experts, not one per 32
  for (int e0 = 0; e0 < E; e0 += 256) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = e0 + lane + 32 * i;
      v[i] = e < E ? __ldg(src + e) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = e0 + lane + 32 * i;
      if (e < E) row[e] = v[i];
    }
  }
  __syncwarp();
  // each lane's best remaining expert (hi = 0: none left)
  uint32_t taken = 0, hi = 0, lo = 0;
  for (int i = 0; i < per_lane; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const uint32_t h = order_bits(row[e]), l = ~static_cast<uint32_t>(e);
      if (h > hi || (h == hi && l > lo)) { hi = h; lo = l; }
    }
  }
  int mine_id = -1;
  float top = 0.f;
  for (int j = 0; j < k; ++j) {
    const uint32_t best_hi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t best_lo = __reduce_max_sync(0xffffffffu, hi == best_hi ? lo : 0u);
    const int id = static_cast<int>(~best_lo);
    if (lane == j) mine_id = id;
    if (j == 0) top = row[id];
    if ((id & 31) == lane) {  // the winner's lane takes the next of its experts
      taken |= 1u << (id >> 5);
      hi = 0;
      lo = 0;
      for (int i = 0; i < per_lane; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !(taken & (1u << i))) {
          const uint32_t h = order_bits(row[e]), l = ~static_cast<uint32_t>(e);
          if (h > hi || (h == hi && l > lo)) { hi = h; lo = l; }
        }
      }
    }
  }
  const float mine_v = lane < k ? row[mine_id] : 0.f;
  // weights: exp(l - l_top) normalised over the selected (or all) experts
  float ex = (lane < k) ? expf(mine_v - top) : 0.f;
  float denom;
  if (renormalize) {
    denom = warp_sum(ex);
  } else {
    float part = 0.f;
    for (int e = lane; e < E; e += 32) part += expf(row[e] - top);
    denom = warp_sum(part);
  }
  if (lane < k) {
    idx_out[lane] = mine_id;
    w_out[lane] = ex / denom;
    if (s_idx) s_idx[lane] = mine_id;
  }
  if (lane < S) {
    idx_out[k + lane] = E + lane;
    w_out[k + lane] = 1.0f;
    if (s_idx) s_idx[k + lane] = E + lane;
  }
  __syncwarp();
}

// One warp per token.
__global__ void __launch_bounds__(kRouteWarps * 32)
route_topk_kernel(const float* __restrict__ logits, int T, int E, int k, int S, int renormalize,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  pdl_enter();
  extern __shared__ float s_logits[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* row = s_logits + static_cast<size_t>(warp) * E;
  const int slots = k + S;
  for (int t = blockIdx.x * kRouteWarps + warp; t < T; t += gridDim.x * kRouteWarps)
    route_token(logits + static_cast<size_t>(t) * E, row, E, k, S, renormalize, lane,
                topk_idx + static_cast<size_t>(t) * slots, topk_w + static_cast<size_t>(t) * slots,
                nullptr);
}

// Per-chunk expert histogram (shared-memory counters) plus index validation:
// an index outside [-1, E) or an expert listed twice by one token is
// recorded in the status word and the route is treated as masked.
__global__ void __launch_bounds__(256)
chunk_histogram_kernel(const int32_t* __restrict__ topk_idx, int T, int E, int k,
                       int32_t* __restrict__ chunk_counts, uint32_t* status,
                       int32_t* __restrict__ counters, int ncnt) {
  pdl_enter();
  extern __shared__ int32_t s_cnt[];
  const int chunk = blockIdx.x;
  const int t0 = chunk * kChunkTokens;
  const int nt = min(kChunkTokens, T - t0);
  if (counters) {
    int32_t* c = counters + static_cast<size_t>(t0) * ncnt;
    for (int i = threadIdx.x; i < nt * ncnt; i += blockDim.x) c[i] = 0;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int nr = nt * k;
  const int32_t* idx = topk_idx + static_cast<size_t>(t0) * k;
  for (int r = threadIdx.x; r < nr; r += blockDim.x) {
    const int e = idx[r];
    if (e == -1) continue;
    if (e < -1 || e >= E) {
      record_status(status, kStatusIndex);
      continue;
    }
    const int t = r / k, j = r - t * k;
    bool dup = false;
    for (int jj = 0; jj < j; ++jj) dup |= (idx[t * k + jj] == e);
    if (dup) {
      record_status(status, kStatusIndex);
      continue;
    }
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[static_cast<size_t>(chunk) * E + e] = s_cnt[e];
}

// Block-wide exclusive scan over up to 1024 values (one per thread).
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    s_warp[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? s_warp[warp - 1] : 0);
  if (total) *total = s_warp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return excl;
}

// One CTA of 1024 threads.  Thread (g, e) = (tid / E, tid % E) owns expert e
// in the g-th of G = 1024 / E runs of chunks: pass 1 sums its run (loads
// batched 16 at a time, so a run costs a few memory round trips), the runs
// and then the experts are scanned in shared memory, and pass 2 rewrites the
// run's counts as global row bases (expert offset + rows of earlier chunks).
constexpr int kScanBatch = 16;
__global__ void __launch_bounds__(1024)
scan_kernel(int32_t* __restrict__ chunk_counts, int nchunks, int E, int R,
            int32_t* __restrict__ tokens_per_expert, int32_t* __restrict__ expert_offsets,
            int32_t* __restrict__ mtile_prefix, int32_t* __restrict__ permuted_token) {
  pdl_enter();
  __shared__ int s_warp[32];
  __shared__ int s_run[1024];   // [g][e]: the run's count, then its exclusive prefix
  __shared__ int s_eoff[1024];  // [e]: the expert's first row
  const int tid = threadIdx.x;
  const int G = max(1, 1024 / max(E, 1));
  const int g = tid / max(E, 1), e = tid - g * max(E, 1);
  const bool active = E > 0 && g < G;
  const int per = (nchunks + G - 1) / G;
  const int c0 = min(nchunks, g * per), c1 = min(nchunks, c0 + per);
  int run = 0;
  if (active) {
    for (int c = c0; c < c1; c += kScanBatch) {
      int v[kScanBatch];
#pragma unroll
      for (int i = 0; i < kScanBatch; ++i)
        v[i] = c + i < c1 ? chunk_counts[static_cast<size_t>(c + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < kScanBatch; ++i) run += v[i];
    }
    s_run[tid] = run;
  }
  __syncthreads();
  int count = 0;  // the expert's total (threads of run 0)
  if (active && g == 0) {
    for (int q = 0; q < G; ++q) {
      const int r = s_run[q * E + e];
      s_run[q * E + e] = count;
      count += r;
    }
  }
  int total = 0;
  const bool owner = active && g == 0;
  const int off = block_exclusive_scan(owner ? count : 0, s_warp, &total);
  const int mt = (count + kBM - 1) / kBM;
  int mt_total = 0;
  const int mt_off = block_exclusive_scan(owner ? mt : 0, s_warp, &mt_total);
  if (owner) {
    tokens_per_expert[e] = count;
    expert_offsets[e] = off;
    mtile_prefix[e] = mt_off;
    s_eoff[e] = off;
  }
  if (tid == 0) {
    expert_offsets[E] = total;
    mtile_prefix[E] = mt_total;
  }
  __syncthreads();
  if (active) {
    // the run's first row: the expert's offset plus the earlier runs' rows
    int base = s_eoff[e] + s_run[g * E + e];
    for (int c = c0; c < c1; c += kScanBatch) {
      int v[kScanBatch];
#pragma unroll
      for (int i = 0; i < kScanBatch; ++i)
        v[i] = c + i < c1 ? chunk_counts[static_cast<size_t>(c + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < kScanBatch; ++i) {
        if (c + i < c1) chunk_counts[static_cast<size_t>(c + i) * E + e] = base;
        base += v[i];
      }
    }
  }
  for (int r = total + tid; r < R; r += blockDim.x) permuted_token[r] = -1;
}

// One warp per chunk.  Routes are visited in (token, slot) order, 32 at a
// time; lanes holding the same expert are grouped with __match_any_sync and
// ranked by lane, and the group's lowest lane advances the expert's running
// row counter.  A token lists an expert at most once, so (token, slot) order
// is token order within every expert: the scatter is stable.
__global__ void __launch_bounds__(32)
scatter_kernel(const int32_t* __restrict__ topk_idx, int T, int E, int k,
               const int32_t* __restrict__ chunk_base, int32_t* __restrict__ row_id_map,
               int32_t* __restrict__ permuted_token) {
  pdl_enter();
  extern __shared__ int32_t s_next[];
  int32_t* s_idx = s_next + E;  // the chunk's routes, staged once
  const int chunk = blockIdx.x, lane = threadIdx.x;
  const int t0 = chunk * kChunkTokens;
  const int nt = min(kChunkTokens, T - t0);
  const int nr = nt * k;
  const size_t base = static_cast<size_t>(t0) * k;
  for (int e0 = 0; e0 < E; e0 += 8 * 32) {  // eight independent loads per lane at a time
    int v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = e0 + lane + 32 * i;
      v[i] = e < E ? chunk_base[static_cast<size_t>(chunk) * E + e] : 0;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = e0 + lane + 32 * i;
      if (e < E) s_next[e] = v[i];
    }
  }
  for (int r0 = 0; r0 < nr; r0 += 8 * 32) {  // eight independent loads per lane at a time
    int v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = r0 + lane + 32 * i;
      v[i] = r < nr ? topk_idx[base + r] : -1;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = r0 + lane + 32 * i;
      if (r < nr) s_idx[r] = v[i];
    }
  }
  __syncwarp();
  for (int r0 = 0; r0 < nr; r0 += 32) {
    const int r = r0 + lane;
    int e = -1;
    if (r < nr) {
      e = s_idx[r];
      const int t = r / k, j = r - t * k;
      bool dup = false;
      for (int jj = 0; jj < j; ++jj) dup |= (s_idx[t * k + jj] == e);
      if (e < 0 || e >= E || dup) e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int leader = __ffs(peers) - 1;
    int start = 0;
    if (e >= 0) start = s_next[e];
    __syncwarp();
    if (e >= 0 && lane == leader) s_next[e] = start + __popc(peers);
    __syncwarp();
    if (r < nr) {
      const int t = t0 + r / k;
      if (e >= 0) {
        const int row = start + rank;
        row_id_map[base + r] = row;
        permuted_token[row] = t;
      } else {
        row_id_map[base + r] = -1;
      }
    }
  }
}

// x_perm[r] = x[permuted_token[r]] in 16-byte vectors; a grid-stride loop
// over rows, one CTA per row at a time.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ permuted_token,
                   int R, int vecs_per_row, uint4* __restrict__ x_perm) {
  pdl_enter();
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const int t = permuted_token[r];
    uint4* dst = x_perm + static_cast<size_t>(r) * vecs_per_row;
    if (t < 0) {
      for (int v = threadIdx.x; v < vecs_per_row; v += blockDim.x) dst[v] = make_uint4(0, 0, 0, 0);
    } else {
      const uint4* src = x + static_cast<size_t>(t) * vecs_per_row;
      for (int v = threadIdx.x; v < vecs_per_row; v += blockDim.x) dst[v] = __ldg(src + v);
    }
  }
}

// x_perm[row_id_map[t][j]] = x[t] for every valid route, driven by the
// source: each token row is read once and written to its (up to k) permuted
// rows, so the copy reads T rows instead of T * k (one HBM read of x rather
// than k).  Rows from expert_offsets[E] to R (the masked tail, no token) are
// zeroed.  One CTA per token at a time; the token's row indices are staged in
// shared memory.
__global__ void __launch_bounds__(256)
scatter_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ row_id_map,
                    const int32_t* __restrict__ expert_offsets, int T, int k, int E, int R,
                    int vecs_per_row, uint4* __restrict__ x_perm) {
  pdl_enter();
  constexpr int kVecs = 4;  // 16-byte vectors per thread loaded before any store
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const uint4* src = x + static_cast<size_t>(t) * vecs_per_row;
    for (int v0 = 0; v0 < vecs_per_row; v0 += kVecs * blockDim.x) {
      uint4 val[kVecs];
#pragma unroll
      for (int i = 0; i < kVecs; ++i) {
        const int v = v0 + i * blockDim.x + threadIdx.x;
        if (v < vecs_per_row) val[i] = __ldcs(src + v);  // read once: streaming
      }
      for (int j = 0; j < k; ++j) {  // the token's rows (the same words for every thread)
        const int32_t r = __ldg(row_id_map + static_cast<size_t>(t) * k + j);
        if (r < 0 || r >= R) continue;
        uint4* dst = x_perm + static_cast<size_t>(r) * vecs_per_row;
#pragma unroll
        for (int i = 0; i < kVecs; ++i) {
          const int v = v0 + i * blockDim.x + threadIdx.x;
          if (v < vecs_per_row) dst[v] = val[i];
        }
      }
    }
  }
  const int first = min(max(expert_offsets[E], 0), R);
  const size_t n = static_cast<size_t>(R - first) * vecs_per_row;
  uint4* tail = x_perm + static_cast<size_t>(first) * vecs_per_row;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    tail[i] = make_uint4(0, 0, 0, 0);
}

// The same for rows of any width that is a multiple of 4 bytes: 16-byte
// copies when the width allows, 4-byte copies otherwise; token indices
// outside [0, T) give zero rows.
template <typename V>
__global__ void __launch_bounds__(256)
gather_row_bytes_kernel(const V* __restrict__ src, const int32_t* __restrict__ permuted_token,
                        int R, int T, int vecs_per_row, V* __restrict__ dst) {
  pdl_enter();
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const int t = permuted_token[r];
    V* d = dst + static_cast<size_t>(r) * vecs_per_row;
    if (t < 0 || t >= T) {
      for (int v = threadIdx.x; v < vecs_per_row; v += blockDim.x) d[v] = V{};
    } else {
      const V* sp = src + static_cast<size_t>(t) * vecs_per_row;
      for (int v = threadIdx.x; v < vecs_per_row; v += blockDim.x) d[v] = __ldg(sp + v);
    }
  }
}

// Validates caller-supplied offsets (non-decreasing, offsets[0] == 0,
// offsets[E] <= R) and builds the m-tile prefix.  Bad offsets are recorded
// and replaced by an empty problem.
__global__ void __launch_bounds__(1024)
mtile_prefix_kernel(const int32_t* __restrict__ offsets, int E, int R,
                    int32_t* __restrict__ mtile_prefix, uint32_t* status) {
  pdl_enter();
  __shared__ int s_warp[32];
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const int e = threadIdx.x;
  int mt = 0;
  if (e < E) {
    const int a = offsets[e], b = offsets[e + 1];
    if (b < a || a < 0 || b > R || (e == 0 && a != 0)) s_bad = 1;
    mt = (b > a) ? (b - a + kBM - 1) / kBM : 0;
  }
  __syncthreads();
  const bool bad = s_bad != 0;
  if (bad) mt = 0;
  int total = 0;
  const int off = block_exclusive_scan(e < E ? mt : 0, s_warp, &total);
  if (e < E) mtile_prefix[e] = off;
  if (e == 0) {
    mtile_prefix[E] = total;
    if (bad) record_status(status, kStatusIndex);
  }
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 p = __bfloat1622float2(h[i]);
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}

// out[t][c..c+8) = sum_{j} w[t][j] * y[row][c..c+8), fp32 in slot order
// (w = 1 when topk_w is null: the plain sum of the token's rows).
__global__ void __launch_bounds__(256)
combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ row_id_map,
               const float* __restrict__ topk_w, int T, int vecs_per_row, int k,
               uint4* __restrict__ out) {
  pdl_enter();
  const int t = blockIdx.x;
  const int v = blockIdx.y * blockDim.x + threadIdx.x;
  if (t >= T || v >= vecs_per_row) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  // up to eight routes at a time: their rows, weights and y vectors are
  // loaded independently, then summed in slot order
  for (int j0 = 0; j0 < k; j0 += 8) {
    int row[8];
    float w[8];
    uint4 yv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = j0 + i;
      row[i] = j < k ? __ldg(row_id_map + static_cast<size_t>(t) * k + j) : -1;
      w[i] = (j < k && topk_w) ? __ldg(topk_w + static_cast<size_t>(t) * k + j) : 1.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      yv[i] = row[i] >= 0 ? __ldcs(y + static_cast<size_t>(row[i]) * vecs_per_row + v)
                          : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (row[i] < 0) continue;
      float f[8];
      bf16x8_to_f32(yv[i], f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(w[i], f[q], acc[q]);
    }
  }
  uint4 o;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
  out[static_cast<size_t>(t) * vecs_per_row + v] = o;
}

// Expert histogram, scan and the stable scatter of R = T*k routes in ONE
// block of 1024 threads: s_idx (shared) holds the routes, s_cnt (shared) E
// zeroed counters.  Same results as chunk_histogram / scan / scatter, bit for
// bit, for routes that are all valid (moe_forward's own routing).  s_ptok,
// when given, receives permuted_token in shared memory too.
__device__ __forceinline__ void permute_block(const int32_t* s_idx, int32_t* s_cnt, int* s_warp,
                                              int T, int E, int k,
                                              int32_t* __restrict__ tokens_per_expert,
                                              int32_t* __restrict__ expert_offsets,
                                              int32_t* __restrict__ mtile_prefix,
                                              int32_t* __restrict__ row_id_map,
                                              int32_t* __restrict__ permuted_token,
                                              int32_t* s_ptok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = T * k;
  // histogram
  for (int r = threadIdx.x; r < R; r += blockDim.x) atomicAdd(&s_cnt[s_idx[r]], 1);
  __syncthreads();
  // scan (thread e owns expert e)
  const int e = threadIdx.x;
  const int count = e < E ? s_cnt[e] : 0;
  int total = 0;
  const int off = block_exclusive_scan(count, s_warp, &total);
  const int mt = (count + kBM - 1) / kBM;
  int mt_total = 0;
  const int mt_off = block_exclusive_scan(e < E ? mt : 0, s_warp, &mt_total);
  if (e < E) {
    tokens_per_expert[e] = count;
    expert_offsets[e] = off;
    mtile_prefix[e] = mt_off;
    s_cnt[e] = off;  // next free row of expert e
  }
  if (e == 0) {
    expert_offsets[E] = total;
    mtile_prefix[E] = mt_total;
  }
  __syncthreads();
  // stable scatter by warp 0, 32 routes at a time in (token, slot) order
  if (warp == 0) {
    for (int r0 = 0; r0 < R; r0 += 32) {
      const int r = r0 + lane;
      const int ex_id = r < R ? s_idx[r] : -1;
      const uint32_t peers = __match_any_sync(0xffffffffu, ex_id);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int leader = __ffs(peers) - 1;
      int start = 0;
      if (ex_id >= 0) start = s_cnt[ex_id];
      __syncwarp();
      if (ex_id >= 0 && lane == leader) s_cnt[ex_id] = start + __popc(peers);
      __syncwarp();
      if (ex_id >= 0) {
        const int row_id = start + rank;
        row_id_map[r] = row_id;
        permuted_token[row_id] = r / k;
        if (s_ptok) s_ptok[row_id] = r / k;
      }
    }
  }
}

// Decode sizes (T*k <= kSmallRoutes, E <= kSmallExperts): the permutation
// after the routing kernel in one launch instead of three.
__global__ void __launch_bounds__(1024)
permute_small_kernel(const int32_t* __restrict__ topk_idx, int T, int E, int k,
                     int32_t* __restrict__ tokens_per_expert,
                     int32_t* __restrict__ expert_offsets, int32_t* __restrict__ mtile_prefix,
                     int32_t* __restrict__ row_id_map, int32_t* __restrict__ permuted_token,
                     int32_t* __restrict__ zero_ints, int n_zero) {
  pdl_enter();
  for (int i = threadIdx.x; i < n_zero; i += blockDim.x) zero_ints[i] = 0;
  extern __shared__ int32_t s_small[];
  __shared__ int s_warp[32];
  const int R = T * k;
  int32_t* s_idx = s_small;
  int32_t* s_cnt = s_small + R;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  for (int r = threadIdx.x; r < R; r += blockDim.x) s_idx[r] = __ldg(topk_idx + r);
  __syncthreads();
  permute_block(s_idx, s_cnt, s_warp, T, E, k, tokens_per_expert, expert_offsets, mtile_prefix,
                row_id_map, permuted_token, nullptr);
}

// The smallest decode steps (T <= kTinyTokens): routing, the permutation and
// (when x is given) the row gather in ONE block, one warp per token for the
// routing -- two kernel boundaries fewer than route + permute + gather.  Same
// arithmetic as route_topk_kernel and permute_small_kernel (shared code).
__global__ void __launch_bounds__(1024)
route_permute_tiny_kernel(const float* __restrict__ logits, int T, int E, int k, int S,
                          int renormalize, int32_t* __restrict__ topk_idx,
                          float* __restrict__ topk_w, int32_t* __restrict__ tokens_per_expert,
                          int32_t* __restrict__ expert_offsets,
                          int32_t* __restrict__ mtile_prefix, int32_t* __restrict__ row_id_map,
                          int32_t* __restrict__ permuted_token, const uint4* __restrict__ x,
                          int vecs_per_row, uint4* __restrict__ x_perm,
                          int32_t* __restrict__ zero_ints, int n_zero) {
  pdl_enter();
  for (int i = threadIdx.x; i < n_zero; i += blockDim.x) zero_ints[i] = 0;
  extern __shared__ int32_t s_tiny[];
  __shared__ int s_warp[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slots = k + S, experts = E + S;  // routed + shared
  const int R = T * slots;
  int32_t* s_idx = s_tiny;
  int32_t* s_cnt = s_idx + R;
  int32_t* s_ptok = s_cnt + experts;
  float* s_rows = reinterpret_cast<float*>(s_ptok + R);
  for (int e = threadIdx.x; e < experts; e += blockDim.x) s_cnt[e] = 0;
  if (warp < T)
    route_token(logits + static_cast<size_t>(warp) * E, s_rows + static_cast<size_t>(warp) * E, E,
                k, S, renormalize, lane, topk_idx + static_cast<size_t>(warp) * slots,
                topk_w + static_cast<size_t>(warp) * slots, s_idx + warp * slots);
  __syncthreads();
  permute_block(s_idx, s_cnt, s_warp, T, experts, slots, tokens_per_expert, expert_offsets,
                mtile_prefix, row_id_map, permuted_token, s_ptok);
  if (x == nullptr) return;
  __syncthreads();
  for (int i = threadIdx.x; i < R * vecs_per_row; i += blockDim.x) {
    const int r = i / vecs_per_row, v = i - r * vecs_per_row;
    x_perm[i] = __ldg(x + static_cast<size_t>(s_ptok[r]) * vecs_per_row + v);
  }
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int renormalize,
                              int32_t* topk_idx, float* topk_w, cudaStream_t s, int S) {
  if (T == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * kRouteWarps * E;
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(route_topk_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  const int blocks = min(ceil_div(T, kRouteWarps), num_sms() * 8);
  return launch_kernel(route_topk_kernel, dim3(blocks), dim3(kRouteWarps * 32), smem, s, 1,
                       logits, T, E, k, S, renormalize, topk_idx, topk_w);
}

cudaError_t launch_chunk_histogram(const int32_t* topk_idx, int T, int E, int k,
                                   int32_t* chunk_counts, uint32_t* status, cudaStream_t s,
                                   int32_t* counters, int ncnt) {
  const int nchunks = ceil_div(T, kChunkTokens);
  if (nchunks == 0) return cudaSuccess;
  return launch_kernel(chunk_histogram_kernel, dim3(nchunks), dim3(256), sizeof(int32_t) * E, s,
                       1, topk_idx, T, E, k, chunk_counts, status, counters, ncnt);
}

cudaError_t launch_scan(int32_t* chunk_counts, int nchunks, int E, int R,
                        int32_t* tokens_per_expert, int32_t* expert_offsets,
                        int32_t* mtile_prefix, int32_t* permuted_token, cudaStream_t s) {
  return launch_kernel(scan_kernel, dim3(1), dim3(1024), 0, s, 1, chunk_counts, nchunks, E, R,
                       tokens_per_expert, expert_offsets, mtile_prefix, permuted_token);
}

cudaError_t launch_scatter(const int32_t* topk_idx, int T, int E, int k,
                           const int32_t* chunk_base, int32_t* row_id_map,
                           int32_t* permuted_token, cudaStream_t s) {
  const int nchunks = ceil_div(T, kChunkTokens);
  if (nchunks == 0) return cudaSuccess;
  return launch_kernel(scatter_kernel, dim3(nchunks), dim3(32),
                       sizeof(int32_t) * (E + static_cast<size_t>(kChunkTokens) * k), s, 1,
                       topk_idx, T, E, k, chunk_base, row_id_map, permuted_token);
}

cudaError_t launch_gather_rows(const void* x, const int32_t* permuted_token, int R, int H,
                               void* x_perm, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const int vecs = H / 8;
  const int blocks = min(R, num_sms() * 8);
  return launch_kernel(gather_rows_kernel, dim3(blocks), dim3(256), 0, s, 1,
                       static_cast<const uint4*>(x), permuted_token, R, vecs,
                       static_cast<uint4*>(x_perm));
}

cudaError_t launch_scatter_rows(const void* x, const int32_t* row_id_map,
                                const int32_t* expert_offsets, int T, int k, int E, int H,
                                void* x_perm, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = min(T, num_sms() * 8);
  return launch_kernel(scatter_rows_kernel, dim3(blocks), dim3(256), 0, s, 1,
                       static_cast<const uint4*>(x), row_id_map, expert_offsets, T, k, E, T * k,
                       H / 8, static_cast<uint4*>(x_perm));
}

cudaError_t launch_gather_row_bytes(const void* src, const int32_t* permuted_token, int R, int T,
                                    int row_bytes, void* dst, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const int blocks = min(R, num_sms() * 8);
  if (row_bytes % 16 == 0)
    return launch_kernel(gather_row_bytes_kernel<uint4>, dim3(blocks), dim3(256), 0, s, 1,
                         static_cast<const uint4*>(src), permuted_token, R, T, row_bytes / 16,
                         static_cast<uint4*>(dst));
  return launch_kernel(gather_row_bytes_kernel<uint32_t>, dim3(blocks), dim3(256), 0, s, 1,
                       static_cast<const uint32_t*>(src), permuted_token, R, T, row_bytes / 4,
                       static_cast<uint32_t*>(dst));
}

cudaError_t launch_mtile_prefix_from_offsets(const int32_t* expert_offsets, int E, int R,
                                             int32_t* mtile_prefix, uint32_t* status,
                                             cudaStream_t s) {
  return launch_kernel(mtile_prefix_kernel, dim3(1), dim3(1024), 0, s, 1, expert_offsets, E, R,
                       mtile_prefix, status);
}

bool permute_small_fits(int T, int E, int k) {
  return static_cast<long>(T) * k <= kSmallRoutes && E <= kSmallExperts && T > 0;
}

cudaError_t launch_permute_small(const int32_t* topk_idx, int T, int E, int k,
                                 int32_t* tokens_per_expert, int32_t* expert_offsets,
                                 int32_t* mtile_prefix, int32_t* row_id_map,
                                 int32_t* permuted_token, cudaStream_t s, int32_t* zero_ints,
                                 int n_zero) {
  const size_t smem = sizeof(int32_t) * (static_cast<size_t>(T) * k + E);
  return launch_kernel(permute_small_kernel, dim3(1), dim3(1024), smem, s, 1, topk_idx, T, E, k,
                       tokens_per_expert, expert_offsets, mtile_prefix, row_id_map,
                       permuted_token, zero_ints, zero_ints ? n_zero : 0);
}

bool route_permute_tiny_fits(int T, int E, int k, int S) {
  return T > 0 && T <= kTinyTokens && E + S <= kTinyExperts && T * (k + S) <= kTinyRoutes;
}

cudaError_t launch_route_permute_tiny(const float* logits, int T, int E, int k, int S,
                                      int renormalize, int32_t* topk_idx, float* topk_w,
                                      int32_t* tokens_per_expert, int32_t* expert_offsets,
                                      int32_t* mtile_prefix, int32_t* row_id_map,
                                      int32_t* permuted_token, const void* x, int H,
                                      void* x_perm, cudaStream_t s, int32_t* zero_ints,
                                      int n_zero) {
  const int R = T * (k + S);
  const size_t smem = sizeof(int32_t) * (2 * static_cast<size_t>(R) + E + S) +
                      sizeof(float) * static_cast<size_t>(T) * E;
  return launch_kernel(route_permute_tiny_kernel, dim3(1), dim3(1024), smem, s, 1, logits, T, E,
                       k, S, renormalize, topk_idx, topk_w, tokens_per_expert, expert_offsets,
                       mtile_prefix, row_id_map, permuted_token, static_cast<const uint4*>(x),
                       H / 8, static_cast<uint4*>(x_perm), zero_ints, zero_ints ? n_zero : 0);
}

cudaError_t launch_combine(const void* y, const int32_t* row_id_map, const float* topk_w,
                           int T, int H, int k, void* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int vecs = H / 8;
  dim3 grid(T, ceil_div(vecs, 256));
  return launch_kernel(combine_kernel, grid, dim3(256), 0, s, 1, static_cast<const uint4*>(y),
                       row_id_map, topk_w, T, vecs, k, static_cast<uint4*>(out));
}

}  // namespace moe
