// C ABI of the MoE expert-FFN library: argument checks, workspace layout and
// the launch sequences of each entry point (declared in include/moe_ffn.h).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/moe_ffn.h"
#include "internal.h"

namespace moe {


int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {
thread_local int g_launches = 0;
}  // namespace

void set_last_launch_count(int n) { g_launches = n; }

namespace {

// Stage names of moe_forward and moe_backward, in launch order.
constexpr int kFwdStages = 8;
constexpr int kBwdStages = 10;
constexpr int kMaxStages = 10;
const char* const kStageNames[kFwdStages] = {"route_topk", "chunk_histogram", "scan",
                                             "scatter",    "permute_rows",    "gemm1_swiglu",
                                             "gemm2",      "combine"};
const char* const kBwdStageNames[kBwdStages] = {
    "route_topk",    "permute", "permute_rows", "gemm1_recompute", "dgrad_h_swiglu",
    "wgrad_w2",      "dgrad_x", "wgrad_w1",    "combine_dx",      "router_backward"};

// Event ring for moe_stage_timing_begin/end (one row of kMaxStages+1 events
// per recorded call).  `kind` is the entry point last recorded (0 forward,
// 1 backward).
struct StageTimer {
  bool on = false;
  int capacity = 0;
  int used = 0;
  int kind = 0;
  cudaEvent_t* ev = nullptr;
  void mark(int call, int i, cudaStream_t s) {
    if (on && call < capacity) cudaEventRecord(ev[call * (kMaxStages + 1) + i], s);
  }
};
thread_local StageTimer g_timer;

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// Byte offsets of every scratch region inside the caller's workspace.
// The problem after routing: the S shared experts become experts E .. E+S-1
// that every token selects in slots k .. k+S-1.
moe_problem expanded(const moe_problem& p) {
  moe_problem q = p;
  q.E = p.E + p.shared_experts;
  q.k = p.k + p.shared_experts;
  q.shared_experts = 0;
  return q;
}

struct Layout {
  size_t status, chunk_counts, tokens_per_expert, expert_offsets, mtile_prefix, topk_idx, topk_w,
      row_id_map, permuted_token, counters, dec_counters, x_perm, h, y, total;
};

Layout layout_of(const moe_problem& p0) {
  const moe_problem p = expanded(p0);
  const size_t T = p.T, E = p.E, R = static_cast<size_t>(p.T) * p.k;
  const size_t nchunks = (T + kChunkTokens - 1) / kChunkTokens;
  Layout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.status = take(sizeof(uint32_t));
  L.chunk_counts = take(sizeof(int32_t) * nchunks * E);
  L.tokens_per_expert = take(sizeof(int32_t) * E);
  L.expert_offsets = take(sizeof(int32_t) * (E + 1));
  L.mtile_prefix = take(sizeof(int32_t) * (E + 1));
  L.topk_idx = take(sizeof(int32_t) * R);
  L.topk_w = take(sizeof(float) * R);
  L.row_id_map = take(sizeof(int32_t) * R);
  L.permuted_token = take(sizeof(int32_t) * R);
  L.counters = take(sizeof(int32_t) * T * (p.H > 0 ? (static_cast<size_t>(p.H) + kBN - 1) / kBN : 0));
  L.dec_counters = take(sizeof(int32_t) * static_cast<size_t>(decode_mlp_counters(p.T, p.E, p.H)));
  L.x_perm = take(2 * R * static_cast<size_t>(p.H));
  L.h = take(2 * R * static_cast<size_t>(p.F));
  L.y = take(2 * R * static_cast<size_t>(p.H));
  L.total = o;
  return L;
}

// The backward's workspace: the forward's regions (routing, x_perm; y holds
// the permuted output gradient, h the weighted activations w*h) plus the fp32
// pre-activations, their bf16 gradient, the routing weight of each permuted
// row and the per-(row, 256-column tile) partials of the router gradient.
struct BwdLayout {
  Layout f;
  size_t act, dact, w_perm, dw_part, total;
};

BwdLayout bwd_layout_of(const moe_problem& p0) {
  const moe_problem p = expanded(p0);
  const size_t R = static_cast<size_t>(p.T) * p.k, F = p.F;
  BwdLayout B;
  B.f = layout_of(p0);
  size_t o = B.f.total;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  B.act = take(sizeof(float) * R * 2 * F);
  B.dact = take(2 * R * 2 * F);
  B.w_perm = take(sizeof(float) * R);
  B.dw_part = take(sizeof(float) * R * bwd_router_parts(static_cast<int>(F)));
  B.total = o;
  return B;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

int check_routing(const moe_problem* p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->E < 1 || p->k < 1 || p->k > p->E) return MOE_ERR_INVALID_ARG;
  if (p->shared_experts < 0) return MOE_ERR_INVALID_ARG;
  const int S = p->shared_experts;
  if (p->E + S > MOE_MAX_EXPERTS || p->k + S > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(p->T) * (p->k + S) > (1LL << 30)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}


int check_full(const moe_problem* p) {
  int rc = check_routing(p);
  if (rc != MOE_OK) return rc;
  if (p->H <= 0 || p->F <= 0) return MOE_ERR_INVALID_ARG;
  if (p->precision != MOE_PREC_BF16 && p->precision != MOE_PREC_FP8_NVFP4)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (p->fusion & ~(MOE_FUSE_GATHER_A | MOE_FUSE_COMBINE)) return MOE_ERR_INVALID_ARG;
  if (p->kernel != MOE_KERNEL_AUTO && p->kernel != MOE_KERNEL_TOKEN_TILES &&
      p->kernel != MOE_KERNEL_WEIGHT_TILES && p->kernel != MOE_KERNEL_WEIGHT_TILES_2CTA &&
      p->kernel != MOE_KERNEL_DECODE_FUSED)
    return MOE_ERR_INVALID_ARG;
  // the FP8/NVFP4 GEMMs come in two tilings
  if (p->precision == MOE_PREC_FP8_NVFP4 && p->kernel != MOE_KERNEL_AUTO &&
      p->kernel != MOE_KERNEL_TOKEN_TILES && p->kernel != MOE_KERNEL_WEIGHT_TILES_2CTA)
    return MOE_ERR_INVALID_ARG;
  // hidden a multiple of 256, intermediate a multiple of 128 (the tile sizes)
  if (p->H % 256 != 0 || p->F % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int I = p->glu_interleave;
  if (I < 0) return MOE_ERR_INVALID_ARG;
  if (I != 0 && (p->F % I != 0 || !(I == 32 || I == 64 || I % 128 == 0)))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long R = static_cast<long long>(p->T) * p->k;
  if (R * p->H >= (1LL << 40) || static_cast<long long>(p->E) * 2 * p->F >= (1LL << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

int check_ws(const moe_problem* p, void* ws, size_t ws_bytes) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_MISALIGNED;
  if (ws_bytes < layout_of(*p).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

#define MOE_REQUIRE_PTR(ptr)                            \
  do {                                                  \
    if (!(ptr)) return MOE_ERR_INVALID_ARG;             \
    if (!aligned16(ptr)) return MOE_ERR_MISALIGNED;     \
  } while (0)

#define MOE_LAUNCH(expr)                          \
  do {                                            \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
    ++launches;                                   \
  } while (0)

// GEMM tiling for this problem.  With at most two routes per expert on
// average the 32-token weight-row tiles give the most CTAs streaming the
// weights; otherwise 2-CTA weight-row tiles, whose N fits each expert's rows
// (a ragged expert pads at most 31 rows) -- on GB300 they match or beat the
// token-row tilings even for experts with thousands of rows.
int gemm_tiling(const moe_problem* p) {
  // the one-launch decode MLP is moe_forward's; elsewhere its tiles run as two GEMMs
  if (p->kernel == MOE_KERNEL_DECODE_FUSED) return MOE_KERNEL_WEIGHT_TILES;
  if (p->kernel != MOE_KERNEL_AUTO) return p->kernel;
  const long long routes = static_cast<long long>(p->T) * p->k;
  if (routes <= 2LL * p->E) return MOE_KERNEL_WEIGHT_TILES;
  return MOE_KERNEL_WEIGHT_TILES_2CTA;
}

// FP8/NVFP4 tiling: 1-CTA token-row tiles unless the 2-CTA weight-row tiles
// are asked for (a cta_group::2 MMA costs the same for every N <= 256, so
// fitting N to ragged experts saves no tensor time; the token-row tiles are
// faster on GB300).
int lowprec_tiling(const moe_problem* p) {
  if (p->kernel == MOE_KERNEL_WEIGHT_TILES_2CTA) return p->kernel;
  return MOE_KERNEL_TOKEN_TILES;
}

// moe_forward at decode sizes: GEMM1, GEMM2 and the combine in one launch
// (grouped_mlp_decode.cu) below one route per expert on average.  From one
// to two routes per expert the two-GEMM 32-token weight tiles measured as
// fast or faster on GB300 (H=2048 F=768 E=128 top-8, CUDA-graph replay:
// T=16 150 us against 147 us, T=32 217 us against 203 us; below: T=1 37.1
// against 38.6 us, T=4 67.6 against 79.3 us, T=8 105.7 against 113.9 us).
bool use_decode_fused(const moe_problem* p) {
  if (p->kernel == MOE_KERNEL_DECODE_FUSED) return true;
  return p->kernel == MOE_KERNEL_AUTO && static_cast<long long>(p->T) * p->k < p->E;
}

bool use_weight_tiles(const moe_problem* p) { return gemm_tiling(p) == MOE_KERNEL_WEIGHT_TILES; }

float clamp_of(const moe_problem* p) {
  const float c = p->swiglu_clamp;
  return (c > 0.f && std::isfinite(c)) ? c : 0.f;
}

// GEMM1 (x_perm -> h with SwiGLU) then GEMM2 (h -> y).
// Fused form (moe_forward): fused != nullptr gathers GEMM1's A rows from x by
// permuted_token and runs the weighted combine in GEMM2's epilogue into out.
struct FusedIO {
  bool gather, combine;
  const int32_t* permuted_token;
  const int32_t* row_id_map;
  const float* topk_w;
  int32_t* counters;
  void* out;
};

int run_mlp(const moe_problem* p, const void* x_perm, const int32_t* offsets,
            const int32_t* mtp, const void* w1, const void* w2, void* h, void* y,
            uint32_t* status, cudaStream_t s, int& launches, StageTimer* tm = nullptr,
            int call = 0, int mark = 0, const FusedIO* fused = nullptr) {
  const int R = p->T * p->k;
  GroupedGemmArgs g1{};
  g1.epi = Epi::kSwiGLU;
  g1.a = x_perm;
  g1.a_rows = R;
  g1.b = w1;
  g1.b_rows_per_expert = 2 * p->F;
  g1.E = p->E;
  g1.K = p->H;
  g1.n_tiles = p->F / (kBN / 2);
  g1.expert_offsets = offsets;
  g1.mtile_prefix = mtp;
  g1.out = h;
  g1.ldo = p->F;
  g1.out_rows = R;
  g1.F = p->F;
  g1.interleave = p->glu_interleave;
  g1.clamp = clamp_of(p);
  g1.status = status;
  const bool swap = use_weight_tiles(p);
  if (fused && fused->gather && !swap) {
    g1.permuted_token = fused->permuted_token;
    g1.x_rows = p->T;
  }
  const bool swap2 = gemm_tiling(p) == MOE_KERNEL_WEIGHT_TILES_2CTA;
  if (swap2) g1.permuted_token = nullptr;  // no gathered-A form
  MOE_LAUNCH(swap    ? launch_grouped_gemm_swap(g1, s)
             : swap2 ? launch_grouped_gemm_swap2(g1, s)
                     : launch_grouped_gemm(g1, s));
  if (tm) tm->mark(call, mark, s);
  GroupedGemmArgs g2{};
  g2.epi = Epi::kPlain;
  g2.a = h;
  g2.a_rows = R;
  g2.b = w2;
  g2.b_rows_per_expert = p->H;
  g2.E = p->E;
  g2.K = p->F;
  g2.n_tiles = p->H / kBN;
  g2.expert_offsets = offsets;
  g2.mtile_prefix = mtp;
  g2.out = y;
  g2.ldo = p->H;
  g2.out_rows = R;
  g2.F = p->F;
  g2.status = status;
  if (fused && fused->combine && !swap && !swap2) {
    g2.epi = Epi::kCombine;
    g2.out = fused->out;
    g2.partials = y;
    g2.permuted_token = fused->permuted_token;
    g2.row_id_map = fused->row_id_map;
    g2.topk_w = fused->topk_w;
    g2.counters = fused->counters;
    g2.k = p->k;
  }
  MOE_LAUNCH(swap    ? launch_grouped_gemm_swap(g2, s)
             : swap2 ? launch_grouped_gemm_swap2(g2, s)
                     : launch_grouped_gemm(g2, s));
  if (tm) tm->mark(call, mark + 1, s);
  return MOE_OK;
}

// histogram -> scan -> scatter; fills row maps, counts and offsets.
int run_permute(const moe_problem* p, const int32_t* topk_idx, int32_t* row_id_map,
                int32_t* permuted_token, int32_t* tokens_per_expert, int32_t* expert_offsets,
                int32_t* mtp, void* ws, const Layout& L, cudaStream_t s, int& launches,
                StageTimer* tm = nullptr, int call = 0, int mark = 0,
                int32_t* counters = nullptr, int ncnt = 0) {
  const int R = p->T * p->k;
  const int nchunks = ceil_div(p->T, kChunkTokens);
  uint32_t* status = at<uint32_t>(ws, L.status);
  int32_t* cc = at<int32_t>(ws, L.chunk_counts);
  if (nchunks > 0)
    MOE_LAUNCH(launch_chunk_histogram(topk_idx, p->T, p->E, p->k, cc, status, s, counters, ncnt));
  if (tm) tm->mark(call, mark, s);
  MOE_LAUNCH(launch_scan(cc, nchunks, p->E, R, tokens_per_expert, expert_offsets, mtp,
                         permuted_token, s));
  if (tm) tm->mark(call, mark + 1, s);
  if (nchunks > 0)
    MOE_LAUNCH(launch_scatter(topk_idx, p->T, p->E, p->k, cc, row_id_map, permuted_token, s));
  if (tm) tm->mark(call, mark + 2, s);
  return MOE_OK;
}

// Checks shared by moe_backward and moe_backward_routed; a non-zero return is
// the status to give the caller.
int check_backward(const moe_problem* p, const void* w1, const void* w2, void* dw1, void* dw2,
                   void* ws, size_t ws_bytes) {
  int rc = check_full(p);
  if (rc != MOE_OK) return rc;
  if (p->precision != MOE_PREC_BF16) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_MISALIGNED;
  if (ws_bytes < bwd_layout_of(*p).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  MOE_REQUIRE_PTR(w1);
  MOE_REQUIRE_PTR(w2);
  MOE_REQUIRE_PTR(dw1);
  MOE_REQUIRE_PTR(dw2);
  return MOE_OK;
}

// No routes: the weight gradients are zero.
int backward_no_tokens(const moe_problem* q, void* dw1, void* dw2, cudaStream_t s) {
  int launches = 0;
  const size_t w1_bytes = sizeof(uint16_t) * q->E * 2 * static_cast<size_t>(q->F) * q->H;
  const size_t w2_bytes = sizeof(uint16_t) * q->E * static_cast<size_t>(q->H) * q->F;
  MOE_LAUNCH(cudaMemsetAsync(dw1, 0, w1_bytes, s));
  MOE_LAUNCH(cudaMemsetAsync(dw2, 0, w2_bytes, s));
  g_launches = launches;
  return MOE_OK;
}

// The backward after routing and permutation (routes in the workspace's
// row maps, weights in `wts` [T, q->k]): the row gathers, the pre-activation
// recompute, dH with the SwiGLU backward, dW2, dXp, dW1 and the dx sum.
// Leaves the per-row router partials in the workspace.
int run_backward_core(const moe_problem* p, const moe_problem* q, const BwdLayout& B,
                      const void* x, const void* d_out, const float* wts, const void* w1,
                      const void* w2, void* dx, void* dw1, void* dw2, void* ws, cudaStream_t s,
                      int& launches, StageTimer& tm, int call) {
  const Layout& L = B.f;
  const int R = q->T * q->k;
  const int H = q->H, F = q->F;
  int32_t* off = at<int32_t>(ws, L.expert_offsets);
  int32_t* mtp = at<int32_t>(ws, L.mtile_prefix);
  int32_t* rmap = at<int32_t>(ws, L.row_id_map);
  int32_t* ptok = at<int32_t>(ws, L.permuted_token);
  uint32_t* status = at<uint32_t>(ws, L.status);
  void* x_perm = at<void>(ws, L.x_perm);
  void* hw = at<void>(ws, L.h);      // [R, F] w * h
  void* dy = at<void>(ws, L.y);      // [R, H] permuted output gradient, later dXp
  float* act = at<float>(ws, B.act);  // [R, 2F] fp32 pre-activations
  void* dact = at<void>(ws, B.dact);  // [R, 2F] bf16 their gradient
  float* w_perm = at<float>(ws, B.w_perm);
  float* dw_part = at<float>(ws, B.dw_part);
  MOE_LAUNCH(launch_scatter_rows(x, rmap, off, q->T, q->k, q->E, H, x_perm, s));
  MOE_LAUNCH(launch_scatter_rows(d_out, rmap, off, q->T, q->k, q->E, H, dy, s));
  MOE_LAUNCH(launch_weights_to_rows(rmap, wts, R, w_perm, s));
  tm.mark(call, 3, s);
  // pre-activations a = x W1_e^T in fp32, recomputed rather than kept from
  // the forward
  BwdGemmArgs ga{};
  ga.mode = kBwdPreact;
  ga.a = x_perm;
  ga.b = w1;
  ga.R = R;
  ga.E = q->E;
  ga.K = H;
  ga.N = 2 * F;
  ga.expert_offsets = off;
  ga.mtile_prefix = mtp;
  ga.out = act;
  ga.status = status;
  MOE_LAUNCH(launch_grouped_gemm_bwd(ga, s));
  tm.mark(call, 4, s);
  // dh = dY W2_e, then the SwiGLU backward: dA, w*h, router partials
  BwdGemmArgs g{};
  g.mode = kBwdDataSwiGLU;
  g.a = dy;
  g.b = w2;
  g.R = R;
  g.E = q->E;
  g.K = H;
  g.N = F;
  g.expert_offsets = off;
  g.mtile_prefix = mtp;
  g.act = act;
  g.dact = dact;
  g.hw = hw;
  g.dw_part = dw_part;
  g.w_perm = w_perm;
  g.F = F;
  g.interleave = p->glu_interleave;
  g.clamp = clamp_of(p);
  g.status = status;
  MOE_LAUNCH(launch_grouped_gemm_bwd(g, s));
  tm.mark(call, 5, s);
  // dW2_e = dY_e^T (w h)_e
  BwdGemmArgs gw2{};
  gw2.mode = kBwdWeight;
  gw2.a = dy;
  gw2.b = hw;
  gw2.R = R;
  gw2.E = q->E;
  gw2.M = H;
  gw2.N = F;
  gw2.expert_offsets = off;
  gw2.out = dw2;
  gw2.status = status;
  MOE_LAUNCH(launch_grouped_gemm_bwd(gw2, s));
  tm.mark(call, 6, s);
  // dXp = dA W1_e (into dY's region, no longer needed)
  BwdGemmArgs gx{};
  gx.mode = kBwdDataPlain;
  gx.a = dact;
  gx.b = w1;
  gx.R = R;
  gx.E = q->E;
  gx.K = 2 * F;
  gx.N = H;
  gx.expert_offsets = off;
  gx.mtile_prefix = mtp;
  gx.out = dy;
  gx.status = status;
  MOE_LAUNCH(launch_grouped_gemm_bwd(gx, s));
  tm.mark(call, 7, s);
  // dW1_e = dA_e^T x_e
  BwdGemmArgs gw1{};
  gw1.mode = kBwdWeight;
  gw1.a = dact;
  gw1.b = x_perm;
  gw1.R = R;
  gw1.E = q->E;
  gw1.M = 2 * F;
  gw1.N = H;
  gw1.expert_offsets = off;
  gw1.out = dw1;
  gw1.status = status;
  MOE_LAUNCH(launch_grouped_gemm_bwd(gw1, s));
  tm.mark(call, 8, s);
  // dx_t = sum over the token's routes of dXp (weights already applied)
  MOE_LAUNCH(launch_combine(dy, rmap, nullptr, q->T, H, q->k, dx, s));
  return MOE_OK;
}

// GEMM1 + SwiGLU (+ the 1x128 E4M3 re-quantisation of h) and GEMM2 of the
// FP8-activation / NVFP4-weight layer on f16 rows x_perm (dequantised
// activations), into h (workspace) and y.
int run_mlp_lowprec(const moe_problem* p, const void* x_perm, const int32_t* off,
                    const int32_t* mtp, const void* w1q, const void* w2q,
                    const moe_fp4_scales& sc, void* h, void* y, uint32_t* status, cudaStream_t s,
                    int& launches, StageTimer* tm = nullptr, int call = 0, int mark = 0) {
  const int R = p->T * p->k;
  const uint8_t* sc1 = static_cast<const uint8_t*>(sc.prepared);
  const uint8_t* sc2 = sc1 + static_cast<size_t>(p->E) * 2 * p->F * p->H / 16;
  GroupedGemmArgs g1{};
  g1.epi = Epi::kSwiGLU;
  g1.a = x_perm;
  g1.a_rows = R;
  g1.b = w1q;
  g1.b_rows_per_expert = 2 * p->F;
  g1.E = p->E;
  g1.K = p->H;
  g1.n_tiles = p->F / (kBN / 2);
  g1.expert_offsets = off;
  g1.mtile_prefix = mtp;
  g1.out = h;
  g1.ldo = p->F;
  g1.out_rows = R;
  g1.F = p->F;
  g1.interleave = p->glu_interleave;
  g1.clamp = clamp_of(p);
  g1.status = status;
  const int lt = lowprec_tiling(p);
  MOE_LAUNCH(lt == MOE_KERNEL_WEIGHT_TILES_2CTA
                 ? launch_grouped_gemm_fp4_pair(g1, sc1, sc.w1_gscale, s)
                 : launch_grouped_gemm_fp4(g1, sc1, sc.w1_gscale, s));
  if (tm) tm->mark(call, mark, s);
  GroupedGemmArgs g2{};
  g2.epi = Epi::kPlain;
  g2.a = h;
  g2.a_rows = R;
  g2.b = w2q;
  g2.b_rows_per_expert = p->H;
  g2.E = p->E;
  g2.K = p->F;
  g2.n_tiles = p->H / kBN;
  g2.expert_offsets = off;
  g2.mtile_prefix = mtp;
  g2.out = y;
  g2.ldo = p->H;
  g2.out_rows = R;
  g2.F = p->F;
  g2.status = status;
  MOE_LAUNCH(lt == MOE_KERNEL_WEIGHT_TILES_2CTA
                 ? launch_grouped_gemm_fp4_pair(g2, sc2, sc.w2_gscale, s)
                 : launch_grouped_gemm_fp4(g2, sc2, sc.w2_gscale, s));
  if (tm) tm->mark(call, mark + 1, s);
  return MOE_OK;
}

// Validation of the FP4 weight scales struct (host) and its device pointers.
int check_fp4_scales(const void* wscales) {
  if (!wscales) return MOE_ERR_INVALID_ARG;
  const moe_fp4_scales* sc = static_cast<const moe_fp4_scales*>(wscales);
  MOE_REQUIRE_PTR(sc->prepared);
  MOE_REQUIRE_PTR(sc->w1_gscale);
  MOE_REQUIRE_PTR(sc->w2_gscale);
  return MOE_OK;
}

// The FP8-activation / NVFP4-weight layer (moe_forward at that precision and
// moe_forward_fp8_nvfp4).
int forward_lowprec(const moe_problem* p, const void* xq_v, const float* xs, const float* logits,
                    const void* w1q, const void* w2q, const moe_fp4_scales* scp, void* out,
                    int32_t* topk_idx_out, float* topk_w_out, int32_t* tokens_per_expert_out,
                    void* ws, size_t ws_bytes, cudaStream_t s) {
  const uint8_t* xq = static_cast<const uint8_t*>(xq_v);
  int rc = check_full(p);
  if (rc != MOE_OK) return rc;
  if (p->shared_experts != 0) return MOE_ERR_INVALID_ARG;  // bf16 moe_forward only
  if (p->precision != MOE_PREC_FP8_NVFP4) return MOE_ERR_INVALID_ARG;
  rc = check_ws(p, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  MOE_REQUIRE_PTR(w1q);
  MOE_REQUIRE_PTR(w2q);
  rc = check_fp4_scales(scp);
  if (rc != MOE_OK) return rc;
  const moe_fp4_scales& sc = *scp;
  if (topk_idx_out && !aligned16(topk_idx_out)) return MOE_ERR_MISALIGNED;
  if (topk_w_out && !aligned16(topk_w_out)) return MOE_ERR_MISALIGNED;
  if (tokens_per_expert_out && !aligned16(tokens_per_expert_out)) return MOE_ERR_MISALIGNED;
  const Layout L = layout_of(*p);
  int launches = 0;
  int32_t* tpe = tokens_per_expert_out ? tokens_per_expert_out
                                       : at<int32_t>(ws, L.tokens_per_expert);
  if (p->T == 0) {
    if (tokens_per_expert_out)
      MOE_LAUNCH(cudaMemsetAsync(tokens_per_expert_out, 0, sizeof(int32_t) * p->E, s));
    g_launches = launches;
    return MOE_OK;
  }
  MOE_REQUIRE_PTR(xq);
  MOE_REQUIRE_PTR(xs);
  MOE_REQUIRE_PTR(logits);
  MOE_REQUIRE_PTR(out);
  const int R = p->T * p->k;
  int32_t* idx = topk_idx_out ? topk_idx_out : at<int32_t>(ws, L.topk_idx);
  float* wts = topk_w_out ? topk_w_out : at<float>(ws, L.topk_w);
  int32_t* off = at<int32_t>(ws, L.expert_offsets);
  int32_t* mtp = at<int32_t>(ws, L.mtile_prefix);
  int32_t* rmap = at<int32_t>(ws, L.row_id_map);
  int32_t* ptok = at<int32_t>(ws, L.permuted_token);
  uint32_t* status = at<uint32_t>(ws, L.status);
  void* x_perm = at<void>(ws, L.x_perm);
  void* h = at<void>(ws, L.h);
  void* y = at<void>(ws, L.y);

  const int call = g_timer.on ? g_timer.used++ : 0;
  StageTimer& tm = g_timer;
  if (tm.on) tm.kind = 0;
  tm.mark(call, 0, s);
  if (route_permute_tiny_fits(p->T, p->E, p->k, 0)) {
    MOE_LAUNCH(launch_route_permute_tiny(logits, p->T, p->E, p->k, 0, p->renormalize ? 1 : 0, idx,
                                         wts, tpe, off, mtp, rmap, ptok, nullptr, p->H, nullptr,
                                         s));
    for (int i = 1; i <= 4; ++i) tm.mark(call, i, s);
  } else {
    MOE_LAUNCH(launch_route_topk(logits, p->T, p->E, p->k, p->renormalize ? 1 : 0, idx, wts, s));
    tm.mark(call, 1, s);
    if (permute_small_fits(p->T, p->E, p->k)) {
      MOE_LAUNCH(launch_permute_small(idx, p->T, p->E, p->k, tpe, off, mtp, rmap, ptok, s));
      for (int i = 2; i <= 4; ++i) tm.mark(call, i, s);
    } else {
      rc = run_permute(p, idx, rmap, ptok, tpe, off, mtp, ws, L, s, launches, &tm, call, 2);
      if (rc != MOE_OK) return rc;
    }
  }
  MOE_LAUNCH(launch_gather_dequant_fp8(xq, xs, ptok, R, p->H, x_perm, s));
  tm.mark(call, 5, s);
  rc = run_mlp_lowprec(p, x_perm, off, mtp, w1q, w2q, sc, h, y, status, s, launches, &tm, call, 6);
  if (rc != MOE_OK) return rc;
  MOE_LAUNCH(launch_combine(y, rmap, wts, p->T, p->H, p->k, out, s));
  tm.mark(call, 8, s);
  g_launches = launches;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_DEVICE_INDEX: return "MOE_ERR_DEVICE_INDEX";
    default: return "MOE_ERR_UNKNOWN";
  }
}

size_t moe_workspace_size(const moe_problem* p) {
  if (check_full(p) != MOE_OK && check_routing(p) != MOE_OK) return 0;
  moe_problem q = *p;
  if (q.H < 0) q.H = 0;
  if (q.F < 0) q.F = 0;
  return layout_of(q).total;
}

int moe_route_topk(const moe_problem* p, const float* logits, int32_t* topk_idx, float* topk_w,
                   void* ws, size_t ws_bytes, void* stream) {
  (void)ws;
  (void)ws_bytes;
  int rc = check_routing(p);
  if (rc != MOE_OK) return rc;
  if (p->shared_experts != 0) return MOE_ERR_INVALID_ARG;  // moe_forward only
  if (p->T == 0) { g_launches = 0; return MOE_OK; }
  MOE_REQUIRE_PTR(logits);
  MOE_REQUIRE_PTR(topk_idx);
  MOE_REQUIRE_PTR(topk_w);
  int launches = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_LAUNCH(launch_route_topk(logits, p->T, p->E, p->k, p->renormalize ? 1 : 0, topk_idx,
                               topk_w, s));
  g_launches = launches;
  return MOE_OK;
}

int moe_permute(const moe_problem* p, const int32_t* topk_idx, const void* x, void* x_perm,
                int32_t* row_id_map, int32_t* permuted_token, int32_t* tokens_per_expert,
                int32_t* expert_offsets, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_routing(p);
  if (rc != MOE_OK) return rc;
  if (p->shared_experts != 0) return MOE_ERR_INVALID_ARG;  // moe_forward only
  if (x_perm) {
    if (p->H <= 0 || p->H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    MOE_REQUIRE_PTR(x);
    MOE_REQUIRE_PTR(x_perm);
  }
  MOE_REQUIRE_PTR(tokens_per_expert);
  MOE_REQUIRE_PTR(expert_offsets);
  if (p->T > 0) {
    MOE_REQUIRE_PTR(topk_idx);
    MOE_REQUIRE_PTR(row_id_map);
    MOE_REQUIRE_PTR(permuted_token);
  }
  moe_problem q = *p;  // permute uses only the routing regions of the workspace
  q.H = 0;
  q.F = 0;
  rc = check_ws(&q, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  const Layout L = layout_of(q);
  int launches = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = run_permute(p, topk_idx, row_id_map, permuted_token, tokens_per_expert, expert_offsets,
                   at<int32_t>(ws, L.mtile_prefix), ws, L, s, launches);
  if (rc != MOE_OK) return rc;
  if (x_perm && p->T > 0)
    MOE_LAUNCH(launch_scatter_rows(x, row_id_map, expert_offsets, p->T, p->k, p->E, p->H, x_perm,
                                   s));
  g_launches = launches;
  return MOE_OK;
}

int moe_grouped_swiglu_mlp(const moe_problem* p, const void* x_perm, const float* x_perm_scale,
                           const int32_t* expert_offsets, const void* w1, const void* w2,
                           const void* wscales, void* y_perm, void* ws, size_t ws_bytes,
                           void* stream) {
  int rc = check_full(p);
  if (rc != MOE_OK) return rc;
  if (p->shared_experts != 0) return MOE_ERR_INVALID_ARG;  // moe_forward only
  const bool lowprec = p->precision == MOE_PREC_FP8_NVFP4;
  if (lowprec) {
    rc = check_fp4_scales(wscales);
    if (rc != MOE_OK) return rc;
  } else if (x_perm_scale || wscales) {
    return MOE_ERR_INVALID_ARG;  // bf16 rows carry no scales
  }
  rc = check_ws(p, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  MOE_REQUIRE_PTR(expert_offsets);
  MOE_REQUIRE_PTR(w1);
  MOE_REQUIRE_PTR(w2);
  if (p->T == 0) { g_launches = 0; return MOE_OK; }
  MOE_REQUIRE_PTR(x_perm);
  MOE_REQUIRE_PTR(y_perm);
  if (lowprec) MOE_REQUIRE_PTR(x_perm_scale);
  const Layout L = layout_of(*p);
  int launches = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* status = at<uint32_t>(ws, L.status);
  int32_t* mtp = at<int32_t>(ws, L.mtile_prefix);
  const int R = p->T * p->k;
  MOE_LAUNCH(launch_mtile_prefix_from_offsets(expert_offsets, p->E, R, mtp, status, s));
  if (lowprec) {
    // the E4M3 rows with their per-128 scales -> f16 rows in the workspace
    // (in place: row r from row r), then the FP4 GEMMs
    void* xf = at<void>(ws, L.x_perm);
    MOE_LAUNCH(launch_gather_dequant_fp8(static_cast<const uint8_t*>(x_perm), x_perm_scale,
                                         nullptr, R, p->H, xf, s));
    rc = run_mlp_lowprec(p, xf, expert_offsets, mtp, w1, w2,
                         *static_cast<const moe_fp4_scales*>(wscales), at<void>(ws, L.h), y_perm,
                         status, s, launches);
  } else {
    rc = run_mlp(p, x_perm, expert_offsets, mtp, w1, w2, at<void>(ws, L.h), y_perm, status, s,
                 launches);
  }
  if (rc != MOE_OK) return rc;
  g_launches = launches;
  return MOE_OK;
}

int moe_permute_rows(const moe_problem* p, const int32_t* permuted_token, const void* src,
                     int32_t row_bytes, void* dst, void* stream) {
  int rc = check_routing(p);
  if (rc != MOE_OK) return rc;
  if (p->shared_experts != 0) return MOE_ERR_INVALID_ARG;  // moe_forward only
  if (row_bytes <= 0 || row_bytes % 4 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (p->T == 0) { g_launches = 0; return MOE_OK; }
  MOE_REQUIRE_PTR(permuted_token);
  MOE_REQUIRE_PTR(src);
  MOE_REQUIRE_PTR(dst);
  int launches = 0;
  MOE_LAUNCH(launch_gather_row_bytes(src, permuted_token, p->T * p->k, p->T, row_bytes, dst,
                                     static_cast<cudaStream_t>(stream)));
  g_launches = launches;
  return MOE_OK;
}

int moe_unpermute_combine(const moe_problem* p, const void* y_perm, const int32_t* row_id_map,
                          const float* topk_w, void* out, void* stream) {
  int rc = check_routing(p);
  if (rc != MOE_OK) return rc;
  if (p->shared_experts != 0) return MOE_ERR_INVALID_ARG;  // moe_forward only
  if (p->H <= 0 || p->H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (p->T == 0) { g_launches = 0; return MOE_OK; }
  MOE_REQUIRE_PTR(y_perm);
  MOE_REQUIRE_PTR(row_id_map);
  MOE_REQUIRE_PTR(topk_w);
  MOE_REQUIRE_PTR(out);
  int launches = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_LAUNCH(launch_combine(y_perm, row_id_map, topk_w, p->T, p->H, p->k, out, s));
  g_launches = launches;
  return MOE_OK;
}

int moe_forward(const moe_problem* p, const void* x, const float* x_scale, const float* logits,
                const void* w1, const void* w2, const void* wscales, void* out,
                int32_t* topk_idx_out, float* topk_w_out, int32_t* tokens_per_expert_out,
                void* ws, size_t ws_bytes, void* stream) {
  int rc = check_full(p);
  if (rc != MOE_OK) return rc;
  if (p->precision == MOE_PREC_FP8_NVFP4)
    return forward_lowprec(p, x, x_scale, logits, w1, w2,
                           static_cast<const moe_fp4_scales*>(wscales), out, topk_idx_out,
                           topk_w_out, tokens_per_expert_out, ws, ws_bytes,
                           static_cast<cudaStream_t>(stream));
  if (p->precision != MOE_PREC_BF16) return MOE_ERR_INVALID_ARG;
  if (x_scale || wscales) return MOE_ERR_INVALID_ARG;  // bf16 rows carry no scales
  rc = check_ws(p, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  MOE_REQUIRE_PTR(w1);
  MOE_REQUIRE_PTR(w2);
  if (topk_idx_out && !aligned16(topk_idx_out)) return MOE_ERR_MISALIGNED;
  if (topk_w_out && !aligned16(topk_w_out)) return MOE_ERR_MISALIGNED;
  if (tokens_per_expert_out && !aligned16(tokens_per_expert_out)) return MOE_ERR_MISALIGNED;
  const Layout L = layout_of(*p);
  const moe_problem pe = expanded(*p);  // after routing: E+S experts, k+S slots
  const moe_problem* q = &pe;
  const int S = p->shared_experts;
  int launches = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* tpe = tokens_per_expert_out ? tokens_per_expert_out
                                       : at<int32_t>(ws, L.tokens_per_expert);
  if (p->T == 0) {
    if (tokens_per_expert_out)
      MOE_LAUNCH(cudaMemsetAsync(tokens_per_expert_out, 0, sizeof(int32_t) * q->E, s));
    g_launches = launches;
    return MOE_OK;
  }
  MOE_REQUIRE_PTR(x);
  MOE_REQUIRE_PTR(logits);
  MOE_REQUIRE_PTR(out);
  const int R = q->T * q->k;
  int32_t* idx = topk_idx_out ? topk_idx_out : at<int32_t>(ws, L.topk_idx);
  float* wts = topk_w_out ? topk_w_out : at<float>(ws, L.topk_w);
  int32_t* off = at<int32_t>(ws, L.expert_offsets);
  int32_t* mtp = at<int32_t>(ws, L.mtile_prefix);
  int32_t* rmap = at<int32_t>(ws, L.row_id_map);
  int32_t* ptok = at<int32_t>(ws, L.permuted_token);
  uint32_t* status = at<uint32_t>(ws, L.status);
  void* x_perm = at<void>(ws, L.x_perm);
  void* h = at<void>(ws, L.h);
  void* y = at<void>(ws, L.y);
  int32_t* counters = at<int32_t>(ws, L.counters);
  const bool plain_tiles = use_weight_tiles(q) || gemm_tiling(q) == MOE_KERNEL_WEIGHT_TILES_2CTA;
  const bool fuse_gather = !plain_tiles && (p->fusion & MOE_FUSE_GATHER_A) != 0;
  const bool fuse_combine = !plain_tiles && (p->fusion & MOE_FUSE_COMBINE) != 0;
  const bool decode_fused = use_decode_fused(q);
  int32_t* dctr = decode_fused ? at<int32_t>(ws, L.dec_counters) : nullptr;
  const int n_dctr = decode_fused ? decode_mlp_counters(q->T, q->E, q->H) : 0;

  const int call = g_timer.on ? g_timer.used++ : 0;
  StageTimer& tm = g_timer;
  if (tm.on) tm.kind = 0;
  tm.mark(call, 0, s);
  if (!fuse_combine && route_permute_tiny_fits(p->T, p->E, p->k, S)) {
    // the smallest decode steps: routing, permutation and (few rows) the
    // gather in one block
    // (the one-launch decode MLP gathers its rows itself)
    const bool gather_here = !fuse_gather && !decode_fused && R <= kTinyGatherRoutes;
    MOE_LAUNCH(launch_route_permute_tiny(logits, p->T, p->E, p->k, S, p->renormalize ? 1 : 0, idx,
                                         wts, tpe, off, mtp, rmap, ptok,
                                         gather_here ? x : nullptr, p->H, x_perm, s, dctr,
                                         n_dctr));
    for (int i = 1; i <= 4; ++i) tm.mark(call, i, s);
    if (!fuse_gather && !decode_fused && !gather_here)
      MOE_LAUNCH(launch_gather_rows(x, ptok, R, p->H, x_perm, s));
  } else {
    MOE_LAUNCH(
        launch_route_topk(logits, p->T, p->E, p->k, p->renormalize ? 1 : 0, idx, wts, s, S));
    tm.mark(call, 1, s);
    if (!fuse_combine && permute_small_fits(q->T, q->E, q->k)) {
      // decode sizes: histogram + scan + scatter in one block
      MOE_LAUNCH(launch_permute_small(idx, q->T, q->E, q->k, tpe, off, mtp, rmap, ptok, s,
                                      dctr, n_dctr));
      for (int i = 2; i <= 4; ++i) tm.mark(call, i, s);
    } else {
      rc = run_permute(q, idx, rmap, ptok, tpe, off, mtp, ws, L, s, launches, &tm, call, 2,
                       fuse_combine ? counters : nullptr, p->H / kBN);
      if (rc != MOE_OK) return rc;
      if (decode_fused)
        MOE_LAUNCH(cudaMemsetAsync(dctr, 0, sizeof(int32_t) * static_cast<size_t>(n_dctr), s));
    }
    if (!fuse_gather && !decode_fused)
      MOE_LAUNCH(launch_scatter_rows(x, rmap, off, q->T, q->k, q->E, q->H, x_perm, s));
  }
  tm.mark(call, 5, s);
  if (decode_fused) {
    // GEMM1, GEMM2 and the combine in one launch (timed as the GEMM1 stage)
    DecodeMlpArgs a{};
    a.x = x;
    a.w1 = w1;
    a.w2 = w2;
    a.expert_offsets = off;
    a.h = h;
    a.y = y;
    a.out = out;
    a.permuted_token = ptok;
    a.row_id_map = rmap;
    a.topk_w = wts;
    a.counters = dctr;
    a.R = R;
    a.T = q->T;
    a.E = q->E;
    a.H = q->H;
    a.F = q->F;
    a.k = q->k;
    a.interleave = q->glu_interleave;
    a.clamp = clamp_of(q);
    a.status = status;
    MOE_LAUNCH(launch_grouped_mlp_decode(a, s));
    for (int i = 6; i <= 8; ++i) tm.mark(call, i, s);
    g_launches = launches;
    return MOE_OK;
  }
  const FusedIO fused{fuse_gather, fuse_combine, ptok, rmap, wts, counters, out};
  rc = run_mlp(q, fuse_gather ? x : x_perm, off, mtp, w1, w2, h, y, status, s, launches, &tm,
               call, 6, &fused);
  if (rc != MOE_OK) return rc;
  if (!fuse_combine) MOE_LAUNCH(launch_combine(y, rmap, wts, q->T, q->H, q->k, out, s));
  tm.mark(call, 8, s);
  g_launches = launches;
  return MOE_OK;
}

int moe_forward_routed(const moe_problem* p, const void* x, const int32_t* topk_idx,
                       const float* topk_w, const void* w1, const void* w2, void* out,
                       int32_t* tokens_per_expert_out, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_full(p);
  if (rc != MOE_OK) return rc;
  if (p->shared_experts != 0) return MOE_ERR_INVALID_ARG;  // moe_forward only
  if (p->precision != MOE_PREC_BF16) return MOE_ERR_INVALID_ARG;
  rc = check_ws(p, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  MOE_REQUIRE_PTR(w1);
  MOE_REQUIRE_PTR(w2);
  if (tokens_per_expert_out && !aligned16(tokens_per_expert_out)) return MOE_ERR_MISALIGNED;
  const Layout L = layout_of(*p);
  int launches = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* tpe = tokens_per_expert_out ? tokens_per_expert_out
                                       : at<int32_t>(ws, L.tokens_per_expert);
  if (p->T == 0) {
    if (tokens_per_expert_out)
      MOE_LAUNCH(cudaMemsetAsync(tokens_per_expert_out, 0, sizeof(int32_t) * p->E, s));
    g_launches = launches;
    return MOE_OK;
  }
  MOE_REQUIRE_PTR(x);
  MOE_REQUIRE_PTR(topk_idx);
  MOE_REQUIRE_PTR(topk_w);
  MOE_REQUIRE_PTR(out);
  int32_t* off = at<int32_t>(ws, L.expert_offsets);
  int32_t* mtp = at<int32_t>(ws, L.mtile_prefix);
  int32_t* rmap = at<int32_t>(ws, L.row_id_map);
  int32_t* ptok = at<int32_t>(ws, L.permuted_token);
  uint32_t* status = at<uint32_t>(ws, L.status);
  void* x_perm = at<void>(ws, L.x_perm);
  void* h = at<void>(ws, L.h);
  void* y = at<void>(ws, L.y);
  // the validating permutation: masked, out-of-range and repeated routes
  rc = run_permute(p, topk_idx, rmap, ptok, tpe, off, mtp, ws, L, s, launches);
  if (rc != MOE_OK) return rc;
  MOE_LAUNCH(launch_scatter_rows(x, rmap, off, p->T, p->k, p->E, p->H, x_perm, s));
  rc = run_mlp(p, x_perm, off, mtp, w1, w2, h, y, status, s, launches);
  if (rc != MOE_OK) return rc;
  MOE_LAUNCH(launch_combine(y, rmap, topk_w, p->T, p->H, p->k, out, s));
  g_launches = launches;
  return MOE_OK;
}

size_t moe_backward_workspace_size(const moe_problem* p) {
  if (check_full(p) != MOE_OK || p->precision != MOE_PREC_BF16) return 0;
  return bwd_layout_of(*p).total;
}

int moe_backward(const moe_problem* p, const void* x, const float* logits, const void* w1,
                 const void* w2, const void* d_out, void* dx, float* d_logits, void* dw1,
                 void* dw2, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_backward(p, w1, w2, dw1, dw2, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  if (d_logits && !aligned16(d_logits)) return MOE_ERR_MISALIGNED;
  const BwdLayout B = bwd_layout_of(*p);
  const Layout& L = B.f;
  const moe_problem pe = expanded(*p);  // after routing: E+S experts, k+S slots
  const moe_problem* q = &pe;
  const int S = p->shared_experts;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->T == 0) return backward_no_tokens(q, dw1, dw2, s);
  MOE_REQUIRE_PTR(x);
  MOE_REQUIRE_PTR(logits);
  MOE_REQUIRE_PTR(d_out);
  MOE_REQUIRE_PTR(dx);
  int launches = 0;
  int32_t* idx = at<int32_t>(ws, L.topk_idx);
  float* wts = at<float>(ws, L.topk_w);
  int32_t* tpe = at<int32_t>(ws, L.tokens_per_expert);
  int32_t* off = at<int32_t>(ws, L.expert_offsets);
  int32_t* mtp = at<int32_t>(ws, L.mtile_prefix);
  int32_t* rmap = at<int32_t>(ws, L.row_id_map);
  int32_t* ptok = at<int32_t>(ws, L.permuted_token);

  const int call = g_timer.on ? g_timer.used++ : 0;
  StageTimer& tm = g_timer;
  if (tm.on) tm.kind = 1;
  tm.mark(call, 0, s);
  // the forward's routing and permutation
  MOE_LAUNCH(launch_route_topk(logits, p->T, p->E, p->k, p->renormalize ? 1 : 0, idx, wts, s, S));
  tm.mark(call, 1, s);
  if (permute_small_fits(q->T, q->E, q->k)) {
    MOE_LAUNCH(launch_permute_small(idx, q->T, q->E, q->k, tpe, off, mtp, rmap, ptok, s));
  } else {
    rc = run_permute(q, idx, rmap, ptok, tpe, off, mtp, ws, L, s, launches);
    if (rc != MOE_OK) return rc;
  }
  tm.mark(call, 2, s);
  rc = run_backward_core(p, q, B, x, d_out, wts, w1, w2, dx, dw1, dw2, ws, s, launches, tm, call);
  if (rc != MOE_OK) return rc;
  tm.mark(call, 9, s);
  if (d_logits)
    MOE_LAUNCH(launch_router_backward(logits, idx, wts, rmap, at<float>(ws, B.dw_part),
                                      bwd_router_parts(q->F), p->T, p->E, p->k, q->k,
                                      p->renormalize ? 1 : 0, d_logits, s));
  tm.mark(call, 10, s);
  g_launches = launches;
  return MOE_OK;
}

int moe_backward_routed(const moe_problem* p, const void* x, const int32_t* topk_idx,
                        const float* topk_w, const void* w1, const void* w2, const void* d_out,
                        void* dx, float* d_topk_w, void* dw1, void* dw2, void* ws,
                        size_t ws_bytes, void* stream) {
  int rc = check_backward(p, w1, w2, dw1, dw2, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  if (p->shared_experts != 0) return MOE_ERR_INVALID_ARG;  // moe_backward only
  if (d_topk_w && !aligned16(d_topk_w)) return MOE_ERR_MISALIGNED;
  const BwdLayout B = bwd_layout_of(*p);
  const Layout& L = B.f;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->T == 0) return backward_no_tokens(p, dw1, dw2, s);
  MOE_REQUIRE_PTR(x);
  MOE_REQUIRE_PTR(topk_idx);
  MOE_REQUIRE_PTR(topk_w);
  MOE_REQUIRE_PTR(d_out);
  MOE_REQUIRE_PTR(dx);
  int launches = 0;
  int32_t* tpe = at<int32_t>(ws, L.tokens_per_expert);
  int32_t* off = at<int32_t>(ws, L.expert_offsets);
  int32_t* mtp = at<int32_t>(ws, L.mtile_prefix);
  int32_t* rmap = at<int32_t>(ws, L.row_id_map);
  int32_t* ptok = at<int32_t>(ws, L.permuted_token);
  const int call = g_timer.on ? g_timer.used++ : 0;
  StageTimer& tm = g_timer;
  if (tm.on) tm.kind = 1;
  tm.mark(call, 0, s);
  tm.mark(call, 1, s);
  // the validating permutation: masked, out-of-range and repeated routes
  rc = run_permute(p, topk_idx, rmap, ptok, tpe, off, mtp, ws, L, s, launches);
  if (rc != MOE_OK) return rc;
  tm.mark(call, 2, s);
  rc = run_backward_core(p, p, B, x, d_out, topk_w, w1, w2, dx, dw1, dw2, ws, s, launches, tm,
                         call);
  if (rc != MOE_OK) return rc;
  tm.mark(call, 9, s);
  if (d_topk_w)
    MOE_LAUNCH(launch_route_weight_grad(rmap, at<float>(ws, B.dw_part),
                                        bwd_router_parts(p->F),
                                        static_cast<long>(p->T) * p->k, d_topk_w, s));
  tm.mark(call, 10, s);
  g_launches = launches;
  return MOE_OK;
}

size_t moe_prepared_scales_size(const moe_problem* p) {
  if (check_full(p) != MOE_OK) return 0;
  return static_cast<size_t>(p->E) * (2 * static_cast<size_t>(p->F) * p->H / 16 +
                                      static_cast<size_t>(p->H) * p->F / 16);
}

int moe_prepare_weights(const moe_problem* p, const uint8_t* w1_scale, const uint8_t* w2_scale,
                        void* prepared, size_t prepared_bytes, void* stream) {
  int rc = check_full(p);
  if (rc != MOE_OK) return rc;
  if (p->shared_experts != 0) return MOE_ERR_INVALID_ARG;  // moe_forward only
  if (p->precision != MOE_PREC_FP8_NVFP4) return MOE_ERR_INVALID_ARG;
  MOE_REQUIRE_PTR(w1_scale);
  MOE_REQUIRE_PTR(w2_scale);
  MOE_REQUIRE_PTR(prepared);
  if (prepared_bytes < moe_prepared_scales_size(p)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  int launches = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* dst = static_cast<uint8_t*>(prepared);
  MOE_LAUNCH(launch_prepare_scales(w1_scale, dst, p->E, 2 * p->F, p->H, s));
  MOE_LAUNCH(launch_prepare_scales(w2_scale, dst + static_cast<size_t>(p->E) * 2 * p->F * p->H / 16,
                                   p->E, p->H, p->F, s));
  g_launches = launches;
  return MOE_OK;
}

int moe_prepare_weights_mxfp4(const moe_problem* p, const uint8_t* w1_scale,
                              const uint8_t* w2_scale, void* prepared, size_t prepared_bytes,
                              float* w1_gscale_out, float* w2_gscale_out, void* stream) {
  int rc = check_full(p);
  if (rc != MOE_OK) return rc;
  if (p->shared_experts != 0) return MOE_ERR_INVALID_ARG;  // moe_forward only
  if (p->precision != MOE_PREC_FP8_NVFP4) return MOE_ERR_INVALID_ARG;
  MOE_REQUIRE_PTR(w1_scale);
  MOE_REQUIRE_PTR(w2_scale);
  MOE_REQUIRE_PTR(prepared);
  MOE_REQUIRE_PTR(w1_gscale_out);
  MOE_REQUIRE_PTR(w2_gscale_out);
  if (prepared_bytes < moe_prepared_scales_size(p)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  int launches = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* dst = static_cast<uint8_t*>(prepared);
  MOE_LAUNCH(launch_prepare_mxfp4_scales(
      w1_scale, w2_scale, dst, dst + static_cast<size_t>(p->E) * 2 * p->F * p->H / 16, p->E,
      p->F, p->H, w1_gscale_out, w2_gscale_out, s));
  g_launches = launches;
  return MOE_OK;
}

int moe_forward_fp8_nvfp4(const moe_problem* p, const uint8_t* xq, const float* xs,
                          const float* logits, const uint8_t* w1q, const float* w1_gscale,
                          const uint8_t* w2q, const float* w2_gscale, const void* prepared_scales,
                          void* out, int32_t* topk_idx_out, float* topk_w_out,
                          int32_t* tokens_per_expert_out, void* ws, size_t ws_bytes,
                          void* stream) {
  const moe_fp4_scales sc{prepared_scales, w1_gscale, w2_gscale};
  return forward_lowprec(p, xq, xs, logits, w1q, w2q, &sc, out, topk_idx_out, topk_w_out,
                         tokens_per_expert_out, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

int moe_get_device_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (word & (1u << MOE_ERR_DEVICE_TIMEOUT)) return MOE_ERR_DEVICE_TIMEOUT;
  if (word & (1u << MOE_ERR_DEVICE_INDEX)) return MOE_ERR_DEVICE_INDEX;
  return MOE_OK;
}

int moe_clear_device_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_last_launch_count(void) { return g_launches; }

int moe_selected_kernel(const moe_problem* p) {
  if (check_full(p) != MOE_OK) return -1;
  if (p->precision == MOE_PREC_FP8_NVFP4) return lowprec_tiling(p);
  const moe_problem q = expanded(*p);
  return use_decode_fused(&q) ? MOE_KERNEL_DECODE_FUSED : gemm_tiling(&q);
}

int moe_stage_timing_begin(int n_calls) {
  if (n_calls <= 0) return MOE_ERR_INVALID_ARG;
  StageTimer& t = g_timer;
  if (n_calls > t.capacity) {
    if (t.ev) {
      for (int i = 0; i < t.capacity * (kMaxStages + 1); ++i) cudaEventDestroy(t.ev[i]);
      delete[] t.ev;
    }
    t.ev = new cudaEvent_t[n_calls * (kMaxStages + 1)];
    for (int i = 0; i < n_calls * (kMaxStages + 1); ++i)
      if (cudaEventCreate(&t.ev[i]) != cudaSuccess) return MOE_ERR_CUDA;
    t.capacity = n_calls;
  }
  t.used = 0;
  t.on = true;
  return MOE_OK;
}

int moe_stage_timing_end(float* ms, int max_stages, int* n_stages, int* n_calls) {
  StageTimer& t = g_timer;
  t.on = false;
  const int calls = t.used < t.capacity ? t.used : t.capacity;
  if (n_calls) *n_calls = calls;
  const int nst = t.kind ? kBwdStages : kFwdStages;
  if (n_stages) *n_stages = nst;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  for (int i = 0; i < nst && i < max_stages; ++i) {
    double acc = 0.0;
    for (int c = 0; c < calls; ++c) {
      float v = 0.f;
      if (cudaEventElapsedTime(&v, t.ev[c * (kMaxStages + 1) + i],
                               t.ev[c * (kMaxStages + 1) + i + 1]) != cudaSuccess)
        return MOE_ERR_CUDA;
      acc += v;
    }
    if (ms) ms[i] = calls ? static_cast<float>(acc / calls) : 0.f;
  }
  return MOE_OK;
}

const char* moe_stage_name(int i) {
  if (g_timer.kind) return (i >= 0 && i < kBwdStages) ? kBwdStageNames[i] : "";
  return (i >= 0 && i < kFwdStages) ? kStageNames[i] : "";
}

}  // extern "C"
