// Internal launcher interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// Tokens per routing chunk: the unit of the per-chunk expert histogram and
// of the stable scatter (one warp scatters one chunk in token order).
constexpr int kChunkTokens = 64;

// Grouped-GEMM tiling (rows of permuted tokens x output columns x K step).
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;

inline int ceil_div(long a, long b) { return static_cast<int>((a + b - 1) / b); }

int num_sms();

// Records the number of kernel launches of the entry point that just
// succeeded on this thread (read back by moe_last_launch_count).
void set_last_launch_count(int n);

// Programmatic dependent launch for every kernel; building with
// -DMOE_NO_PDL turns it off (for comparison timings only).
constexpr bool pdl_enabled() {
#ifdef MOE_NO_PDL
  return false;
#else
  return true;
#endif
}

// cudaLaunchKernelEx with programmatic stream serialization allowed (the
// kernels wait with griddepcontrol.wait before touching global memory) and an
// optional cluster of cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Step 1: routing.
cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int renormalize,
                              int32_t* topk_idx, float* topk_w, cudaStream_t s, int S = 0);

// Step 2a: per-chunk expert histogram of topk_idx (also validates indices).
// When `counters` is not NULL the kernel also zeroes counters[t * ncnt ..
// (t+1) * ncnt) for the tokens of its chunk (the fused combine's arrival
// counters).
cudaError_t launch_chunk_histogram(const int32_t* topk_idx, int T, int E, int k,
                                   int32_t* chunk_counts, uint32_t* status, cudaStream_t s,
                                   int32_t* counters = nullptr, int ncnt = 0);

// Step 2b: turn chunk histograms into per-(chunk, expert) row bases and
// produce tokens_per_expert, expert_offsets, the m-tile prefix and the
// masked-tail fill of permuted_token.
cudaError_t launch_scan(int32_t* chunk_counts, int nchunks, int E, int R,
                        int32_t* tokens_per_expert, int32_t* expert_offsets,
                        int32_t* mtile_prefix, int32_t* permuted_token, cudaStream_t s);

// Step 2 in one block for decode sizes when every route is valid: same
// outputs as histogram + scan + scatter.
constexpr int kSmallRoutes = 4096;
constexpr int kSmallExperts = 1024;
// The smallest decode steps: routing + permutation (+ the row gather when x is
// not null) in one single-block launch.
constexpr int kTinyTokens = 32;     // one routing warp per token
constexpr int kTinyExperts = 256;   // staged logits: T * E floats of shared memory
constexpr int kTinyRoutes = 256;
constexpr int kTinyGatherRoutes = 64;  // rows one block gathers faster than a launch
bool route_permute_tiny_fits(int T, int E, int k, int S);
// Both single-block forms also zero zero_ints[0 .. n_zero) when given (the
// counters of the one-launch decode MLP that follows them).
cudaError_t launch_route_permute_tiny(const float* logits, int T, int E, int k, int S,
                                      int renormalize,
                                      int32_t* topk_idx, float* topk_w,
                                      int32_t* tokens_per_expert, int32_t* expert_offsets,
                                      int32_t* mtile_prefix, int32_t* row_id_map,
                                      int32_t* permuted_token, const void* x, int H,
                                      void* x_perm, cudaStream_t s,
                                      int32_t* zero_ints = nullptr, int n_zero = 0);
bool permute_small_fits(int T, int E, int k);
cudaError_t launch_permute_small(const int32_t* topk_idx, int T, int E, int k,
                                 int32_t* tokens_per_expert, int32_t* expert_offsets,
                                 int32_t* mtile_prefix, int32_t* row_id_map,
                                 int32_t* permuted_token, cudaStream_t s,
                                 int32_t* zero_ints = nullptr, int n_zero = 0);

// Step 2c: stable scatter -> row_id_map and permuted_token.
cudaError_t launch_scatter(const int32_t* topk_idx, int T, int E, int k,
                           const int32_t* chunk_base, int32_t* row_id_map,
                           int32_t* permuted_token, cudaStream_t s);

// x_perm[r] = x[permuted_token[r]] (zero row for -1).
cudaError_t launch_gather_rows(const void* x, const int32_t* permuted_token, int R, int H,
                               void* x_perm, cudaStream_t s);

// The same rows written from the source side: x_perm[row_id_map[t][j]] =
// x[t] (each token row read once), zero rows for [expert_offsets[E], T*k).
cudaError_t launch_scatter_rows(const void* x, const int32_t* row_id_map,
                                const int32_t* expert_offsets, int T, int k, int E, int H,
                                void* x_perm, cudaStream_t s);

// dst[r] = src[permuted_token[r]] for rows of row_bytes bytes (a multiple of
// 4); zero row for -1 or a token outside [0, T).
cudaError_t launch_gather_row_bytes(const void* src, const int32_t* permuted_token, int R, int T,
                                    int row_bytes, void* dst, cudaStream_t s);

// m-tile prefix from caller-supplied expert offsets (validated on device).
cudaError_t launch_mtile_prefix_from_offsets(const int32_t* expert_offsets, int E, int R,
                                             int32_t* mtile_prefix, uint32_t* status,
                                             cudaStream_t s);

// Step 6: out[t] = sum_j w[t][j] * y[row_id_map[t][j]] in slot order (w = 1
// when topk_w is null).
cudaError_t launch_combine(const void* y, const int32_t* row_id_map, const float* topk_w,
                           int T, int H, int k, void* out, cudaStream_t s);

// Steps 3-5: grouped GEMMs on tcgen05.
enum class Epi : int { kSwiGLU = 0, kPlain = 1, kCombine = 2 };

struct GroupedGemmArgs {
  Epi epi;
  const void* a;               // [a_rows, K] bf16 (permuted rows)
  int a_rows;
  const void* b;               // [E * b_rows_per_expert, K] bf16
  int b_rows_per_expert;
  int E;
  int K;
  int n_tiles;                 // output tiles per expert along N
  const int32_t* expert_offsets;
  const int32_t* mtile_prefix;
  void* out;                   // bf16 rows of ldo elements
  int ldo;
  int out_rows;                // rows >= expert_offsets[E] .. out_rows are zeroed (kPlain)
  int F;                       // SwiGLU: intermediate width
  int interleave;              // SwiGLU: GLU interleave (0, 32, 64 or multiple of 128)
  float clamp;                 // SwiGLU clamp (<= 0: none)
  uint32_t* status;
  // kSwiGLU with permuted_token != NULL: A rows are gathered from a = x [x_rows, K]
  // kCombine: the fused weighted top-k reduction into out = [T, ldo]
  const int32_t* permuted_token = nullptr;
  int x_rows = 0;
  const int32_t* row_id_map = nullptr;
  const float* topk_w = nullptr;
  int32_t* counters = nullptr;  // [T, n_tiles], zero before the launch
  void* partials = nullptr;     // [R, ldo] bf16
  int k = 0;
};

cudaError_t launch_grouped_gemm(const GroupedGemmArgs& g, cudaStream_t s);

// The same GEMMs with weight rows on the MMA's M side and up to 32 tokens on
// N (kSwiGLU and kPlain epilogues; no gather / combine fusion).
cudaError_t launch_grouped_gemm_swap(const GroupedGemmArgs& g, cudaStream_t s);

// Decode sizes in one launch: GEMM1 + SwiGLU, GEMM2 and (out != NULL) the
// weighted combine, 128 weight rows x up to 32 token rows per tile
// (grouped_mlp_decode.cu).  counters: decode_mlp_counters(T, E, H) int32,
// zero at launch; with the combine every route of every token must be valid.
struct DecodeMlpArgs {
  const void* x;                  // [T, H] bf16 token rows (gathered by permuted_token)
  const void* w1;                 // [E * 2F, H] bf16
  const void* w2;                 // [E * H, F] bf16
  const int32_t* expert_offsets;  // [E + 1]
  void* h;                        // [R, F] bf16 (scratch)
  void* y;                        // [R, H] bf16 (the output without the combine)
  void* out;                      // [T, H] bf16 or NULL
  const int32_t* permuted_token;  // [R]
  const int32_t* row_id_map;      // [T, k]
  const float* topk_w;            // [T, k]
  int32_t* counters;
  int R, T, E, H, F, k, interleave;
  float clamp;
  uint32_t* status;
};
int decode_mlp_counters(int T, int E, int H);
cudaError_t launch_grouped_mlp_decode(const DecodeMlpArgs& g, cudaStream_t s);

// Weight-row tiles on CTA pairs (cta_group::2), tokens on N fitted per tile.
cudaError_t launch_grouped_gemm_swap2(const GroupedGemmArgs& g, cudaStream_t s);

// NVFP4-weight GEMMs (a = f16 rows, b = packed E2M1 codes [E * rows, K / 2],
// scales in the prepared layout, gscale = per-expert fp32 tensor scales).
// kSwiGLU stores FP8-requantised h as f16; kPlain stores bf16 y.
cudaError_t launch_grouped_gemm_fp4(const GroupedGemmArgs& g, const uint8_t* scales,
                                    const float* gscale, cudaStream_t s);
// The same GEMMs with weight-row tiles on CTA pairs (cta_group::2, N fitted per
// expert); needs rows per expert a multiple of 128.
cudaError_t launch_grouped_gemm_fp4_pair(const GroupedGemmArgs& g, const uint8_t* scales,
                                         const float* gscale, cudaStream_t s);
// [E][N][K/16] E4M3 scales -> [E][N/128][K/64][128][4]
cudaError_t launch_prepare_scales(const uint8_t* src, uint8_t* dst, int E, int N, int K,
                                  cudaStream_t s);
// MXFP4 E8M0 scales [E][2F][H/32] and [E][H][F/32] -> the prepared E4M3 layout
// (exact powers of two) plus per-expert fp32 scales g1[E], g2[E].
cudaError_t launch_prepare_mxfp4_scales(const uint8_t* s1, const uint8_t* s2, uint8_t* dst1,
                                        uint8_t* dst2, int E, int F, int H, float* g1, float* g2,
                                        cudaStream_t s);
// ---- backward -------------------------------------------------------------
// Grouped GEMMs of the backward (grouped_gemm_bwd.cu):
//   kBwdDataPlain   out[r, :N] = a[r, :K] b_e[K, N]       (b read MN-major)
//   kBwdDataSwiGLU  the same product dh, then the SwiGLU backward epilogue
//                   over act (pre-activations -> dA in place), hw and dw_part
//   kBwdWeight      out[e, :M, :N] = a_e^T b_e over the rows of expert e
//   kBwdPreact      out[r, :N] = a[r, :K] b_e[N, K]^T in fp32 (the forward's
//                   GEMM1 without its activation; b read K-major)
constexpr int kBwdDataPlain = 0;
constexpr int kBwdDataSwiGLU = 1;
constexpr int kBwdWeight = 2;
constexpr int kBwdPreact = 3;

struct BwdGemmArgs {
  int mode;
  const void* a;  // data: [R, K]; weight: [R, M] bf16
  const void* b;  // data: [E * K, N] stacked weights; weight: [R, N] bf16;
                  // pre-activations: [E * N, K] weights
  int R, E, K, N, M;
  const int32_t* expert_offsets;  // [E + 1]
  const int32_t* mtile_prefix;    // [E + 1] (data modes)
  void* out;                      // data: [R, N]; weight: [E, M, N] bf16; [R, N] fp32
  // kBwdDataSwiGLU
  const void* act = nullptr;      // [R, 2F] fp32 pre-activations
  void* dact = nullptr;           // [R, 2F] bf16 out: their gradient dA
  void* hw = nullptr;             // [R, F] bf16 out: w * h
  float* dw_part = nullptr;       // [R, bwd_router_parts(N)] fp32 out
  const float* w_perm = nullptr;  // [R] routing weight per permuted row
  int F = 0, interleave = 0;
  float clamp = 0.f;
  uint32_t* status = nullptr;
};

cudaError_t launch_grouped_gemm_bwd(const BwdGemmArgs& g, cudaStream_t s);

// Epilogue warps per TMEM lane quadrant in the SwiGLU-backward GEMM (they
// split a tile's 32-column chunks), and the router-gradient partials it
// writes per permuted row for N = F columns: one per tile and warp of a
// quadrant.
constexpr int kBwdSwiGLUSplit = 1;
inline int bwd_router_parts(int F) { return kBwdSwiGLUSplit * ((F + kBN - 1) / kBN); }

// w_perm[row_id_map[t][j]] = topk_w[t][j] for every valid route.
cudaError_t launch_weights_to_rows(const int32_t* row_id_map, const float* topk_w, long routes,
                                   float* w_perm, cudaStream_t s);

// d topk_w[t][j] = sum of the dw_part row of route (t, j) (fixed order), 0
// for a masked slot: the routing-weight gradient of caller-supplied routes.
cudaError_t launch_route_weight_grad(const int32_t* row_id_map, const float* dw_part,
                                     int n_parts, long routes, float* d_topk_w,
                                     cudaStream_t s);

// Router backward, one warp per token: dw_j = sum of the dw_part row of the
// route (fixed order), then the softmax backward over the first k slots of
// the `slots` per token into dlogits [T, E] fp32.
cudaError_t launch_router_backward(const float* logits, const int32_t* topk_idx,
                                   const float* topk_w, const int32_t* row_id_map,
                                   const float* dw_part, int n_parts, int T, int E, int k,
                                   int slots, int renormalize, float* dlogits, cudaStream_t s);

// FP8 rows (E4M3 codes + fp32 scales per 128) gathered by permuted_token into
// f16 (permuted_token NULL: row r from row r).
cudaError_t launch_gather_dequant_fp8(const uint8_t* xq, const float* xs,
                                      const int32_t* permuted_token, int R, int H, void* x_perm,
                                      cudaStream_t s);

}  // namespace moe
