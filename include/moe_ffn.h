/*
 * moe_ffn.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts expert-FFN
 * forward: top-k routing -> permute -> grouped GEMM1 + SwiGLU -> grouped
 * GEMM2 -> weighted unpermute/combine, on one GPU.
 *
 * The layer is the one the "[SM90] Add W4A8 MegaMoE support" page (FlashInfer)
 * describes in its description and Usage section: expert indices per token
 * with -1 masking a route, fp32 routing weights, two expert GEMMs, clamped
 * SwiGLU and a top-k reduction; hidden width a multiple of 256 and
 * intermediate width a multiple of 128.  Permute/unpermute are the row
 * reorderings of "add permute fusion into hybrid ep" (Megatron-LM, PR
 * description); the gate/up pairing and its interleave option follow
 * "Support GEMM + Swiglu fused MLP" (Megatron-LM, description and the review
 * of moe_mlp_glu_interleave_size).
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, row-major
 *     and dense, 16-byte aligned.  The library never allocates device memory
 *     and never frees caller memory.  Inputs are never written; every output
 *     element is overwritten.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is
 *     enqueued asynchronously on it; no entry point synchronises the host or
 *     reads device data on the host, except moe_get_device_status.
 *   - `ws` is caller-provided scratch of at least moe_workspace_size() bytes,
 *     256-byte aligned.  It may be reused by consecutive calls on the same
 *     stream; calls that overlap in time must not share a workspace.
 *   - Argument checks run on the host before any launch and return a status
 *     without touching the GPU.  A failed launch returns MOE_ERR_CUDA.
 *     Device-side faults the kernels detect themselves (a bounded wait that
 *     ran out, an index out of range) are recorded in the workspace status
 *     word and read back with moe_get_device_status.
 *   - bf16 tensors are raw 16-bit bfloat16 values.
 *
 * Shapes: T tokens, H hidden, F expert intermediate, E experts, k routes per
 * token, R = T*k permuted rows.
 */
#ifndef MOE_FFN_H_
#define MOE_FFN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* null pointer, k > E, negative size ... */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* H % 256, F % 128, interleave rule, E/k limits */
  MOE_ERR_MISALIGNED = 3,         /* a pointer not 16-byte (ws: 256-byte) aligned */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4,
  MOE_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 6,     /* a kernel's bounded wait ran out (device status) */
  MOE_ERR_DEVICE_INDEX = 7        /* a kernel saw an out-of-range index (device status) */
} moe_status;

typedef enum { MOE_PREC_BF16 = 0, MOE_PREC_FP8_NVFP4 = 1 } moe_precision;

/* Problem description shared by all entry points. */
typedef struct moe_problem {
  int32_t T, H, F, E, k;
  /* 1: routing weights = softmax over the k selected logits (default);
     0: the full-softmax probability of each selected expert. */
  int32_t renormalize;
  /* Row order of W1 [E, 2F, H]:
     0  -> rows [gate_0 .. gate_{F-1} | up_0 .. up_{F-1}];
     I  -> alternating blocks of I gate rows then I up rows.
     I must divide F and be 32, 64 or a multiple of 128. */
  int32_t glu_interleave;
  /* SwiGLU clamp c: h = silu(min(g, c)) * clamp(u, -c, c); <= 0 or non-finite
     means no clamp. */
  float swiglu_clamp;
  int32_t precision; /* moe_precision */
  /* Fusion options of moe_forward (bit mask; 0 = the default, fastest
     measured form: permuted copy of x and a separate combine kernel):
       MOE_FUSE_GATHER_A  GEMM1 gathers its A rows straight from x with TMA
                          tile::gather4, so no permuted copy of x is written;
       MOE_FUSE_COMBINE   the weighted top-k reduction runs in GEMM2's
                          epilogue (bf16 partials + per-token arrival counters,
                          slot-ordered sum by the last arrival).
     Both give results within the same tolerance of the exact layer.  They
     apply to the 1-CTA token-row tilings only. */
  int32_t fusion;
  /* GEMM tiling (moe_problem.kernel):
       MOE_KERNEL_AUTO          T*k <= 2*E (at most two routes per expert on
                                average): weight-row tiles (in moe_forward at
                                T*k < E: the one-launch decode MLP below);
                                else 2-CTA weight-row tiles
       MOE_KERNEL_TOKEN_TILES   128 permuted token rows x 256 weight rows per tile
                                (the tiling the fusion options apply to)
       MOE_KERNEL_WEIGHT_TILES  128 weight rows x up to 32 token rows per tile
                                (decode sizes: weights stream once at HBM speed)
       MOE_KERNEL_WEIGHT_TILES_2CTA  256 weight rows x up to 256 token rows per
                                CTA pair (cta_group::2), N fitted to the
                                expert's rows (pads at most 31 rows); tiles of
                                experts with one token tile (weight-streaming)
                                interleaved with those of experts with more
                                (MMA-bound)
       MOE_KERNEL_DECODE_FUSED  moe_forward only (the other entry points run
                                MOE_KERNEL_WEIGHT_TILES): the 32-token weight
                                tiles of GEMM1 + SwiGLU and of GEMM2 and the
                                weighted combine in ONE persistent launch
                                (GEMM1 gathers its token rows from x with
                                TMA tile::gather4: no permuted copy of x).
                                Tiles are claimed from a global counter,
                                GEMM1's first; a GEMM2 tile streams its
                                weights at once and waits for its expert's h
                                rows on a per-expert count; the tile that
                                completes a token's k routes of a 128-feature
                                block sums them in slot order (bit-identical
                                to the separate combine)
     The fusion options do not apply to the weight-row tilings.  Any other
     value is MOE_ERR_INVALID_ARG. */
  int32_t kernel;
  /* Shared experts (moe_forward only; 0 elsewhere): S >= 0 experts, stored
     after the E routed ones in w1/w2 (experts E .. E+S-1, same shapes), that
     every token uses with weight 1 in addition to its k routed experts.  The
     routing outputs then have k+S slots per token (the shared ones last, ids
     E .. E+S-1, weight 1) and tokens_per_expert has E+S entries.  Needs
     k+S <= MOE_MAX_TOPK and E+S <= MOE_MAX_EXPERTS. */
  int32_t shared_experts;
} moe_problem;

#define MOE_FUSE_GATHER_A 1
#define MOE_FUSE_COMBINE 2
#define MOE_KERNEL_AUTO 0
#define MOE_KERNEL_TOKEN_TILES 1
#define MOE_KERNEL_WEIGHT_TILES 2
/* 3, 4 and 5 named tilings that are no longer built */
#define MOE_KERNEL_WEIGHT_TILES_2CTA 6
#define MOE_KERNEL_DECODE_FUSED 7

/* Limits checked by every entry point. */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 32

/* Human-readable name of a status code (static storage, never NULL). */
MOE_API const char* moe_status_string(int status);

/* Bytes of scratch every entry point needs for this problem (0 if the
 * problem itself is invalid).  Sized for the worst case of the routing, so
 * one workspace serves every call with the same sizes. */
MOE_API size_t moe_workspace_size(const moe_problem* p);

/* Step 1 -- top-k routing ("[SM90] Add W4A8 MegaMoE support", Usage: int
 * expert indices and fp32 weights per route).
 *   logits   [T, E] fp32
 *   topk_idx [T, k] int32 out: experts by logit descending, ties to the lower
 *            expert id (exact fp32 comparisons)
 *   topk_w   [T, k] fp32  out: softmax over the selected logits
 *            (renormalize=1) or full-softmax probabilities (renormalize=0). */
MOE_API int moe_route_topk(const moe_problem* p, const float* logits, int32_t* topk_idx,
                           float* topk_w, void* ws, size_t ws_bytes, void* stream);

/* Step 2 -- permute ("add permute fusion into hybrid ep", PR description):
 * stable scatter of routes into expert-contiguous rows, experts ascending,
 * tokens ascending within an expert.
 *   topk_idx          [T, k] int32, -1 = masked route (not counted)
 *   x                 [T, H] bf16, may be NULL when x_perm is NULL
 *   x_perm            [R, H] bf16 out or NULL: x_perm[r] = x[permuted_token[r]],
 *                     zero rows for the masked tail
 *   row_id_map        [T, k] int32 out: permuted row of route (t, j), -1 masked
 *   permuted_token    [R] int32 out: token of each row, -1 for the masked tail
 *   tokens_per_expert [E] int32 out
 *   expert_offsets    [E + 1] int32 out: exclusive prefix sum of the counts
 * A route index outside [-1, E) or an expert listed twice by one token is
 * recorded as MOE_ERR_DEVICE_INDEX in the device status. */
MOE_API int moe_permute(const moe_problem* p, const int32_t* topk_idx, const void* x,
                        void* x_perm, int32_t* row_id_map, int32_t* permuted_token,
                        int32_t* tokens_per_expert, int32_t* expert_offsets, void* ws,
                        size_t ws_bytes, void* stream);

/* Scales of NVFP4 weights as the low-precision entry points take them
 * ("[SM90] Add W4A8 MegaMoE support", Usage: E4M3 scales per 16 values,
 * transformed before the call, and one fp32 scale per expert tensor).  A
 * HOST struct holding DEVICE pointers:
 *   prepared   the block scales of W1 and W2 as moe_prepare_weights (or
 *              moe_prepare_weights_mxfp4) wrote them
 *   w1_gscale  [E] fp32 per-expert scale of W1
 *   w2_gscale  [E] fp32 per-expert scale of W2 */
typedef struct moe_fp4_scales {
  const void* prepared;
  const float* w1_gscale;
  const float* w2_gscale;
} moe_fp4_scales;

/* Steps 3-5 -- grouped expert MLP on permuted rows ("Support GEMM + Swiglu
 * fused MLP"; MegaMoE description: two expert GEMMs and clamped SwiGLU).
 *   expert_offsets [E + 1] int32 (device), non-decreasing, offsets[E] <= R
 *   y_perm         [R, H] bf16 out: y = silu-glu(x W1^T) W2^T per row, NOT
 *                  weighted; rows >= expert_offsets[E] are set to zero.
 * precision = MOE_PREC_BF16:
 *   x_perm         [R, H] bf16, rows of expert e at
 *                  [expert_offsets[e], expert_offsets[e+1])
 *   x_perm_scale   must be NULL
 *   w1             [E, 2F, H] bf16 (gate/up rows per glu_interleave)
 *   w2             [E, H, F] bf16
 *   wscales        must be NULL
 * precision = MOE_PREC_FP8_NVFP4 (the MegaMoE page's W4A8 formats; see the
 * low-precision section below):
 *   x_perm         [R, H] E4M3 codes (one byte each), permuted rows
 *   x_perm_scale   [R, H/128] fp32 scale of every 128 values of a row
 *   w1, w2         packed E2M1 codes [E, 2F, H/2] and [E, H, F/2]
 *   wscales        const moe_fp4_scales* (host struct of device pointers)
 *   GEMM1's SwiGLU output is re-quantised to E4M3 per 1x128 before GEMM2, as
 *   in moe_forward_fp8_nvfp4.  H a multiple of 256, F of 128. */
MOE_API int moe_grouped_swiglu_mlp(const moe_problem* p, const void* x_perm,
                                   const float* x_perm_scale, const int32_t* expert_offsets,
                                   const void* w1, const void* w2, const void* wscales,
                                   void* y_perm, void* ws, size_t ws_bytes, void* stream);

/* Row gather for payloads other than bf16 hidden rows (the permute of "add
 * permute fusion into hybrid ep", PR description, applied to any fixed-width
 * row): dst[r] = src[permuted_token[r]] for r < T*k, a zero row where
 * permuted_token[r] is -1.  For the low-precision layer's staged form: the
 * E4M3 code rows (row_bytes = H) and their fp32 scale rows (row_bytes =
 * 4*H/128) of x, gathered with the permuted_token moe_permute wrote.
 *   permuted_token [T*k] int32 (device), values in [-1, T)
 *   src [T, row_bytes] bytes, dst [T*k, row_bytes] bytes out (device)
 *   row_bytes a positive multiple of 4 (pointers 16-byte aligned).
 * A token index outside [-1, T) gives a zero row (not reported). */
MOE_API int moe_permute_rows(const moe_problem* p, const int32_t* permuted_token,
                             const void* src, int32_t row_bytes, void* dst, void* stream);

/* Step 6 -- weighted unpermute/combine (MegaMoE description: top-k
 * reduction):  out[t] = sum_{j=0..k-1, row_id_map[t][j] >= 0}
 *                        topk_w[t][j] * y_perm[row_id_map[t][j]],
 * summed in fp32 in slot order j = 0..k-1 and rounded once to bf16, so the
 * result is bitwise reproducible.
 *   y_perm [R, H] bf16, row_id_map [T, k] int32, topk_w [T, k] fp32,
 *   out [T, H] bf16 out. */
MOE_API int moe_unpermute_combine(const moe_problem* p, const void* y_perm,
                                  const int32_t* row_id_map, const float* topk_w, void* out,
                                  void* stream);

/* The whole layer, steps 1-6, enqueued on `stream` with no host round trip.
 *   logits [T, E] fp32, out [T, H] bf16 out
 *   topk_idx_out [T, k] int32, topk_w_out [T, k] fp32,
 *   tokens_per_expert_out [E] int32: optional copies of the routing (NULL to
 *   skip).
 * precision = MOE_PREC_BF16: x [T, H] bf16, x_scale NULL, w1 [E, 2F, H] and
 *   w2 [E, H, F] bf16, wscales NULL.
 * precision = MOE_PREC_FP8_NVFP4: x [T, H] E4M3 codes, x_scale [T, H/128]
 *   fp32, w1 / w2 packed E2M1 codes, wscales a const moe_fp4_scales* -- the
 *   same layer as moe_forward_fp8_nvfp4 (bit-identical results); shared
 *   experts are bf16 only. */
MOE_API int moe_forward(const moe_problem* p, const void* x, const float* x_scale,
                        const float* logits, const void* w1, const void* w2,
                        const void* wscales, void* out, int32_t* topk_idx_out,
                        float* topk_w_out, int32_t* tokens_per_expert_out, void* ws,
                        size_t ws_bytes, void* stream);

/* The layer with the routing supplied by the caller (steps 2-6): the staged
 * top-k indices and weights of the MegaMoE page's interface (description,
 * item 5 of the changes; Usage: INT64 indices with -1 for a masked route and
 * FP32 routing weights -- int32 indices here).
 *   x [T, H] bf16, topk_idx [T, k] int32, topk_w [T, k] fp32,
 *   w1 [E, 2F, H] bf16, w2 [E, H, F] bf16, out [T, H] bf16 out,
 *   tokens_per_expert_out [E] int32 (optional).
 * A slot with index -1 is skipped; a token whose slots are all masked gets a
 * zero row.  An index outside [-1, E), or an expert repeated in a later slot
 * of the same token, is treated as masked and recorded as
 * MOE_ERR_DEVICE_INDEX in the workspace status word (moe_get_device_status).
 * The weights are used as given (no normalisation).  bf16 precision only;
 * moe_problem.fusion is ignored; moe_problem.kernel picks the GEMM tiling as
 * for moe_forward. */
MOE_API int moe_forward_routed(const moe_problem* p, const void* x, const int32_t* topk_idx,
                               const float* topk_w, const void* w1, const void* w2, void* out,
                               int32_t* tokens_per_expert_out, void* ws, size_t ws_bytes,
                               void* stream);

/* ---- Backward (bf16 precision) -------------------------------------------
 * Gradients of a scalar loss L given G = dL/d out, for the layer moe_forward
 * computes (training use: the Megatron-LM pages, "add permute fusion into
 * hybrid ep" and "Support GEMM + Swiglu fused MLP", place the layer in
 * training; they print no backward formulas, so these are the derivatives of
 * the forward).  Per route (token t, expert e, weight w), with g, u the gate
 * and up pre-activations, gc = min(g, c), uc = clamp(u, -c, c) and
 * h = silu(gc) uc:
 *   dh = W2_e^T (w G_t);  du = dh silu(gc) [-c <= u <= c];
 *   dg = dh uc silu'(gc) [g <= c];  dW2_e += (w G_t) h^T;
 *   dW1_e += [dg | du] x_t^T (rows per glu_interleave);  dx_t += W1_e^T [dg | du];
 *   d w = <G_t, y>, then the softmax backward of the routing weights
 *   (renormalize = 1: over the selected logits; 0: over all E).
 * The top-k selection passes no gradient.  The forward's intermediates are
 * recomputed, not stored: the pre-activations x W1_e^T are recomputed in fp32
 * and the clamp decisions are taken on those fp32 values.  Every output is
 * written by one thread in a fixed order (no atomics): bitwise reproducible.
 *   x [T, H] bf16, logits [T, E] fp32, w1 [E+S, 2F, H] bf16,
 *   w2 [E+S, H, F] bf16, d_out [T, H] bf16 (G);
 *   dx [T, H] bf16 out; d_logits [T, E] fp32 out (NULL to skip);
 *   dw1 [E+S, 2F, H] bf16 out, dw2 [E+S, H, F] bf16 out (shared experts
 *   included; an expert no token selects gets zero gradients);
 *   ws of at least moe_backward_workspace_size(p) bytes.
 * p->precision must be MOE_PREC_BF16; p->fusion and p->kernel are ignored. */
MOE_API size_t moe_backward_workspace_size(const moe_problem* p);
MOE_API int moe_backward(const moe_problem* p, const void* x, const float* logits,
                         const void* w1, const void* w2, const void* d_out, void* dx,
                         float* d_logits, void* dw1, void* dw2, void* ws, size_t ws_bytes,
                         void* stream);

/* The backward of moe_forward_routed (routing supplied by the caller): the
 * same gradients with topk_idx / topk_w as given (int32 [T, k], -1 = masked
 * slot; fp32 [T, k]) and, instead of the logit gradient, the gradient of
 * every routing weight:
 *   d_topk_w [T, k] fp32 out (NULL to skip): dL/d topk_w[t][j] = <G_t, y_tj>,
 *   the unweighted output of the slot's expert for token t; 0 for a masked
 *   slot.
 * Masked, out-of-range and repeated slots are handled and reported as in
 * moe_forward_routed.  shared_experts must be 0; bf16 precision only;
 * workspace of moe_backward_workspace_size(p) bytes. */
MOE_API int moe_backward_routed(const moe_problem* p, const void* x, const int32_t* topk_idx,
                                const float* topk_w, const void* w1, const void* w2,
                                const void* d_out, void* dx, float* d_topk_w, void* dw1,
                                void* dw2, void* ws, size_t ws_bytes, void* stream);

/* Self-test of the bounded waits (the pages have no counterpart: this checks
 * the library's own failure detection).  Launches one CTA that waits on an
 * mbarrier nothing arrives on, through the same bounded wait every kernel
 * uses, with a limit of limit_ns nanoseconds (1 .. 2e9); the wait runs out,
 * MOE_ERR_DEVICE_TIMEOUT is recorded in the status word of `ws` (a workspace
 * from moe_workspace_size; read it with moe_get_device_status) and the kernel
 * returns normally, leaving the context usable.  Asynchronous on `stream`.
 * Returns MOE_ERR_INVALID_ARG for a null ws or a limit out of range. */
MOE_API int moe_selftest_wait_timeout(void* ws, uint64_t limit_ns, void* stream);

/* Capacity, in int32 entries, of the fixed device scratch that
 * moe_permute_noalloc uses: ceil(T / 64) * E + E + 1 must not exceed it. */
#define MOE_NOALLOC_SCRATCH_INTS (1 << 18)

/* moe_permute for callers that cannot allocate device memory or hand the
 * library a workspace -- for example code that runs while a stream is being
 * captured into a CUDA graph (cudaMalloc is not allowed there), or a host
 * framework whose device memory all belongs to its own pool and which has
 * no way to pass scratch through a plain C call.  It takes the same
 * arguments as moe_permute minus the workspace and writes the same outputs.
 * Its scratch (the per-chunk expert histograms and the m-tile prefix) lives
 * in one fixed array of MOE_NOALLOC_SCRATCH_INTS int32 (1 MiB) that every GPU
 * loading this library keeps until the process exits; nothing is allocated
 * or freed, by this call or by anything it calls.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress, with that device current) and keeps it for
 *     every later call; make that first call before any stream capture on
 *     the device.  Resetting the device (cudaDeviceReset) after it is not
 *     supported: the kept address may no longer be the array's.
 *   - Every call on a device shares the one array.  Calls whose work can
 *     overlap on the GPU (different streams without ordering between them)
 *     race on it and give wrong results; serialise them.  Each call
 *     overwrites every scratch entry it reads, so stale contents from an
 *     earlier call do no harm.
 *   - Problems needing more scratch than the array holds are rejected with
 *     MOE_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   - Index errors are handled as in moe_permute (bad routes are treated
 *     as masked) but are not reported: there is no workspace status word.
 * The source pages have no counterpart to this entry point; it exists only
 * for callers without an allocator. */
MOE_API int moe_permute_noalloc(const moe_problem* p, const int32_t* topk_idx, const void* x,
                                void* x_perm, int32_t* row_id_map, int32_t* permuted_token,
                                int32_t* tokens_per_expert, int32_t* expert_offsets,
                                void* stream);

/* ---- Low-precision layer (precision = MOE_PREC_FP8_NVFP4) ----------------
 * The formats of the "[SM90] Add W4A8 MegaMoE support" page's Usage section:
 * FP8 E4M3 activations with one fp32 scale per 128 channels, NVFP4 weights =
 * E2M1 codes (two per byte, the even index in the low nibble) with one E4M3
 * scale per 16 values along K and one fp32 scale per expert weight tensor.
 * The weights stay 4-bit in HBM.  GEMM1's SwiGLU output is re-quantised to
 * E4M3 with one fp32 scale (amax / 448) per 128 values of a row before
 * GEMM2, as that page's split GEMM1 does.  Output bf16.  Tilings
 * (moe_problem.kernel): MOE_KERNEL_AUTO or MOE_KERNEL_TOKEN_TILES run 1-CTA
 * 128-token x 256-weight-row tiles; MOE_KERNEL_WEIGHT_TILES_2CTA runs 2-CTA
 * weight-row tiles (each CTA expands its 128 weight rows; the 1x128
 * re-quantisation block of h spans both CTAs of a pair, whose per-token
 * maxima are exchanged through distributed shared memory); any other value
 * is MOE_ERR_INVALID_ARG.  moe_problem.fusion is ignored. */

/* Bytes of the prepared scale buffer for W1 and W2 together. */
MOE_API size_t moe_prepared_scales_size(const moe_problem* p);

/* Re-lays the E4M3 block scales of both weight tensors into the order the
 * kernels stream them (per expert, per 128 weight rows, per 64-deep K step:
 * 128 rows x 4 scales), the analogue of the page's weight transform before
 * the call.  Run once per set of weights.
 *   w1_scale [E, 2F, H/16] bytes, w2_scale [E, H, F/16] bytes (device)
 *   prepared  device buffer of moe_prepared_scales_size() bytes, 16-aligned */
MOE_API int moe_prepare_weights(const moe_problem* p, const uint8_t* w1_scale,
                                const uint8_t* w2_scale, void* prepared, size_t prepared_bytes,
                                void* stream);

/* MXFP4 weights (the MegaMoE page's Usage: raw weight scales E8M0 per 32
 * values; the page prepares them with a weight transform before the call):
 * re-encodes them exactly for moe_forward_fp8_nvfp4.  The packed E2M1 codes
 * are used as they are (w1q / w2q); the scales become the prepared layout of
 * moe_prepare_weights plus one fp32 scale per expert tensor:
 *   w1_scale [E, 2F, H/32], w2_scale [E, H, F/32]: E8M0 bytes, 2^(s - 127);
 *   prepared: moe_prepared_scales_size(p) bytes out;
 *   w1_gscale_out [E], w2_gscale_out [E]: fp32 out, to pass to
 *   moe_forward_fp8_nvfp4 as the expert scales.
 * With e_max the expert tensor's largest scale byte, its fp32 scale is
 * 2^(e_max - 135) and each block's scale becomes the E4M3 power of two
 * 2^(s - e_max + 8) in [2^-9, 2^8], exact; a block more than 17 binades
 * below e_max is set to zero.  The byte 255 (not a number) is out of contract.
 * p->precision must be MOE_PREC_FP8_NVFP4. */
MOE_API int moe_prepare_weights_mxfp4(const moe_problem* p, const uint8_t* w1_scale,
                                      const uint8_t* w2_scale, void* prepared,
                                      size_t prepared_bytes, float* w1_gscale_out,
                                      float* w2_gscale_out, void* stream);

/* The whole low-precision layer.
 *   xq [T, H] E4M3 codes, xs [T, H/128] fp32, logits [T, E] fp32
 *   w1q [E, 2F, H/2], w2q [E, H, F/2] packed E2M1 codes (GLU interleave as
 *   in moe_problem), w1_gscale / w2_gscale [E] fp32, prepared scales from
 *   moe_prepare_weights; out [T, H] bf16; optional routing copies as in
 *   moe_forward; ws of moe_workspace_size(p) bytes. */
MOE_API int moe_forward_fp8_nvfp4(const moe_problem* p, const uint8_t* xq, const float* xs,
                                  const float* logits, const uint8_t* w1q,
                                  const float* w1_gscale, const uint8_t* w2q,
                                  const float* w2_gscale, const void* prepared_scales, void* out,
                                  int32_t* topk_idx_out, float* topk_w_out,
                                  int32_t* tokens_per_expert_out, void* ws, size_t ws_bytes,
                                  void* stream);

/* Synchronises `stream`, returns the status the kernels recorded in `ws`
 * since the last moe_clear_device_status (MOE_OK if none). */
MOE_API int moe_get_device_status(void* ws, void* stream);

/* Resets the workspace status word (enqueued on `stream`). */
MOE_API int moe_clear_device_status(void* ws, void* stream);

/* The GEMM tiling moe_forward uses for this problem (a MOE_KERNEL_* value
 * other than MOE_KERNEL_AUTO), or -1 for an invalid problem. */
MOE_API int moe_selected_kernel(const moe_problem* p);

/* Number of kernel launches the last successful call on this thread
 * enqueued (for launch accounting in benchmarks). */
MOE_API int moe_last_launch_count(void);

/* Per-stage timing of moe_forward / moe_backward with CUDA events (for
 * benchmarks).  moe_stage_timing_begin(n) makes the next n moe_forward or
 * moe_backward calls on this thread record an event on their stream before
 * each stage and after the last (events created once, reused);
 * moe_stage_timing_end synchronises the device, writes the average
 * milliseconds of each stage over the recorded calls into ms[0 .. *n_stages)
 * (at most max_stages entries) and stops recording.  Stage i is named by
 * moe_stage_name(i), for the entry point recorded last (time one kind of
 * call per session).  Returns a status. */
MOE_API int moe_stage_timing_begin(int n_calls);
MOE_API int moe_stage_timing_end(float* ms, int max_stages, int* n_stages, int* n_calls);
MOE_API const char* moe_stage_name(int i);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H_ */
