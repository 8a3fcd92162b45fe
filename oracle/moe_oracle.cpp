// CPU ORACLE for the single-GPU MoE expert-FFN forward -- TEST INFRASTRUCTURE.
//
// Plain, slow, fp64 C++ written straight from the definitions of the layer.
// Only tests, the package's smoke check and the benchmark's CPU-baseline leg
// may load this library; the product path never calls it.  It shares no code,
// header, table or constant with the CUDA path.
//
// Sources for what each step computes (page titles and sections):
//   * "[SM90] Add W4A8 MegaMoE support" (FlashInfer), description + Usage:
//     the layer is routing -> two expert GEMMs -> clamped SwiGLU -> top-k
//     reduction; routes are expert indices with -1 masking a route, routing
//     weights are fp32, activation scales are fp32 per 128 channels, NVFP4
//     weight scales are E4M3 per 16 values.
//   * "add permute fusion into hybrid ep" (Megatron-LM), PR description:
//     permute = reorder token rows into expert-contiguous order, unpermute =
//     the inverse reorder that feeds the combine.
//   * "Support GEMM + Swiglu fused MLP" (Megatron-LM), description and the
//     review thread on moe_mlp_glu_interleave_size: fc1 produces gate and up
//     and SwiGLU consumes them; the interleave option reorders W1's rows.
//
// Readings where the pages are silent (each is also listed in the design
// notes): selection on raw fp32 logits with ties to the lowest expert id;
// weights = softmax over the k selected logits (renormalize=1) or the full
// softmax probabilities (renormalize=0); stable (token-ascending) order inside
// an expert; interleave I = alternating blocks of I gate rows and I up rows;
// clamp c: silu(min(g, c)) * clamp(u, -c, c).
//
// Pins: every function here is checked by the CPU test-suite against brute
// force, closed forms, library routines (numpy / torch) and invariants.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// bf16 is the top half of an IEEE binary32; widening is exact.
inline double bf16_value(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Row of W1 holding gate (resp. up) output column f.
//   interleave 0: W1 = [gate rows 0..F-1 | up rows 0..F-1]
//   interleave I: blocks of I gate rows followed by I up rows, repeated.
inline long gate_row(long f, long F, long I) {
  if (I <= 0) return f;
  return (f / I) * 2 * I + f % I;
}
inline long up_row(long f, long F, long I) {
  if (I <= 0) return F + f;
  return gate_row(f, F, I) + I;
}

inline double silu(double z) { return z / (1.0 + std::exp(-z)); }

// ---- low-precision formats (OCP 8-bit and 4-bit floating point) ----------
// E4M3 ("fn" variant, no infinities): sign, 4 exponent bits (bias 7), 3
// mantissa bits; exponent field 0 is subnormal; S.1111.111 is NaN.
inline double e4m3_value(uint8_t c) {
  const int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return std::nan("");
  const double v = (e == 0) ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return sgn ? -v : v;
}

// E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 subnormal.
inline double e2m1_value(uint8_t n) {
  const int sgn = (n >> 3) & 1, e = (n >> 1) & 3, m = n & 1;
  const double v = (e == 0) ? 0.5 * m : std::ldexp(1.0 + m / 2.0, e - 1);
  return sgn ? -v : v;
}

// Nearest E4M3 code to x, ties to the even code, magnitudes above the
// largest finite value (448) saturate to it.  Found by trying every finite
// code: slow and plain.
inline uint8_t e4m3_encode(float x) {
  if (std::isnan(x)) return 0x7F;
  const double a = std::fabs(static_cast<double>(x));
  int best = 0;
  double best_d = a;  // distance to code 0 (value 0)
  for (int c = 1; c < 127; ++c) {  // 127 = NaN
    const double d = std::fabs(e4m3_value(static_cast<uint8_t>(c)) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_d = d;
    }
  }
  if (a >= 448.0) best = 0x7E;
  return static_cast<uint8_t>(best | (std::signbit(x) && best != 0 ? 0x80 : 0));
}

// Decoded values of every code, filled once from the functions above (a
// speed-up of the same definitions, nothing else).
struct CodeTables {
  double e4m3[256];
  double e2m1[16];
  CodeTables() {
    for (int c = 0; c < 256; ++c) e4m3[c] = e4m3_value(static_cast<uint8_t>(c));
    for (int c = 0; c < 16; ++c) e2m1[c] = e2m1_value(static_cast<uint8_t>(c));
  }
};
const CodeTables kCodes;

// NVFP4 weight element k of a packed row: two E2M1 values per byte, the even
// index in the low nibble; one E4M3 scale per 16 values; times the tensor's
// fp32 scale g.
inline double nvfp4_value(const uint8_t* q_row, const uint8_t* s_row, long k, double g) {
  const uint8_t byte = q_row[k >> 1];
  const uint8_t nib = (k & 1) ? (byte >> 4) : (byte & 15);
  return kCodes.e2m1[nib] * kCodes.e4m3[s_row[k >> 4]] * g;
}

// E8M0 scale byte: 2^(e - 127) (the byte 255 is not a number; out of contract).
inline double e8m0_value(uint8_t e) { return std::ldexp(1.0, static_cast<int>(e) - 127); }

// MXFP4 (the MegaMoE page's Usage: raw weight scales E8M0 per 32 values):
// w = E2M1(q) * 2^(s - 127), s the scale byte of the 32-value block.
inline double mxfp4_value(const uint8_t* q_row, const uint8_t* s_row, long k) {
  const uint8_t byte = q_row[k >> 1];
  const uint8_t nib = (k & 1) ? (byte >> 4) : (byte & 15);
  return kCodes.e2m1[nib] * e8m0_value(s_row[k >> 5]);
}

// Weight formats of the low-precision oracle: 0 NVFP4 (E4M3 scale per 16 values
// times the expert's fp32 scale g), 1 MXFP4 (E8M0 scale per 32 values; g unused).
inline double fp4_value(int wfmt, const uint8_t* q_row, const uint8_t* s_row, long k, double g) {
  return wfmt == 1 ? mxfp4_value(q_row, s_row, k) : nvfp4_value(q_row, s_row, k, g);
}
inline int scale_block(int wfmt) { return wfmt == 1 ? 32 : 16; }

// clamp <= 0 or non-finite means "no clamp".
inline double swiglu(double g, double u, double c) {
  if (c > 0 && std::isfinite(c)) {
    g = std::fmin(g, c);
    u = std::fmax(std::fmin(u, c), -c);
  }
  return silu(g) * u;
}

}  // namespace

extern "C" {

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

int oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

double oracle_bf16_value(uint16_t bits) { return bf16_value(bits); }

// ---------------------------------------------------------------------------
// Step 1: top-k routing.
// For token t the selected set is the k experts with the largest logits,
// listed by (logit descending, expert id ascending).  Comparisons are exact
// fp32 comparisons (+0 == -0).  Weights, in fp64:
//   renormalize = 1: softmax over the k selected logits;
//   renormalize = 0: the full softmax probability of each selected expert.
// Returns 0, or -1 on bad sizes.
int oracle_route_topk(int T, int E, int k, int renormalize, const float* logits,
                      int32_t* topk_idx, double* topk_w) {
  if (T < 0 || E < 1 || k < 1 || k > E) return -1;
  for (int t = 0; t < T; ++t) {
    const float* l = logits + static_cast<long>(t) * E;
    std::vector<char> taken(E, 0);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;  // strict: ties keep the lower id
      }
      taken[best] = 1;
      topk_idx[static_cast<long>(t) * k + j] = best;
    }
    const double lmax = l[topk_idx[static_cast<long>(t) * k]];
    double denom = 0.0;
    if (renormalize) {
      for (int j = 0; j < k; ++j)
        denom += std::exp(static_cast<double>(l[topk_idx[static_cast<long>(t) * k + j]]) - lmax);
    } else {
      for (int e = 0; e < E; ++e) denom += std::exp(static_cast<double>(l[e]) - lmax);
    }
    for (int j = 0; j < k; ++j) {
      double v = std::exp(static_cast<double>(l[topk_idx[static_cast<long>(t) * k + j]]) - lmax);
      topk_w[static_cast<long>(t) * k + j] = v / denom;
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Step 2: permute bookkeeping.
//   tokens_per_expert[e] = number of routes (t, j) with topk_idx[t][j] == e
//   expert_offsets       = exclusive prefix sum (E + 1 entries)
//   rows are handed out in (expert ascending, token ascending) order:
//     row_id_map[t][j]    = the permuted row of route (t, j), -1 if masked
//     permuted_token[row] = t, and -1 for the unused tail rows when some
//                           routes are masked.
// Returns 0, -1 on bad sizes, -2 on an index outside [-1, E), -3 when a token
// lists the same expert twice.
int oracle_permute(int T, int E, int k, const int32_t* topk_idx, int32_t* tokens_per_expert,
                   int32_t* expert_offsets, int32_t* row_id_map, int32_t* permuted_token) {
  if (T < 0 || E < 1 || k < 1) return -1;
  const long R = static_cast<long>(T) * k;
  for (long i = 0; i < R; ++i)
    if (topk_idx[i] < -1 || topk_idx[i] >= E) return -2;
  for (int t = 0; t < T; ++t)
    for (int a = 0; a < k; ++a)
      for (int b = a + 1; b < k; ++b) {
        int32_t ea = topk_idx[static_cast<long>(t) * k + a];
        if (ea >= 0 && ea == topk_idx[static_cast<long>(t) * k + b]) return -3;
      }
  for (int e = 0; e < E; ++e) tokens_per_expert[e] = 0;
  for (long i = 0; i < R; ++i)
    if (topk_idx[i] >= 0) tokens_per_expert[topk_idx[i]] += 1;
  expert_offsets[0] = 0;
  for (int e = 0; e < E; ++e) expert_offsets[e + 1] = expert_offsets[e] + tokens_per_expert[e];
  for (long i = 0; i < R; ++i) row_id_map[i] = -1;
  for (long r = 0; r < R; ++r) permuted_token[r] = -1;
  for (int e = 0; e < E; ++e) {
    int32_t next = expert_offsets[e];
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (topk_idx[static_cast<long>(t) * k + j] == e) {
          row_id_map[static_cast<long>(t) * k + j] = next;
          permuted_token[next] = t;
          ++next;
        }
  }
  return 0;
}

// Materialise the permuted activations: x_perm[r] = x[permuted_token[r]]
// (rows with permuted_token = -1 are zero).
int oracle_gather_rows(long R, int H, const uint16_t* x, const int32_t* permuted_token,
                       uint16_t* x_perm) {
  for (long r = 0; r < R; ++r) {
    uint16_t* dst = x_perm + r * H;
    if (permuted_token[r] < 0) {
      std::memset(dst, 0, sizeof(uint16_t) * H);
    } else {
      std::memcpy(dst, x + static_cast<long>(permuted_token[r]) * H, sizeof(uint16_t) * H);
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Steps 3+4: GEMM1 and SwiGLU for the rows of each expert, in fp64.
// For permuted row r in expert e's segment [expert_offsets[e], expert_offsets[e+1]):
//   g_f = sum_h x_perm[r][h] * W1_e[gate_row(f)][h]
//   u_f = sum_h x_perm[r][h] * W1_e[up_row(f)][h]
//   h[r][f] = silu(min(g_f, c)) * clamp(u_f, -c, c)        (no clamp if c <= 0)
// w1_experts[e] points at expert e's [2F, H] bf16 matrix (NULL allowed for an
// expert with no rows).  Rows beyond expert_offsets[E] are set to 0.
int oracle_gemm1_swiglu(long R, int H, int F, int E, int interleave, double clamp,
                        const int32_t* expert_offsets, const uint16_t* x_perm,
                        const uint16_t* const* w1_experts, double* h) {
  if (interleave > 0 && F % interleave != 0) return -1;
  for (int e = 0; e < E; ++e)
    if (expert_offsets[e + 1] > expert_offsets[e] && w1_experts[e] == nullptr) return -2;
  for (long r = expert_offsets[E]; r < R; ++r)
    for (int f = 0; f < F; ++f) h[r * F + f] = 0.0;
  for (int e = 0; e < E; ++e) {
    const long r0 = expert_offsets[e], r1 = expert_offsets[e + 1];
    if (r1 <= r0) continue;
    const uint16_t* W = w1_experts[e];
#pragma omp parallel for schedule(dynamic)
    for (long r = r0; r < r1; ++r) {
      std::vector<double> xr(H);
      for (int c = 0; c < H; ++c) xr[c] = bf16_value(x_perm[r * H + c]);
      for (int f = 0; f < F; ++f) {
        const uint16_t* wg = W + gate_row(f, F, interleave) * static_cast<long>(H);
        const uint16_t* wu = W + up_row(f, F, interleave) * static_cast<long>(H);
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
          g += xr[c] * bf16_value(wg[c]);
          u += xr[c] * bf16_value(wu[c]);
        }
        h[r * F + f] = swiglu(g, u, clamp);
      }
    }
  }
  return 0;
}

// Step 5: GEMM2, y[r][n] = sum_f h[r][f] * W2_e[n][f] (W2_e is [H, F]).
int oracle_gemm2(long R, int H, int F, int E, const int32_t* expert_offsets, const double* h,
                 const uint16_t* const* w2_experts, double* y) {
  for (int e = 0; e < E; ++e)
    if (expert_offsets[e + 1] > expert_offsets[e] && w2_experts[e] == nullptr) return -2;
  for (long r = expert_offsets[E]; r < R; ++r)
    for (int n = 0; n < H; ++n) y[r * H + n] = 0.0;
  for (int e = 0; e < E; ++e) {
    const long r0 = expert_offsets[e], r1 = expert_offsets[e + 1];
    if (r1 <= r0) continue;
    const uint16_t* W = w2_experts[e];
#pragma omp parallel for schedule(dynamic)
    for (long r = r0; r < r1; ++r) {
      const double* hr = h + r * F;
      for (int n = 0; n < H; ++n) {
        const uint16_t* wn = W + static_cast<long>(n) * F;
        double acc = 0.0;
        for (int f = 0; f < F; ++f) acc += hr[f] * bf16_value(wn[f]);
        y[r * H + n] = acc;
      }
    }
  }
  return 0;
}

// Step 6: weighted unpermute / combine.
//   out[t][n] = sum over slots j = 0..k-1 with row_id_map[t][j] >= 0 of
//               topk_w[t][j] * y[row_id_map[t][j]][n]
int oracle_unpermute_combine(int T, int H, int k, const double* y, const int32_t* row_id_map,
                             const double* topk_w, double* out) {
#pragma omp parallel for
  for (int t = 0; t < T; ++t) {
    double* o = out + static_cast<long>(t) * H;
    for (int n = 0; n < H; ++n) o[n] = 0.0;
    for (int j = 0; j < k; ++j) {
      const long row = row_id_map[static_cast<long>(t) * k + j];
      if (row < 0) continue;
      const double w = topk_w[static_cast<long>(t) * k + j];
      for (int n = 0; n < H; ++n) o[n] += w * y[row * H + n];
    }
  }
  return 0;
}

// The whole layer: route -> permute -> gather -> GEMM1+SwiGLU -> GEMM2 -> combine.
// topk_idx_out / topk_w_out / tokens_per_expert_out may be NULL.
int oracle_moe_forward(int T, int H, int F, int E, int k, int renormalize, int interleave,
                       double clamp, const float* logits, const uint16_t* x,
                       const uint16_t* const* w1_experts, const uint16_t* const* w2_experts,
                       double* out, int32_t* topk_idx_out, double* topk_w_out,
                       int32_t* tokens_per_expert_out) {
  const long R = static_cast<long>(T) * k;
  std::vector<int32_t> idx(R), row_id_map(R), permuted_token(R), counts(E), offsets(E + 1);
  std::vector<double> w(R);
  int rc = oracle_route_topk(T, E, k, renormalize, logits, idx.data(), w.data());
  if (rc) return rc;
  rc = oracle_permute(T, E, k, idx.data(), counts.data(), offsets.data(), row_id_map.data(),
                      permuted_token.data());
  if (rc) return rc;
  std::vector<uint16_t> x_perm(static_cast<size_t>(R) * H);
  oracle_gather_rows(R, H, x, permuted_token.data(), x_perm.data());
  std::vector<double> h(static_cast<size_t>(R) * F), y(static_cast<size_t>(R) * H);
  rc = oracle_gemm1_swiglu(R, H, F, E, interleave, clamp, offsets.data(), x_perm.data(),
                           w1_experts, h.data());
  if (rc) return rc;
  rc = oracle_gemm2(R, H, F, E, offsets.data(), h.data(), w2_experts, y.data());
  if (rc) return rc;
  oracle_unpermute_combine(T, H, k, y.data(), row_id_map.data(), w.data(), out);
  if (topk_idx_out) std::memcpy(topk_idx_out, idx.data(), sizeof(int32_t) * R);
  if (topk_w_out) std::memcpy(topk_w_out, w.data(), sizeof(double) * R);
  if (tokens_per_expert_out) std::memcpy(tokens_per_expert_out, counts.data(), sizeof(int32_t) * E);
  return 0;
}

// Second, permutation-free evaluation of the same layer for given routes: for
// every token and slot, run the selected expert's MLP on the token's own row
// and accumulate the weighted result.  Used to cross-check the permuted form.
int oracle_dense_bruteforce(int T, int H, int F, int E, int k, int interleave, double clamp,
                            const int32_t* topk_idx, const double* topk_w, const uint16_t* x,
                            const uint16_t* const* w1_experts,
                            const uint16_t* const* w2_experts, double* out) {
#pragma omp parallel for schedule(dynamic)
  for (int t = 0; t < T; ++t) {
    std::vector<double> xr(H), hv(F);
    for (int c = 0; c < H; ++c) xr[c] = bf16_value(x[static_cast<long>(t) * H + c]);
    double* o = out + static_cast<long>(t) * H;
    for (int n = 0; n < H; ++n) o[n] = 0.0;
    for (int j = 0; j < k; ++j) {
      const int e = topk_idx[static_cast<long>(t) * k + j];
      if (e < 0) continue;
      const uint16_t* W1 = w1_experts[e];
      const uint16_t* W2 = w2_experts[e];
      for (int f = 0; f < F; ++f) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
          g += xr[c] * bf16_value(W1[gate_row(f, F, interleave) * static_cast<long>(H) + c]);
          u += xr[c] * bf16_value(W1[up_row(f, F, interleave) * static_cast<long>(H) + c]);
        }
        hv[f] = swiglu(g, u, clamp);
      }
      const double w = topk_w[static_cast<long>(t) * k + j];
      for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int f = 0; f < F; ++f) acc += hv[f] * bf16_value(W2[static_cast<long>(n) * F + f]);
        o[n] += w * acc;
      }
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Low-precision variant (the MegaMoE page's formats: FP8 E4M3 activations
// with fp32 scales per 128 channels, NVFP4 weights = E2M1 values with E4M3
// scales per 16 values and an fp32 scale per expert weight tensor).

double oracle_e4m3_value(uint8_t c) { return e4m3_value(c); }
double oracle_e2m1_value(uint8_t n) { return e2m1_value(n); }
double oracle_e8m0_value(uint8_t e) { return e8m0_value(e); }
uint8_t oracle_e4m3_encode(float x) { return e4m3_encode(x); }

// Re-quantisation of one row block of h to FP8 (the split GEMM1 epilogue of
// the MegaMoE page stores its output with per-128 scales): s = amax / 448 in
// fp32 (s = 1 when the block is all zero), code = E4M3(h / s) computed in
// fp32, returned value = E4M3 value * s.  n <= 128 values.
void oracle_requant_fp8_block(const double* h, int n, double* out) {
  float amax = 0.f;
  for (int i = 0; i < n; ++i) amax = std::fmax(amax, std::fabs(static_cast<float>(h[i])));
  const float s = amax > 0.f ? amax / 448.0f : 1.0f;
  for (int i = 0; i < n; ++i) {
    const float v = static_cast<float>(h[i]) / s;
    out[i] = e4m3_value(e4m3_encode(v)) * static_cast<double>(s);
  }
}

// GEMM1 + SwiGLU on dequantised operands, rows of each expert:
//   x_hat[r][c]  = E4M3(xq[r][c]) * xs[r][c / 128]
//   w_hat[n][c]  = E2M1(q) * E4M3(s[n][c / 16]) * g1[e]
//   h = silu(min(g, clamp)) * clamp(u, -clamp, clamp), then (requant != 0)
//   every 128-wide block of a row re-quantised to FP8 as above.
// w1q[e]: [2F, H/2] bytes, w1s[e]: [2F, H/16] bytes.
int oracle_gemm1_swiglu_lowprec(long R, int H, int F, int E, int interleave, double clamp,
                                const int32_t* expert_offsets, const uint8_t* xq_perm,
                                const float* xs_perm, const uint8_t* const* w1q,
                                const uint8_t* const* w1s, const float* g1, int requant,
                                int wfmt, double* h) {
  const int sb = scale_block(wfmt);
  if (interleave > 0 && F % interleave != 0) return -1;
  if (H % 128 != 0 || F % 128 != 0) return -1;
  for (int e = 0; e < E; ++e)
    if (expert_offsets[e + 1] > expert_offsets[e] && (!w1q[e] || !w1s[e])) return -2;
  for (long r = expert_offsets[E]; r < R; ++r)
    for (int f = 0; f < F; ++f) h[r * F + f] = 0.0;
  for (int e = 0; e < E; ++e) {
    const long r0 = expert_offsets[e], r1 = expert_offsets[e + 1];
    if (r1 <= r0) continue;
    const long nr = r1 - r0;
    std::vector<double> xhat(static_cast<size_t>(nr) * H), hraw(static_cast<size_t>(nr) * F);
    for (long r = r0; r < r1; ++r)
      for (int c = 0; c < H; ++c)
        xhat[(r - r0) * H + c] =
            kCodes.e4m3[xq_perm[r * H + c]] * static_cast<double>(xs_perm[r * (H / 128) + c / 128]);
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
    for (long r = r0; r < r1; ++r) {
      for (int f = 0; f < F; ++f) {
        const double* xr = &xhat[(r - r0) * H];
        const long rg = gate_row(f, F, interleave), ru = up_row(f, F, interleave);
        const uint8_t* qg = w1q[e] + rg * (H / 2);
        const uint8_t* sg = w1s[e] + rg * (H / sb);
        const uint8_t* qu = w1q[e] + ru * (H / 2);
        const uint8_t* su = w1s[e] + ru * (H / sb);
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
          g += xr[c] * fp4_value(wfmt, qg, sg, c, g1[e]);
          u += xr[c] * fp4_value(wfmt, qu, su, c, g1[e]);
        }
        hraw[(r - r0) * F + f] = swiglu(g, u, clamp);
      }
    }
    for (long r = r0; r < r1; ++r) {
      const double* hr = &hraw[(r - r0) * F];
      if (requant) {
        for (int b = 0; b < F; b += 128) oracle_requant_fp8_block(&hr[b], 128, &h[r * F + b]);
      } else {
        for (int f = 0; f < F; ++f) h[r * F + f] = hr[f];
      }
    }
  }
  return 0;
}

// GEMM2 on dequantised NVFP4 weights: y[r][n] = sum_f h[r][f] * w2_hat[n][f].
// w2q[e]: [H, F/2] bytes, w2s[e]: [H, F/16] bytes.
int oracle_gemm2_lowprec(long R, int H, int F, int E, const int32_t* expert_offsets,
                         const double* h, const uint8_t* const* w2q, const uint8_t* const* w2s,
                         const float* g2, int wfmt, double* y) {
  const int sb = scale_block(wfmt);
  for (int e = 0; e < E; ++e)
    if (expert_offsets[e + 1] > expert_offsets[e] && (!w2q[e] || !w2s[e])) return -2;
  for (long r = expert_offsets[E]; r < R; ++r)
    for (int n = 0; n < H; ++n) y[r * H + n] = 0.0;
  for (int e = 0; e < E; ++e) {
    const long r0 = expert_offsets[e], r1 = expert_offsets[e + 1];
    if (r1 <= r0) continue;
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
    for (long r = r0; r < r1; ++r) {
      for (int n = 0; n < H; ++n) {
        const uint8_t* q = w2q[e] + static_cast<long>(n) * (F / 2);
        const uint8_t* sc = w2s[e] + static_cast<long>(n) * (F / sb);
        double acc = 0.0;
        for (int f = 0; f < F; ++f) acc += h[r * F + f] * fp4_value(wfmt, q, sc, f, g2[e]);
        y[r * H + n] = acc;
      }
    }
  }
  return 0;
}

// The whole low-precision layer: route -> permute -> gather (codes and
// scales) -> GEMM1 + SwiGLU + FP8 re-quantisation -> GEMM2 -> combine.
int oracle_moe_forward_lowprec(int T, int H, int F, int E, int k, int renormalize,
                               int interleave, double clamp, const float* logits,
                               const uint8_t* xq, const float* xs, const uint8_t* const* w1q,
                               const uint8_t* const* w1s, const float* g1,
                               const uint8_t* const* w2q, const uint8_t* const* w2s,
                               const float* g2, int wfmt, double* out, int32_t* topk_idx_out,
                               double* topk_w_out) {
  const long R = static_cast<long>(T) * k;
  std::vector<int32_t> idx(R), row_id_map(R), permuted_token(R), counts(E), offsets(E + 1);
  std::vector<double> w(R);
  int rc = oracle_route_topk(T, E, k, renormalize, logits, idx.data(), w.data());
  if (rc) return rc;
  rc = oracle_permute(T, E, k, idx.data(), counts.data(), offsets.data(), row_id_map.data(),
                      permuted_token.data());
  if (rc) return rc;
  std::vector<uint8_t> xq_perm(static_cast<size_t>(R) * H, 0);
  std::vector<float> xs_perm(static_cast<size_t>(R) * (H / 128), 1.0f);
  for (long r = 0; r < R; ++r) {
    const int t = permuted_token[r];
    if (t < 0) continue;
    std::memcpy(&xq_perm[r * H], xq + static_cast<long>(t) * H, H);
    std::memcpy(&xs_perm[r * (H / 128)], xs + static_cast<long>(t) * (H / 128),
                sizeof(float) * (H / 128));
  }
  std::vector<double> h(static_cast<size_t>(R) * F), y(static_cast<size_t>(R) * H);
  rc = oracle_gemm1_swiglu_lowprec(R, H, F, E, interleave, clamp, offsets.data(), xq_perm.data(),
                                   xs_perm.data(), w1q, w1s, g1, 1, wfmt, h.data());
  if (rc) return rc;
  rc = oracle_gemm2_lowprec(R, H, F, E, offsets.data(), h.data(), w2q, w2s, g2, wfmt, y.data());
  if (rc) return rc;
  oracle_unpermute_combine(T, H, k, y.data(), row_id_map.data(), w.data(), out);
  if (topk_idx_out) std::memcpy(topk_idx_out, idx.data(), sizeof(int32_t) * R);
  if (topk_w_out) std::memcpy(topk_w_out, w.data(), sizeof(double) * R);
  return 0;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward of the layer.  The Megatron-LM pages ("add permute fusion into
// hybrid ep", "Support GEMM + Swiglu fused MLP") use the layer in training,
// where the gradients of its inputs are needed; the pages print no backward
// formulas, so these are the derivatives of the forward above, taken route by
// route.  For a route (token t, slot j) to expert e with weight w:
//   g_f, u_f = rows gate_row(f), up_row(f) of W1_e times x_t
//   gc_f = min(g_f, c), uc_f = clamp(u_f, -c, c), h_f = silu(gc_f) uc_f
//   y = W2_e h,  out_t = sum over the token's routes of w y
// and with G = dL/d out_t:
//   dy = w G,  dw = <G, y>
//   dh_f = sum_n W2_e[n][f] dy[n]
//   du_f = dh_f silu(gc_f)          where -c <= u_f <= c, else 0
//   dg_f = dh_f uc_f silu'(gc_f)    where g_f <= c, else 0
//   silu'(z) = s (1 + z (1 - s)),  s = 1 / (1 + exp(-z))
//   dW2_e[n][f] += dy[n] h_f
//   dW1_e[gate_row(f)][:] += dg_f x_t,  dW1_e[up_row(f)][:] += du_f x_t
//   dx_t += sum_f dg_f W1_e[gate_row(f)] + du_f W1_e[up_row(f)]
// Without a clamp both masks are 1.  The top-k selection is piecewise
// constant and passes no gradient; the routing weights do (router backward
// below).  mask_f32 = 1 takes the two clamp decisions on g and u rounded to
// fp32 (the precision a caller may keep the pre-activations in); 0 takes
// them on the exact values.
// magnitude = 1 returns, instead of each output, the sum of the absolute
// values of the terms that make it up (|a| |b| for every product a b of the
// sums above): the scale of the rounding error a finite-precision evaluation
// of the same sums may make.
namespace {

inline double silu_grad(double z) {
  const double s = 1.0 / (1.0 + std::exp(-z));
  return s * (1.0 + z * (1.0 - s));
}

// Column f of the SwiGLU and its backward for one route.
inline void swiglu_backward(double g, double u, double dh, double c, int mask_f32, double* h,
                            double* dg, double* du) {
  double gc = g, uc = u;
  bool pass_g = true, pass_u = true;
  if (c > 0 && std::isfinite(c)) {
    const double gm = mask_f32 ? static_cast<double>(static_cast<float>(g)) : g;
    const double um = mask_f32 ? static_cast<double>(static_cast<float>(u)) : u;
    pass_g = gm <= c;
    pass_u = um >= -c && um <= c;
    gc = std::fmin(g, c);
    uc = std::fmax(std::fmin(u, c), -c);
  }
  *h = silu(gc) * uc;
  *du = pass_u ? dh * silu(gc) : 0.0;
  *dg = pass_g ? dh * uc * silu_grad(gc) : 0.0;
}

// Which output column f (and gate or up) row `row` of W1 holds: the inverse
// of gate_row / up_row.
inline long w1_row_column(long row, long F, long I, bool* is_gate) {
  if (I == 0) {
    *is_gate = row < F;
    return row < F ? row : row - F;
  }
  const long block = row / I;
  *is_gate = (block % 2) == 0;
  return (block / 2) * I + row % I;
}

// Gate and up pre-activations of column f for the widened row xr.
inline void preact(const double* xr, const uint16_t* W1, long H, long F, long I, long f,
                   double* g, double* u) {
  const uint16_t* wg = W1 + gate_row(f, F, I) * H;
  const uint16_t* wu = W1 + up_row(f, F, I) * H;
  double a = 0.0, b = 0.0;
  for (long c = 0; c < H; ++c) {
    a += xr[c] * bf16_value(wg[c]);
    b += xr[c] * bf16_value(wu[c]);
  }
  *g = a;
  *u = b;
}

// dh_f = sum_n W2[n][f] dy[n].
inline double dh_at(const double* dy, const uint16_t* W2, long H, long F, long f) {
  double acc = 0.0;
  for (long n = 0; n < H; ++n) acc += bf16_value(W2[n * F + f]) * dy[n];
  return acc;
}

// Every backward quantity of one route: the W1-row-ordered dA (2F), h (F),
// dy (H) and dw = <G, y> (its magnitude sum |G| |y| when `magnitude`).
// Optionally adds the route's dx contribution (|dA| |W1| when `magnitude`).
void route_backward(long H, long F, long I, double c, int mask_f32, int magnitude, double w,
                    const uint16_t* x_row, const uint16_t* g_row, const uint16_t* W1,
                    const uint16_t* W2, double* dA, double* h, double* dy, double* dw,
                    double* dx_add) {
  std::vector<double> xr(H), G(H), gv(F), uv(F), y(H);
  for (long c2 = 0; c2 < H; ++c2) {
    xr[c2] = bf16_value(x_row[c2]);
    G[c2] = bf16_value(g_row[c2]);
  }
  for (long f = 0; f < F; ++f) {
    preact(xr.data(), W1, H, F, I, f, &gv[f], &uv[f]);
    double hf, dg, du;
    swiglu_backward(gv[f], uv[f], 0.0, c, mask_f32, &hf, &dg, &du);
    h[f] = hf;
  }
  double d = 0.0;
  for (long n = 0; n < H; ++n) {
    double acc = 0.0;
    for (long f = 0; f < F; ++f) acc += bf16_value(W2[n * F + f]) * h[f];
    y[n] = acc;
    d += magnitude ? std::fabs(G[n] * acc) : G[n] * acc;
  }
  *dw = d;
  for (long n = 0; n < H; ++n) dy[n] = w * G[n];
  for (long f = 0; f < F; ++f) {
    const double dh = dh_at(dy, W2, H, F, f);
    double hf, dg, du;
    swiglu_backward(gv[f], uv[f], dh, c, mask_f32, &hf, &dg, &du);
    dA[gate_row(f, F, I)] = dg;
    dA[up_row(f, F, I)] = du;
  }
  if (dx_add) {
    for (long row = 0; row < 2 * F; ++row) {
      const double a = dA[row];
      if (a == 0.0) continue;
      const uint16_t* wr = W1 + row * H;
      for (long c2 = 0; c2 < H; ++c2)
        dx_add[c2] += magnitude ? std::fabs(a * bf16_value(wr[c2])) : a * bf16_value(wr[c2]);
    }
  }
}

}  // namespace

extern "C" {

// Expert backward for given routes.  topk_idx / topk_w are [T, slots] (-1 =
// masked slot); expert e uses w1_experts[e] [2F, H] and w2_experts[e] [H, F]
// (NULL allowed for an expert no route selects); d_out is G as bf16 [T, H].
// Outputs (fp64): dx [T, H], dw_route [T, slots] (= <G_t, y> per route, 0 for
// a masked slot), dw1 [E, 2F, H], dw2 [E, H, F].  Returns 0, -1 on bad sizes,
// -2 on a route to an expert without weights or outside [-1, E).
int oracle_moe_backward(int T, int H, int F, int E, int slots, int interleave, double clamp,
                        int mask_f32, int magnitude, const int32_t* topk_idx,
                        const double* topk_w,
                        const uint16_t* x, const uint16_t* const* w1_experts,
                        const uint16_t* const* w2_experts, const uint16_t* d_out, double* dx,
                        double* dw_route, double* dw1, double* dw2) {
  if (T < 0 || H <= 0 || F <= 0 || E <= 0 || slots <= 0) return -1;
  const long R = static_cast<long>(T) * slots, HH = H, FF = F;
  for (long r = 0; r < R; ++r) {
    const int e = topk_idx[r];
    if (e < -1 || e >= E) return -2;
    if (e >= 0 && (w1_experts[e] == nullptr || w2_experts[e] == nullptr)) return -2;
  }
  std::vector<double> dA(static_cast<size_t>(R) * 2 * FF, 0.0), hr(static_cast<size_t>(R) * FF, 0.0),
      dy(static_cast<size_t>(R) * HH, 0.0), dxr(static_cast<size_t>(R) * HH, 0.0);
#pragma omp parallel for schedule(dynamic)
  for (long r = 0; r < R; ++r) {
    const int e = topk_idx[r];
    dw_route[r] = 0.0;
    if (e < 0) continue;
    const long t = r / slots;
    route_backward(HH, FF, interleave, clamp, mask_f32, magnitude, topk_w[r], x + t * HH,
                   d_out + t * HH, w1_experts[e], w2_experts[e], &dA[r * 2 * FF], &hr[r * FF],
                   &dy[r * HH], &dw_route[r], &dxr[r * HH]);
  }
#pragma omp parallel for
  for (long t = 0; t < T; ++t)
    for (long c = 0; c < HH; ++c) {
      double acc = 0.0;
      for (int j = 0; j < slots; ++j) acc += dxr[(t * slots + j) * HH + c];
      dx[t * HH + c] = acc;
    }
#pragma omp parallel for schedule(dynamic)
  for (long er = 0; er < static_cast<long>(E) * 2 * FF; ++er) {
    const long e = er / (2 * FF), row = er % (2 * FF);
    double* out = dw1 + er * HH;
    for (long c = 0; c < HH; ++c) out[c] = 0.0;
    for (long r = 0; r < R; ++r) {
      if (topk_idx[r] != e) continue;
      const double a = dA[r * 2 * FF + row];
      const uint16_t* xr = x + (r / slots) * HH;
      for (long c = 0; c < HH; ++c)
        out[c] += magnitude ? std::fabs(a * bf16_value(xr[c])) : a * bf16_value(xr[c]);
    }
  }
#pragma omp parallel for schedule(dynamic)
  for (long en = 0; en < static_cast<long>(E) * HH; ++en) {
    const long e = en / HH, n = en % HH;
    double* out = dw2 + en * FF;
    for (long f = 0; f < FF; ++f) out[f] = 0.0;
    for (long r = 0; r < R; ++r) {
      if (topk_idx[r] != e) continue;
      const double d = dy[r * HH + n];
      for (long f = 0; f < FF; ++f)
        out[f] += magnitude ? std::fabs(d * hr[r * FF + f]) : d * hr[r * FF + f];
    }
  }
  return 0;
}

// dx rows and per-route dw of the listed tokens only (the same definitions as
// oracle_moe_backward, for sizes where the whole backward is too slow).
//   tokens [n], dx_rows [n, H] (slots summed in order j = 0, 1, ...),
//   dw_rows [n, slots].
int oracle_backward_tokens(int T, int H, int F, int E, int slots, int interleave, double clamp,
                           int mask_f32, int magnitude, const int32_t* topk_idx,
                           const double* topk_w,
                           const uint16_t* x, const uint16_t* const* w1_experts,
                           const uint16_t* const* w2_experts, const uint16_t* d_out, int n,
                           const int32_t* tokens, double* dx_rows, double* dw_rows) {
  if (T < 0 || H <= 0 || F <= 0 || E <= 0 || slots <= 0 || n < 0) return -1;
  const long HH = H, FF = F;
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= T) return -1;
  std::vector<double> part(static_cast<size_t>(n) * slots * HH, 0.0);
#pragma omp parallel for schedule(dynamic)
  for (long q = 0; q < static_cast<long>(n) * slots; ++q) {
    const long i = q / slots, j = q % slots, t = tokens[i], r = t * slots + j;
    dw_rows[q] = 0.0;
    const int e = topk_idx[r];
    if (e < 0 || e >= E || !w1_experts[e] || !w2_experts[e]) continue;
    std::vector<double> dA(2 * FF), h(FF), dy(HH);
    route_backward(HH, FF, interleave, clamp, mask_f32, magnitude, topk_w[r], x + t * HH,
                   d_out + t * HH, w1_experts[e], w2_experts[e], dA.data(), h.data(), dy.data(),
                   &dw_rows[q], &part[q * HH]);
  }
  for (long i = 0; i < n; ++i)
    for (long c = 0; c < HH; ++c) {
      double acc = 0.0;
      for (long j = 0; j < slots; ++j) acc += part[(i * slots + j) * HH + c];
      dx_rows[i * HH + c] = acc;
    }
  return 0;
}

// Whole rows of dW1 for the listed (expert, W1 row) pairs:
//   dW1_e[row][:] = sum over the routes of e of dA[row] x_t   (rows [n, H]).
int oracle_backward_dw1_rows(int T, int H, int F, int E, int slots, int interleave,
                             double clamp, int mask_f32, int magnitude,
                             const int32_t* topk_idx, const double* topk_w, const uint16_t* x,
                             const uint16_t* const* w1_experts,
                             const uint16_t* const* w2_experts, const uint16_t* d_out, int n,
                             const int32_t* pairs, double* rows) {
  if (T < 0 || H <= 0 || F <= 0 || E <= 0 || slots <= 0 || n < 0) return -1;
  const long HH = H, FF = F, R = static_cast<long>(T) * slots;
  for (int i = 0; i < n; ++i) {
    const int e = pairs[2 * i], row = pairs[2 * i + 1];
    if (e < 0 || e >= E || row < 0 || row >= 2 * F) return -1;
  }
  for (int i = 0; i < n; ++i) {
    const int e = pairs[2 * i];
    const long row = pairs[2 * i + 1];
    bool is_gate = true;
    const long f = w1_row_column(row, FF, interleave, &is_gate);
    std::vector<long> routes;
    for (long r = 0; r < R; ++r)
      if (topk_idx[r] == e) routes.push_back(r);
    std::vector<double> a(routes.size(), 0.0);
    if (!routes.empty() && (!w1_experts[e] || !w2_experts[e])) return -2;
#pragma omp parallel for schedule(dynamic)
    for (long q = 0; q < static_cast<long>(routes.size()); ++q) {
      const long r = routes[q], t = r / slots;
      std::vector<double> xr(HH), dy(HH);
      for (long c = 0; c < HH; ++c) {
        xr[c] = bf16_value(x[t * HH + c]);
        dy[c] = topk_w[r] * bf16_value(d_out[t * HH + c]);
      }
      double g, u, h, dg, du;
      preact(xr.data(), w1_experts[e], HH, FF, interleave, f, &g, &u);
      swiglu_backward(g, u, dh_at(dy.data(), w2_experts[e], HH, FF, f), clamp, mask_f32, &h,
                      &dg, &du);
      a[q] = is_gate ? dg : du;
      if (magnitude) a[q] = std::fabs(a[q]);
    }
#pragma omp parallel for
    for (long c = 0; c < HH; ++c) {
      double acc = 0.0;
      for (size_t q = 0; q < routes.size(); ++q) {
        const double xv = bf16_value(x[(routes[q] / slots) * HH + c]);
        acc += a[q] * (magnitude ? std::fabs(xv) : xv);
      }
      rows[i * HH + c] = acc;
    }
  }
  return 0;
}

// Whole columns of dW2 for the listed (expert, f) pairs:
//   dW2_e[:][f] = sum over the routes of e of w G_t h_f   (cols [n, H]).
int oracle_backward_dw2_cols(int T, int H, int F, int E, int slots, int interleave,
                             double clamp, int mask_f32, int magnitude,
                             const int32_t* topk_idx, const double* topk_w, const uint16_t* x,
                             const uint16_t* const* w1_experts, const uint16_t* d_out, int n,
                             const int32_t* pairs, double* cols) {
  if (T < 0 || H <= 0 || F <= 0 || E <= 0 || slots <= 0 || n < 0) return -1;
  const long HH = H, FF = F, R = static_cast<long>(T) * slots;
  for (int i = 0; i < n; ++i) {
    const int e = pairs[2 * i], f = pairs[2 * i + 1];
    if (e < 0 || e >= E || f < 0 || f >= F) return -1;
  }
  for (int i = 0; i < n; ++i) {
    const int e = pairs[2 * i];
    const long f = pairs[2 * i + 1];
    std::vector<long> routes;
    for (long r = 0; r < R; ++r)
      if (topk_idx[r] == e) routes.push_back(r);
    if (!routes.empty() && !w1_experts[e]) return -2;
    std::vector<double> wh(routes.size(), 0.0);
#pragma omp parallel for schedule(dynamic)
    for (long q = 0; q < static_cast<long>(routes.size()); ++q) {
      const long r = routes[q], t = r / slots;
      std::vector<double> xr(HH);
      for (long c = 0; c < HH; ++c) xr[c] = bf16_value(x[t * HH + c]);
      double g, u, h, dg, du;
      preact(xr.data(), w1_experts[e], HH, FF, interleave, f, &g, &u);
      swiglu_backward(g, u, 0.0, clamp, mask_f32, &h, &dg, &du);
      wh[q] = magnitude ? std::fabs(topk_w[r] * h) : topk_w[r] * h;
    }
#pragma omp parallel for
    for (long nn = 0; nn < HH; ++nn) {
      double acc = 0.0;
      for (size_t q = 0; q < routes.size(); ++q) {
        const double gv = bf16_value(d_out[(routes[q] / slots) * HH + nn]);
        acc += (magnitude ? std::fabs(gv) : gv) * wh[q];
      }
      cols[i * HH + nn] = acc;
    }
  }
  return 0;
}

// Router backward: the gradient of the loss with respect to the logits given
// dw = dL/d topk_w for the first k slots of each token (slots >= k are shared
// experts with the constant weight 1 and pass nothing).
//   renormalize = 1: dl_{e_j} = w_j (dw_j - sum_i w_i dw_i), 0 elsewhere;
//   renormalize = 0: dl_e = p_e ([e selected by slot j] dw_j - sum_i w_i dw_i),
//                    p = softmax of the token's E logits (fp64).
// A masked slot (-1) is left out of both sums.  dlogits [T, E] fp64.
// magnitude = 1: dw holds the magnitudes m_j of the per-route gradients and
// the result is the magnitude of each logit's gradient, the two sums added
// instead of subtracted: w_j (m_j + sum_i w_i m_i), resp.
// p_e ([e = e_j] m_j + sum_i w_i m_i).
int oracle_router_backward(int T, int E, int k, int slots, int renormalize, int magnitude,
                           const float* logits, const int32_t* topk_idx, const double* topk_w,
                           const double* dw, double* dlogits) {
  if (T < 0 || E <= 0 || k <= 0 || slots < k) return -1;
#pragma omp parallel for
  for (long t = 0; t < T; ++t) {
    double* dl = dlogits + t * E;
    for (int e = 0; e < E; ++e) dl[e] = 0.0;
    double s = 0.0;
    for (int j = 0; j < k; ++j) {
      const long r = t * slots + j;
      if (topk_idx[r] >= 0) s += topk_w[r] * dw[r];
    }
    if (renormalize) {
      for (int j = 0; j < k; ++j) {
        const long r = t * slots + j;
        if (topk_idx[r] >= 0) dl[topk_idx[r]] = topk_w[r] * (magnitude ? dw[r] + s : dw[r] - s);
      }
    } else {
      const float* l = logits + t * E;
      double lmax = l[0];
      for (int e = 1; e < E; ++e) lmax = std::fmax(lmax, static_cast<double>(l[e]));
      double denom = 0.0;
      for (int e = 0; e < E; ++e) denom += std::exp(static_cast<double>(l[e]) - lmax);
      for (int e = 0; e < E; ++e)
        dl[e] = (magnitude ? 1.0 : -1.0) * (std::exp(static_cast<double>(l[e]) - lmax) / denom) * s;
      for (int j = 0; j < k; ++j) {
        const long r = t * slots + j;
        const int e = topk_idx[r];
        if (e >= 0) dl[e] += std::exp(static_cast<double>(l[e]) - lmax) / denom * dw[r];
      }
    }
  }
  return 0;
}

}  // extern "C"
