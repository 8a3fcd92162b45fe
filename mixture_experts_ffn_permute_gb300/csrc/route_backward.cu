// Small kernels of the layer's backward around the routing: the routing
// weights in permuted-row order, and the router backward (the gradient of the
// loss with respect to the logits given d loss / d weight of each route).
//
// The top-k selection is piecewise constant and passes no gradient; the
// weights do.  For the k routed slots of a token, with dw_j the gradient of
// slot j's weight and s = sum_j w_j dw_j:
//   renormalised weights (softmax over the selected logits):
//     dl[e_j] = w_j (dw_j - s), every other expert 0;
//   full-softmax probabilities p:
//     dl[e] = p_e ([e = e_j] dw_j - s) for every expert e.
// Shared-expert slots (weight 1, after the k routed ones) pass nothing.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(256)
weights_to_rows_kernel(const int32_t* __restrict__ row_id_map, const float* __restrict__ topk_w,
                       long routes, float* __restrict__ w_perm) {
  pdl_enter();
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < routes;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const int r = row_id_map[i];
    if (r >= 0) w_perm[r] = topk_w[i];
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One warp per token.  Lane j < k holds slot j; every expert e is owned by
// lane e % 32, which alone writes dlogits[t][e].
__global__ void __launch_bounds__(256)
router_backward_kernel(const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                       const float* __restrict__ topk_w, const int32_t* __restrict__ row_id_map,
                       const float* __restrict__ dw_part, int n_parts, int T, int E, int k,
                       int slots, int renormalize, float* __restrict__ dlogits) {
  pdl_enter();
  const long t = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;  // whole warps leave together
  int ej = -1;
  float wj = 0.f, dwj = 0.f;
  if (lane < k) {
    const int e = topk_idx[t * slots + lane];
    const int r = row_id_map[t * slots + lane];
    if (e >= 0 && e < E && r >= 0) {
      ej = e;
      wj = topk_w[t * slots + lane];
      const float* part = dw_part + static_cast<long>(r) * n_parts;
      float acc = 0.f;
      for (int i = 0; i < n_parts; ++i) acc += part[i];  // fixed order
      dwj = acc;
    }
  }
  const float s = warp_sum(wj * dwj);
  float* dl = dlogits + t * E;
  if (renormalize) {
    for (int e = lane; e < E; e += 32) dl[e] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int e = __shfl_sync(0xffffffffu, ej, j);
      const float v = __shfl_sync(0xffffffffu, wj * (dwj - s), j);
      if (e >= 0 && (e & 31) == lane) dl[e] = v;
    }
  } else {
    const float* l = logits + t * E;
    float m = -INFINITY;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, l[e]);
    m = warp_max(m);
    float den = 0.f;
    for (int e = lane; e < E; e += 32) den += expf(l[e] - m);
    den = warp_sum(den);
    for (int e = lane; e < E; e += 32) dl[e] = -(expf(l[e] - m) / den) * s;
    for (int j = 0; j < k; ++j) {
      const int e = __shfl_sync(0xffffffffu, ej, j);
      const float d = __shfl_sync(0xffffffffu, dwj, j);
      if (e >= 0 && (e & 31) == lane) dl[e] += (expf(l[e] - m) / den) * d;
    }
  }
}

// d topk_w[t][j] = the route's <dOut_t, y>: the fixed-order sum of its
// row's partials; 0 for a masked slot.  One thread per slot.
__global__ void __launch_bounds__(256)
route_weight_grad_kernel(const int32_t* __restrict__ row_id_map,
                         const float* __restrict__ dw_part, int n_parts, long routes,
                         float* __restrict__ d_topk_w) {
  pdl_enter();
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < routes;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const int r = row_id_map[i];
    float acc = 0.f;
    if (r >= 0) {
      const float* part = dw_part + static_cast<long>(r) * n_parts;
      for (int q = 0; q < n_parts; ++q) acc += part[q];
    }
    d_topk_w[i] = acc;
  }
}

}  // namespace

cudaError_t launch_route_weight_grad(const int32_t* row_id_map, const float* dw_part,
                                     int n_parts, long routes, float* d_topk_w,
                                     cudaStream_t s) {
  if (routes <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<long>((routes + 255) / 256, num_sms() * 8L));
  return launch_kernel(route_weight_grad_kernel, dim3(blocks), dim3(256), 0, s, 1, row_id_map,
                       dw_part, n_parts, routes, d_topk_w);
}

cudaError_t launch_weights_to_rows(const int32_t* row_id_map, const float* topk_w, long routes,
                                   float* w_perm, cudaStream_t s) {
  if (routes <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<long>((routes + 255) / 256, num_sms() * 8L));
  return launch_kernel(weights_to_rows_kernel, dim3(blocks), dim3(256), 0, s, 1, row_id_map,
                       topk_w, routes, w_perm);
}

cudaError_t launch_router_backward(const float* logits, const int32_t* topk_idx,
                                   const float* topk_w, const int32_t* row_id_map,
                                   const float* dw_part, int n_parts, int T, int E, int k,
                                   int slots, int renormalize, float* dlogits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = ceil_div(static_cast<long>(T) * 32, 256);
  return launch_kernel(router_backward_kernel, dim3(blocks), dim3(256), 0, s, 1, logits,
                       topk_idx, topk_w, row_id_map, dw_part, n_parts, T, E, k, slots,
                       renormalize, dlogits);
}

}  // namespace moe
