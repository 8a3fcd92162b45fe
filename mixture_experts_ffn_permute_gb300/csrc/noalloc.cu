// moe_permute_noalloc: the permute of moe_permute with its scratch in a
// fixed device array instead of a caller workspace, for callers that cannot
// allocate device memory (see include/moe_ffn.h).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/moe_ffn.h"
#include "internal.h"

namespace moe {
namespace {

// The one scratch array: per-chunk expert histograms (turned into row bases
// in place) followed by the m-tile prefix.  Lives as long as the library is
// loaded, on every device that loads it.
static __device__ __align__(256) int32_t g_noalloc_scratch[MOE_NOALLOC_SCRATCH_INTS];

constexpr int kMaxDevices = 64;
int32_t* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on the current device.  Host code only
// sees a host-side stand-in under the array's name, so the address is looked
// up once per device with that device current and kept for later calls (a
// device reset after that first call is therefore not supported).
int scratch_on_current_device(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
      return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<int32_t*>(ptr);
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_permute_noalloc(const moe_problem* p, const int32_t* topk_idx, const void* x,
                                   void* x_perm, int32_t* row_id_map, int32_t* permuted_token,
                                   int32_t* tokens_per_expert, int32_t* expert_offsets,
                                   void* stream) {
  using namespace moe;
  if (!p) return MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->E < 1 || p->k < 1 || p->k > p->E) return MOE_ERR_INVALID_ARG;
  if (p->shared_experts != 0) return MOE_ERR_INVALID_ARG;  // moe_forward only
  if (p->E > MOE_MAX_EXPERTS || p->k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(p->T) * p->k > (1LL << 30)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long nchunks = (static_cast<long long>(p->T) + kChunkTokens - 1) / kChunkTokens;
  const long long need = nchunks * p->E + p->E + 1;
  if (need > MOE_NOALLOC_SCRATCH_INTS) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (x_perm) {
    if (p->H <= 0 || p->H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!x || !x_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_MISALIGNED;
  }
  if (!tokens_per_expert || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if (!aligned16(tokens_per_expert) || !aligned16(expert_offsets)) return MOE_ERR_MISALIGNED;
  if (p->T > 0) {
    if (!topk_idx || !row_id_map || !permuted_token) return MOE_ERR_INVALID_ARG;
    if (!aligned16(topk_idx) || !aligned16(row_id_map) || !aligned16(permuted_token))
      return MOE_ERR_MISALIGNED;
  }
  int32_t* scratch = nullptr;
  int rc = scratch_on_current_device(&scratch);
  if (rc != MOE_OK) return rc;
  int32_t* chunk_counts = scratch;
  int32_t* mtile_prefix = scratch + nchunks * p->E;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int R = p->T * p->k;
  int launches = 0;
  // Every chunk's histogram row is written in full before the scan reads it,
  // and the scan writes the whole m-tile prefix: nothing needs clearing.
  if (nchunks > 0) {
    if (launch_chunk_histogram(topk_idx, p->T, p->E, p->k, chunk_counts, nullptr, s) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    ++launches;
  }
  if (launch_scan(chunk_counts, static_cast<int>(nchunks), p->E, R, tokens_per_expert,
                  expert_offsets, mtile_prefix, permuted_token, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  ++launches;
  if (nchunks > 0) {
    if (launch_scatter(topk_idx, p->T, p->E, p->k, chunk_counts, row_id_map, permuted_token,
                       s) != cudaSuccess)
      return MOE_ERR_CUDA;
    ++launches;
  }
  if (x_perm && p->T > 0) {
    if (launch_gather_rows(x, permuted_token, R, p->H, x_perm, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    ++launches;
  }
  set_last_launch_count(launches);
  return MOE_OK;
}
