// Hardware probe: the HBM streaming rate of K-major bulk-tensor weight loads
// as the GEMM producers issue them -- 64-column boxes of 128 rows (128-byte
// rows, mode 0) against 3-D boxes of two 64-column planes (256-byte rows,
// mode 1) -- for two row strides, 8 to 152 streaming CTAs and two ring
// depths.  Each CTA streams its own block of rows; a consumer thread releases
// every stage as soon as it lands.  Every wait is bounded, and the consumer
// drains every issued copy before the CTA exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>
#include <vector>
#include "ptx.cuh"
using namespace moe;

typedef CUresult (*EncFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                          const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                          CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

__device__ __forceinline__ void tma3(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// mode 0: 2-D boxes 64 cols x 128 rows (16 KB) per stage
// mode 1: 3-D boxes 64 cols x 128 rows x 2 column blocks (32 KB) per stage
__global__ void __launch_bounds__(64, 1)
stream_kernel(const __grid_constant__ CUtensorMap map, int mode, int stages, int rows_per_cta, int K,
              uint32_t* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t full[16], empty[16];
  const uint32_t sbytes = mode == 0 ? 16384u : 32768u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    fence_mbarrier_init();
  }
  __syncthreads();
  const int kblk_per = mode == 0 ? 1 : 2;
  const int nkb = K / 64 / kblk_per;
  const int tiles = rows_per_cta / 128;
  const int row0 = blockIdx.x * rows_per_cta;
  if (threadIdx.x == 0) {
    int stage = 0; uint32_t phase = 0;
    for (int t = 0; t < tiles; ++t)
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1, status)) return;
        mbar_arrive_expect_tx(&full[stage], sbytes);
        uint8_t* dst = smem + stage * sbytes;
        if (mode == 0) tma_load_2d(dst, &map, kb * 64, row0 + t * 128, &full[stage], policy_evict_first());
        else tma3(dst, &map, 0, row0 + t * 128, kb * 2, &full[stage]);
        if (++stage == stages) { stage = 0; phase ^= 1; }
      }
  } else if (threadIdx.x == 32) {
    int stage = 0; uint32_t phase = 0;
    for (int t = 0; t < tiles; ++t)
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&full[stage], phase, status)) return;
        mbar_arrive(&empty[stage]);
        if (++stage == stages) { stage = 0; phase ^= 1; }
      }
  }
}

int main() {
  cudaSetDevice(0);
  int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  EncFn enc = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&enc, 12000, cudaEnableDefault, &q);
  if (!enc) { printf("no encode fn\n"); return 1; }
  uint32_t* status; cudaMalloc(&status, 4); cudaMemset(status, 0, 4);
  const int Ks[] = {2048, 7168};
  const size_t max_bytes = (size_t)3 << 30;
  void* buf; if (cudaMalloc(&buf, max_bytes) != cudaSuccess) { printf("alloc\n"); return 1; }
  cudaMemset(buf, 0, max_bytes);
  cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  for (int K : Ks) {
    // rows per CTA: about 8 MB per CTA, a multiple of 128
    int rows_per_cta = (int)((8u << 20) / (K * 2)) / 128 * 128;
    if (rows_per_cta < 128) rows_per_cta = 128;
    size_t rows = (size_t)rows_per_cta * sms;
    if (rows * K * 2 > max_bytes) { printf("K=%d too big\n", K); continue; }
    for (int mode = 0; mode < 2; ++mode) {
      CUtensorMap map;
      CUresult r;
      if (mode == 0) {
        cuuint64_t dims[2] = {(cuuint64_t)K, rows};
        cuuint64_t str[1] = {(cuuint64_t)K * 2};
        cuuint32_t box[2] = {64, 128}, es[2] = {1, 1};
        r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, buf, dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      } else {
        cuuint64_t dims[3] = {64, rows, (cuuint64_t)K / 64};
        cuuint64_t str[2] = {(cuuint64_t)K * 2, 128};
        cuuint32_t box[3] = {64, 128, 2}, es[3] = {1, 1, 1};
        r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, buf, dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      }
      if (r != CUDA_SUCCESS) { printf("K=%d mode=%d encode failed %d\n", K, mode, (int)r); continue; }
      const int stage_list[] = {6, 10};
      const int grid_list[] = {8, 32, 64, 96, 152};
      for (int grid : grid_list)
      for (int stages : stage_list) {
        const uint32_t sbytes = mode == 0 ? 16384u : 32768u;
        int st = stages;
        if (mode == 1) st = stages / 2 > 0 ? stages / 2 : 1;  // same bytes in flight
        size_t smem = 1024 + (size_t)st * sbytes;
        cudaEvent_t a, b; cudaEventCreate(&a); cudaEventCreate(&b);
        float best = 1e9f;
        for (int rep = 0; rep < 4; ++rep) {
          cudaEventRecord(a);
          stream_kernel<<<grid, 64, smem>>>(map, mode, st, rows_per_cta, K, status);
          cudaEventRecord(b);
          cudaEventSynchronize(b);
          float ms; cudaEventElapsedTime(&ms, a, b);
          if (rep > 0 && ms < best) best = ms;
        }
        cudaError_t e = cudaGetLastError();
        uint32_t hs = 0; cudaMemcpy(&hs, status, 4, cudaMemcpyDeviceToHost);
        double gb = (double)rows_per_cta * grid * K * 2 / 1e9;
        printf("K=%5d mode=%d grid=%3d stages=%2d (%3zu KB/SM): %.3f ms  %.0f GB/s total, %.1f GB/s per CTA err=%d status=%u\n", K, mode, grid, st,
               (size_t)st * sbytes / 1024, best, gb / (best / 1e3), gb / (best / 1e3) / grid, (int)e, hs);
      }
    }
  }
  return 0;
}
