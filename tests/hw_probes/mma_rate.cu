// Hardware probe: the tcgen05.mma kind::f16 rate for M = 128 (one CTA) and
// M = 256 (a cta_group::2 pair) at N = 16 .. 256, issued back to back by one
// thread with no wait between K steps, on zeroed shared-memory operands on
// every SM.  It bounds what the GEMM kernels' MMA issuers can reach for each
// tile shape.  Two variants measure the cost of `commits` tcgen05.commit
// per K step (arriving on an mbarrier nobody waits on) and of spreading a K
// step's four MMAs over `chains` independent accumulators.  Prints one line
// per configuration; every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>
#include "ptx.cuh"
#include "pair_tiles.cuh"
using namespace moe;

constexpr int kSteps = 4000;  // 64-deep K steps per CTA (4 MMAs each)

template <bool kPair>
__global__ void __launch_bounds__(128, 1) probe(uint32_t n, uint32_t* status, unsigned long long* ns,
                                                 int commits, int chains) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;              // 128 x 64 bf16 = 16 KB
  uint8_t* sB = smem + 16384;      // up to 256 x 64 bf16 = 32 KB
  __shared__ uint64_t bar, bar2;
  __shared__ uint32_t slot;
  for (int i = threadIdx.x; i < 49152 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) { mbar_init(&bar, 1); mbar_init(&bar2, 1); fence_mbarrier_init(); }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  if (warp == 1) {
    if (kPair) pair::tmem_alloc2<256>(&slot); else tmem_alloc<256>(&slot);
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = slot;
  const bool leader = !kPair || cluster_ctarank() == 0;
  if (threadIdx.x == 0 && leader) {
    const uint32_t idesc = kPair ? idesc_bf16_f32(256, n) : idesc_bf16_f32(128, n);
    const uint64_t a = sw128_kmajor_desc(smem_u32(sA));
    const uint64_t b = sw128_kmajor_desc(smem_u32(sB));
    const uint64_t t0 = globaltimer_ns();
    for (int s = 0; s < kSteps; ++s) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t acc = tmem + static_cast<uint32_t>((kk % chains) * 32);
        if (kPair) pair::mma(acc, a + 2 * kk, b + 2 * kk, idesc, (s | (kk / chains)) != 0);
        else mma_bf16_ss(acc, a + 2 * kk, b + 2 * kk, idesc, (s | (kk / chains)) != 0);
      }
      for (int c = 0; c < commits; ++c) {
        if (kPair) pair::commit_local(&bar2); else mma_commit(&bar2);
      }
    }
    if (kPair) pair::commit_local(&bar); else mma_commit(&bar);
    mbar_wait(&bar, 0, status);
    const uint64_t t1 = globaltimer_ns();
    ns[blockIdx.x] = t1 - t0;
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if (kPair) pair::tmem_dealloc2<256>(tmem); else tmem_dealloc<256>(tmem);
  }
}

template <bool kPair>
void run(uint32_t n, int grid, uint32_t* status, unsigned long long* ns, int commits = 0,
         int chains = 1) {
  auto k = probe<kPair>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 50 * 1024);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 50 * 1024;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaMemset(ns, 0, sizeof(unsigned long long) * grid);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0); cudaEventCreate(&e1);
  cudaLaunchKernelEx(&cfg, k, n, status, ns, commits, chains);  // warm
  cudaEventRecord(e0);
  cudaLaunchKernelEx(&cfg, k, n, status, ns, commits, chains);
  cudaEventRecord(e1);
  cudaError_t err = cudaDeviceSynchronize();
  float ms = 0; cudaEventElapsedTime(&ms, e0, e1);
  unsigned long long h[256]; cudaMemcpy(h, ns, sizeof(unsigned long long) * grid, cudaMemcpyDeviceToHost);
  unsigned long long mx = 0; for (int i = 0; i < grid; ++i) if (h[i] > mx) mx = h[i];
  uint32_t st = 0; cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost);
  const double M = kPair ? 256 : 128;
  const int units = kPair ? grid / 2 : grid;
  const double flop = 2.0 * M * n * 64 * kSteps * units;
  printf("%s N=%3u commits=%d chains=%d grid=%3d: event %.3f ms, max in-kernel %.3f ms, %.3f us/Kstep, %.0f TFLOP/s, err=%d status=%u\n",
         kPair ? "pair  M=256" : "1-CTA M=128", n, commits, chains, grid, ms, mx / 1e6, mx / 1e3 / kSteps,
         flop / (mx * 1e-9) / 1e12, (int)err, st);
}

int main() {
  uint32_t* status; unsigned long long* ns;
  cudaMalloc(&status, 4); cudaMemset(status, 0, 4);
  cudaMalloc(&ns, 256 * sizeof(unsigned long long));
  int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  sms &= ~1;
  for (uint32_t n : {32u, 64u, 128u, 256u}) run<false>(n, sms, status, ns);
  for (uint32_t n : {32u, 64u, 128u, 256u}) run<true>(n, sms, status, ns);
  for (int c : {1, 2}) {
    for (uint32_t n : {16u, 32u, 256u}) run<false>(n, sms, status, ns, c, 1);
    for (uint32_t n : {32u, 256u}) run<true>(n, sms, status, ns, c, 1);
  }
  for (int ch : {2, 4}) {
    for (uint32_t n : {16u, 32u}) run<false>(n, sms, status, ns, 0, ch);
    run<true>(32u, sms, status, ns, 0, ch);
  }
  return 0;
}
