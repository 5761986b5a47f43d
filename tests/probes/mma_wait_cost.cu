// mma_wait_cost.cu - what an mbarrier wait between groups of tcgen05 MMAs
// costs the tensor pipe, with the issuing loop in a lane-0 branch or run by
// the whole warp (elect.sync picking the issuing lane).
//
// One CTA per SM.  A step is four groups of eight 128x128x16 bf16 MMAs in
// the forward kernel's shapes (P V with A from tensor memory, then S = Q K^T
// from shared memory, for two query tiles), 2048 cycles of tensor work;
// each group is committed to its own mbarrier.  Modes:
//   0  no waits
//   1  one thread (lane 0 branch) waits on an already-completed mbarrier
//      before every group
//   2  the whole warp waits on it before every group; MMAs and commits
//      issued by the elected lane
// Prints "mode M err=E cycles_per_step C" per mode (average over SMs).
// Every loop is bounded; operands are constant bf16 values in shared memory.
#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sm100_ptx.cuh"
#include "tc_attn_mma.cuh"

using namespace osattn;

namespace {

__device__ __forceinline__ bool gate(uint64_t* bar) {
  for (uint32_t it = 0; it < (1u << 26); ++it)
    if (mbar_try_wait(bar, 0)) return true;
  return false;
}

template <int kMode>
__global__ void __launch_bounds__(128, 1) wait_cost(int steps, unsigned long long* cycles,
                                                    unsigned int* bad) {
  constexpr bool kWarp = kMode == 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t done_bar, bars[4], drain;
  __shared__ uint32_t tbase;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Q0, Q1 (32 KB each) and two K/V stages (32 KB each): bf16 1.0 everywhere
  for (int i = threadIdx.x; i < 131072 / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(smem)[i] = 0x3f803f80u;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
    mbar_init(&drain, 1);
    mbar_init(&done_bar, 1);
    fence_barrier_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {
    tmem_alloc(&tbase, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tbase;
  if (threadIdx.x == 0) mbar_arrive(&done_bar);  // its phase 0 is complete from here on
  __syncthreads();
  const uint64_t q0 = sdesc_sw128(smem_u32(smem), 16, 1024), q1 = q0 + (32768 >> 4);
  const uint64_t kd = sdesc_sw128(smem_u32(smem + 65536), 16, 1024);
  const uint64_t vd = sdesc_sw128(smem_u32(smem + 65536), 128 * 128, 1024);
  const bool issuer = kWarp ? warp == 1 : (warp == 1 && lane == 0);
  if (issuer) {
    unsigned int nbad = 0;
    const unsigned long long t0 = clock64();
    for (int j = 0; j < steps; ++j) {
      const uint64_t stage = static_cast<uint64_t>((j % 2) * (32768 >> 4));
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int t = g >> 1;
        if constexpr (kMode != 0) {
          bool ok = gate(&done_bar);
          if constexpr (kWarp) ok = __all_sync(0xffffffffu, ok);
          nbad += ok ? 0u : 1u;
        }
        if ((g & 1) == 0)  // O_t += P_t V
          mma_tmem_a_128<128, false, kWarp>(tmem + 256 + t * 128, tmem + t * 128, vd + stage,
                                            true);
        else  // S_t = Q_t K^T
          mma_abt_128<128, false, kWarp>(tmem + t * 128, t ? q1 : q0, kd + stage);
        mma_commit<kWarp>(&bars[g]);
      }
    }
    mma_commit<kWarp>(&drain);
    for (long it = 0; it < 100000000 && !mbar_try_wait(&drain, 0); ++it) {
    }
    if (lane == 0) {
      cycles[blockIdx.x] = clock64() - t0;
      if (nbad) atomicAdd(bad, nbad);
    }
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int kMode>
int run(int sms, unsigned long long* d_cycles, unsigned int* d_bad) {
  const int smem = 131072 + 2048, steps = 500;
  cudaFuncSetAttribute(wait_cost<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaMemset(d_bad, 0, sizeof(unsigned int));
  wait_cost<kMode><<<sms, 128, smem>>>(steps, d_cycles, d_bad);
  const cudaError_t e = cudaDeviceSynchronize();
  unsigned long long h[1024] = {};
  unsigned int hb = 0;
  cudaMemcpy(h, d_cycles, sms * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  cudaMemcpy(&hb, d_bad, sizeof(unsigned int), cudaMemcpyDeviceToHost);
  double avg = 0;
  for (int i = 0; i < sms; ++i) avg += static_cast<double>(h[i]);
  avg /= sms;
  std::printf("mode %d err=%d bad=%u cycles_per_step %.0f\n", kMode, static_cast<int>(e), hb,
              avg / steps);
  return e == cudaSuccess && hb == 0 ? 0 : 1;
}

}  // namespace

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  if (sms <= 0 || sms > 1024) return 2;
  unsigned long long* d_cycles = nullptr;
  unsigned int* d_bad = nullptr;
  cudaMalloc(&d_cycles, 1024 * sizeof(unsigned long long));
  cudaMalloc(&d_bad, sizeof(unsigned int));
  int rc = run<0>(sms, d_cycles, d_bad);
  if (rc == 0) rc = run<1>(sms, d_cycles, d_bad);
  if (rc == 0) rc = run<2>(sms, d_cycles, d_bad);
  cudaFree(d_cycles);
  cudaFree(d_bad);
  return rc;
}
