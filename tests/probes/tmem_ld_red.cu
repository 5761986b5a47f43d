// tmem_ld_red.cu - what tcgen05.ld.red returns, against the values stored.
//
// The forward kernel takes the row max (or min, for a negative scale) of an
// unmasked score tile from its tensor-memory loads (tmem_ld_red_32x32b_x32)
// instead of a pass over the 128 values, so the result must be exactly the
// max / min of the 32 values each thread receives, with the values
// themselves unchanged.  One CTA of four warps stores a 128 x 32 fp32 tile
// (each warp its own 32 lanes) and loads it back with both reductions.
// Rows include all-negative values, -inf, an all -inf row, 1e30 and 3e38.
// Prints "values_mismatched V max_mismatched A min_mismatched B"; exit 0 when
// all three are 0.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <cuda_runtime.h>

#include "sm100_ptx.cuh"

using namespace osattn;

namespace {

constexpr int kRows = 128, kCols = 32;

__global__ void __launch_bounds__(128, 1) ld_red(const float* in, float* out_vals, float* out_max,
                                                 float* out_min) {
  __shared__ uint32_t base_s;
  const int warp = threadIdx.x >> 5, row = threadIdx.x;
  if (warp == 0) {
    tmem_alloc(&base_s, kCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t base = base_s;
  const uint32_t taddr = base + (static_cast<uint32_t>(warp * 32) << 16);  // lanes of this warp
  uint32_t v[kCols];
  for (int c = 0; c < kCols; ++c) v[c] = __float_as_uint(in[row * kCols + c]);
  tmem_st_32x32b_x32(taddr, v);
  tmem_st_wait();
  uint32_t r[kCols];
  float mx, mn;
  tmem_ld_red_32x32b_x32<true>(taddr, r, mx);
  tmem_ld_wait();
  reg_fence32(r);
  for (int c = 0; c < kCols; ++c) out_vals[row * kCols + c] = __uint_as_float(r[c]);
  tmem_ld_red_32x32b_x32<false>(taddr, r, mn);
  tmem_ld_wait();
  reg_fence32(r);
  out_max[row] = mx;
  out_min[row] = mn;
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(base, kCols);
}

uint32_t bits(float x) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  return u;
}

}  // namespace

int main() {
  constexpr int n = kRows * kCols;
  static float h[n], hv[n], hmax[kRows], hmin[kRows];
  uint32_t s = 12345u;
  for (int i = 0; i < n; ++i) {
    s = s * 1664525u + 1013904223u;
    h[i] = static_cast<float>(static_cast<int>((s >> 8) % 20001u) - 10000) * 0.37f;
  }
  for (int c = 0; c < kCols; ++c) h[5 * kCols + c] = -1.0f - c;      // all negative
  h[6 * kCols + 7] = -INFINITY;
  h[7 * kCols + 31] = 1e30f;
  h[8 * kCols + 0] = 3e38f;
  for (int c = 0; c < kCols; ++c) h[9 * kCols + c] = -INFINITY;      // all -inf
  float *din = nullptr, *dv = nullptr, *dmax = nullptr, *dmin = nullptr;
  if (cudaMalloc(&din, n * 4) || cudaMalloc(&dv, n * 4) || cudaMalloc(&dmax, kRows * 4) ||
      cudaMalloc(&dmin, kRows * 4)) {
    std::printf("cudaMalloc failed\n");
    return 2;
  }
  cudaMemcpy(din, h, n * 4, cudaMemcpyHostToDevice);
  ld_red<<<1, 128>>>(din, dv, dmax, dmin);
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    std::printf("cuda error %s\n", cudaGetErrorString(e));
    return 2;
  }
  cudaMemcpy(hv, dv, n * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(hmax, dmax, kRows * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(hmin, dmin, kRows * 4, cudaMemcpyDeviceToHost);
  int bad_v = 0, bad_max = 0, bad_min = 0;
  for (int i = 0; i < n; ++i) bad_v += bits(hv[i]) != bits(h[i]);
  for (int r = 0; r < kRows; ++r) {
    float mx = -INFINITY, mn = INFINITY;
    for (int c = 0; c < kCols; ++c) {
      mx = std::fmax(mx, h[r * kCols + c]);
      mn = std::fmin(mn, h[r * kCols + c]);
    }
    bad_max += bits(mx) != bits(hmax[r]);
    bad_min += bits(mn) != bits(hmin[r]);
  }
  std::printf("values_mismatched %d max_mismatched %d min_mismatched %d\n", bad_v, bad_max, bad_min);
  return (bad_v || bad_max || bad_min) ? 1 : 0;
}
