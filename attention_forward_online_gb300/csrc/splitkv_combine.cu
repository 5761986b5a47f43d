// splitkv_combine.cu - merges split-KV partial results of the attention
// forward pass.
//
// Each key range s of a query row left a normalised partial O_s and its
// lse_s = m_s + ln l_s.  As an online-softmax state that partial is the pair
// (m, l) = (lse_s, 1) carrying O_s; the pairs are folded with the combine of
// chapter 6 "Softmax 与 Online Softmax" §6.4.1 (yangyitao.com):
//   M = max(m, lse_s); if M == -inf keep the empty state;
//   alpha = e^{m - M}, beta = e^{lse_s - M};
//   l = l alpha + beta, O = O alpha + beta O_s, m = M,
// and O / l, LSE = m + ln l at the end (a row no range could see keeps the
// (-inf, 0) identity and gets O = 0, LSE = -inf).  The fold order is the
// split order; the combine is associative, so any order gives the same
// result up to rounding.
//
// One warp per row; each lane owns d/32 consecutive columns (a float4 or
// float2 per partial), so each partial row is one coalesced 256/512-byte
// read.  O is written as bf16 or fp16, the type of the inputs.
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "osattn_internal.h"

namespace osattn {
namespace {

template <typename T>
__device__ __forceinline__ void store2(T* dst, float a, float b);
template <>
__device__ __forceinline__ void store2<__nv_bfloat16>(__nv_bfloat16* dst, float a, float b) {
  *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(a, b);
}
template <>
__device__ __forceinline__ void store2<__half>(__half* dst, float a, float b) {
  *reinterpret_cast<__half2*>(dst) = __floats2half2_rn(a, b);
}

template <int HD, typename T>
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const float* __restrict__ o_part,
                                                              const float* __restrict__ lse_part,
                                                              T* __restrict__ O,
                                                              float* __restrict__ LSE,
                                                              long long rows, int num_splits) {
  constexpr int CPL = HD / 32;  // columns per lane
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  float m = -INFINITY, l = 0.f, acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  for (int s = 0; s < num_splits; ++s) {
    const long long prow = static_cast<long long>(s) * rows + row;
    const float lse_s = lse_part[prow];
    const float M = fmaxf(m, lse_s);
    if (M == -INFINITY) continue;  // both states empty: keep (-inf, 0)
    const float alpha = expf(m - M), beta = expf(lse_s - M);
    const float* src = o_part + prow * HD + lane * CPL;
    float o_s[CPL];
    if constexpr (CPL == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      o_s[0] = v.x; o_s[1] = v.y; o_s[2] = v.z; o_s[3] = v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      o_s[0] = v.x; o_s[1] = v.y;
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = fmaf(acc[c], alpha, beta * o_s[c]);
    l = fmaf(l, alpha, beta);
    m = M;
  }
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
  T* dst = O + row * HD + lane * CPL;
#pragma unroll
  for (int c = 0; c < CPL; c += 2) store2<T>(dst + c, acc[c] * inv_l, acc[c + 1] * inv_l);
  if (lane == 0) LSE[row] = l > 0.f ? m + logf(l) : -INFINITY;
}

}  // namespace

cudaError_t launch_splitkv_combine(const float* o_part, const float* lse_part, void* O,
                                   float* LSE, long long rows, int d, int num_splits, int fp16,
                                   cudaStream_t stream) {
  constexpr int kRowsPerBlock = 8;
  const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(blocks)), b(kRowsPerBlock * 32);
  if (fp16) {
    __half* o = static_cast<__half*>(O);
    if (d == 64)
      splitkv_combine_kernel<64, __half><<<g, b, 0, stream>>>(o_part, lse_part, o, LSE, rows, num_splits);
    else
      splitkv_combine_kernel<128, __half><<<g, b, 0, stream>>>(o_part, lse_part, o, LSE, rows, num_splits);
  } else {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(O);
    if (d == 64)
      splitkv_combine_kernel<64, __nv_bfloat16><<<g, b, 0, stream>>>(o_part, lse_part, o, LSE, rows,
                                                                    num_splits);
    else
      splitkv_combine_kernel<128, __nv_bfloat16><<<g, b, 0, stream>>>(o_part, lse_part, o, LSE, rows,
                                                                     num_splits);
  }
  return cudaGetLastError();
}

}  // namespace osattn
