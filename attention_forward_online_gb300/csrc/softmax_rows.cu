// softmax_rows.cu - standalone row softmax with the online (m, l) normaliser.
//
// The kernel of chapter 6 "Softmax 与 Online Softmax" (yangyitao.com) §6.4,
// re-done for GB300: every thread keeps its own (m, l) state, the states of a
// row are merged with the guarded combine of §6.4.1 (a warp butterfly, then
// across the CTA's warps through shared memory), and the row is normalised
// with the merged state.  The pages' kernel reads each element twice (§6.4,
// last paragraph); here a row of up to 32768 elements stays in registers
// between the statistics and the normalisation, so each element is read once
// and written once - the lower bound §6.2 states.  Longer rows use a
// streaming variant that reads twice (the online softmax's three accesses per
// element, §6.7.4).
//
// Inside one thread the elements are a block: its max first, then
// sum e^{x - m_t}, which is the blocked form of the recurrence (§6.6); the
// exponentials are kept and rescaled by e^{m_t - M} / L at the end, so each
// element costs one exponential.  A row whose elements are all -inf keeps the
// (-inf, 0) state; its output is 0 and its LSE -inf (never NaN).
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "osattn_internal.h"

namespace osattn {
namespace {

constexpr int kThreads = 256;  // streaming kernel
constexpr unsigned kFull = 0xffffffffu;

// The combine of two (m, l) states, branch-free: when both are empty the
// exponent base is taken as 0 instead of -inf, so e^{-inf - 0} = 0 keeps
// (-inf, 0) with no -inf - (-inf) = NaN (the guard of the combine).
__device__ __forceinline__ void combine(float& m, float& l, float m2, float l2) {
  const float M = fmaxf(m, m2);
  const float base = M == -INFINITY ? 0.f : M;
  l = l * __expf(m - base) + l2 * __expf(m2 - base);
  m = M;
}

// Merges the per-thread states of a CTA of `warps` warps; every thread
// returns the row's (M, L).
__device__ __forceinline__ void block_combine(float& m, float& l, float* sm, int warps) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    combine(m, l, __shfl_xor_sync(kFull, m, off), __shfl_xor_sync(kFull, l, off));
  if (warps == 1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sm[2 * warp] = m;
    sm[2 * warp + 1] = l;
  }
  __syncthreads();
  m = lane < warps ? sm[2 * lane] : -INFINITY;
  l = lane < warps ? sm[2 * lane + 1] : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    combine(m, l, __shfl_xor_sync(kFull, m, off), __shfl_xor_sync(kFull, l, off));
  __syncthreads();  // sm is reused for the next row
}

template <typename T>
struct Vec;  // 16-byte vector of T
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void load(const float* p, float* v) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  }
  __device__ static void store(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
  __device__ static float get(const float* p, long long i) { return p[i]; }
  __device__ static void put(float* p, long long i, float v) { p[i] = v; }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16* p, float* v) {
    const uint4 x = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float* v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ static float get(const __nv_bfloat16* p, long long i) { return __bfloat162float(p[i]); }
  __device__ static void put(__nv_bfloat16* p, long long i, float v) { p[i] = __float2bfloat16_rn(v); }
};
template <>
struct Vec<__half> {
  static constexpr int N = 8;
  __device__ static void load(const __half* p, float* v) {
    const uint4 x = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
  __device__ static void store(__half* p, const float* v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ static float get(const __half* p, long long i) { return __half2float(p[i]); }
  __device__ static void put(__half* p, long long i, float v) { p[i] = __float2half_rn(v); }
};

// Row held in registers: each thread owns NV 16-byte vectors (32 elements),
// the CTA has just enough warps for the row (blockDim = 32 * warps), so a
// short row costs a small combine and many rows run per SM.  Vector access
// when the row start is 16-byte aligned and N a multiple of the vector
// width; element access otherwise.  Grid-strides over rows.
template <typename T, int NV, bool kVec>
__global__ void __launch_bounds__(1024) softmax_rows_regs(const T* __restrict__ in,
                                                          T* __restrict__ out,
                                                          float* __restrict__ lse,
                                                          long long rows, int N) {
  constexpr int EPV = Vec<T>::N;
  constexpr int E = NV * EPV;  // elements per thread
  __shared__ float sm[64];
  const int nt = blockDim.x, warps = nt >> 5;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const T* x = in + row * N;
    T* y = out + row * N;
    float v[E];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int base = (i * nt + threadIdx.x) * EPV;  // vector-strided over the CTA
      if (kVec) {
        if (base < N) Vec<T>::load(x + base, v + i * EPV);
        else
#pragma unroll
          for (int e = 0; e < EPV; ++e) v[i * EPV + e] = -INFINITY;
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          v[i * EPV + e] = base + e < N ? Vec<T>::get(x, base + e) : -INFINITY;
      }
    }
    // this thread's block: max, then the exponentials and their sum
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < E; ++e) m = fmaxf(m, v[e]);
    const float base_t = m == -INFINITY ? 0.f : m;  // all-masked thread: every e^{-inf} = 0
    float l = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      v[e] = __expf(v[e] - base_t);
      l += v[e];
    }
    const float m_t = m;
    block_combine(m, l, sm, warps);
    // y = e^{x - m_t} * e^{m_t - M} / L  (0 for a row with no finite entry)
    const float f = l > 0.f ? __expf(m_t - m) / l : 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int base = (i * nt + threadIdx.x) * EPV;
      float o[EPV];
#pragma unroll
      for (int e = 0; e < EPV; ++e) o[e] = v[i * EPV + e] * f;
      if (kVec) {
        if (base < N) Vec<T>::store(y + base, o);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          if (base + e < N) Vec<T>::put(y, base + e, o[e]);
      }
    }
    if (lse && threadIdx.x == 0) lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
  }
}

// Rows longer than the register budget: pass 1 streams the row once for the
// per-thread (m, l) (blockwise per element run, combined as it goes), pass 2
// reads it again and writes y.  Scalar element access (any N, any alignment).
template <typename T>
__global__ void __launch_bounds__(kThreads) softmax_rows_stream(const T* __restrict__ in,
                                                                T* __restrict__ out,
                                                                float* __restrict__ lse,
                                                                long long rows, int N) {
  constexpr int kRun = 8;  // elements folded per combine step
  __shared__ float sm[64];
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const T* x = in + row * N;
    T* y = out + row * N;
    float m = -INFINITY, l = 0.f;
    for (int i0 = threadIdx.x * kRun; i0 < N; i0 += kThreads * kRun) {
      float r[kRun];
      float rm = -INFINITY;
#pragma unroll
      for (int e = 0; e < kRun; ++e) {
        r[e] = i0 + e < N ? Vec<T>::get(x, i0 + e) : -INFINITY;
        rm = fmaxf(rm, r[e]);
      }
      if (rm == -INFINITY) continue;  // an all-masked run leaves the state alone
      float rl = 0.f;
#pragma unroll
      for (int e = 0; e < kRun; ++e) rl += __expf(r[e] - rm);
      combine(m, l, rm, rl);
    }
    block_combine(m, l, sm, kThreads / 32);
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    for (int i0 = threadIdx.x * kRun; i0 < N; i0 += kThreads * kRun) {
#pragma unroll
      for (int e = 0; e < kRun; ++e)
        if (i0 + e < N) {
          const float xv = Vec<T>::get(x, i0 + e);
          Vec<T>::put(y, i0 + e, l > 0.f ? __expf(xv - m) * inv_l : 0.f);
        }
    }
    if (lse && threadIdx.x == 0) lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
  }
}

template <typename T, int NV>
cudaError_t launch_regs(const void* in, void* out, float* lse, long long rows, int N, bool vec,
                        int threads, int num_sms, cudaStream_t s) {
  const T* x = static_cast<const T*>(in);
  T* y = static_cast<T*>(out);
  // enough CTAs for every SM to keep many rows' loads in flight
  const long long want = static_cast<long long>(num_sms) * (2048 / threads) * 2;
  const int grid = static_cast<int>(rows < want ? rows : want);
  if (vec)
    softmax_rows_regs<T, NV, true><<<grid, threads, 0, s>>>(x, y, lse, rows, N);
  else
    softmax_rows_regs<T, NV, false><<<grid, threads, 0, s>>>(x, y, lse, rows, N);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_any(const void* in, void* out, float* lse, long long rows, int N, int num_sms,
                       cudaStream_t s) {
  constexpr int EPV = Vec<T>::N;
  constexpr int NV = 32 / EPV;  // 32 elements per thread
  const bool vec = (N % EPV) == 0 && (reinterpret_cast<uintptr_t>(in) % 16) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) % 16) == 0;
  if (N <= 1024 * 32) {
    const int warps = (N + 32 * 32 - 1) / (32 * 32);  // one warp per 1024 elements
    return launch_regs<T, NV>(in, out, lse, rows, N, vec, warps * 32, num_sms, s);
  }
  const long long want = static_cast<long long>(num_sms) * 8;
  const int grid = static_cast<int>(rows < want ? rows : want);
  softmax_rows_stream<T><<<grid, kThreads, 0, s>>>(static_cast<const T*>(in), static_cast<T*>(out),
                                                  lse, rows, N);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_softmax_rows(const void* in, void* out, float* lse, long long rows, int N,
                                int elem, int num_sms, cudaStream_t stream) {
  if (elem == 1) return launch_any<float>(in, out, lse, rows, N, num_sms, stream);
  if (elem == 2) return launch_any<__half>(in, out, lse, rows, N, num_sms, stream);
  return launch_any<__nv_bfloat16>(in, out, lse, rows, N, num_sms, stream);
}

}  // namespace osattn
