// softmax_rows.cu - standalone row softmax with the online (m, l) normaliser.
//
// The kernel of chapter 6 "Softmax 与 Online Softmax" (yangyitao.com) §6.4,
// re-done for GB300: every thread keeps its own (m, l) state, the states of a
// row are merged with the guarded combine of §6.4.1 (a warp butterfly, then
// across the CTA's warps through shared memory), and the row is normalised
// with the merged state.  The pages' kernel reads each element twice (§6.4,
// last paragraph); here a row of up to 32768 elements stays in registers
// between the statistics and the normalisation, so each element is read once
// and written once - the lower bound §6.2 states.
//
// Longer rows are split across the CTAs of a thread-block cluster, the
// "split-row" case of §6.7.1 with the cluster reduction it names: each CTA
// reduces its part of the row to one (m, l) state, the states meet through
// distributed shared memory and every CTA merges them with the same guarded
// combine.  Up to (cluster size) x 32768 elements the parts stay in the
// CTAs' registers (one read, one write per element); beyond that each CTA
// streams its part twice (the three accesses of §6.7.4), the second read
// served mostly by L2 because a cluster's part of the row was just read,
// with two CTAs per SM so that one part's reads overlap another's writes.
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
#include "sm100_ptx.cuh"

namespace osattn {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

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

// ---- thread-block cluster primitives (PTX)
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives, then waits; shared
// memory writes before the arrival are visible to the cluster after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// Reads a float at the same shared-memory offset in the cluster's CTA `rank`.
__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Merges the CTA-wide states (m, l) of the C CTAs of the cluster; every
// thread of every CTA returns the row's (M, L), merged in the same order
// everywhere.  sm[64..67] is this CTA's slot and a broadcast buffer.
__device__ __forceinline__ void cluster_combine(float& m, float& l, float* sm, int C) {
  if (threadIdx.x == 0) {
    sm[64] = m;
    sm[65] = l;
  }
  cluster_sync();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float mm = -INFINITY, ll = 0.f;
    if (lane < C) {
      mm = ld_dsmem_f32(sm + 64, lane);
      ll = ld_dsmem_f32(sm + 65, lane);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      combine(mm, ll, __shfl_xor_sync(kFull, mm, off), __shfl_xor_sync(kFull, ll, off));
    if (lane == 0) {
      sm[66] = mm;
      sm[67] = ll;
    }
  }
  __syncthreads();
  m = sm[66];
  l = sm[67];
  // no CTA may overwrite its slot (next row) or exit while another reads it
  cluster_sync();
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
  __shared__ float sm[68];
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
    // this thread's block: max, then the exponentials and their sum.  The
    // arithmetic runs on pairs (f32x2: one instruction for two elements,
    // the same rounding as scalar code): 16-bit rows are bound by issue.
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < E; e += 2) m = fmax3(m, v[e], v[e + 1]);
    const float base_t = m == -INFINITY ? 0.f : m;  // all-masked thread: every e^{-inf} = 0
    // e^{x - base} = 2^{x log2(e) - base log2(e)}: one fused multiply-add a pair
    const uint64_t k2 = f2_pack(kLog2e, kLog2e), nb2 = f2_pack(-base_t * kLog2e, -base_t * kLog2e);
    uint64_t l2 = 0;  // bit pattern 0 = (0.0f, 0.0f)
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      float a, b;
      f2_unpack(f2_fma(f2_pack(v[e], v[e + 1]), k2, nb2), a, b);
      v[e] = ex2_approx(a);
      v[e + 1] = ex2_approx(b);
      l2 = f2_add(l2, f2_pack(v[e], v[e + 1]));
    }
    float la, lb;
    f2_unpack(l2, la, lb);
    float l = la + lb;
    const float m_t = m;
    block_combine(m, l, sm, warps);
    // y = e^{x - m_t} * e^{m_t - M} / L  (0 for a row with no finite entry)
    const float f = l > 0.f ? __expf(m_t - m) / l : 0.f;
    const uint64_t f2 = f2_pack(f, f);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int base = (i * nt + threadIdx.x) * EPV;
      float o[EPV];
#pragma unroll
      for (int e = 0; e < EPV; e += 2)
        f2_unpack(f2_mul(f2_pack(v[i * EPV + e], v[i * EPV + e + 1]), f2), o[e], o[e + 1]);
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

// ---- rows split across a cluster of C CTAs (C = %cluster_nctarank)
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Part of the row in registers: CTA `rank` of the cluster owns elements
// [rank * chunk, rank * chunk + chunk) with chunk = blockDim.x * 32, laid out
// like softmax_rows_regs within its part.  One read and one write per
// element.  Grid-strides over rows by cluster.
template <typename T, int NV, bool kVec>
__global__ void __launch_bounds__(1024) softmax_rows_cluster_regs(const T* __restrict__ in,
                                                                  T* __restrict__ out,
                                                                  float* __restrict__ lse,
                                                                  long long rows, int N) {
  constexpr int EPV = Vec<T>::N;
  constexpr int E = NV * EPV;
  __shared__ float sm[68];
  const int nt = blockDim.x, warps = nt >> 5;
  const int C = static_cast<int>(cluster_size());
  const uint32_t rank = cluster_rank();
  const long long c0 = static_cast<long long>(rank) * nt * E;
  const int n_here = static_cast<int>(max(0LL, min(static_cast<long long>(nt) * E, N - c0)));
  for (long long row = cluster_id(); row < rows; row += cluster_count()) {
    const T* x = in + row * N + c0;
    T* y = out + row * N + c0;
    float v[E];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int base = (i * nt + threadIdx.x) * EPV;
      if (kVec) {
        if (base < n_here) Vec<T>::load(x + base, v + i * EPV);
        else
#pragma unroll
          for (int e = 0; e < EPV; ++e) v[i * EPV + e] = -INFINITY;
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          v[i * EPV + e] = base + e < n_here ? Vec<T>::get(x, base + e) : -INFINITY;
      }
    }
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < E; ++e) m = fmaxf(m, v[e]);
    const float base_t = m == -INFINITY ? 0.f : m;
    float l = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      v[e] = __expf(v[e] - base_t);
      l += v[e];
    }
    const float m_t = m;
    block_combine(m, l, sm, warps);
    cluster_combine(m, l, sm, C);
    const float f = l > 0.f ? __expf(m_t - m) / l : 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int base = (i * nt + threadIdx.x) * EPV;
      float o[EPV];
#pragma unroll
      for (int e = 0; e < EPV; ++e) o[e] = v[i * EPV + e] * f;
      if (kVec) {
        if (base < n_here) Vec<T>::store(y + base, o);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          if (base + e < n_here) Vec<T>::put(y, base + e, o[e]);
      }
    }
    if (lse && rank == 0 && threadIdx.x == 0) lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
  }
}

// Rows beyond the cluster's registers: CTA `rank` owns elements
// [rank * chunk, rank * chunk + chunk) and streams them twice - pass 1 for
// its (m, l), folded per run of kU vectors (each run's max, then the sum of
// its exponentials, combined into the thread's state), pass 2 after the
// cluster combine to write y.  Every thread keeps kU 16-byte loads in flight.
template <typename T, bool kVec>
__global__ void __launch_bounds__(1024) softmax_rows_cluster_stream(const T* __restrict__ in,
                                                                    T* __restrict__ out,
                                                                    float* __restrict__ lse,
                                                                    long long rows, int N,
                                                                    int chunk) {
  constexpr int EPV = Vec<T>::N;
  constexpr int kU = 4;
  constexpr int R = kU * EPV;  // elements per run
  __shared__ float sm[68];
  const int nt = blockDim.x, warps = nt >> 5;
  const int C = static_cast<int>(cluster_size());
  const uint32_t rank = cluster_rank();
  const long long c0 = static_cast<long long>(rank) * chunk;
  const int n_here = static_cast<int>(max(0LL, min(static_cast<long long>(chunk), N - c0)));
  const int step = nt * R;  // elements per iteration of the CTA
  for (long long row = cluster_id(); row < rows; row += cluster_count()) {
    const T* x = in + row * N + c0;
    T* y = out + row * N + c0;
    float m = -INFINITY, l = 0.f;
    for (int k0 = 0; k0 < n_here; k0 += step) {
      float r[R];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int base = k0 + (u * nt + threadIdx.x) * EPV;
        if (kVec) {
          if (base < n_here) Vec<T>::load(x + base, r + u * EPV);
          else
#pragma unroll
            for (int e = 0; e < EPV; ++e) r[u * EPV + e] = -INFINITY;
        } else {
#pragma unroll
          for (int e = 0; e < EPV; ++e)
            r[u * EPV + e] = base + e < n_here ? Vec<T>::get(x, base + e) : -INFINITY;
        }
      }
      float rm = -INFINITY;
#pragma unroll
      for (int e = 0; e < R; e += 2) rm = fmax3(rm, r[e], r[e + 1]);
      if (rm == -INFINITY) continue;  // an all-masked run leaves the state alone
      const uint64_t k2 = f2_pack(kLog2e, kLog2e), nb2 = f2_pack(-rm * kLog2e, -rm * kLog2e);
      uint64_t rl2 = 0;
#pragma unroll
      for (int e = 0; e < R; e += 2) {
        float a, b;
        f2_unpack(f2_fma(f2_pack(r[e], r[e + 1]), k2, nb2), a, b);
        rl2 = f2_add(rl2, f2_pack(ex2_approx(a), ex2_approx(b)));
      }
      float ra, rb;
      f2_unpack(rl2, ra, rb);
      combine(m, l, rm, ra + rb);
    }
    block_combine(m, l, sm, warps);
    cluster_combine(m, l, sm, C);
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    const float mb = m == -INFINITY ? 0.f : m;
    const uint64_t k2 = f2_pack(kLog2e, kLog2e), nb2 = f2_pack(-mb * kLog2e, -mb * kLog2e),
                   inv2 = f2_pack(inv_l, inv_l);
    for (int k0 = 0; k0 < n_here; k0 += step) {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int base = k0 + (u * nt + threadIdx.x) * EPV;
        float o[EPV];
        if (kVec) {
          if (base < n_here) {
            Vec<T>::load(x + base, o);
#pragma unroll
            for (int e = 0; e < EPV; e += 2) {
              float a, b;
              f2_unpack(f2_fma(f2_pack(o[e], o[e + 1]), k2, nb2), a, b);
              f2_unpack(f2_mul(f2_pack(ex2_approx(a), ex2_approx(b)), inv2), o[e], o[e + 1]);
            }
            Vec<T>::store(y + base, o);
          }
        } else {
#pragma unroll
          for (int e = 0; e < EPV; ++e)
            if (base + e < n_here) Vec<T>::put(y, base + e, __expf(Vec<T>::get(x, base + e) - mb) * inv_l);
        }
      }
    }
    if (lse && rank == 0 && threadIdx.x == 0) lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
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

// Launches `kernel` with clusters of C CTAs of `threads` threads along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kernel)(KArgs...), int C, int threads, long long rows,
                           int num_sms, cudaStream_t s, Args... args) {
  // enough clusters to cover the SMs a few times over; rows grid-stride
  const long long want = 4LL * num_sms / C;
  const long long nclusters = rows < want ? rows : (want > 0 ? want : 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * C));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kRegElems = 1024 * 32;  // elements one CTA holds in registers

template <typename T>
cudaError_t launch_any(const void* in, void* out, float* lse, long long rows, int N, int num_sms,
                       int max_cluster, cudaStream_t s) {
  constexpr int EPV = Vec<T>::N;
  constexpr int NV = 32 / EPV;  // 32 elements per thread
  const bool vec = (N % EPV) == 0 && (reinterpret_cast<uintptr_t>(in) % 16) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) % 16) == 0;
  const T* x = static_cast<const T*>(in);
  T* y = static_cast<T*>(out);
  if (N <= kRegElems) {
    const int warps = (N + 32 * 32 - 1) / (32 * 32);  // one warp per 1024 elements
    return launch_regs<T, NV>(in, out, lse, rows, N, vec, warps * 32, num_sms, s);
  }
  if (N <= static_cast<long long>(max_cluster) * kRegElems) {
    // C CTAs, each with just enough warps for its part (32 elements a thread)
    const int C = (N + kRegElems - 1) / kRegElems;
    const int per = (N + C - 1) / C;
    const int threads = ((per + 32 * 32 - 1) / (32 * 32)) * 32;
    return vec ? launch_cluster(softmax_rows_cluster_regs<T, NV, true>, C, threads, rows, num_sms,
                                s, x, y, lse, rows, N)
               : launch_cluster(softmax_rows_cluster_regs<T, NV, false>, C, threads, rows, num_sms,
                                s, x, y, lse, rows, N);
  }
  const int C = max_cluster;
  const int chunk = ((N + C - 1) / C + 7) / 8 * 8;  // a whole number of 16-byte vectors
  // 512 threads a CTA: two CTAs (two rows' parts) per SM, so one part's
  // reads overlap the other's writes and cluster barriers
  return vec ? launch_cluster(softmax_rows_cluster_stream<T, true>, C, 512, rows, 2 * num_sms, s,
                              x, y, lse, rows, N, chunk)
             : launch_cluster(softmax_rows_cluster_stream<T, false>, C, 512, rows, 2 * num_sms, s,
                              x, y, lse, rows, N, chunk);
}

template <typename T>
cudaError_t allow_large_clusters() {
  constexpr int NV = 32 / Vec<T>::N;
  cudaError_t e;

  if ((e = cudaFuncSetAttribute(softmax_rows_cluster_regs<T, NV, true>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(softmax_rows_cluster_regs<T, NV, false>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(softmax_rows_cluster_stream<T, true>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(softmax_rows_cluster_stream<T, false>,
                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

}  // namespace

cudaError_t prepare_softmax_rows(int* max_cluster) {
  cudaError_t e;
  if ((e = allow_large_clusters<float>()) != cudaSuccess ||
      (e = allow_large_clusters<__half>()) != cudaSuccess ||
      (e = allow_large_clusters<__nv_bfloat16>()) != cudaSuccess)
    return e;
  // 16 CTAs of 1024 threads where the GPU can co-schedule such a cluster,
  // else the portable 8.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(16);
  cfg.blockDim = dim3(1024);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 16;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, softmax_rows_cluster_stream<float, true>, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // a refused query is not an error: fall back to 8
    n = 0;
  }
  *max_cluster = n >= 1 ? 16 : 8;
  return cudaSuccess;
}

cudaError_t launch_softmax_rows(const void* in, void* out, float* lse, long long rows, int N,
                                int elem, int num_sms, int max_cluster, cudaStream_t stream) {
  if (elem == 1) return launch_any<float>(in, out, lse, rows, N, num_sms, max_cluster, stream);
  if (elem == 2) return launch_any<__half>(in, out, lse, rows, N, num_sms, max_cluster, stream);
  return launch_any<__nv_bfloat16>(in, out, lse, rows, N, num_sms, max_cluster, stream);
}

}  // namespace osattn
