// bwd_fp32_simt.cu - fp32 gradients of the attention forward pass (dQ, dK,
// dV) on the SIMT pipes, for callers of the fp32 forward: full-precision
// FMAs and expf, no tensor cores (TF32 cannot hold fp32 accuracy).
//
// Same chain rule as the tensor-core kernels (the forward keeps one number
// per query row, LSE = m + ln l: chapter 6 "Softmax 与 Online Softmax" of the
// hand-written FlashAttention v2 book, §6.5; the scores are recomputed, as
// m.xxqk.cn/news/563265 §5.2 describes):
//   P_ij = e^{scale <Q_i, K_j> - LSE_i} on the visible keys,
//   dS_ij = P_ij (<dO_i, V_j> - D_i),  D_i = <dO_i, O_i>  (bwd_rowdot_kernel),
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij Q_i,  dQ_i = scale sum_j dS_ij K_j.
//
// bwd_fp32_dkdv_kernel: one CTA of 8 warps per 32 keys of a (b, h), K and V
//   of those keys in shared memory; query rows stream through shared memory
//   32 at a time.  Lane i scores query i against each of its warp's 4 keys,
//   then the warp folds P and dS of the 32 queries into dV and dK, each lane
//   holding d/32 columns.
// bwd_fp32_dq_kernel: one CTA of 8 warps per 32 queries, key rows streaming;
//   lane j scores key j against each of its warp's 4 queries and the warp
//   folds dS into dQ the same way.
// Every output element is written once by one thread: no atomics, results
// are deterministic.  Tensors are addressed through element strides of their
// (b, h, row) axes (multiples of 4, so rows stay 16-byte aligned).
#include <cmath>
#include <cstdint>

#include "osattn_internal.h"

namespace osattn {
namespace {

constexpr int kTile = 32;                 // keys (dK/dV) or queries (dQ) per CTA; streamed rows per step
constexpr int kWarps = 8;
constexpr int kPerWarp = kTile / kWarps;  // rows a warp owns
constexpr unsigned kFull = 0xffffffffu;

struct Strides8 {
  long long q[3], k[3], v[3], g[3], dq[3], dk[3], dv[3];  // (b, h, row); g = dO
};

template <int HD>
constexpr int fp32_bwd_smem_bytes() {
  return (4 * kTile * (HD + 1) + 2 * kTile) * static_cast<int>(sizeof(float));
}

// rows row0 .. row0 + 31 of a [N, HD] slice into dst[32][HD + 1] (zeros past N)
template <int HD>
__device__ __forceinline__ void load_tile(float (*dst)[HD + 1], const float* base, long long rs,
                                          int row0, int N) {
  for (int idx = threadIdx.x; idx < kTile * HD; idx += blockDim.x) {
    const int r = idx / HD, c = idx - r * HD;
    const int row = row0 + r;
    dst[r][c] = row < N ? base[row * rs + c] : 0.f;
  }
}

__device__ __forceinline__ bool visible(int i, int j, int Nq, int kv_len, int causal) {
  return i < Nq && j < kv_len && (!causal || j <= i);
}

template <int HD>
__global__ void __launch_bounds__(kWarps * 32) bwd_fp32_dkdv_kernel(
    const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
    const float* __restrict__ dO, const float* __restrict__ LSE, const float* __restrict__ D,
    float* __restrict__ dK, float* __restrict__ dV, const int32_t* __restrict__ key_len, int H,
    int Nq, int Nkv, float scale, int causal, int num_tiles, const Strides8 st) {
  constexpr int CPL = HD / 32;
  extern __shared__ float sm[];
  float(*sK)[HD + 1] = reinterpret_cast<float(*)[HD + 1]>(sm);
  float(*sV)[HD + 1] = sK + kTile;
  float(*sQ)[HD + 1] = sV + kTile;
  float(*sG)[HD + 1] = sQ + kTile;
  float* sL = reinterpret_cast<float*>(sG + kTile);
  float* sD = sL + kTile;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long bh = blockIdx.x / num_tiles;
  const int kt = blockIdx.x % num_tiles;
  const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
  const int kv_len = key_len ? min(max(key_len[b], 0), Nkv) : Nkv;
  const int k0 = kt * kTile;

  load_tile<HD>(sK, K + b * st.k[0] + h * st.k[1], st.k[2], k0, Nkv);
  load_tile<HD>(sV, V + b * st.v[0] + h * st.v[1], st.v[2], k0, Nkv);
  const float* Qbh = Q + b * st.q[0] + h * st.q[1];
  const float* Gbh = dO + b * st.g[0] + h * st.g[1];

  float accV[kPerWarp][CPL], accK[kPerWarp][CPL];
#pragma unroll
  for (int r = 0; r < kPerWarp; ++r)
#pragma unroll
    for (int m = 0; m < CPL; ++m) accV[r][m] = accK[r][m] = 0.f;

  // Queries that can see a key of this tile: all, or (causal) those at or
  // after its first key.
  const int i_first = k0 < kv_len ? (causal ? (k0 / kTile) * kTile : 0) : Nq;
  for (int i0 = i_first; i0 < Nq; i0 += kTile) {
    __syncthreads();  // the previous query tile is consumed (and K, V are loaded)
    load_tile<HD>(sQ, Qbh, st.q[2], i0, Nq);
    load_tile<HD>(sG, Gbh, st.g[2], i0, Nq);
    if (threadIdx.x < kTile) {
      const int i = i0 + threadIdx.x;
      sL[threadIdx.x] = i < Nq ? LSE[bh * Nq + i] : -INFINITY;
      sD[threadIdx.x] = i < Nq ? D[bh * Nq + i] : 0.f;
    }
    __syncthreads();
    const int i = i0 + lane;  // this lane's query
    const float Li = sL[lane], Di = sD[lane];
#pragma unroll
    for (int r = 0; r < kPerWarp; ++r) {
      const int kr = warp * kPerWarp + r;  // key row in the tile
      float s = 0.f, dp = 0.f;
#pragma unroll 4
      for (int c = 0; c < HD; ++c) {
        s = fmaf(sQ[lane][c], sK[kr][c], s);
        dp = fmaf(sG[lane][c], sV[kr][c], dp);
      }
      const bool vis = visible(i, k0 + kr, Nq, kv_len, causal) && Li != -INFINITY;
      const float p = vis ? expf(s * scale - Li) : 0.f;
      const float ds = p * (dp - Di);
#pragma unroll 2
      for (int qq = 0; qq < kTile; ++qq) {
        const float pq = __shfl_sync(kFull, p, qq), dq = __shfl_sync(kFull, ds, qq);
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
          accV[r][m] = fmaf(pq, sG[qq][lane + 32 * m], accV[r][m]);
          accK[r][m] = fmaf(dq, sQ[qq][lane + 32 * m], accK[r][m]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kPerWarp; ++r) {
    const int j = k0 + warp * kPerWarp + r;
    if (j >= Nkv) continue;
    float* dv = dV + b * st.dv[0] + h * st.dv[1] + j * st.dv[2];
    float* dk = dK + b * st.dk[0] + h * st.dk[1] + j * st.dk[2];
#pragma unroll
    for (int m = 0; m < CPL; ++m) {
      dv[lane + 32 * m] = accV[r][m];
      dk[lane + 32 * m] = accK[r][m] * scale;
    }
  }
}

template <int HD>
__global__ void __launch_bounds__(kWarps * 32) bwd_fp32_dq_kernel(
    const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
    const float* __restrict__ dO, const float* __restrict__ LSE, const float* __restrict__ D,
    float* __restrict__ dQ, const int32_t* __restrict__ key_len, int H, int Nq, int Nkv,
    float scale, int causal, int num_tiles, const Strides8 st) {
  constexpr int CPL = HD / 32;
  extern __shared__ float sm[];
  float(*sQ)[HD + 1] = reinterpret_cast<float(*)[HD + 1]>(sm);
  float(*sG)[HD + 1] = sQ + kTile;
  float(*sK)[HD + 1] = sG + kTile;
  float(*sV)[HD + 1] = sK + kTile;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long bh = blockIdx.x / num_tiles;
  int qt = blockIdx.x % num_tiles;
  if (causal) qt = num_tiles - 1 - qt;  // the longest key loops first
  const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
  const int kv_len = key_len ? min(max(key_len[b], 0), Nkv) : Nkv;
  const int q0 = qt * kTile;
  int kv_end = kv_len;
  if (causal) kv_end = min(kv_end, q0 + kTile);

  load_tile<HD>(sQ, Q + b * st.q[0] + h * st.q[1], st.q[2], q0, Nq);
  load_tile<HD>(sG, dO + b * st.g[0] + h * st.g[1], st.g[2], q0, Nq);
  float Lr[kPerWarp], Dr[kPerWarp];
#pragma unroll
  for (int r = 0; r < kPerWarp; ++r) {
    const int i = q0 + warp * kPerWarp + r;
    Lr[r] = i < Nq ? LSE[bh * Nq + i] : -INFINITY;
    Dr[r] = i < Nq ? D[bh * Nq + i] : 0.f;
  }
  const float* Kbh = K + b * st.k[0] + h * st.k[1];
  const float* Vbh = V + b * st.v[0] + h * st.v[1];

  float acc[kPerWarp][CPL];
#pragma unroll
  for (int r = 0; r < kPerWarp; ++r)
#pragma unroll
    for (int m = 0; m < CPL; ++m) acc[r][m] = 0.f;

  for (int j0 = 0; j0 < kv_end; j0 += kTile) {
    __syncthreads();  // the previous key tile is consumed (and Q, dO are loaded)
    load_tile<HD>(sK, Kbh, st.k[2], j0, Nkv);
    load_tile<HD>(sV, Vbh, st.v[2], j0, Nkv);
    __syncthreads();
    const int j = j0 + lane;  // this lane's key
#pragma unroll
    for (int r = 0; r < kPerWarp; ++r) {
      const int qr = warp * kPerWarp + r;
      float s = 0.f, dp = 0.f;
#pragma unroll 4
      for (int c = 0; c < HD; ++c) {
        s = fmaf(sQ[qr][c], sK[lane][c], s);
        dp = fmaf(sG[qr][c], sV[lane][c], dp);
      }
      const bool vis = visible(q0 + qr, j, Nq, kv_len, causal) && Lr[r] != -INFINITY;
      const float p = vis ? expf(s * scale - Lr[r]) : 0.f;
      const float ds = p * (dp - Dr[r]);
#pragma unroll 2
      for (int kk = 0; kk < kTile; ++kk) {
        const float dk = __shfl_sync(kFull, ds, kk);
#pragma unroll
        for (int m = 0; m < CPL; ++m) acc[r][m] = fmaf(dk, sK[kk][lane + 32 * m], acc[r][m]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kPerWarp; ++r) {
    const int i = q0 + warp * kPerWarp + r;
    if (i >= Nq) continue;
    float* dq = dQ + b * st.dq[0] + h * st.dq[1] + i * st.dq[2];
#pragma unroll
    for (int m = 0; m < CPL; ++m) dq[lane + 32 * m] = acc[r][m] * scale;
  }
}

template <int HD>
cudaError_t set_fp32_attrs() {
  cudaError_t e = cudaFuncSetAttribute(bwd_fp32_dkdv_kernel<HD>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       fp32_bwd_smem_bytes<HD>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(bwd_fp32_dq_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fp32_bwd_smem_bytes<HD>());
}

template <int HD>
cudaError_t launch_fp32_t(const BwdArgs& a, const Strides8& st) {
  const int nk = (a.Nkv + kTile - 1) / kTile, nq = (a.Nq + kTile - 1) / kTile;
  const long long gk = static_cast<long long>(nk) * a.B * a.H;
  const long long gq = static_cast<long long>(nq) * a.B * a.H;
  if (gk > 0x7fffffffLL || gq > 0x7fffffffLL) return cudaErrorInvalidValue;
  const float* Q = static_cast<const float*>(a.Q);
  const float* K = static_cast<const float*>(a.K);
  const float* V = static_cast<const float*>(a.V);
  const float* G = static_cast<const float*>(a.dO);
  bwd_fp32_dkdv_kernel<HD><<<static_cast<unsigned>(gk), kWarps * 32, fp32_bwd_smem_bytes<HD>(),
                             a.stream>>>(Q, K, V, G, a.LSE, a.D, static_cast<float*>(a.dK),
                                         static_cast<float*>(a.dV), a.key_len, a.H, a.Nq, a.Nkv,
                                         a.scale, a.causal, nk, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_fp32_dq_kernel<HD><<<static_cast<unsigned>(gq), kWarps * 32, fp32_bwd_smem_bytes<HD>(),
                           a.stream>>>(Q, K, V, G, a.LSE, a.D, static_cast<float*>(a.dQ), a.key_len,
                                       a.H, a.Nq, a.Nkv, a.scale, a.causal, nq, st);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prepare_bwd_fp32() {
  cudaError_t e = set_fp32_attrs<64>();
  if (e != cudaSuccess) return e;
  return set_fp32_attrs<128>();
}

cudaError_t launch_bwd_fp32(const BwdArgs& a) {
  Strides8 st;
  for (int i = 0; i < 3; ++i) {
    st.q[i] = a.q_strides[i];
    st.k[i] = a.k_strides[i];
    st.v[i] = a.v_strides[i];
    st.g[i] = a.do_strides[i];
    st.dq[i] = a.dq_strides[i];
    st.dk[i] = a.dk_strides[i];
    st.dv[i] = a.dv_strides[i];
  }
  cudaError_t e = launch_bwd_rowdot_fp32(a);
  if (e != cudaSuccess) return e;
  return a.d == 64 ? launch_fp32_t<64>(a, st) : launch_fp32_t<128>(a, st);
}

}  // namespace osattn
