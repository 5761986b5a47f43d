// fwd_fp32_simt.cu - fp32 attention forward with online softmax on the SIMT
// pipes (full-precision FMA; no tensor cores, since TF32 cannot hold the
// 1e-5 tolerance fp32 callers expect).
//
// Follows chapter 6 "Softmax 与 Online Softmax" of the hand-written
// FlashAttention v2 book (yangyitao.com): the running (m, l) state and its
// rescale by e^{m_old - m_new} (§6.3.1), the -inf guard (§6.4), the blocked
// loop carrying (m, l, O) (§6.6, exponentiating against the new max), the
// fused additive mask (§6.7.3), and LSE = m + log l (§6.5).
//
// Work split: one CTA of 4 warps owns 16 query rows of one (b, h); each warp
// owns 4 rows.  Keys stream through shared memory 32 at a time; lane j
// scores key j against the warp's rows, the warp reduces the tile max and sum
// with shuffles, and each lane accumulates d/32 output columns.  Q, K, V and
// O are addressed through element strides of their (b, h, row) axes, each a
// multiple of 4 so every row stays 16-byte aligned.
#include <cmath>
#include <cstdint>

#include "osattn_internal.h"

namespace osattn {
namespace {

constexpr int kRowsPerCta = 16;
constexpr int kRowsPerWarp = 4;
constexpr int kKeysPerTile = 32;
constexpr unsigned kFull = 0xffffffffu;

struct Strides {
  long long q[3], k[3], v[3], o[3];  // element strides of (b, h, row)
};

template <int HD>
__global__ void __launch_bounds__(128) fwd_fp32_kernel(const float* __restrict__ Q,
                                                       const float* __restrict__ K,
                                                       const float* __restrict__ V,
                                                       float* __restrict__ O,
                                                       float* __restrict__ LSE,
                                                       const int32_t* __restrict__ key_len,
                                                       int H, int Nq, int Nkv, float scale,
                                                       int causal, int num_q_tiles,
                                                       const Strides st) {
  constexpr int CPL = HD / 32;  // output columns per lane
  __shared__ float sQ[kRowsPerCta][HD];
  __shared__ float sK[kKeysPerTile][HD + 1];  // +1: lane j reads row j conflict-free
  __shared__ float sV[kKeysPerTile][HD];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long bh = blockIdx.x / num_q_tiles;
  int qt = blockIdx.x % num_q_tiles;
  if (causal) qt = num_q_tiles - 1 - qt;  // heaviest query tiles of a head first
  const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
  int kv_len = Nkv;
  if (key_len) kv_len = min(max(key_len[b], 0), Nkv);
  const int q0 = qt * kRowsPerCta;
  int kv_end = kv_len;
  if (causal) kv_end = min(kv_end, q0 + kRowsPerCta);

  const float* Qbh = Q + b * st.q[0] + h * st.q[1];
  const float* Kbh = K + b * st.k[0] + h * st.k[1];
  const float* Vbh = V + b * st.v[0] + h * st.v[1];

  for (int e = threadIdx.x; e < kRowsPerCta * HD / 4; e += blockDim.x) {
    const int r = (e * 4) / HD, c = (e * 4) % HD;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q0 + r < Nq) v = *reinterpret_cast<const float4*>(Qbh + (q0 + r) * st.q[2] + c);
    *reinterpret_cast<float4*>(&sQ[r][c]) = v;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], o[kRowsPerWarp][CPL];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) o[rr][c] = 0.f;
  }

  for (int k0 = 0; k0 < kv_end; k0 += kKeysPerTile) {
    __syncthreads();  // previous tile fully consumed (and sQ written on entry)
    for (int e = threadIdx.x; e < kKeysPerTile * HD / 4; e += blockDim.x) {
      const int r = (e * 4) / HD, c = (e * 4) % HD;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
      if (k0 + r < Nkv) {
        kv = *reinterpret_cast<const float4*>(Kbh + (k0 + r) * st.k[2] + c);
        vv = *reinterpret_cast<const float4*>(Vbh + (k0 + r) * st.v[2] + c);
      }
      sK[r][c] = kv.x; sK[r][c + 1] = kv.y; sK[r][c + 2] = kv.z; sK[r][c + 3] = kv.w;
      *reinterpret_cast<float4*>(&sV[r][c]) = vv;
    }
    __syncthreads();

    // Lane `lane` scores key k0 + lane against the warp's rows.  Four
    // interleaved partial sums per row keep the partial magnitudes (and so
    // the fp32 rounding of the logit) about four times smaller than one
    // running sum over all d products.
    const int j = k0 + lane;
    float s[kRowsPerWarp];
    {
      float acc[kRowsPerWarp][4];
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[rr][t] = 0.f;
#pragma unroll 2
      for (int c = 0; c < HD; c += 4) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float kc = sK[lane][c + t];
#pragma unroll
          for (int rr = 0; rr < kRowsPerWarp; ++rr)
            acc[rr][t] = fmaf(sQ[warp * kRowsPerWarp + rr][c + t], kc, acc[rr][t]);
        }
      }
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr)
        s[rr] = (acc[rr][0] + acc[rr][1]) + (acc[rr][2] + acc[rr][3]);
    }
    float p[kRowsPerWarp], alpha[kRowsPerWarp];
    bool changed[kRowsPerWarp];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int qi = q0 + warp * kRowsPerWarp + rr;
      float x = s[rr] * scale;
      if (j >= kv_len || (causal && j > qi)) x = -INFINITY;  // additive -inf mask
      float mx = x;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
      const float m_new = fmaxf(m[rr], mx);
      changed[rr] = false;
      alpha[rr] = 1.f;
      p[rr] = 0.f;
      if (m_new == -INFINITY) continue;  // nothing visible yet: keep (-inf, 0)
      if (m_new != m[rr]) {
        alpha[rr] = expf(m[rr] - m_new);
        changed[rr] = true;
      }
      p[rr] = expf(x - m_new);  // masked keys give exactly 0
      float ps = p[rr];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(kFull, ps, off);
      l[rr] = l[rr] * alpha[rr] + ps;
      m[rr] = m_new;
    }
    // O = O * alpha (only rows whose max moved) + P V_tile
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr)
      if (changed[rr]) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) o[rr][c] *= alpha[rr];
      }
    const int nkeys = min(kKeysPerTile, kv_end - k0);
    for (int jj = 0; jj < nkeys; ++jj) {
      float vj[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) vj[c] = sV[jj][lane + 32 * c];
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const float pj = __shfl_sync(kFull, p[rr], jj);
#pragma unroll
        for (int c = 0; c < CPL; ++c) o[rr][c] = fmaf(pj, vj[c], o[rr][c]);
      }
    }
  }

  // Epilogue: the single final O / l; a row that saw no key gets O = 0 and
  // LSE = -inf.
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int qi = q0 + warp * kRowsPerWarp + rr;
    if (qi >= Nq) continue;
    const float inv_l = l[rr] > 0.f ? 1.f / l[rr] : 0.f;
    float* orow = O + b * st.o[0] + h * st.o[1] + qi * st.o[2];
#pragma unroll
    for (int c = 0; c < CPL; ++c) orow[lane + 32 * c] = o[rr][c] * inv_l;
    if (lane == 0) LSE[bh * Nq + qi] = l[rr] > 0.f ? m[rr] + logf(l[rr]) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_fwd_fp32(const FwdArgs& a) {
  const int num_q_tiles = (a.Nq + kRowsPerCta - 1) / kRowsPerCta;
  const long long grid = static_cast<long long>(num_q_tiles) * a.B * a.H;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(grid)), blk(128);
  const float* q = static_cast<const float*>(a.Q);
  const float* k = static_cast<const float*>(a.K);
  const float* v = static_cast<const float*>(a.V);
  float* o = static_cast<float*>(a.O);
  Strides st;
  for (int i = 0; i < 3; ++i) {
    st.q[i] = a.q_strides[i];
    st.k[i] = a.k_strides[i];
    st.v[i] = a.v_strides[i];
    st.o[i] = a.o_strides[i];
  }
  if (a.d == 64)
    fwd_fp32_kernel<64><<<g, blk, 0, a.stream>>>(q, k, v, o, a.LSE, a.key_len, a.H, a.Nq, a.Nkv,
                                                 a.scale, a.causal, num_q_tiles, st);
  else
    fwd_fp32_kernel<128><<<g, blk, 0, a.stream>>>(q, k, v, o, a.LSE, a.key_len, a.H, a.Nq,
                                                  a.Nkv, a.scale, a.causal, num_q_tiles, st);
  return cudaGetLastError();
}

}  // namespace osattn
