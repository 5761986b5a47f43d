// fwd_bf16_tcgen05.cu - bf16 attention forward with online softmax on the
// Blackwell tensor cores (tcgen05 MMAs, accumulators in tensor memory,
// operands staged by TMA through an mbarrier ring).  Built for sm_103a.
//
// The method is the blocked online-softmax loop of chapter 6 "Softmax 与
// Online Softmax" of the hand-written FlashAttention v2 book (yangyitao.com):
// a running row max m and adjusted sum l (§6.3.1), the guarded update when
// every key so far is masked (§6.4), O rescaled by alpha = e^{m_old - m_new}
// and P = e^{S - m_new} exponentiated against the new max (§6.6, the form
// without beta), LSE = m + log l (§6.5); the scale and additive mask precede
// the softmax and O / l happens once at the end (m.xxqk.cn/news/563265 §4.1).
// Exponentials run in base 2 with scale * log2(e) folded into one multiply;
// m and l live in those units and LSE converts back to natural log.
//
// CTA layout (192 threads, one CTA per 128-row query tile of one (b, h)):
//   warp 0        TMA producer: Q once, then K_0, K_1, V_0, K_2, V_1, ...
//                 into a STAGES-deep ring of K/V tiles (one tile per stage),
//                 in exactly the order the MMA warp consumes them.
//   warp 1        allocates tensor memory; one thread issues the MMAs:
//                 S_0, S_1, PV_0, S_2, PV_1, ... so S_{t+1} runs on the
//                 tensor core while the softmax works on S_t.
//   warps 2..5    softmax warpgroup, one query row per thread (tensor-memory
//                 lane = row): reads S_t, masks, updates (m, l), writes
//                 P_t = bf16(2^{x - m}) over S_t in tensor memory, rescales
//                 O in tensor memory when some row's m moved, then the
//                 epilogue O / l and LSE.
// Tensor memory (512 columns): S double buffer at columns 0 and 128 (fp32,
// 128 x 128 each; P_t overwrites the first 64 columns of its S buffer as
// packed bf16 pairs), O at column 256 (fp32, 128 x d).
//
// Tiles wholly outside the mask are never loaded or multiplied: the key loop
// stops at min(key_len, last visible key of the tile's last row).  Only tiles
// crossing key_len or the causal diagonal pay for element masking.
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>

#include "osattn_internal.h"
#include "sm100_ptx.cuh"

namespace osattn {
namespace {

constexpr int BM = 128;  // query rows per tile (MMA M, tensor-memory lanes)
constexpr int BN = 128;  // keys per tile (MMA N of S = Q K^T, K of P V)
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol0 = 0, kSCol1 = 128, kOCol = 256;
constexpr float kLn2 = 0.6931471805599453f;

// Give-up sites recorded in the status word's second slot.
enum : uint32_t {
  kSiteProdEmpty = 1,
  kSiteMmaQ = 2,
  kSiteMmaKV = 3,
  kSiteMmaP = 4,
  kSiteSoftS = 5,
  kSiteSoftO = 6,
  kSiteEpiO = 7
};

template <int HD>
struct Cfg {
  static constexpr int kColBlocks = HD / 64;           // 128-byte (64-element) column blocks
  static constexpr int kTileBytes = BN * HD * 2;       // one K or V tile
  static constexpr int kQBytes = BM * HD * 2;
  static constexpr int kStages = HD == 128 ? 6 : 10;
  static constexpr int kTileRegion = kQBytes + kStages * kTileBytes;
};

struct __align__(8) Bars {
  uint64_t q_full;
  uint64_t kv_full[16];
  uint64_t kv_empty[16];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full;
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int HD>
constexpr int smem_bytes() {
  return Cfg<HD>::kTileRegion + static_cast<int>(sizeof(Bars)) + 1024;  // +1024: alignment slack
}

struct Params {
  __nv_bfloat16* O;
  float* LSE;
  const int32_t* key_len;
  int H, Nq, Nkv;
  int num_q_tiles;
  float scale_log2;  // scale * log2(e)
  int causal;
  unsigned int* status;
  uint64_t wait_limit_ns;
};

// Waits on an mbarrier ignoring the abort flag (used only while draining
// work that is already in flight), bounded by the wait limit.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return;
  }
}

// Position of K_t / V_t in the producer's load sequence
// K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}.
__device__ __forceinline__ int seq_of_k(int t) { return t == 0 ? 0 : 2 * t - 1; }
__device__ __forceinline__ int seq_of_v(int t, int n) { return t == n - 1 ? 2 * n - 1 : 2 * t + 2; }

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Params p) {
  using C = Cfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::kQBytes;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kTileRegion);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Work tile: all query tiles of one (b, h) are adjacent in launch order so
  // CTAs running together share that head's K/V in L2; causal heads start
  // with their longest query tiles.
  const int bh = blockIdx.x / p.num_q_tiles;
  int qt = blockIdx.x % p.num_q_tiles;
  if (p.causal) qt = p.num_q_tiles - 1 - qt;
  const int b = bh / p.H;
  int kv_len = p.Nkv;
  if (p.key_len) kv_len = min(max(p.key_len[b], 0), p.Nkv);
  const int q0 = qt * BM;
  int kv_end = kv_len;
  if (p.causal) kv_end = min(kv_end, q0 + BM);
  const int n_tiles = (kv_end + BN - 1) / BN;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 128);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->mma_drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort_flag, p.status, p.status + 1, p.wait_limit_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_tiles > 0) {
      mbar_arrive_expect_tx(&bars->q_full, C::kQBytes);
#pragma unroll
      for (int cb = 0; cb < C::kColBlocks; ++cb)
        tma_load_3d(sQ + cb * BM * 128, &tmQ, &bars->q_full, cb * 64, q0, bh);
      const int total = 2 * n_tiles;
      int u = 0;
      for (; u < total; ++u) {
        // Decode which tile sequence slot u holds.
        int kt;
        bool is_v;
        if (u == 0) {
          kt = 0;
          is_v = false;
        } else if (u == total - 1) {
          kt = n_tiles - 1;
          is_v = true;
        } else {
          is_v = (u % 2) == 0;
          kt = is_v ? (u - 2) / 2 : (u + 1) / 2;
        }
        const int s = u % C::kStages;
        const uint32_t round = static_cast<uint32_t>(u / C::kStages);
        if (!mbar_wait(&bars->kv_empty[s], (round & 1u) ^ 1u, wc, kSiteProdEmpty)) break;
        mbar_arrive_expect_tx(&bars->kv_full[s], C::kTileBytes);
        uint8_t* dst = sKV + s * C::kTileBytes;
        const CUtensorMap* map = is_v ? &tmV : &tmK;
#pragma unroll
        for (int cb = 0; cb < C::kColBlocks; ++cb)
          tma_load_3d(dst + cb * BN * 128, map, &bars->kv_full[s], cb * 64, kt * BN, bh);
      }
      // Let every load this thread issued land before the CTA can exit.
      drain_wait(&bars->q_full, 0, p.wait_limit_ns);
      for (int v = (u > C::kStages ? u - C::kStages : 0); v < u; ++v)
        drain_wait(&bars->kv_full[v % C::kStages], static_cast<uint32_t>(v / C::kStages) & 1u,
                   p.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0);   // K-major A and B
      constexpr uint32_t idPV = idesc_bf16_f32(BM, HD, 1);  // B (V) is MN-major
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t kv_base = smem_u32(sKV);
      bool ok = mbar_wait(&bars->q_full, 0, wc, kSiteMmaQ);
      if (ok) tc_fence_after_sync();

      auto issue_s = [&](int t) -> bool {
        const int u = seq_of_k(t);
        const int s = u % C::kStages;
        if (!mbar_wait(&bars->kv_full[s], static_cast<uint32_t>(u / C::kStages) & 1u, wc,
                       kSiteMmaKV))
          return false;
        tc_fence_after_sync();
        const uint32_t d_col = tmem + ((t & 1) ? kSCol1 : kSCol0);
        const uint32_t k_base = kv_base + s * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk / 4) * (BM * 128) + (kk % 4) * 32;
          const uint64_t a = sdesc_sw128(q_base + off, 16, 1024);
          const uint64_t bdesc = sdesc_sw128(k_base + (kk / 4) * (BN * 128) + (kk % 4) * 32, 16, 1024);
          mma_bf16_ss(d_col, a, bdesc, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->kv_empty[s]);
        mma_commit(&bars->s_full[t & 1]);
        return true;
      };
      auto issue_pv = [&](int t) -> bool {
        if (!mbar_wait(&bars->p_full[t & 1], static_cast<uint32_t>(t >> 1) & 1u, wc, kSiteMmaP))
          return false;
        const int u = seq_of_v(t, n_tiles);
        const int s = u % C::kStages;
        if (!mbar_wait(&bars->kv_full[s], static_cast<uint32_t>(u / C::kStages) & 1u, wc,
                       kSiteMmaKV))
          return false;
        tc_fence_after_sync();
        const uint32_t p_col = tmem + ((t & 1) ? kSCol1 : kSCol0);
        const uint32_t v_base = kv_base + s * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // 16 keys per step = two 8-row swizzle atoms (2 KB); the d axis
          // crosses 64-element column blocks BN * 128 bytes apart.
          const uint64_t bdesc = sdesc_sw128(v_base + kk * 2048, BN * 128, 1024);
          mma_bf16_ts(tmem + kOCol, p_col + kk * 8, bdesc, idPV, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->kv_empty[s]);
        mma_commit(&bars->o_full);
        return true;
      };

      if (ok) ok = issue_s(0);
      for (int t = 1; ok && t < n_tiles; ++t) {
        ok = issue_s(t);
        if (ok) ok = issue_pv(t - 1);
      }
      if (ok) issue_pv(n_tiles - 1);
      // Every MMA this thread issued must complete before tensor memory is freed.
      mma_commit(&bars->mma_drain);
      drain_wait(&bars->mma_drain, 0, p.wait_limit_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax WG
    const int quarter = warp & 3;  // tensor-memory lanes [32*quarter, 32*quarter+32)
    const int row = quarter * 32 + lane;
    const int qi = q0 + row;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;

    for (int t = 0; t < n_tiles; ++t) {
      ok = mbar_wait(&bars->s_full[t & 1], static_cast<uint32_t>(t >> 1) & 1u, wc, kSiteSoftS);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t s_addr = lane_base + ((t & 1) ? kSCol1 : kSCol0);
      uint32_t sr[BN];
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch) tmem_ld_32x32b_x32(s_addr + ch * 32, sr + ch * 32);
      tmem_ld_wait();
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch) reg_fence32(sr + ch * 32);

      float x[BN];
#pragma unroll
      for (int j = 0; j < BN; ++j) x[j] = __uint_as_float(sr[j]) * c;
      const int k0 = t * BN;
      if (k0 + BN > kv_len || (p.causal && k0 + BN - 1 > q0)) {
        // Tile crosses key_len or the causal diagonal: additive -inf mask.
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          const int kj = k0 + j;
          if (kj >= kv_len || (p.causal && kj > qi)) x[j] = -INFINITY;
        }
      }
      float mx = x[0];
#pragma unroll
      for (int j = 1; j < BN; ++j) mx = fmaxf(mx, x[j]);
      const float m_new = fmaxf(m, mx);
      const bool changed = (m_new != m);
      float alpha = 1.f;
      uint32_t pk[BN / 2];
      float rs = 0.f;
      if (m_new == -INFINITY) {
        // Every key so far is masked: the state stays (-inf, 0) and P = 0.
#pragma unroll
        for (int j = 0; j < BN / 2; ++j) pk[j] = 0u;
      } else {
        if (changed) alpha = ex2_approx(m - m_new);
#pragma unroll
        for (int j = 0; j < BN / 2; ++j) {
          const float p0 = ex2_approx(x[2 * j] - m_new);
          const float p1 = ex2_approx(x[2 * j + 1] - m_new);
          rs += p0 + p1;
          pk[j] = pack_bf16x2(p0, p1);
        }
      }
      l = l * alpha + rs;
      m = m_new;
      tmem_st_32x32b_x32(s_addr, pk);
      tmem_st_32x32b_x32(s_addr + 32, pk + 32);

      if (t > 0) {
        // O holds the sum through PV_{t-1}; rescale it by alpha once that
        // MMA has finished, and only if some row of this warp moved its max.
        bool okw = mbar_wait(&bars->o_full, static_cast<uint32_t>(t - 1) & 1u, wc, kSiteSoftO);
        okw = __all_sync(0xffffffffu, okw);
        if (!okw) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (__any_sync(0xffffffffu, changed)) {
#pragma unroll
          for (int ch = 0; ch < HD / 32; ++ch) {
            uint32_t orr[32];
            const uint32_t o_addr = lane_base + kOCol + ch * 32;
            tmem_ld_32x32b_x32(o_addr, orr);
            tmem_ld_wait();
            reg_fence32(orr);
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
            tmem_st_32x32b_x32(o_addr, orr);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars->p_full[t & 1]);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n_tiles > 0) {
      ok = mbar_wait(&bars->o_full, static_cast<uint32_t>(n_tiles - 1) & 1u, wc, kSiteEpiO);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) tc_fence_after_sync();
    }
    if (ok) {
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool store = qi < p.Nq;
      __nv_bfloat16* orow = p.O + (static_cast<long long>(bh) * p.Nq + qi) * HD;
#pragma unroll
      for (int ch = 0; ch < HD / 32; ++ch) {
        uint32_t orr[32];
        if (n_tiles > 0) {
          tmem_ld_32x32b_x32(lane_base + kOCol + ch * 32, orr);
          tmem_ld_wait();
          reg_fence32(orr);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = 0u;
        }
        uint32_t packed[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          packed[e] = pack_bf16x2(__uint_as_float(orr[2 * e]) * inv_l,
                                  __uint_as_float(orr[2 * e + 1]) * inv_l);
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
        }
      }
      if (store)
        p.LSE[static_cast<long long>(bh) * p.Nq + qi] =
            l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int HD>
cudaError_t set_attrs() {
  return cudaFuncSetAttribute(fwd_bf16_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem_bytes<HD>());
}

}  // namespace

cudaError_t prepare_fwd_bf16() {
  cudaError_t e = set_attrs<64>();
  if (e != cudaSuccess) return e;
  return set_attrs<128>();
}

cudaError_t launch_fwd_bf16(const FwdArgs& a, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV) {
  Params p;
  p.O = static_cast<__nv_bfloat16*>(a.O);
  p.LSE = a.LSE;
  p.key_len = a.key_len;
  p.H = a.H;
  p.Nq = a.Nq;
  p.Nkv = a.Nkv;
  p.num_q_tiles = (a.Nq + BM - 1) / BM;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.causal = a.causal;
  p.status = a.status;
  p.wait_limit_ns = a.wait_limit_ns;
  const long long grid = static_cast<long long>(p.num_q_tiles) * a.B * a.H;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(grid)), blk(kThreads);
  if (a.d == 64)
    fwd_bf16_kernel<64><<<g, blk, smem_bytes<64>(), a.stream>>>(tmQ, tmK, tmV, p);
  else
    fwd_bf16_kernel<128><<<g, blk, smem_bytes<128>(), a.stream>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace osattn
