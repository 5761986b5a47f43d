// bwd_tcgen05.cu - gradients of the attention forward pass (dQ, dK, dV) on
// the Blackwell tensor cores (tcgen05 MMAs, accumulators in tensor memory,
// operands staged by TMA).  Built for sm_103a.
//
// The forward pass keeps one number per query row, LSE = m + ln l (chapter 6
// "Softmax 与 Online Softmax" of the hand-written FlashAttention v2 book,
// §6.5), and the backward pass rebuilds the scores from Q and K instead of
// storing them (m.xxqk.cn/news/563265 §5.2, last paragraph).  With
// P_ij = e^{s_ij - LSE_i} on the visible keys the chain rule gives
//   D_i   = <dO_i, O_i>                 (= sum_j P_ij dP_ij)
//   dP_ij = <dO_i, V_j>,  dS_ij = P_ij (dP_ij - D_i)
//   dV_j  = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij Q_i,  dQ_i = scale sum_j dS_ij K_j.
//
// Two launches on one stream:
//   bwd_dq_kernel      one CTA per 128-row query tile: Q and dO stay, the
//                      visible K/V tiles stream.  Per key tile:
//                        S = Q K^T  and  dP = dO V^T;  dS in 16-bit over dP
//                        dQ += dS K                            (A from tensor memory)
//                      It also forms D = rowsum(dO * O) of its rows (dO from
//                      its resident tile, O read once) and writes it for:
//   bwd_dkdv_kernel    one CTA per 128-key tile of a (b, h): K and V stay in
//                      shared memory while the query tiles that can see
//                      those keys stream through a TMA ring.  Per query tile:
//                        S^T  = K Q^T   and  dP^T = V dO^T   (tensor memory)
//                        P^T, dS^T in 16-bit over the first 64 columns of each
//                        dV += P^T dO   and  dK += dS^T Q     (A from tensor memory)
// (bwd_rowdot_kernel forms D on its own for the fp32 path.)
// S and dP are computed twice (once per kernel) so that no kernel needs
// atomics: each output element is written once, by one CTA.
//
// CTA layout (320 threads): warps 0-7 elementwise in two warpgroups, group g
// taking columns 64g .. 64g + 63 of every score tile (one tile row per
// thread, tensor-memory lane = row), warp 8 producer (TMA; its lanes stage
// LSE and D of the dK/dV kernel's query tiles), warp 9 allocates tensor
// memory and one of its threads issues the MMAs.  Every wait is bounded as in the
// forward kernel: a wait past the limit records OSATTN_ERR_TIMEOUT, the CTA
// drains its own copies and MMAs, frees tensor memory and returns.
//
// Tensor memory (512 columns), dK/dV kernel: [0, 128) S^T, [128, 256) dP^T,
// [256, 256 + d) dV, [256 + d, 256 + 2d) dK.  dQ kernel: [0, 256) two S
// buffers, [256, 384) dP, [384, 384 + d) dQ.
#include <cmath>
#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "osattn_internal.h"
#include "sm100_ptx.cuh"
#include "tc_attn_mma.cuh"

namespace osattn {
namespace {

constexpr int kT = 128;            // rows of every tile (keys or queries)
constexpr int kBwdThreads = 320;   // warps 0-7 elementwise, 8 producer, 9 MMA
constexpr int kProdWarp = 8, kMmaWarp = 9;
constexpr uint32_t kCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

// Give-up sites recorded in the status word's second slot.
enum : uint32_t { kSiteBwdLoad = 21, kSiteBwdMma = 22, kSiteBwdElem = 23, kSiteBwdEpi = 24 };

template <int HD>
struct BwdCfg {
  static constexpr int kTileBytes = kT * HD * 2;       // one 128-row tile
  // dK/dV kernel: K, V, then kStages stages of (Q_i, dO_i), then LSE and D
  // of each stage's queries.
  static constexpr int kStages = HD == 128 ? 2 : 4;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kDkdvLse = 2 * kTileBytes + kStages * kStageBytes;
  static constexpr int kDkdvRegion = kDkdvLse + 2 * kStages * kT * 4;
  // dQ kernel: Q, dO, then kKSlots K tiles and kVSlots V tiles (K_j is read
  // until dQ_j, V_j only until dP_j, so K needs the deeper ring).
  static constexpr int kKSlots = HD == 128 ? 3 : 4;
  static constexpr int kVSlots = HD == 128 ? 2 : 4;
  static constexpr int kDqRegion = (2 + kKSlots + kVSlots) * kTileBytes;
  static constexpr uint32_t kColAcc0 = 256;            // dV
  static constexpr uint32_t kColAcc1 = 256 + HD;       // dK
};

struct __align__(16) BwdBars {
  uint64_t fixed_full;            // the tile pair loaded once (K, V or Q, dO)
  uint64_t full[4];               // per ring tile: its loads landed (dK/dV: and LSE, D staged)
  uint64_t empty[4];              // dK/dV: Q slot free (after dK); dQ: K slot free (after dQ)
  uint64_t empty2[4];             // dK/dV: dO slot free (after dV); dQ: V slot free (after dP)
  uint64_t s_full[2];             // MMA -> elementwise: a score tile (S or S^T) is ready
                                  //   (the dQ kernel alternates two S buffers)
  uint64_t dp_full;               // MMA -> elementwise: dP or dP^T is ready
  uint64_t p_full;                // elementwise -> MMA: P^T written (dK/dV kernel; 256 arrivals)
  uint64_t ds_full;               // elementwise -> MMA: dS or dS^T written (256 arrivals)
  uint64_t acc_full;              // MMA -> epilogue: the last accumulation is done
  uint64_t mma_drain;
  uint64_t d_full;                // dQ kernel: both warpgroups' halves of D stored (256)
  uint32_t tmem_base;
  int abort_flag;
  float d_part[2][kT];            // dQ kernel: D of each row over each warpgroup's columns
};

template <int HD>
constexpr int dkdv_smem_bytes() {
  return BwdCfg<HD>::kDkdvRegion + static_cast<int>(sizeof(BwdBars)) + 1024;
}
template <int HD>
constexpr int dq_smem_bytes() {
  return BwdCfg<HD>::kDqRegion + static_cast<int>(sizeof(BwdBars)) + 1024;
}
static_assert(dkdv_smem_bytes<128>() <= 232448 && dq_smem_bytes<128>() <= 232448 &&
                  dkdv_smem_bytes<64>() <= 232448 && dq_smem_bytes<64>() <= 232448,
              "shared memory per CTA");

struct BwdParams {
  uint16_t* dQ;
  uint16_t* dK;
  uint16_t* dV;
  long long dq_s[3], dk_s[3], dv_s[3];  // element strides of the b, h and row axes
  const float* LSE;
  float* D;              // [B*H*Nq]: written by the dQ kernel, read by the dK/dV kernel
  const uint16_t* O;     // forward output (for D), with its b, h, row element strides
  long long o_s[3];
  const int32_t* key_len;
  int H, Nq, Nkv;
  int num_tiles;     // 128-row tiles per (b, h): of keys (dK/dV) or queries (dQ)
  int BH;            // B * H
  int group_heads;   // causal: heads per longest-first group of CTAs
  float scale;
  float scale_log2;  // scale * log2(e)
  int causal;
  unsigned int* status;
  uint64_t wait_limit_ns;
};

template <bool kF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kF16) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return;
  }
}

// Counts tx_bytes of an mbarrier's expected transaction bytes as arrived
// (for a copy that will not be issued after all).
__device__ __forceinline__ void mbar_complete_tx(uint64_t* bar, uint32_t tx_bytes) {
  asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(tx_bytes)
               : "memory");
}

// The (b, h) and the rank by length (0 = longest loop) of this CTA's tile.
// Causal tiles differ in length: they run longest first within groups of
// group_heads heads (whose streamed tiles fit in L2 together), so the
// launch does not end on the last heads' longest loops.  Otherwise heads
// run one after another.
__device__ __forceinline__ void unit_of(const BwdParams& p, int& bh, int& rank) {
  const int nt = p.num_tiles;
  if (p.causal) {
    const int G = p.group_heads;
    const int g0 = (static_cast<int>(blockIdx.x) / (G * nt)) * G;
    const int gsize = min(G, p.BH - g0);
    const int r = static_cast<int>(blockIdx.x) - g0 * nt;
    bh = g0 + r % gsize;
    rank = r / gsize;
  } else {
    bh = static_cast<int>(blockIdx.x) / nt;
    rank = static_cast<int>(blockIdx.x) % nt;
  }
}

__device__ __forceinline__ int clamp_key_len(const int32_t* key_len, int b, int Nkv) {
  return key_len ? min(max(key_len[b], 0), Nkv) : Nkv;
}

// Writes NC fp32 tensor-memory columns of one tile row, starting at taddr,
// times `mul`, as 16-bit values to dst (or zeros when has_acc is false).
// The loads are warp-wide; only the stores depend on `store`.
template <int NC, bool kF16>
__device__ __forceinline__ void write_row(uint16_t* dst, uint32_t taddr, bool has_acc, bool store,
                                          float mul) {
#pragma unroll
  for (int ch = 0; ch < NC / 32; ++ch) {
    uint32_t r[32];
    if (has_acc) {
      tmem_ld_32x32b_x32(taddr + ch * 32, r);
      tmem_ld_wait();
      reg_fence32(r);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = 0u;
    }
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      pk[e] = pack2<kF16>(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
    if (store) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + ch * 32);
#pragma unroll
      for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
    }
  }
}

// ------------------------------------------------------------------ D = rowsum(dO * O)
struct RowStrides {
  long long o[3], g[3];  // element strides of the b, h and row axes of O and dO
};

// Two 16-bit values packed in one 32-bit word, as floats.
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w);
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}
template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// D = rowsum(dO * O) in fp32.  A row is d * sizeof(T) / 16 16-byte
// vectors, read by that many consecutive lanes (every row starts 16-byte
// aligned: the entry points require 16-byte aligned bases and strides), so
// a warp covers several rows per pass; each warp issues the loads of
// kPasses passes before using any, to keep enough bytes in flight for the
// HBM stream.  The lanes of a row sum their partial dots by shuffles.
template <typename T>
__global__ void __launch_bounds__(256, 3) bwd_rowdot_kernel(const T* __restrict__ O,
                                                         const T* __restrict__ dO,
                                                         float* __restrict__ D, long long rows,
                                                         int d, int H, int Nq, RowStrides st) {
  constexpr int kPasses = 4;
  constexpr int kEpv = 16 / static_cast<int>(sizeof(T));  // elements per vector
  const int lane = threadIdx.x & 31;
  const int lpr = d / kEpv;                 // lanes per row
  const int rpw = 32 / lpr;                 // rows per warp pass
  const int sub = lane / lpr, vec = lane - sub * lpr;
  const long long warp = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long step = static_cast<long long>(gridDim.x) * (blockDim.x >> 5) * rpw * kPasses;
  for (long long base = warp * rpw * kPasses; base < rows; base += step) {
    uint4 a[kPasses], g[kPasses];
#pragma unroll
    for (int u = 0; u < kPasses; ++u) {
      const long long row = base + u * rpw + sub;
      a[u] = make_uint4(0u, 0u, 0u, 0u);
      g[u] = make_uint4(0u, 0u, 0u, 0u);
      if (row < rows) {
        const long long bh = row / Nq;
        const long long i = row - bh * Nq, b = bh / H, h = bh - b * H;
        a[u] = reinterpret_cast<const uint4*>(O + b * st.o[0] + h * st.o[1] + i * st.o[2])[vec];
        g[u] = reinterpret_cast<const uint4*>(dO + b * st.g[0] + h * st.g[1] + i * st.g[2])[vec];
      }
    }
#pragma unroll
    for (int u = 0; u < kPasses; ++u) {
      const uint32_t aw[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
      const uint32_t gw[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (sizeof(T) == 4) {
          acc = fmaf(__uint_as_float(aw[e]), __uint_as_float(gw[e]), acc);
        } else {
          const float2 x = unpack2<T>(aw[e]), y = unpack2<T>(gw[e]);
          acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
        }
      }
      for (int off = lpr >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const long long row = base + u * rpw + sub;
      if (vec == 0 && row < rows) D[row] = acc;
    }
  }
}

// Both kernels issue every score product at full width (128 x 128, N = 128
// MMAs) and overlap it with the elementwise work in two parts per tile: the
// P part (P = 2^{s * scale * log2(e) - LSE * log2(e)} on the visible
// entries, kept in fp32 registers) needs only the scores, the dS part
// (dS = P (dP - D), rounded to 16 bits) then waits for dP.  Warpgroup g
// handles columns 64g .. 64g + 63 and writes its 16-bit results over the
// first 32 of them (column pair (2e, 2e + 1) of the group in column e), so
// the two groups never touch each other's columns; the MMAs that read those
// results take 16-element steps 0-3 from columns 0-31 and 4-7 from 64-95.

// P part over the 64 columns of this thread's group at tile column c0:
// pr[x] = P of column c0 + x; kMask applies vis(column), nl2of4(column)
// gives -LSE * log2(e) of 4 columns (stored negated, so the exponent
// argument is one FMA).  With kWriteP the 16-bit P is written
// over columns c0 .. c0 + 31.
template <bool kF16, bool kWriteP, bool kMask, typename Vis, typename L2of4>
__device__ __forceinline__ void bwd_p_part(uint32_t s_addr, int c0, float c, Vis&& vis,
                                           L2of4&& nl2of4, float (&pr)[64]) {
  uint32_t sa[32], sb[32];
  tmem_ld_32x32b_x32(s_addr + c0, sa);
  tmem_ld_wait();
  reg_fence32(sa);
  // the second half's load lands while the first half is computed
  tmem_ld_32x32b_x32(s_addr + c0 + 32, sb);
  const uint64_t c2 = f2_pack(c, c);
  // Half h: columns c0 + 32h .. + 31 from sv; exponent arguments
  // s * c - LSE * log2(e) two at a time (packed fp32 FMA: the same rounding
  // as two scalar FMAs).  With kWriteP its 16-bit P goes over columns
  // c0 + 16h .. + 15, which only the first half's load covered.
  auto half = [&](const uint32_t(&sv)[32], int h) {
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const float4 L = nl2of4(c0 + 32 * h + 4 * g);
#pragma unroll
      for (int u = 0; u < 4; u += 2) {
        const int x = 32 * h + 4 * g + u;
        const uint64_t s2 =
            f2_pack(__uint_as_float(sv[4 * g + u]), __uint_as_float(sv[4 * g + u + 1]));
        const uint64_t a2 = f2_fma(s2, c2, u == 0 ? f2_pack(L.x, L.y) : f2_pack(L.z, L.w));
        float a0, a1;
        f2_unpack(a2, a0, a1);
        const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
        if constexpr (kMask) {
          pr[x] = vis(c0 + x) ? e0 : 0.f;
          pr[x + 1] = vis(c0 + x + 1) ? e1 : 0.f;
        } else {
          pr[x] = e0;
          pr[x + 1] = e1;
        }
      }
    }
    if constexpr (kWriteP) {
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = pack2<kF16>(pr[32 * h + 2 * e], pr[32 * h + 2 * e + 1]);
      tmem_st_32x32b_x16(s_addr + c0 + 16 * h, pk);
    }
  };
  half(sa, 0);
  tmem_ld_wait();
  reg_fence32(sb);
  half(sb, 1);
}

// dS part over the same 64 columns of the dP tile at dp_addr, written as
// 16-bit pairs over columns c0 .. c0 + 31; ndof4(column) gives -D of 4
// columns (stored negated: dP - D is one add).  Chunk ch reads columns
// c0 + 32ch .. + 31 and writes c0 + 16ch .. + 15, which only the first
// chunk's load covered.
template <bool kF16, typename Dof4>
__device__ __forceinline__ void bwd_ds_part(uint32_t dp_addr, int c0, Dof4&& ndof4,
                                            const float (&pr)[64]) {
  uint32_t dva[32], dvb[32];
  tmem_ld_32x32b_x32(dp_addr + c0, dva);
  tmem_ld_wait();
  reg_fence32(dva);
  // the second chunk's load lands while the first is computed
  tmem_ld_32x32b_x32(dp_addr + c0 + 32, dvb);
  auto chunk = [&](const uint32_t(&dv)[32], int ch) {
    uint32_t gk[16];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const float4 D = ndof4(c0 + 32 * ch + 4 * g);
      const int x = 32 * ch + 4 * g;
      // dS = P (dP - D), two at a time (packed fp32: same rounding as scalar)
      const uint64_t d01 = f2_add(
          f2_pack(__uint_as_float(dv[4 * g]), __uint_as_float(dv[4 * g + 1])), f2_pack(D.x, D.y));
      const uint64_t d23 = f2_add(
          f2_pack(__uint_as_float(dv[4 * g + 2]), __uint_as_float(dv[4 * g + 3])), f2_pack(D.z, D.w));
      float gr[4];
      f2_unpack(f2_mul(f2_pack(pr[x], pr[x + 1]), d01), gr[0], gr[1]);
      f2_unpack(f2_mul(f2_pack(pr[x + 2], pr[x + 3]), d23), gr[2], gr[3]);
      gk[2 * g] = pack2<kF16>(gr[0], gr[1]);
      gk[2 * g + 1] = pack2<kF16>(gr[2], gr[3]);
    }
    tmem_st_32x32b_x16(dp_addr + c0 + 16 * ch, gk);
  };
  chunk(dva, 0);
  tmem_ld_wait();
  reg_fence32(dvb);
  chunk(dvb, 1);
}

// D (128 x N fp32) (+)= A B over 128 inner elements: A the 16-bit operand
// the two warpgroups wrote (elements 0-63 in columns 0-31 of a_tmem,
// 64-127 in 64-95), B an MN-major tile, 16 rows (2 KB) per MMA.
// Issued warp-wide (one elected lane, see mma_ss_k).
template <int N, bool kF16>
__device__ __forceinline__ void mma_tmem_a_groups(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                  bool accumulate) {
  constexpr uint32_t id = idesc_f16_f32(128, N, 1, kF16);  // B is MN-major
  mma_bf16_ts<true>(d_tmem, a_tmem, b_desc, id, accumulate ? 1u : 0u);
#pragma unroll
  for (int kk = 1; kk < 8; ++kk)
    mma_ts_k<1, true>(d_tmem, a_tmem + (kk / 4) * 64 + (kk % 4) * 8,
                      sdesc_add(b_desc, static_cast<uint32_t>((kk * 2048) >> 4)), id);
}

// ------------------------------------------------------------------ dK, dV
template <int HD, bool kF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const BwdParams p) {
  using C = BwdCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kTileBytes;
  uint8_t* ring = smem + 2 * C::kTileBytes;  // stage s: Q_i at +0, dO_i at +kTileBytes
  float* lse2 = reinterpret_cast<float*>(smem + C::kDkdvLse);  // [stage][query]: -LSE * log2(e)
  float* dsum = lse2 + C::kStages * kT;                        //   and -D (-inf, 0 past Nq)
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kDkdvRegion);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int bh, kt;
  unit_of(p, bh, kt);  // causal: key tile 0 meets the most query tiles
  const int b = bh / p.H, h = bh % p.H;
  const int k0 = kt * kT;
  const int kv_len = clamp_key_len(p.key_len, b, p.Nkv);
  const int nqt = (p.Nq + kT - 1) / kT;
  // Query tiles that can see this key tile: causal ones start at the tile
  // holding query k0 (key j is visible to query i iff j <= i).
  const int it0 = p.causal ? k0 / kT : 0;
  const int n_it = k0 < kv_len ? max(0, nqt - it0) : 0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->fixed_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->full[s], 2);  // the dO load's expect-tx, then the Q load's arrival
      mbar_init(&bars->empty[s], 1);
      mbar_init(&bars->empty2[s], 1);
    }
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->mma_drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort_flag, p.status, p.status + 1, p.wait_limit_ns};

  if (warp == kProdWarp) {
    // ---------------------------------------------------------------- producer
    int issued = 0;
    if (n_it > 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->fixed_full, 2 * C::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb) {
          tma_load_4d(sK + cb * kT * 128, &tmK, &bars->fixed_full, cb * 64, k0, h, b);
          tma_load_4d(sV + cb * kT * 128, &tmV, &bars->fixed_full, cb * 64, k0, h, b);
        }
      }
      for (int it = 0; it < n_it; ++it) {
        const int s = it % C::kStages;
        const int q0 = (it0 + it) * kT;
        const long long rowbase = static_cast<long long>(bh) * p.Nq;
        // LSE and D of the tile's queries: read before waiting for the
        // stage, so their latency hides behind the wait.
        float l2[kT / 32], dd[kT / 32];
#pragma unroll
        for (int r = 0; r < kT / 32; ++r) {
          const int q = q0 + lane + 32 * r;
          l2[r] = -INFINITY;  // staged negated: -LSE * log2(e) and -D
          dd[r] = 0.f;
          if (q < p.Nq) {
            const float L = p.LSE[rowbase + q];
            l2[r] = (L == -INFINITY) ? -INFINITY : -(L * kLog2e);
            dd[r] = -p.D[rowbase + q];
          }
        }
        uint8_t* st = ring + s * C::kStageBytes;
        // dO_i's slot frees after dV of the tile before (half a tile before
        // Q_i's, which frees after dK): load it first.
        bool ok = true;
        if (it >= C::kStages)
          ok = mbar_wait(&bars->empty2[s], static_cast<uint32_t>(it / C::kStages - 1) & 1u, wc,
                         kSiteBwdLoad);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->full[s], 2 * C::kTileBytes);
#pragma unroll
          for (int cb = 0; cb < HD / 64; ++cb)
            tma_load_4d(st + C::kTileBytes + cb * kT * 128, &tmdO, &bars->full[s], cb * 64, q0, h, b);
        }
        issued = it + 1;  // dO_i is in flight: the drain below must cover this tile
        if (it >= C::kStages)
          ok = mbar_wait(&bars->empty[s], static_cast<uint32_t>(it / C::kStages - 1) & 1u, wc,
                         kSiteBwdLoad);
        if (!__all_sync(0xffffffffu, ok)) {
          // Q_i will not be loaded: count its bytes and arrival as done, so
          // the phase completes once dO_i has landed.
          if (lane == 0) {
            mbar_complete_tx(&bars->full[s], C::kTileBytes);
            mbar_arrive(&bars->full[s]);
          }
          break;
        }
#pragma unroll
        for (int r = 0; r < kT / 32; ++r) {
          lse2[s * kT + lane + 32 * r] = l2[r];
          dsum[s * kT + lane + 32 * r] = dd[r];
        }
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int cb = 0; cb < HD / 64; ++cb)
            tma_load_4d(st + cb * kT * 128, &tmQ, &bars->full[s], cb * 64, q0, h, b);
          mbar_arrive(&bars->full[s]);  // releases the LSE and D writes above
        }
      }
      // Let every load of this CTA land before it can exit.
      if (lane == 0) {
        drain(&bars->fixed_full, 0, wc.limit_ns);
        for (int it = (issued > C::kStages ? issued - C::kStages : 0); it < issued; ++it)
          drain(&bars->full[it % C::kStages], static_cast<uint32_t>(it / C::kStages) & 1u,
                wc.limit_ns);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    // Tensor memory: S^T at column 0 (P^T packed over its first 64 columns),
    // dP^T at 128 (dS^T packed over its first 64), dV and dK after them.
    // Order: S^T_0, dP^T_0; then per query tile it: dV += P^T_it dO_it,
    // S^T_{it+1}, dK += dS^T_it Q_it, dP^T_{it+1}.  The tensor core runs
    // them in issue order, so a product that overwrites a tile follows the
    // one that reads it.
    if (n_it > 0) {  // the whole warp; one elected lane issues
      const uint64_t kA = sdesc_sw128(smem_u32(sK), 16, 1024);  // K-major A
      const uint64_t vA = sdesc_sw128(smem_u32(sV), 16, 1024);
      bool ok = warp_wait(&bars->fixed_full, 0, wc, kSiteBwdMma);
      if (ok) ok = warp_wait(&bars->full[0], 0, wc, kSiteBwdMma);
      if (ok) {
        tc_fence_after_sync();
        const uint32_t sq = smem_u32(ring), sdo = sq + C::kTileBytes;
        mma_abt<128, HD, kF16, true>(tmem, kA, sdesc_sw128(sq, 16, 1024));
        mma_commit<true>(&bars->s_full[0]);
        mma_abt<128, HD, kF16, true>(tmem + 128, vA, sdesc_sw128(sdo, 16, 1024));
        mma_commit<true>(&bars->dp_full);
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int s = it % C::kStages, s1 = (it + 1) % C::kStages;
        const uint32_t sq = smem_u32(ring + s * C::kStageBytes), sdo = sq + C::kTileBytes;
        const uint32_t nq = smem_u32(ring + s1 * C::kStageBytes), ndo = nq + C::kTileBytes;
        const bool more = it + 1 < n_it;
        ok = warp_wait(&bars->p_full, static_cast<uint32_t>(it) & 1u, wc, kSiteBwdMma);
        if (!ok) break;
        tc_fence_after_sync();
        // dV += P^T dO: B = dO read MN-major
        mma_tmem_a_groups<HD, kF16>(tmem + C::kColAcc0, tmem, sdesc_sw128(sdo, kT * 128, 1024), it > 0);
        mma_commit<true>(&bars->empty2[s]);
        if (more) {
          ok = warp_wait(&bars->full[s1], static_cast<uint32_t>((it + 1) / C::kStages) & 1u, wc,
                         kSiteBwdMma);
          if (!ok) break;
          tc_fence_after_sync();
          mma_abt<128, HD, kF16, true>(tmem, kA, sdesc_sw128(nq, 16, 1024));
          mma_commit<true>(&bars->s_full[0]);
        }
        ok = warp_wait(&bars->ds_full, static_cast<uint32_t>(it) & 1u, wc, kSiteBwdMma);
        if (!ok) break;
        tc_fence_after_sync();
        // dK += dS^T Q: B = Q read MN-major
        mma_tmem_a_groups<HD, kF16>(tmem + C::kColAcc1, tmem + 128, sdesc_sw128(sq, kT * 128, 1024),
                                    it > 0);
        mma_commit<true>(&bars->empty[s]);
        if (more) {
          mma_abt<128, HD, kF16, true>(tmem + 128, vA, sdesc_sw128(ndo, 16, 1024));
          mma_commit<true>(&bars->dp_full);
        }
      }
      if (ok) mma_commit<true>(&bars->acc_full);
      // Every MMA the warp issued must complete before tensor memory is freed.
      mma_commit<true>(&bars->mma_drain);
      drain(&bars->mma_drain, 0, wc.limit_ns);
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------------- elementwise
    const int c0 = 64 * (warp >> 2);  // this warpgroup's columns (queries) of each tile
    const int row = (warp & 3) * 32 + lane;  // key row of the tile = tensor-memory lane
    const int kabs = k0 + row;
    const bool row_live = kabs < kv_len;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      const int s = it % C::kStages;
      const int q0 = (it0 + it) * kT;
      ok = mbar_wait(&bars->s_full[0], static_cast<uint32_t>(it) & 1u, wc, kSiteBwdElem);
      // LSE and D of this query tile were staged with the stage's loads.
      if (ok)
        ok = mbar_wait(&bars->full[s], static_cast<uint32_t>(it / C::kStages) & 1u, wc, kSiteBwdElem);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const float4* l2 = reinterpret_cast<const float4*>(lse2 + s * kT);
      const float4* dd = reinterpret_cast<const float4*>(dsum + s * kT);
      auto vis = [&](int col) { return row_live && (!p.causal || kabs <= q0 + col); };
      auto l2of4 = [&](int col) { return l2[col >> 2]; };
      float pr[64];
      // No mask when every column of the group is visible to every row of
      // the warp.  The branch must be warp-uniform: the tensor-memory loads
      // inside are warp-collective.
      if (__all_sync(0xffffffffu, row_live && (!p.causal || kabs <= q0 + c0)))
        bwd_p_part<kF16, true, false>(lane_base, c0, p.scale_log2, vis, l2of4, pr);
      else
        bwd_p_part<kF16, true, true>(lane_base, c0, p.scale_log2, vis, l2of4, pr);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars->p_full);
      ok = mbar_wait(&bars->dp_full, static_cast<uint32_t>(it) & 1u, wc, kSiteBwdElem);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      bwd_ds_part<kF16>(lane_base + 128, c0, [&](int col) { return dd[col >> 2]; }, pr);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars->ds_full);
    }
    // epilogue: warpgroup 0 writes dV = sum P^T dO, warpgroup 1 dK = scale * sum dS^T Q
    bool has_acc = false;
    if (ok && n_it > 0) {
      ok = mbar_wait(&bars->acc_full, 0, wc, kSiteBwdEpi);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) tc_fence_after_sync();
      has_acc = ok;
    }
    if (ok) {
      const bool store = kabs < p.Nkv;
      if (c0 == 0)
        write_row<HD, kF16>(p.dV + b * p.dv_s[0] + h * p.dv_s[1] + kabs * p.dv_s[2],
                            lane_base + C::kColAcc0, has_acc, store, 1.f);
      else
        write_row<HD, kF16>(p.dK + b * p.dk_s[0] + h * p.dk_s[1] + kabs * p.dk_s[2],
                            lane_base + C::kColAcc1, has_acc, store, p.scale);
    }
  }

  __syncwarp();
  tmem_st_wait();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kCols);
  }
}

// ------------------------------------------------------------------ dQ
// Tensor memory: S in two 128-column buffers (S_j at 128 (j mod 2)), dP at
// 256 (dS packed over its first 64 columns), dQ at 384.
constexpr uint32_t kDqColDP = 256, kDqColAcc = 384;

template <int HD, bool kF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const BwdParams p) {
  using C = BwdCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = smem + C::kTileBytes;
  uint8_t* kring = smem + 2 * C::kTileBytes;            // K_j in slot j mod kKSlots
  uint8_t* vring = kring + C::kKSlots * C::kTileBytes;  // V_j in slot j mod kVSlots
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kDqRegion);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int bh, qt;
  unit_of(p, bh, qt);
  if (p.causal) qt = p.num_tiles - 1 - qt;  // the last query tile has the longest key loop
  const int b = bh / p.H, h = bh % p.H;
  const int q0 = qt * kT;
  const int kv_len = clamp_key_len(p.key_len, b, p.Nkv);
  int kv_end = kv_len;
  if (p.causal) kv_end = min(kv_end, q0 + kT);
  const int n_kt = q0 < p.Nq ? (kv_end + kT - 1) / kT : 0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->fixed_full, 1);
    for (int s = 0; s < C::kKSlots; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int s = 0; s < C::kVSlots; ++s) mbar_init(&bars->empty2[s], 1);
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->mma_drain, 1);
    mbar_init(&bars->d_full, 256);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort_flag, p.status, p.status + 1, p.wait_limit_ns};

  if (warp == kProdWarp) {
    if (lane == 0 && n_kt > 0) {
      mbar_arrive_expect_tx(&bars->fixed_full, 2 * C::kTileBytes);
#pragma unroll
      for (int cb = 0; cb < HD / 64; ++cb) {
        tma_load_4d(sQ + cb * kT * 128, &tmQ, &bars->fixed_full, cb * 64, q0, h, b);
        tma_load_4d(sdO + cb * kT * 128, &tmdO, &bars->fixed_full, cb * 64, q0, h, b);
      }
      // Tile j: K_j and V_j on full[j mod kKSlots], once both slots are free.
      int issued = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int a = j % C::kKSlots, v = j % C::kVSlots;
        if (j >= C::kKSlots &&
            !mbar_wait(&bars->empty[a], static_cast<uint32_t>(j / C::kKSlots - 1) & 1u, wc,
                       kSiteBwdLoad))
          break;
        if (j >= C::kVSlots &&
            !mbar_wait(&bars->empty2[v], static_cast<uint32_t>(j / C::kVSlots - 1) & 1u, wc,
                       kSiteBwdLoad))
          break;
        mbar_arrive_expect_tx(&bars->full[a], 2 * C::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb) {
          tma_load_4d(kring + a * C::kTileBytes + cb * kT * 128, &tmK, &bars->full[a], cb * 64, j * kT,
                      h, b);
          tma_load_4d(vring + v * C::kTileBytes + cb * kT * 128, &tmV, &bars->full[a], cb * 64, j * kT,
                      h, b);
        }
        issued = j + 1;
      }
      drain(&bars->fixed_full, 0, wc.limit_ns);
      for (int j = (issued > C::kKSlots ? issued - C::kKSlots : 0); j < issued; ++j)
        drain(&bars->full[j % C::kKSlots], static_cast<uint32_t>(j / C::kKSlots) & 1u, wc.limit_ns);
    }
  } else if (warp == kMmaWarp) {
    // Order: S_0, dP_0; then per key tile j: S_{j+1} (other S buffer),
    // dQ += dS_j K_j, dP_{j+1}.  S_{j+1} overwrites S_{j-1}, whose reader
    // signalled ds_full for tile j - 1 before the previous dQ product.
    if (n_kt > 0) {  // the whole warp; one elected lane issues
      const uint64_t qA = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dA = sdesc_sw128(smem_u32(sdO), 16, 1024);
      bool ok = warp_wait(&bars->fixed_full, 0, wc, kSiteBwdMma);
      if (ok) ok = warp_wait(&bars->full[0], 0, wc, kSiteBwdMma);
      if (ok) {
        tc_fence_after_sync();
        mma_abt<128, HD, kF16, true>(tmem, qA, sdesc_sw128(smem_u32(kring), 16, 1024));
        mma_commit<true>(&bars->s_full[0]);
        mma_abt<128, HD, kF16, true>(tmem + kDqColDP, dA, sdesc_sw128(smem_u32(vring), 16, 1024));
        mma_commit<true>(&bars->dp_full);
        mma_commit<true>(&bars->empty2[0]);
      }
      for (int j = 0; ok && j < n_kt; ++j) {
        const int a = j % C::kKSlots, a1 = (j + 1) % C::kKSlots, v1 = (j + 1) % C::kVSlots;
        const uint32_t sk = smem_u32(kring + a * C::kTileBytes);
        const uint32_t nk = smem_u32(kring + a1 * C::kTileBytes);
        const uint32_t nv = smem_u32(vring + v1 * C::kTileBytes);
        const bool more = j + 1 < n_kt;
        if (more) {
          ok = warp_wait(&bars->full[a1], static_cast<uint32_t>((j + 1) / C::kKSlots) & 1u, wc,
                         kSiteBwdMma);
          if (!ok) break;
          tc_fence_after_sync();
          mma_abt<128, HD, kF16, true>(tmem + 128 * ((j + 1) & 1), qA, sdesc_sw128(nk, 16, 1024));
          mma_commit<true>(&bars->s_full[(j + 1) & 1]);
        }
        ok = warp_wait(&bars->ds_full, static_cast<uint32_t>(j) & 1u, wc, kSiteBwdMma);
        if (!ok) break;
        tc_fence_after_sync();
        // dQ += dS K: B = K_j read MN-major
        mma_tmem_a_groups<HD, kF16>(tmem + kDqColAcc, tmem + kDqColDP,
                                    sdesc_sw128(sk, kT * 128, 1024), j > 0);
        mma_commit<true>(&bars->empty[a]);
        if (more) {
          mma_abt<128, HD, kF16, true>(tmem + kDqColDP, dA, sdesc_sw128(nv, 16, 1024));
          mma_commit<true>(&bars->dp_full);
          mma_commit<true>(&bars->empty2[v1]);
        }
      }
      if (ok) mma_commit<true>(&bars->acc_full);
      mma_commit<true>(&bars->mma_drain);
      drain(&bars->mma_drain, 0, wc.limit_ns);
      __syncwarp();
    }
  } else {
    const int c0 = 64 * (warp >> 2);  // this warpgroup's columns (keys) of each tile
    const int row = (warp & 3) * 32 + lane;  // query row of the tile = tensor-memory lane
    const int q = q0 + row;
    const bool row_live = q < p.Nq;
    const long long rix = static_cast<long long>(bh) * p.Nq + q;
    float l2 = -INFINITY;  // negated: -LSE * log2(e)
    // D = rowsum(dO * O) of this row: warpgroup g takes columns
    // g * d/2 .. (g + 1) * d/2 - 1, O from global memory (loaded now, used
    // after the first P part), dO from the resident tile.
    using T = typename std::conditional<kF16, __half, __nv_bfloat16>::type;
    constexpr int kHalfD = HD / 2, kNv = kHalfD / 8;  // 16-byte vectors of the half row
    const int g = warp >> 2;
    uint4 ov[kNv];
#pragma unroll
    for (int v = 0; v < kNv; ++v) ov[v] = make_uint4(0u, 0u, 0u, 0u);
    if (row_live && n_kt > 0) {
      const float L = p.LSE[rix];
      l2 = (L == -INFINITY) ? -INFINITY : -(L * kLog2e);
      const uint4* orow = reinterpret_cast<const uint4*>(
          p.O + b * p.o_s[0] + h * p.o_s[1] + static_cast<long long>(q) * p.o_s[2] + g * kHalfD);
#pragma unroll
      for (int v = 0; v < kNv; ++v) ov[v] = orow[v];
    }
    const float4 l2v = make_float4(l2, l2, l2, l2);
    float4 dv4 = make_float4(0.f, 0.f, 0.f, 0.f);  // -D
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    bool ok = true;
    for (int j = 0; ok && j < n_kt; ++j) {
      ok = mbar_wait(&bars->s_full[j & 1], static_cast<uint32_t>(j >> 1) & 1u, wc, kSiteBwdElem);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const int kx = j * kT;
      auto vis = [&](int col) { return kx + col < kv_len && (!p.causal || kx + col <= q); };
      auto l2of4 = [&](int) { return l2v; };
      const int last = kx + c0 + 63;  // the group's last key
      float pr[64];
      // No mask when every key of the group is visible to every row of the
      // warp (a warp-uniform branch: the tensor-memory loads inside are
      // warp-collective).
      if (__all_sync(0xffffffffu, last < kv_len && (!p.causal || last <= q)))
        bwd_p_part<kF16, false, false>(lane_base + 128 * (j & 1), c0, p.scale_log2, vis, l2of4, pr);
      else
        bwd_p_part<kF16, false, true>(lane_base + 128 * (j & 1), c0, p.scale_log2, vis, l2of4, pr);
      if (j == 0) {
        // the half dot product of D over this warpgroup's columns of the
        // swizzled dO tile (16-byte chunk c of a 128-byte row sits at
        // chunk c ^ (row mod 8)), then both halves through shared memory
        ok = mbar_wait(&bars->fixed_full, 0, wc, kSiteBwdElem);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        float part = 0.f;
#pragma unroll
        for (int v = 0; v < kNv; ++v) {
          const int col = g * kHalfD + v * 8;  // first of the vector's 8 columns
          const uint4 gv = *reinterpret_cast<const uint4*>(
              sdO + (col / 64) * kT * 128 + row * 128 + ((((col % 64) / 8) ^ (row & 7)) * 16));
          const uint32_t ow[4] = {ov[v].x, ov[v].y, ov[v].z, ov[v].w};
          const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = unpack2<T>(ow[e]), y = unpack2<T>(gw[e]);
            part = fmaf(x.x, y.x, fmaf(x.y, y.y, part));
          }
        }
        bars->d_part[g][row] = part;
        mbar_arrive(&bars->d_full);
        ok = mbar_wait(&bars->d_full, 0, wc, kSiteBwdElem);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const float D = bars->d_part[0][row] + bars->d_part[1][row];
        dv4 = make_float4(-D, -D, -D, -D);
        if (g == 0 && row_live) p.D[rix] = D;
      }
      ok = mbar_wait(&bars->dp_full, static_cast<uint32_t>(j) & 1u, wc, kSiteBwdElem);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      bwd_ds_part<kF16>(lane_base + kDqColDP, c0, [&](int) { return dv4; }, pr);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars->ds_full);
    }
    bool has_acc = false;
    if (ok && n_kt > 0) {
      ok = mbar_wait(&bars->acc_full, 0, wc, kSiteBwdEpi);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) tc_fence_after_sync();
      has_acc = ok;
    }
    // warpgroup g writes dQ columns g * d/2 .. (g + 1) * d/2 - 1
    if (ok)
      write_row<HD / 2, kF16>(p.dQ + b * p.dq_s[0] + h * p.dq_s[1] + q * p.dq_s[2] + c0 * HD / 128,
                              lane_base + kDqColAcc + c0 * HD / 128, has_acc, row_live, p.scale);
  }

  __syncwarp();
  tmem_st_wait();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kCols);
  }
}

template <int HD, bool kF16>
cudaError_t set_bwd_attrs() {
  cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_kernel<HD, kF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, dkdv_smem_bytes<HD>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(bwd_dq_kernel<HD, kF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              dq_smem_bytes<HD>());
}

// D = rowsum(dO * O) into a.D, for element type T.
template <typename T>
cudaError_t launch_rowdot(const BwdArgs& a) {
  const long long rows = static_cast<long long>(a.B) * a.H * a.Nq;
  // 8 warps a block, each taking 4 passes of 32 / (lanes per row) rows at
  // a time; 3 blocks per SM, all resident at once
  const long long lanes_per_row = static_cast<long long>(a.d) * sizeof(T) / 16;
  const long long per_block = 8ll * 4 * (32 / lanes_per_row);
  const long long want = static_cast<long long>(a.num_sms) * 3;
  const long long need = (rows + per_block - 1) / per_block;
  const int rgrid = static_cast<int>(need < want ? need : want);
  RowStrides rs;
  for (int i = 0; i < 3; ++i) {
    rs.o[i] = a.o_strides[i];
    rs.g[i] = a.do_strides[i];
  }
  bwd_rowdot_kernel<T><<<rgrid, 256, 0, a.stream>>>(static_cast<const T*>(a.O),
                                                    static_cast<const T*>(a.dO), a.D, rows, a.d,
                                                    a.H, a.Nq, rs);
  return cudaGetLastError();
}

template <int HD, bool kF16>
cudaError_t launch_bwd_t(const BwdArgs& a, const BwdParams& base, const CUtensorMap& tmQ,
                         const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmdO) {
  // Causal CTA groups: heads whose streamed tiles (Q and dO for dK/dV, K
  // and V for dQ) take about 32 MB of L2 together.
  auto group = [&](int rows) {
    const long long head = 2ll * rows * a.d * 2;
    const long long g = (32ll << 20) / (head > 0 ? head : 1);
    const long long bh = static_cast<long long>(a.B) * a.H;
    return static_cast<int>(g < 1 ? 1 : (g > bh ? bh : g));
  };
  BwdParams pk = base;
  pk.BH = a.B * a.H;
  pk.group_heads = group(a.Nq);
  pk.num_tiles = (a.Nkv + kT - 1) / kT;
  const long long gk = static_cast<long long>(pk.num_tiles) * a.B * a.H;
  BwdParams pq = base;
  pq.BH = a.B * a.H;
  pq.group_heads = group(a.Nkv);
  pq.num_tiles = (a.Nq + kT - 1) / kT;
  const long long gq = static_cast<long long>(pq.num_tiles) * a.B * a.H;
  if (gk > 0x7fffffffLL || gq > 0x7fffffffLL) return cudaErrorInvalidValue;
  // dQ first: it also writes D, which the dK/dV kernel reads
  bwd_dq_kernel<HD, kF16><<<static_cast<unsigned>(gq), kBwdThreads, dq_smem_bytes<HD>(), a.stream>>>(
      tmQ, tmK, tmV, tmdO, pq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_dkdv_kernel<HD, kF16><<<static_cast<unsigned>(gk), kBwdThreads, dkdv_smem_bytes<HD>(), a.stream>>>(
      tmQ, tmK, tmV, tmdO, pk);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_rowdot_fp32(const BwdArgs& a) { return launch_rowdot<float>(a); }

cudaError_t prepare_bwd() {
  cudaError_t e;
  if ((e = set_bwd_attrs<64, false>()) != cudaSuccess) return e;
  if ((e = set_bwd_attrs<128, false>()) != cudaSuccess) return e;
  if ((e = set_bwd_attrs<64, true>()) != cudaSuccess) return e;
  return set_bwd_attrs<128, true>();
}

cudaError_t launch_bwd(const BwdArgs& a, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const CUtensorMap& tmdO) {
  BwdParams p;
  p.dQ = static_cast<uint16_t*>(a.dQ);
  p.dK = static_cast<uint16_t*>(a.dK);
  p.dV = static_cast<uint16_t*>(a.dV);
  for (int i = 0; i < 3; ++i) {
    p.dq_s[i] = a.dq_strides[i];
    p.dk_s[i] = a.dk_strides[i];
    p.dv_s[i] = a.dv_strides[i];
  }
  p.LSE = a.LSE;
  p.D = a.D;
  p.O = static_cast<const uint16_t*>(a.O);
  for (int i = 0; i < 3; ++i) p.o_s[i] = a.o_strides[i];
  p.key_len = a.key_len;
  p.H = a.H;
  p.Nq = a.Nq;
  p.Nkv = a.Nkv;
  p.num_tiles = 0;
  p.BH = a.B * a.H;
  p.group_heads = 1;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.causal = a.causal;
  p.status = a.status;
  p.wait_limit_ns = a.wait_limit_ns;
  if (a.d == 64)
    return a.fp16 ? launch_bwd_t<64, true>(a, p, tmQ, tmK, tmV, tmdO)
                  : launch_bwd_t<64, false>(a, p, tmQ, tmK, tmV, tmdO);
  return a.fp16 ? launch_bwd_t<128, true>(a, p, tmQ, tmK, tmV, tmdO)
                : launch_bwd_t<128, false>(a, p, tmQ, tmK, tmV, tmdO);
}

}  // namespace osattn
