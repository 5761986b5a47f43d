// fwd_bf16_tcgen05.cu - bf16 attention forward with online softmax on the
// Blackwell tensor cores (tcgen05 MMAs, accumulators in tensor memory,
// operands staged by TMA through an mbarrier ring).  Built for sm_103a.
//
// The method is the blocked online-softmax loop of chapter 6 "Softmax 与
// Online Softmax" of the hand-written FlashAttention v2 book (yangyitao.com):
// a running row max m and adjusted sum l (§6.3.1), the guarded update while
// every key so far is masked (§6.4), O rescaled by alpha = e^{m_old - m_new}
// and P = e^{S - m_new} exponentiated against the new max (§6.6, the form
// without beta), LSE = m + log l (§6.5); the scale and additive mask precede
// the softmax and O / l happens once at the end (m.xxqk.cn/news/563265 §4.1).
// Exponentials run in base 2 with scale * log2(e) folded into one FMA; m and
// l live in those units and LSE converts back to natural log.
//
// Element type: bf16 or IEEE fp16 (template kF16), the same for Q, K, V, P
// and O; the MMAs accumulate in fp32 either way.  Q, K and V are read through
// 4-D tensor maps (d, N, H, B) with the caller's strides and O is written
// through its own strides, so [B, N, H, d] tensors need no transposing copy.
//
// CTA layout: 512 threads own two 128-row query tiles (Q0, Q1) of one (b, h)
// and stream that head's K/V tiles once for both.
//   warps 0-3   softmax for tile 0, one query row per thread (tensor-memory
//               lane = row); warps 4-7 the same for tile 1.  Per K/V tile:
//               read S_t, mask if the tile crosses key_len or the diagonal,
//               new row max, publish alpha, P_t = bf16(2^(x - m)) written
//               over S_t in tensor memory, l = l * alpha + rowsum(P).
//               At the end, the epilogue O / l and LSE for the tile.
//   warps 8-11  correction: once S_t of this K/V tile (and so PV_t of the
//               previous one) is done, multiply O_t by alpha in tensor memory - only warps holding
//               a row whose max moved do it.  Off the softmax's path.
//   warp 12     TMA producer: Q0, Q1 once, then K_0, V_0, K_1, V_1, ... into
//               a STAGES-deep ring.  MMA iteration j reads V_{j-1} and K_j,
//               so one barrier per iteration covers both loads and one
//               commit per iteration frees both stages: the MMA thread
//               (whose issue of one MMA takes most of the MMA's 64 cycles)
//               spends as little as possible on barrier checks.
//   warp 13     allocates tensor memory and issues the MMAs (warp-wide
//               loop, one elected lane issuing) in the order S0_0, S1_0,
//               PV0_0, S0_1, PV1_0, S1_1, PV0_1, ... so the tensor core
//               computes one tile's S while the other tile's softmax runs
//               (ping-pong between the two query tiles).
// Tensor memory (512 columns): S0 at 0, S1 at 128 (fp32, 128 x 128 each; P_t
// overwrites the first 64 columns of S_t as packed bf16 pairs), O0 at 256,
// O1 at 256 + d (fp32, 128 x d).
// Registers are rebalanced with setmaxnreg: softmax warps 184, correction 88,
// producer / MMA warpgroup 56 (256x184 + 128x88 + 128x56 = 65536 = 512 threads
// x 128 at launch; the host refuses a build with any other launch count).
//
// Tiles wholly outside the mask are never loaded or multiplied: each query
// tile's key loop stops at min(key_len, last visible key of its last row).
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>

#include "osattn_internal.h"
#include "sm100_ptx.cuh"
#include "tc_attn_mma.cuh"

namespace osattn {

// Profiling builds (OSATTN_STEP_TRACE=1, a separate library; never the
// product) stamp the SM clock at each phase of every K/V step of the first
// kTraceCtas CTAs: per softmax warpgroup t (role t, its first warp) S seen /
// S in registers / alpha published / P published; in the MMA warp (role 2)
// K/V seen / P_0 seen / P_1 seen / step issued; P published by each of the
// four softmax warps of tile t (role 3 + t, one stamp per warp); and per
// correction of tile t (role 5 + t, its first warp) alpha seen / O rescaled
// / arrived, with the fourth entry 1 if that warp rescaled O (not a clock).
// Every CTA below kTraceCtaTimes also records, in global-timer
// nanoseconds, when it started, finished its setup, saw its first S, began
// its epilogue (tile 0) and ended, and the SM it ran on.
// osattn_step_trace_read copies both out.
#ifndef OSATTN_STEP_TRACE
#define OSATTN_STEP_TRACE 0
#endif
constexpr int kTraceCtas = 8, kTraceRoles = 7, kTraceSteps = 128, kTraceCtaTimes = 4096;
#if OSATTN_STEP_TRACE
__device__ long long g_step_trace[kTraceCtas][kTraceRoles][kTraceSteps][4];
__device__ long long g_cta_times[kTraceCtaTimes][6];
#define OSATTN_CTA_TIME(cond, k)                                                        \
  do {                                                                                  \
    if ((cond) && blockIdx.x < kTraceCtaTimes)                                          \
      g_cta_times[blockIdx.x][k] = static_cast<long long>(global_timer_ns());           \
  } while (0)
#define OSATTN_STAMP_VALUE(cond, role, j, k, value)                                     \
  do {                                                                                  \
    if ((cond) && blockIdx.x < kTraceCtas && (j) < kTraceSteps)                         \
      g_step_trace[blockIdx.x][role][j][k] = (value);                                   \
  } while (0)
#else
#define OSATTN_STAMP_VALUE(cond, role, j, k, value) \
  do {                                              \
  } while (0)
#define OSATTN_CTA_TIME(cond, k) \
  do {                           \
  } while (0)
#endif
#define OSATTN_STAMP(cond, role, j, k) OSATTN_STAMP_VALUE(cond, role, j, k, clock64())

namespace {

constexpr int BM = 128;     // query rows per tile (MMA M, tensor-memory lanes)
constexpr int BN = 128;     // keys per K/V tile
constexpr int kQTiles = 2;  // query tiles per CTA
constexpr int kThreads = 512;
constexpr int kCorrWarp0 = 8, kProducerWarp = 12, kMmaWarp = 13;
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.6931471805599453f;

// Give-up sites recorded in the status word's second slot.
enum : uint32_t {
  kSiteProdEmpty = 1,
  kSiteMmaQ = 2,
  kSiteMmaKV = 3,
  kSiteMmaP = 4,
  kSiteSoftS = 5,
  kSiteCorrAlpha = 6,
  kSiteEpiO = 8
};

template <int HD>
struct Cfg {
  static constexpr int kTileBytes = BN * HD * 2;  // one K or V tile
  static constexpr int kQBytes = BM * HD * 2;     // one query tile
  static constexpr int kStages = HD == 128 ? 5 : 12;
  // Ring of per-iteration K/V barriers.  The producer arms iteration i after
  // iteration i - kStages/2 - 1 has released its stages, so the MMA has
  // passed iteration i - kIters by then (kIters > kStages/2 + 1).
  static constexpr int kIters = HD == 128 ? 4 : 8;
  static constexpr int kTileRegion = kQTiles * kQBytes + kStages * kTileBytes;
  static constexpr uint32_t kOCol0 = 256;
};

struct __align__(8) Bars {
  uint64_t q_full[kQTiles];
  uint64_t kv_full[8];    // [i % kIters]: V_{i-1} and K_i, which MMA iteration i reads, have landed
  uint64_t kv_empty[8];   // [i % kIters]: the MMAs of iteration i are done (their stages are free)
  uint64_t s_full[kQTiles];      // MMA -> softmax: S_t ready
  uint64_t alpha_full[kQTiles];  // softmax -> correction: alpha published (128 arrivals)
  uint64_t p_full[kQTiles];      // softmax + correction -> MMA: P_t written, O_t rescaled (256)
  uint64_t o_full[kQTiles];      // MMA -> epilogue: the tile's last PV done
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  float alpha[kQTiles][BM];
};

template <int HD>
constexpr int smem_bytes() {
  return Cfg<HD>::kTileRegion + static_cast<int>(sizeof(Bars)) + 1024;  // +1024: alignment slack
}

struct Params {
  uint16_t* O;      // bf16 or fp16 elements
  long long o_sb, o_sh, o_sn;  // O strides (elements) of the b, h and row axes
  float* LSE;
  float* o_part;    // split-KV only: [splits, B*H, Nq, d] fp32 partial O (already / l_s)
  float* lse_part;  // split-KV only: [splits, B*H, Nq] fp32 partial LSE
  const int32_t* key_len;
  int H, Nq, Nkv, BH;
  int num_splits;
  int num_q_blocks;  // ceil(Nq / 256)
  int group_heads;   // causal, unsplit: heads per longest-first group of units
  float scale_log2;  // scale * log2(e)
  int causal;
  unsigned int* status;
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return;
  }
}

template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Packs two fp32 values into the kernel's 16-bit element type.
template <bool kF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kF16) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}

// Number of K/V tiles a query tile starting at row q0 must visit: keys
// [0, min(key_len, q0 + BM if causal)); 0 when the tile lies beyond Nq or
// sees no key.
__device__ __forceinline__ int tile_kv_count(int q0, int Nq, int kv_len, int causal) {
  if (q0 >= Nq) return 0;
  int kv_end = kv_len;
  if (causal) kv_end = min(kv_end, q0 + BM);
  return (kv_end + BN - 1) / BN;
}

// Row max over 128 values (tiles crossing the mask): 3-input instructions in
// 8 chains.
__device__ __forceinline__ float max128(const uint32_t* v) {
  float a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = fmaxf(__uint_as_float(v[i]), __uint_as_float(v[i + 8]));
#pragma unroll
  for (int j = 16; j < BN; j += 16)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      a[i] = fmax3(a[i], __uint_as_float(v[j + i]), __uint_as_float(v[j + 8 + i]));
  return fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

// ------------------------------------------------------------------ softmax
// One thread per query row of tile t (tensor-memory lane = row).
template <int HD, bool kSplit, bool kF16>
__device__ __forceinline__ void softmax_role(const Params& p, Bars* bars, uint32_t tmem, int t,
                                             int b, int h, int q0, int n_t, int kv_len, int sb,
                                             int split, WaitCtl wc) {
  const int bh = b * p.H + h;
  using C = Cfg<HD>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;  // tensor-memory lanes [32*quarter, 32*quarter+32)
  const int row = quarter * 32 + lane;
  const int qi = q0 + row;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const uint32_t s_addr = lane_base + static_cast<uint32_t>(t * BN);
  const float c = p.scale_log2;
  float m = -INFINITY, l = 0.f;
  bool ok = true;

  for (int j = 0; j < n_t; ++j) {
    ok = mbar_wait(&bars->s_full[t], static_cast<uint32_t>(j) & 1u, wc, kSiteSoftS);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    OSATTN_STAMP(row == 0, t, j, 0);
    OSATTN_CTA_TIME(j == 0 && t == 0 && row == 0, 2);
    tc_fence_after_sync();
    // S in registers, with the max (scale >= 0) or min (scale < 0) of each
    // 32-column chunk formed by the loads: an unmasked tile's row max needs
    // no pass over the 128 values.
    uint32_t v[BN];
    float ext[BN / 32];
    if (c >= 0.f) {
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch)
        tmem_ld_red_32x32b_x32<true>(s_addr + ch * 32, v + ch * 32, ext[ch]);
    } else {
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch)
        tmem_ld_red_32x32b_x32<false>(s_addr + ch * 32, v + ch * 32, ext[ch]);
    }
    tmem_ld_wait();
#pragma unroll
    for (int ch = 0; ch < BN / 32; ++ch) {
      reg_fence32(v + ch * 32);
      asm volatile("" : "+f"(ext[ch]));
    }
    OSATTN_STAMP(row == 0, t, j, 1);

    // x_j = s_j * c (log2 units).  Unmasked tiles keep raw s in v and fold
    // the scale into the exponent's FMA (cm = c); tiles crossing key_len or
    // the causal diagonal store x with -inf at masked keys (cm = 1).
    const int k0 = (sb + j) * BN;
    float cm = c, m_new;
    if (k0 + BN > kv_len || (p.causal && k0 + BN - 1 > q0)) {
      const int lim = min(kv_len, p.causal ? qi + 1 : kv_len) - k0;  // visible: e < lim
#pragma unroll
      for (int e = 0; e < BN; ++e)
        v[e] = __float_as_uint(e < lim ? __uint_as_float(v[e]) * c : -INFINITY);
      cm = 1.f;
      m_new = fmaxf(m, max128(v));
    } else {
      // max_j(s_j * c) = c * max_j s_j for c >= 0, c * min_j s_j otherwise
      static_assert(BN == 128, "four 32-column chunks");
      const float e4 = c >= 0.f ? fmaxf(fmaxf(ext[0], ext[1]), fmaxf(ext[2], ext[3]))
                                : fminf(fminf(ext[0], ext[1]), fminf(ext[2], ext[3]));
      m_new = fmaxf(m, e4 * c);
    }
    const float alpha = (m_new == m) ? 1.f : ex2_approx(m - m_new);
    bars->alpha[t][row] = alpha;
    mbar_arrive(&bars->alpha_full[t]);
    OSATTN_STAMP(row == 0, t, j, 2);

    // P = 2^(x - m_new) in pairs (f32x2 FMA, two MUFU ex2, f32x2 add for the
    // row sum), packed to bf16 and stored over S in two halves of 32
    // columns.  A row with no visible key so far has m_new = -inf and x all
    // -inf, so with neg_m = 0 every p is exactly 0 and (m, l) stays (-inf, 0).
    const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
    const uint64_t cm2 = f2_pack(cm, cm), nm2 = f2_pack(neg_m, neg_m);
    uint64_t rs_a = 0, rs_b = 0;  // packed partial row sums (bit pattern 0 = 0.0f)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int i = half * 64 + 2 * e;
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), cm2, nm2),
                  x0, x1);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        const uint64_t pp = f2_pack(p0, p1);
        if (e & 1)
          rs_b = f2_add(rs_b, pp);
        else
          rs_a = f2_add(rs_a, pp);
        pk[e] = pack2<kF16>(p0, p1);
      }
      tmem_st_32x32b_x32(s_addr + half * 32, pk);
    }
    float r0, r1, r2, r3;
    f2_unpack(rs_a, r0, r1);
    f2_unpack(rs_b, r2, r3);
    l = fmaf(l, alpha, (r0 + r1) + (r2 + r3));
    m = m_new;
    tmem_st_wait();
    tc_fence_before_sync();
    mbar_arrive(&bars->p_full[t]);
    OSATTN_STAMP(row == 0, t, j, 3);
    OSATTN_STAMP(lane == 0, 3 + t, j, quarter);
  }

  // ---------------------------------------------------------------- epilogue
  OSATTN_CTA_TIME(t == 0 && row == 0, 3);
  if (ok && n_t > 0) {
    ok = mbar_wait(&bars->o_full[t], 0u, wc, kSiteEpiO);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) tc_fence_after_sync();
  }
  if (!ok) return;
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
  const uint32_t o_addr_t = lane_base + C::kOCol0 + static_cast<uint32_t>(t * HD);
  if constexpr (kSplit) {
    // Partial result of this key range: O_s = O / l_s in fp32 and
    // lse_s = m + ln l_s (or 0 and -inf for a range with no visible key),
    // merged later by the combine kernel.  The tensor-memory loads are
    // warp-wide; only the stores depend on the row.
    const bool store = qi < p.Nq;
    const long long prow = (static_cast<long long>(split) * p.BH + bh) * p.Nq + qi;
    float4* dst = reinterpret_cast<float4*>(p.o_part + prow * HD);
#pragma unroll
    for (int ch = 0; ch < HD / 32; ++ch) {
      uint32_t orr[32];
      if (n_t > 0) {
        tmem_ld_32x32b_x32(o_addr_t + ch * 32, orr);
        tmem_ld_wait();
        reg_fence32(orr);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) orr[e] = 0u;
      }
      if (store) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          dst[ch * 8 + e] = make_float4(
              __uint_as_float(orr[4 * e]) * inv_l, __uint_as_float(orr[4 * e + 1]) * inv_l,
              __uint_as_float(orr[4 * e + 2]) * inv_l, __uint_as_float(orr[4 * e + 3]) * inv_l);
      }
    }
    if (store) p.lse_part[prow] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    return;
  }
  const uint64_t inv2 = f2_pack(inv_l, inv_l);
  const bool store = qi < p.Nq;
  uint16_t* orow = p.O + b * p.o_sb + h * p.o_sh + qi * p.o_sn;
  const uint32_t o_addr = lane_base + C::kOCol0 + static_cast<uint32_t>(t * HD);
#pragma unroll
  for (int ch = 0; ch < HD / 32; ++ch) {
    uint32_t orr[32];
    if (n_t > 0) {
      tmem_ld_32x32b_x32(o_addr + ch * 32, orr);
      tmem_ld_wait();
      reg_fence32(orr);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) orr[e] = 0u;
    }
    uint32_t packed[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float a0, a1;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(orr[2 * e]), __uint_as_float(orr[2 * e + 1])), inv2),
                a0, a1);
      packed[e] = pack2<kF16>(a0, a1);
    }
    if (store) {
      uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        dst[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
    }
  }
  if (store)
    p.LSE[static_cast<long long>(bh) * p.Nq + qi] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// ------------------------------------------------------------------ correction
// Multiplies O_t by alpha in tensor memory once PV_t of the previous K/V
// tile has completed (implied by alpha_full, see below), for warps holding a row whose max moved; then signals
// the MMA warp (together with the softmax) that PV_t may run.
template <int HD>
__device__ __forceinline__ void correction_tile(Bars* bars, uint32_t lane_base, int row, int t,
                                                int j, bool& ok, WaitCtl wc) {
  using C = Cfg<HD>;
  // alpha_full(j) follows s_full(j): S_t(j) is complete, and so is PV_t(j-1),
  // issued before it (the MMA pipe runs in issue order and a commit tracks
  // every earlier MMA of the thread), so O_t may be rescaled now.
  ok = mbar_wait(&bars->alpha_full[t], static_cast<uint32_t>(j) & 1u, wc, kSiteCorrAlpha);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) return;
  OSATTN_STAMP(row == 0, 5 + t, j, 0);
  const float alpha = bars->alpha[t][row];
  const bool rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
  OSATTN_STAMP_VALUE(row == 0, 5 + t, j, 3, rescale ? 1 : 0);
  if (rescale) {
    tc_fence_after_sync();
    const uint64_t a2 = f2_pack(alpha, alpha);
    const uint32_t o_addr = lane_base + C::kOCol0 + static_cast<uint32_t>(t * HD);
    // 64 columns per round trip (two loads, one wait, two stores).  Unrolled,
    // so the next pair's loads can be issued before this pair's stores have
    // read their registers; that overlap is worth a few spilled registers
    // at d = 128 (measured: +1.5 % on the causal 16K workload, the same
    // loop kept rolled and spill-free gained nothing).  The profiling build
    // keeps 32 columns per round trip: with its stamps' registers the wider
    // form spills hundreds of bytes there and would distort the timings.
    constexpr int kPair = OSATTN_STEP_TRACE ? 1 : 2;
#pragma unroll
    for (int ch = 0; ch < HD / 32; ch += kPair) {
      uint32_t orr[64];
#pragma unroll
      for (int k = 0; k < kPair; ++k) tmem_ld_32x32b_x32(o_addr + (ch + k) * 32, orr + k * 32);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < kPair; ++k) reg_fence32(orr + k * 32);
#pragma unroll
      for (int e = 0; e < 16 * kPair; ++e) {
        float a0, a1;
        f2_unpack(f2_mul(f2_pack(__uint_as_float(orr[2 * e]), __uint_as_float(orr[2 * e + 1])), a2),
                  a0, a1);
        orr[2 * e] = __float_as_uint(a0);
        orr[2 * e + 1] = __float_as_uint(a1);
      }
#pragma unroll
      for (int k = 0; k < kPair; ++k) tmem_st_32x32b_x32(o_addr + (ch + k) * 32, orr + k * 32);
    }
    tmem_st_wait();
  }
  OSATTN_STAMP(row == 0, 5 + t, j, 1);
  tc_fence_before_sync();
  mbar_arrive(&bars->p_full[t]);
  OSATTN_STAMP(row == 0, 5 + t, j, 2);
}

template <int HD>
__device__ __forceinline__ void correction_role(Bars* bars, uint32_t tmem, int n0, int n1,
                                                WaitCtl wc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const int n = max(n0, n1);
  bool ok = true;
  for (int j = 0; ok && j < n; ++j) {
    if (j < n0) correction_tile<HD>(bars, lane_base, row, 0, j, ok, wc);
    if (ok && j < n1) correction_tile<HD>(bars, lane_base, row, 1, j, ok, wc);
  }
}

// ------------------------------------------------------------------ producer
template <int HD>
__device__ __forceinline__ void producer_role(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV, Bars* bars, uint8_t* sQ,
                                              uint8_t* sKV, int b, int h, int q0, int n0, int n1,
                                              int sb, WaitCtl wc) {
  using C = Cfg<HD>;
  if (n0 > 0) {
    mbar_arrive_expect_tx(&bars->q_full[0], C::kQBytes);
#pragma unroll
    for (int cb = 0; cb < HD / 64; ++cb)
      tma_load_4d(sQ + cb * BM * 128, tmQ, &bars->q_full[0], cb * 64, q0, h, b);
  }
  if (n1 > 0) {
    mbar_arrive_expect_tx(&bars->q_full[1], C::kQBytes);
#pragma unroll
    for (int cb = 0; cb < HD / 64; ++cb)
      tma_load_4d(sQ + C::kQBytes + cb * BM * 128, tmQ, &bars->q_full[1], cb * 64, q0 + BM, h, b);
  }
  // Load u goes to stage u % kStages: K_j for u = 2j, V_j for u = 2j + 1.
  // MMA iteration i reads V_{i-1} and K_i (loads 2i - 1 and 2i), so both
  // signal kv_full[i % kIters], armed once with their combined size, and
  // load u waits only for the iteration that last read its stage.
  const int n = max(n0, n1);
  const int total = 2 * n;
  int u = 0, armed = 0;
  for (; u < total; ++u) {
    const int s = u % C::kStages;
    if (u >= C::kStages) {
      const int r = (u - C::kStages + 1) >> 1;  // iteration that read load u - kStages
      if (!mbar_wait(&bars->kv_empty[r % C::kIters], static_cast<uint32_t>(r / C::kIters) & 1u, wc,
                     kSiteProdEmpty))
        break;
    }
    const int i = (u + 1) >> 1;  // iteration that reads load u
    uint64_t* full = &bars->kv_full[i % C::kIters];
    if (u == 0 || (u & 1)) {  // first load of iteration i
      mbar_arrive_expect_tx(full, ((i < n) ? C::kTileBytes : 0) + ((i >= 1) ? C::kTileBytes : 0));
      armed = i + 1;
    }
    uint8_t* dst = sKV + s * C::kTileBytes;
    const CUtensorMap* map = (u & 1) ? tmV : tmK;
#pragma unroll
    for (int cb = 0; cb < HD / 64; ++cb)
      tma_load_4d(dst + cb * BN * 128, map, full, cb * 64, (sb + (u >> 1)) * BN, h, b);
  }
  // Let every load this thread issued land before the CTA can exit.
  if (n0 > 0) drain_wait(&bars->q_full[0], 0, wc.limit_ns);
  if (n1 > 0) drain_wait(&bars->q_full[1], 0, wc.limit_ns);
  for (int i = (armed > C::kIters ? armed - C::kIters : 0); i < armed; ++i)
    drain_wait(&bars->kv_full[i % C::kIters], static_cast<uint32_t>(i / C::kIters) & 1u,
               wc.limit_ns);
}

// ------------------------------------------------------------------ MMA issuer
// S_t = Q_t K^T (128 x 128 fp32 into tensor-memory columns [t*128, t*128+128))
// is mma_abt_128; O_t (+)= P_t V, with P from tensor memory (bf16 pairs over
// S_t) and V read MN-major from shared memory, is mma_tmem_a_128.
//
// The whole MMA warp runs this loop: every wait is warp-wide and each MMA
// and commit is issued by the one lane elect.sync picks, so the loop's
// control flow stays warp-uniform (a lane-0-only issuer let the tensor pipe
// idle for about 150 cycles at each barrier wait).

template <int HD, bool kF16>
__device__ __forceinline__ void mma_role(Bars* bars, uint32_t tmem, uint8_t* sQ, uint8_t* sKV,
                                         int n0, int n1, WaitCtl wc) {
  using C = Cfg<HD>;
  [[maybe_unused]] const bool lead = (threadIdx.x & 31) == 0;  // stamps only
  const uint64_t q_desc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
  const uint64_t q_desc1 = q_desc0 + static_cast<uint64_t>(C::kQBytes >> 4);
  const uint64_t k_desc = sdesc_sw128(smem_u32(sKV), 16, 1024);       // stage 0, K-major
  const uint64_t v_desc = sdesc_sw128(smem_u32(sKV), BN * 128, 1024);  // stage 0, MN-major
  constexpr uint64_t kStageStep = static_cast<uint64_t>(C::kTileBytes >> 4);
  const uint32_t s_col0 = tmem, s_col1 = tmem + BN;
  const uint32_t o_col0 = tmem + C::kOCol0, o_col1 = tmem + C::kOCol0 + HD;
  const int n = max(n0, n1);
  bool ok = true;

  for (int j = 0; ok && j <= n; ++j) {
    // K_j sits at load slot 2j, V_{j-1} at 2j - 1; one barrier covers both.
    const uint32_t vs = j > 0 ? static_cast<uint32_t>((2 * j - 1) % C::kStages) : 0u;
    const uint32_t ks = static_cast<uint32_t>((2 * j) % C::kStages);
    ok = warp_wait(&bars->kv_full[j % C::kIters], static_cast<uint32_t>(j / C::kIters) & 1u, wc,
                   kSiteMmaKV);
    OSATTN_STAMP(lead, 2, j, 0);
    if (ok && j == 0) {
      if (n0 > 0) ok = warp_wait(&bars->q_full[0], 0, wc, kSiteMmaQ);
      if (ok && n1 > 0) ok = warp_wait(&bars->q_full[1], 0, wc, kSiteMmaQ);
    }
    if (!ok) break;
    tc_fence_after_sync();
    // tile 0: PV0(j-1), then S0(j)
    if (j > 0 && j - 1 < n0) {
      ok = warp_wait(&bars->p_full[0], static_cast<uint32_t>(j - 1) & 1u, wc, kSiteMmaP);
      OSATTN_STAMP(lead, 2, j, 1);
      if (!ok) break;
      tc_fence_after_sync();
      mma_tmem_a_128<HD, kF16, true>(o_col0, s_col0, v_desc + vs * kStageStep, j > 1);
      if (j == n0) mma_commit<true>(&bars->o_full[0]);
    }
    if (j < n0) {
      mma_abt_128<HD, kF16, true>(s_col0, q_desc0, k_desc + ks * kStageStep);
      mma_commit<true>(&bars->s_full[0]);
    }
    // tile 1: PV1(j-1), then S1(j)
    if (j > 0 && j - 1 < n1) {
      ok = warp_wait(&bars->p_full[1], static_cast<uint32_t>(j - 1) & 1u, wc, kSiteMmaP);
      OSATTN_STAMP(lead, 2, j, 2);
      if (!ok) break;
      tc_fence_after_sync();
      mma_tmem_a_128<HD, kF16, true>(o_col1, s_col1, v_desc + vs * kStageStep, j > 1);
      if (j == n1) mma_commit<true>(&bars->o_full[1]);
    }
    if (j < n1) {
      mma_abt_128<HD, kF16, true>(s_col1, q_desc1, k_desc + ks * kStageStep);
      mma_commit<true>(&bars->s_full[1]);
    }
    mma_commit<true>(&bars->kv_empty[j % C::kIters]);
    OSATTN_STAMP(lead, 2, j, 3);
  }
  // Every MMA the warp issued must complete before tensor memory is freed.
  mma_commit<true>(&bars->mma_drain);
  drain_wait(&bars->mma_drain, 0, wc.limit_ns);
  __syncwarp();
}

template <int HD, bool kSplit, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Params p) {
  using C = Cfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  OSATTN_CTA_TIME(threadIdx.x == 0, 0);
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + kQTiles * C::kQBytes;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kTileRegion);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Work unit: 256 query rows (two tiles) of one (b, h).  Units of a head
  // are adjacent in launch order so concurrently running CTAs share that
  // head's K/V in L2.  Causal units differ in length; unsplit, they run
  // longest first within groups of group_heads heads (whose K/V fits in L2
  // together), so the launch does not end on the last heads' longest units.
  int unit = blockIdx.x, split = 0;
  if constexpr (kSplit) {  // key-range split fastest: splits of one unit run together
    split = unit % p.num_splits;
    unit /= p.num_splits;
  }
  int bh, qb;
  if (!kSplit && p.causal) {
    const int nqb = p.num_q_blocks, G = p.group_heads;
    const int g0 = (unit / (G * nqb)) * G;    // first head of this unit's group
    const int gsize = min(G, p.BH - g0);      // the last group may be smaller
    const int r = unit - g0 * nqb;            // rank within the group
    bh = g0 + r % gsize;
    qb = nqb - 1 - r / gsize;                 // rank 0: the longest units
  } else {
    bh = unit / p.num_q_blocks;
    qb = unit % p.num_q_blocks;
    if (p.causal) qb = p.num_q_blocks - 1 - qb;
  }
  const int b = bh / p.H, h = bh % p.H;
  int kv_len = p.Nkv;
  if (p.key_len) kv_len = min(max(p.key_len[b], 0), p.Nkv);
  const int q0 = qb * (kQTiles * BM);
  int n0 = tile_kv_count(q0, p.Nq, kv_len, p.causal);
  int n1 = tile_kv_count(q0 + BM, p.Nq, kv_len, p.causal);
  int sb = 0;  // first K/V tile of this CTA's key range
  if constexpr (kSplit) {
    // The unit's K/V tiles [0, max(n0, n1)) are cut into num_splits equal
    // ranges; each query tile visits the part of its own range inside ours.
    const int n_all = max(n0, n1);
    const int per = (n_all + p.num_splits - 1) / p.num_splits;
    sb = min(n_all, split * per);
    const int se = min(n_all, sb + per);
    n0 = max(0, min(se, n0) - sb);
    n1 = max(0, min(se, n1) - sb);
  }
  const int n = max(n0, n1);

  if (threadIdx.x == 0) {
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->alpha_full[t], 128);
      mbar_init(&bars->p_full[t], 256);
      mbar_init(&bars->o_full[t], 1);
    }
    for (int i = 0; i < C::kIters; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    mbar_init(&bars->mma_drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort_flag, p.status, p.status + 1, p.wait_limit_ns};
  OSATTN_CTA_TIME(threadIdx.x == 0, 1);
#if OSATTN_STEP_TRACE
  if (threadIdx.x == 0 && blockIdx.x < kTraceCtaTimes) {
    uint32_t sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    g_cta_times[blockIdx.x][5] = sm;
  }
#endif

  if (warp < kCorrWarp0) {
    regs_inc<184>();
    const int t = warp >> 2;
    softmax_role<HD, kSplit, kF16>(p, bars, tmem, t, b, h, q0 + t * BM, t ? n1 : n0, kv_len, sb,
                                   split, wc);
  } else if (warp < kProducerWarp) {
    regs_dec<88>();
    correction_role<HD>(bars, tmem, n0, n1, wc);
  } else {
    regs_dec<56>();
    if (warp == kProducerWarp && lane == 0 && n > 0)
      producer_role<HD>(&tmQ, &tmK, &tmV, bars, sQ, sKV, b, h, q0, n0, n1, sb, wc);
    else if (warp == kMmaWarp && n > 0)
      mma_role<HD, kF16>(bars, tmem, sQ, sKV, n0, n1, wc);
  }

  __syncwarp();
  tmem_st_wait();
  tc_fence_before_sync();
  __syncthreads();
  OSATTN_CTA_TIME(threadIdx.x == 0, 4);
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The setmaxnreg split above hands out exactly 512 x 128 registers; a build
// whose launch register count differs would make setmaxnreg.inc wait
// forever, so such a build is refused here instead of launched.
constexpr int kLaunchRegs = 128;

template <int HD, bool kSplit, bool kF16>
cudaError_t set_attrs() {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, fwd_bf16_kernel<HD, kSplit, kF16>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(fwd_bf16_kernel<HD, kSplit, kF16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<HD>());
}

template <int HD, bool kSplit, bool kF16>
void launch_one(dim3 g, dim3 blk, cudaStream_t s, const CUtensorMap& q, const CUtensorMap& k,
                const CUtensorMap& v, const Params& p) {
  fwd_bf16_kernel<HD, kSplit, kF16><<<g, blk, smem_bytes<HD>(), s>>>(q, k, v, p);
}

}  // namespace

cudaError_t prepare_fwd_bf16() {
  cudaError_t e;
  if ((e = set_attrs<64, false, false>()) != cudaSuccess) return e;
  if ((e = set_attrs<128, false, false>()) != cudaSuccess) return e;
  if ((e = set_attrs<64, true, false>()) != cudaSuccess) return e;
  if ((e = set_attrs<128, true, false>()) != cudaSuccess) return e;
  if ((e = set_attrs<64, false, true>()) != cudaSuccess) return e;
  if ((e = set_attrs<128, false, true>()) != cudaSuccess) return e;
  if ((e = set_attrs<64, true, true>()) != cudaSuccess) return e;
  return set_attrs<128, true, true>();
}

cudaError_t read_step_trace(void* host, size_t bytes, size_t* needed) {
  constexpr size_t kSteps = static_cast<size_t>(kTraceCtas) * kTraceRoles * kTraceSteps * 4;
  constexpr size_t kCtas = static_cast<size_t>(kTraceCtaTimes) * 6;
  *needed = (kSteps + kCtas) * sizeof(long long);
#if OSATTN_STEP_TRACE
  if (bytes < *needed) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemcpyFromSymbol(host, g_step_trace, kSteps * sizeof(long long));
  if (e != cudaSuccess) return e;
  return cudaMemcpyFromSymbol(static_cast<long long*>(host) + kSteps, g_cta_times,
                              kCtas * sizeof(long long));
#else
  (void)host;
  (void)bytes;
  return cudaErrorNotSupported;
#endif
}

cudaError_t launch_fwd_bf16(const FwdArgs& a, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV) {
  Params p;
  p.O = static_cast<uint16_t*>(a.O);
  p.o_sb = a.o_strides[0];
  p.o_sh = a.o_strides[1];
  p.o_sn = a.o_strides[2];
  p.LSE = a.LSE;
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.key_len = a.key_len;
  p.H = a.H;
  p.Nq = a.Nq;
  p.Nkv = a.Nkv;
  p.BH = a.B * a.H;
  p.num_splits = a.num_splits > 0 ? a.num_splits : 1;
  p.num_q_blocks = (a.Nq + kQTiles * BM - 1) / (kQTiles * BM);
  {
    // heads whose K and V together take about kGroupKVBytes of L2
    constexpr long long kGroupKVBytes = 32ll << 20;
    const long long kv_head = 2ll * a.Nkv * a.d * 2;
    const long long gh = kGroupKVBytes / (kv_head > 0 ? kv_head : 1);
    p.group_heads = static_cast<int>(gh < 1 ? 1 : (gh > p.BH ? p.BH : gh));
  }
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.causal = a.causal;
  p.status = a.status;
  p.wait_limit_ns = a.wait_limit_ns;
  const bool split = a.num_splits > 0, f16 = a.fp16 != 0;
  const long long grid = static_cast<long long>(p.num_q_blocks) * a.B * a.H * p.num_splits;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(grid)), blk(kThreads);
  if (a.d == 64) {
    if (f16) split ? launch_one<64, true, true>(g, blk, a.stream, tmQ, tmK, tmV, p)
                   : launch_one<64, false, true>(g, blk, a.stream, tmQ, tmK, tmV, p);
    else split ? launch_one<64, true, false>(g, blk, a.stream, tmQ, tmK, tmV, p)
               : launch_one<64, false, false>(g, blk, a.stream, tmQ, tmK, tmV, p);
  } else {
    if (f16) split ? launch_one<128, true, true>(g, blk, a.stream, tmQ, tmK, tmV, p)
                   : launch_one<128, false, true>(g, blk, a.stream, tmQ, tmK, tmV, p);
    else split ? launch_one<128, true, false>(g, blk, a.stream, tmQ, tmK, tmV, p)
               : launch_one<128, false, false>(g, blk, a.stream, tmQ, tmK, tmV, p);
  }
  return cudaGetLastError();
}

}  // namespace osattn
