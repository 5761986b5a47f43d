// tc_attn_mma.cuh - the two tcgen05 MMA shapes the attention kernels issue.
//
// Shared-memory tiles are the layout the TMA loads write: a 128-row tile of
// d elements is stored as d/64 column blocks, each 128 rows x 128 bytes with
// the 128-byte swizzle (an 8-row atom is 1024 bytes).  Read along d it is a
// K-major operand; read along the rows it is an MN-major one.
#pragma once

#include <cstdint>

#include "sm100_ptx.cuh"

namespace osattn {

// D (128 x 128 fp32, tensor memory) = A B^T over KD elements of the inner
// axis: A and B are 128-row K-major tiles (a_desc / b_desc address their
// first 16-element slice; later slices move 32 bytes within a swizzle row,
// or to the next 64-column block).  Eight MMAs of K = 16 for KD = 128.
template <int KD, bool kF16>
__device__ __forceinline__ void mma_abt_128(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  constexpr uint32_t id = idesc_f16_f32(128, 128, 0, kF16);  // K-major A and B
  mma_ss_k<0>(d_tmem, a_desc, b_desc, id);
#pragma unroll
  for (int kk = 1; kk < KD / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>(((kk / 4) * (128 * 128) + (kk % 4) * 32) >> 4);
    mma_ss_k<1>(d_tmem, sdesc_add(a_desc, off), sdesc_add(b_desc, off), id);
  }
}

// D (128 x N fp32) (+)= A B over 128 inner elements: A from tensor memory
// (a 128 x 128 16-bit tile packed in pairs over 64 columns), B a 128-row
// MN-major shared-memory tile (b_desc: leading offset = distance between its
// 64-column blocks); 16 inner elements per MMA = two 8-row swizzle atoms.
template <int N, bool kF16>
__device__ __forceinline__ void mma_tmem_a_128(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               bool accumulate) {
  constexpr uint32_t id = idesc_f16_f32(128, N, 1, kF16);  // B is MN-major
  mma_bf16_ts(d_tmem, a_tmem, b_desc, id, accumulate ? 1u : 0u);
#pragma unroll
  for (int kk = 1; kk < 128 / 16; ++kk)
    mma_ts_k<1>(d_tmem, a_tmem + kk * 8, sdesc_add(b_desc, static_cast<uint32_t>((kk * 2048) >> 4)),
                id);
}

}  // namespace osattn
