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

// D (128 x N fp32, tensor memory) = A B^T over KD elements of the inner
// axis: A is a 128-row and B an N-row K-major tile (a_desc / b_desc address
// their first 16-element slice; later slices move 32 bytes within a swizzle
// row, or to the next 64-column block, 128 rows = 16 KB on).  B may be a
// row range of a 128-row tile: the block offsets are those of the tile.
// kWarp: issued warp-wide (one elected lane; see mma_ss_k).
template <int N, int KD, bool kF16, bool kWarp = false>
__device__ __forceinline__ void mma_abt(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  constexpr uint32_t id = idesc_f16_f32(128, N, 0, kF16);  // K-major A and B
  mma_ss_k<0, kWarp>(d_tmem, a_desc, b_desc, id);
#pragma unroll
  for (int kk = 1; kk < KD / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>(((kk / 4) * (128 * 128) + (kk % 4) * 32) >> 4);
    mma_ss_k<1, kWarp>(d_tmem, sdesc_add(a_desc, off), sdesc_add(b_desc, off), id);
  }
}

template <int KD, bool kF16, bool kWarp = false>
__device__ __forceinline__ void mma_abt_128(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  mma_abt<128, KD, kF16, kWarp>(d_tmem, a_desc, b_desc);
}

// D (128 x N fp32) (+)= A B over 16 * KSTEPS inner elements: A from tensor
// memory (16-bit pairs, 8 columns per 16 elements), B an MN-major
// shared-memory tile read from its row b_desc points at (leading offset =
// distance between its 64-column blocks); 16 inner elements per MMA = two
// 8-row swizzle atoms (2 KB).
template <int N, int KSTEPS, bool kF16, bool kWarp = false>
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           bool accumulate) {
  constexpr uint32_t id = idesc_f16_f32(128, N, 1, kF16);  // B is MN-major
  mma_bf16_ts<kWarp>(d_tmem, a_tmem, b_desc, id, accumulate ? 1u : 0u);
#pragma unroll
  for (int kk = 1; kk < KSTEPS; ++kk)
    mma_ts_k<1, kWarp>(d_tmem, a_tmem + kk * 8,
                       sdesc_add(b_desc, static_cast<uint32_t>((kk * 2048) >> 4)), id);
}

// The forward's P V: A a 128 x 128 tile (64 columns of pairs).
template <int N, bool kF16, bool kWarp = false>
__device__ __forceinline__ void mma_tmem_a_128(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               bool accumulate) {
  mma_tmem_a<N, 8, kF16, kWarp>(d_tmem, a_tmem, b_desc, accumulate);
}

}  // namespace osattn
