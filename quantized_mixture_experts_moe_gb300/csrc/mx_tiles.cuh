// The MX activation tile layout shared by the permute/quantise kernel and the
// block-scaled tensor-core GEMMs.
//
// Tokens of an expert are cut into tiles of up to NMAX slots; tile_start[e]
// is the prefix over experts of ceil(count[e] / NMAX).  NMAX is 16, 112 or 224:
// the first matching rule of the tile table (qmoe_set_tile_rules) picks it,
// else 224 when the average expert load exceeds 96 pairs.  For a reduction length K an
// activation buffer holds, per (tile t, K step kt of 128 elements), one block
//   [NMAX rows x 128 bytes]  E4M3 codes, row r at r*128, its 16-byte chunk c
//                            at ((c ^ (r & 7)) * 16)  (128-byte swizzle)
//   [NSFB x 512 bytes]       E8M0 scales: row r, block b (0..3) of the step at
//                            (r / 128) * 512 + 16 * (r % 32) + 4 * ((r % 128) / 32) + b
// so a GEMM step fetches its activations with two contiguous bulk copies and
// hands them to the MMA unchanged.
#pragma once
#include <stdint.h>

#include "../../include/qmoe.h"

namespace qmoe {
namespace mxt {

// the rule used when no tile-table rule matches
inline int nmax_default(const qmoe_dims* d) { return ((int64_t)d->T * d->k > (int64_t)96 * d->E) ? 224 : 112; }
// the token tile for these dims (tile_table.cu; host only)
int nmax_for(const qmoe_dims* d);
__host__ __device__ inline int nsfb(int nmax) { return (nmax + 127) / 128; }
__host__ __device__ inline int64_t block_bytes(int nmax) { return (int64_t)nmax * 128 + nsfb(nmax) * 512; }
__host__ __device__ inline int64_t max_tiles(const qmoe_dims* d, int nmax) {
    return ((int64_t)d->T * d->k + nmax - 1) / nmax + d->E;
}
inline int64_t buffer_bytes(const qmoe_dims* d, int64_t K) {
    const int nmax = nmax_for(d);
    return max_tiles(d, nmax) * (K / 128) * block_bytes(nmax);
}
__host__ __device__ inline uint32_t code_offset(int r, int col_in_step) {
    return (uint32_t)r * 128u + (((uint32_t)(col_in_step >> 4) ^ (uint32_t)(r & 7)) << 4) + (uint32_t)(col_in_step & 15);
}
__host__ __device__ inline uint32_t scale_offset(int nmax, int r, int block_in_step) {
    return (uint32_t)nmax * 128u + (uint32_t)(r >> 7) * 512u + 16u * (uint32_t)(r & 31) + 4u * (uint32_t)((r >> 5) & 3) +
           (uint32_t)block_in_step;
}

}  // namespace mxt
}  // namespace qmoe

namespace qmoe {
namespace bft {

// W4A16 activation tiles: the same token tiles as above; per (tile t, K step
// kt of 64 elements) one block of NMAX rows x 128 bytes at
// (t * K/64 + kt) * NMAX*128, row r at r*128 with its 16-byte chunk c at
// ((c ^ (r & 7)) * 16).  After the blocks, a per-row tail:
//   x tiles (stage-1 input): fp16 values v * 2^-e_r, tail = one fp32 2^e_r
//     per (tile, row);
//   h tiles (stage-1 output): bf16 values, tail = K/32 fp32 |max| values per
//     (tile, row), one per 32-column group.
__host__ __device__ inline int64_t block_bytes(int nmax) { return (int64_t)nmax * 128; }
inline int64_t blocks_bytes(const qmoe_dims* d, int64_t K) {
    const int nmax = mxt::nmax_for(d);
    return mxt::max_tiles(d, nmax) * (K / 64) * block_bytes(nmax);
}
inline int64_t x_tiles_bytes(const qmoe_dims* d) {
    const int nmax = mxt::nmax_for(d);
    return blocks_bytes(d, d->H) + mxt::max_tiles(d, nmax) * nmax * 4;
}
inline int64_t h_tiles_bytes(const qmoe_dims* d) {
    const int nmax = mxt::nmax_for(d);
    return blocks_bytes(d, d->I) + mxt::max_tiles(d, nmax) * nmax * (int64_t)(d->I / 32) * 4;
}
// byte offset of element `col` (0..63) of row r inside a block
__host__ __device__ inline uint32_t elem_offset(int r, int col) {
    const uint32_t b = (uint32_t)col * 2u;
    return (uint32_t)r * 128u + (((b >> 4) ^ (uint32_t)(r & 7)) << 4) + (b & 15u);
}

// Pre-packed int4 weights (W4A16): per (128-row tile rt, 64-element K step
// kt) a 4608-byte block at (rt * ceil(K/64) + kt) * 4608: 128 rows x 32 bytes
// of codes, then 128 rows x 2 fp16 scales (the two 32-element blocks of the
// step) multiplied by the row's power of two 2^p_r.  Inside each 32-bit code
// word the eight nibbles are reordered so the low half holds elements 0, 2,
// 4, 6 and the high half 1, 3, 5, 7: nibbles j and j + 4 are the pair
// (2j, 2j+1), which one mask lifts into the two halves of an f16x2.  After all blocks, one fp32
// 2^-p_r per row (ceil(rows/128)*128 of them).
constexpr int kW4Block = 4608;
__host__ __device__ inline int64_t w4_blocks_bytes(int64_t rows, int64_t K) {
    return ((rows + 127) / 128) * ((K + 63) / 64) * kW4Block;
}

}  // namespace bft
}  // namespace qmoe
