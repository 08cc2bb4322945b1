// One-time weight preparation: E8M0 block scales rearranged into the order
// in which the block-scaled tensor-core MMA consumes them.
//
// Row-major scales s[row][kb] (one byte per 32 K elements) become 512-byte
// atoms, one per (128-row tile rt, group of 4 scale blocks kg), stored atom
// after atom with kg fastest.  Inside an atom the byte for tile row r and
// block kb (0..3) sits at 16*(r % 32) + 4*(r / 32) + kb: copying an atom to
// tensor memory with one 32x128b.warpx4 copy places the scale of row r in
// lane r, column r / 32, byte kb -- where the MMA reads it.  Rows and blocks
// beyond the tensor are padded with 127 (scale 1.0).
#include "qmoe_common.cuh"
#include "mx_tiles.cuh"

namespace qmoe {

__host__ __device__ inline int64_t mx_packed_bytes(int64_t rows, int64_t K) {
    return ((rows + 127) / 128) * ((K + 127) / 128) * 512;
}

__global__ void prepack_mx_scales_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t rows,
                                         int64_t KB, int64_t KG, int64_t total) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int64_t atom = i >> 9;
    const int off = (int)(i & 511);
    const int64_t rt = atom / KG, kg = atom - rt * KG;
    const int r = (off >> 4) + 32 * ((off >> 2) & 3);
    const int kb = off & 3;
    const int64_t row = rt * 128 + r, blk = kg * 4 + kb;
    dst[i] = (row < rows && blk < KB) ? src[row * KB + blk] : (uint8_t)127;
}

}  // namespace qmoe

extern "C" size_t qmoe_mx_scales_packed_bytes(int64_t rows, int64_t K) {
    if (rows <= 0 || K <= 0 || K % 32 != 0) return 0;
    return (size_t)qmoe::mx_packed_bytes(rows, K);
}

extern "C" int qmoe_prepack_mx_scales(int64_t rows, int64_t K, const uint8_t* s_rowmajor, uint8_t* s_packed,
                                      qmoe_stream_t stream) {
    using namespace qmoe;
    if (rows <= 0 || K <= 0 || K % 32 != 0 || !s_rowmajor || !s_packed || !aligned16(s_packed)) return QMOE_ERR_ARG;
    const int64_t total = mx_packed_bytes(rows, K);
    const int64_t blocks = (total + 255) / 256;
    prepack_mx_scales_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(s_rowmajor, s_packed, rows, K / 32,
                                                                                (K + 127) / 128, total);
    return launch_status();
}

// ------------------------------------------------------------------ 4-bit weights, tile-major
//
// Packed 4-bit weights W[rows][K/2 bytes] (element 2i in the low nibble of
// byte i) rearranged so that every 128-row x 128-element tile is one
// contiguous 8 KiB block: tile (rt, kt) at ((rt * KT) + kt) * 8192, tile row r
// at r * 64 inside it, same nibble order.  A tensor-core kernel then streams
// each tile with one contiguous read instead of 128 scattered 64-byte pieces.
// Rows and columns beyond the tensor are zero.
namespace qmoe {

__global__ void prepack_fp4_kernel(const uint8_t* __restrict__ src, uint4* __restrict__ dst, int64_t rows,
                                   int64_t Kbytes, int64_t KT, int64_t total16) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total16) return;
    const int64_t tile = i >> 9;          // 512 chunks of 16 B per tile
    const int within = (int)(i & 511);
    const int r = within >> 2, part = within & 3;
    const int64_t rt = tile / KT, kt = tile - rt * KT;
    const int64_t row = rt * 128 + r;
    const int64_t b0 = kt * 64 + part * 16;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < rows && b0 + 16 <= Kbytes) v = *reinterpret_cast<const uint4*>(src + row * Kbytes + b0);
    dst[i] = v;
}

}  // namespace qmoe

extern "C" size_t qmoe_fp4_weights_packed_bytes(int64_t rows, int64_t K) {
    if (rows <= 0 || K <= 0 || K % 32 != 0) return 0;
    return (size_t)(((rows + 127) / 128) * ((K + 127) / 128) * 8192);
}

extern "C" int qmoe_prepack_fp4_weights(int64_t rows, int64_t K, const uint8_t* w_rowmajor, uint8_t* w_packed,
                                        qmoe_stream_t stream) {
    using namespace qmoe;
    if (rows <= 0 || K <= 0 || K % 32 != 0 || !w_rowmajor || !w_packed || !aligned16(w_rowmajor) ||
        !aligned16(w_packed))
        return QMOE_ERR_ARG;
    const int64_t KT = (K + 127) / 128;
    const int64_t total16 = ((rows + 127) / 128) * KT * 512;
    prepack_fp4_kernel<<<(unsigned)((total16 + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
        w_rowmajor, reinterpret_cast<uint4*>(w_packed), rows, K / 2, KT, total16);
    return launch_status();
}

// ------------------------------------------------------------------ int4 weights for the fp16 tensor-core path
namespace qmoe {

// One thread per (padded) row: the power of two 2^p_r that moves the row's
// largest scale into [2^10, 2^11), so every product (n - 8) * s * 2^p_r
// (|n - 8| <= 8) stays below 2^14 in fp16 and small scales keep their
// precision.  Stores 2^-p_r (1 for an all-zero or padding row).
__global__ void prepack_int4_rowfac_kernel(const uint16_t* __restrict__ s, float* __restrict__ rowfac, int64_t rows,
                                           int64_t K, int64_t rows_padded) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows_padded) return;
    float smax = 0.f;
    if (r < rows)
        for (int64_t b = 0; b < K / 32; ++b)
            smax = fmaxf(smax, fabsf(__half2float(__ushort_as_half(s[r * (K / 32) + b]))));
    int p = 0;
    if (smax > 0.f) p = 10 - floor_log2_pos(smax);  // smax is an fp16 value: p in [-5, 34]
    rowfac[r] = exp2i(-p);
}

// One thread per 32-bit output word of a block (1024 code words + 128 scale words).
__global__ void prepack_int4_kernel(const uint8_t* __restrict__ w, const uint16_t* __restrict__ s,
                                    const float* __restrict__ rowfac, uint32_t* __restrict__ dst, int64_t rows,
                                    int64_t K, int64_t KT, int64_t total_words) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total_words) return;
    const int64_t blk = i / (bft::kW4Block / 4);
    const int wi = (int)(i % (bft::kW4Block / 4));
    const int64_t rt = blk / KT, kt = blk - rt * KT;
    uint32_t out = 0;
    if (wi < 1024) {
        const int r = wi >> 3, word = wi & 7;
        const int64_t row = rt * 128 + r;
        const int64_t k0 = kt * 64 + word * 8;  // eight elements k0..k0+7
        if (row < rows && k0 < K) {
            const uint32_t v = *reinterpret_cast<const uint32_t*>(w + row * (K / 2) + k0 / 2);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint32_t nib = (v >> (4 * m)) & 15u;
                const int pos = (m & 1) ? 4 + (m >> 1) : (m >> 1);
                out |= nib << (4 * pos);
            }
        } else {
            out = 0x88888888u;  // padding decodes to 0
        }
    } else {
        const int r = wi - 1024;
        const int64_t row = rt * 128 + r;
        const int64_t kb = kt * 2;
        const float f = rowfac[row];  // 2^-p_r: dividing by it is exact
        uint32_t s0 = 0, s1 = 0;
        if (row < rows && kb * 32 < K)
            s0 = __half_as_ushort(__float2half_rn(__fdiv_rn(__half2float(__ushort_as_half(s[row * (K / 32) + kb])), f)));
        if (row < rows && (kb + 1) * 32 < K)
            s1 = __half_as_ushort(
                __float2half_rn(__fdiv_rn(__half2float(__ushort_as_half(s[row * (K / 32) + kb + 1])), f)));
        out = s0 | (s1 << 16);
    }
    dst[i] = out;
}

}  // namespace qmoe

extern "C" size_t qmoe_int4_weights_packed_bytes(int64_t rows, int64_t K) {
    if (rows <= 0 || K <= 0 || K % 32 != 0) return 0;
    return (size_t)(qmoe::bft::w4_blocks_bytes(rows, K) + ((rows + 127) / 128) * 128 * 4);
}

extern "C" int qmoe_prepack_int4_weights(int64_t rows, int64_t K, const uint8_t* w_rowmajor, const uint16_t* s_fp16,
                                         uint8_t* packed, qmoe_stream_t stream) {
    using namespace qmoe;
    if (rows <= 0 || K <= 0 || K % 32 != 0 || !w_rowmajor || !s_fp16 || !packed || !aligned16(packed) ||
        (reinterpret_cast<uintptr_t>(w_rowmajor) & 3u))
        return QMOE_ERR_ARG;
    const int64_t KT = (K + 63) / 64;
    const int64_t rows_padded = ((rows + 127) / 128) * 128;
    float* rowfac = reinterpret_cast<float*>(packed + bft::w4_blocks_bytes(rows, K));
    prepack_int4_rowfac_kernel<<<(unsigned)((rows_padded + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
        s_fp16, rowfac, rows, K, rows_padded);
    int rc = launch_status();
    if (rc != QMOE_OK) return rc;
    const int64_t words = ((rows + 127) / 128) * KT * (bft::kW4Block / 4);
    prepack_int4_kernel<<<(unsigned)((words + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
        w_rowmajor, s_fp16, rowfac, reinterpret_cast<uint32_t*>(packed), rows, K, KT, words);
    return launch_status();
}
