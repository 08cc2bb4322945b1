// Activation / intermediate quantisation kernels.
//
//  * MX (E4M3 codes + one E8M0 scale per 32 columns) for the fp8 activations
//    that feed the MXFP4 expert GEMMs (aiter tuned grouped-fmoe page,
//    Changes: fp8 activations with MXFP4 weights).  Rule (OCP MX v1.0): per block,
//    X = 2^(floor(log2 amax) - 8), code = nearest-even E4M3 of v / X,
//    saturated to +-448; amax = 0 -> scale byte 127, zero codes.
//  * Per-row symmetric int8 for the W8A8 scheme ("Evaluate native IU4/IU8
//    WMMA ... on gfx1151", Constraint: integer MMAs need quantised
//    activations): s = amax / 127 (1 if amax = 0), q = clamp(rint(v/s), +-127),
//    all in fp32 with IEEE division.
#include <algorithm>

#include "qmoe_common.cuh"
#include "mx_tiles.cuh"

namespace qmoe {

// One thread per 8 consecutive bf16 values; 4 lanes form one 32-block.
__global__ void __launch_bounds__(256)
quant_mx_bf16_kernel(const uint4* __restrict__ x, int64_t n8, uint2* __restrict__ q, uint8_t* __restrict__ s) {
    pdl_sync();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool active = i < n8;
    uint4 v = active ? x[i] : make_uint4(0, 0, 0, 0);
    float f[8];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = __uint_as_float(w[j] << 16);
        f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    if (!active) return;
    uint2 codes = make_uint2(0, 0);
    uint8_t sb = 127;
    if (amax > 0.f) {
        const int X = mx_block_exponent(amax);
        const float m = exp2i(-X);
        sb = (uint8_t)(X + 127);
        codes.x = (uint32_t)e4m3x2_from_float(f[0] * m, f[1] * m) | ((uint32_t)e4m3x2_from_float(f[2] * m, f[3] * m) << 16);
        codes.y = (uint32_t)e4m3x2_from_float(f[4] * m, f[5] * m) | ((uint32_t)e4m3x2_from_float(f[6] * m, f[7] * m) << 16);
    }
    q[i] = codes;
    if ((threadIdx.x & 3) == 0) s[i >> 2] = sb;
}

template <typename In>
__device__ __forceinline__ float load_as_float(const In* p, int64_t i);
template <>
__device__ __forceinline__ float load_as_float<uint16_t>(const uint16_t* p, int64_t i) {
    return bf16_bits_to_float(p[i]);
}
template <>
__device__ __forceinline__ float load_as_float<float>(const float* p, int64_t i) {
    return p[i];
}

// One CTA per row.
template <typename In>
__global__ void __launch_bounds__(256)
quant_rows_int8_kernel(const In* __restrict__ x, int64_t cols, int8_t* __restrict__ q, float* __restrict__ s) {
    pdl_sync();
    __shared__ float red[8];
    const int64_t row = blockIdx.x;
    const In* xr = x + row * cols;
    float amax = 0.f;
    for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) amax = fmaxf(amax, fabsf(load_as_float(xr, c)));
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, red[w]);
    const float sc = (amax == 0.f) ? 1.0f : __fdiv_rn(amax, 127.0f);
    int8_t* qr = q + row * cols;
    for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) {
        float t = rintf(__fdiv_rn(load_as_float(xr, c), sc));
        t = fminf(fmaxf(t, -127.f), 127.f);
        qr[c] = (int8_t)(int)t;
    }
    if (threadIdx.x == 0) s[row] = sc;
}

// Permute + MX-quantise, token-major: one warp per (token, 1024-element
// segment of its row), 8 per CTA.  The segment of bf16 x is read once,
// quantised with the same rule as quant_mx_bf16_kernel, and written to the
// slot of each of the token's k routed pairs in the MX activation tile layout
// (mx_tiles.cuh), so the tensor-core GEMM reads it with bulk copies.  A lane
// owns 16 consecutive elements of each half of the segment; neighbouring
// lanes pair up into one 32-element block.
constexpr int kPqWarps = 8;

__device__ __forceinline__ void mx_quant16(const uint4 v0, const uint4 v1, uint4& codes, uint8_t& sb) {
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    codes = make_uint4(0, 0, 0, 0);
    sb = 127;
    if (amax > 0.f) {
        const int X = mx_block_exponent(amax);
        const float m = exp2i(-X);
        sb = (uint8_t)(X + 127);
        uint32_t c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            c[i] = (uint32_t)e4m3x2_from_float(f[4 * i] * m, f[4 * i + 1] * m) |
                   ((uint32_t)e4m3x2_from_float(f[4 * i + 2] * m, f[4 * i + 3] * m) << 16);
        codes = make_uint4(c[0], c[1], c[2], c[3]);
    }
}

// One (token, segment) item of the permute; wid < T * nseg, warp-uniform.
__device__ __forceinline__ void permute_quant_mx_item(int64_t wid, const uint16_t* __restrict__ x,
                                                      const int32_t* __restrict__ pair_dest, int k, int H, int nmax,
                                                      uint8_t* __restrict__ tiles) {
    const int lane = threadIdx.x & 31;
    const int nseg = H / 1024 + (H % 1024 != 0);  // 1024-element segments of a row
    const int tok = (int)(wid / nseg), seg = (int)(wid % nseg);
    const uint16_t* xr = x + (int64_t)tok * H;
    const int KT = H / 128;
    const int64_t bb = mxt::block_bytes(nmax);
    const int nchunk = H / 16;
    // this segment's 64 chunks of 16 elements, two per lane; every lane
    // reaches the pairwise shuffle
    uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0, b0 = a0, b1 = a0;
    const int ja = seg * 64 + lane, jb = seg * 64 + 32 + lane;
    if (ja < nchunk) {
        a0 = *reinterpret_cast<const uint4*>(xr + 16 * ja);
        a1 = *reinterpret_cast<const uint4*>(xr + 16 * ja + 8);
    }
    if (jb < nchunk) {
        b0 = *reinterpret_cast<const uint4*>(xr + 16 * jb);
        b1 = *reinterpret_cast<const uint4*>(xr + 16 * jb + 8);
    }
    uint4 ca, cb;
    uint8_t sa, sbb;
    mx_quant16(a0, a1, ca, sa);
    mx_quant16(b0, b1, cb, sbb);
    // a K step's four scale bytes are contiguous in a row's atom: the first lane of each 8-lane group
    // (one 128-element step) gathers them from the group's even lanes and stores one word
    uint32_t wa = 0, wb = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        wa |= (uint32_t)(__shfl_sync(0xFFFFFFFFu, (uint32_t)sa, (lane & ~7) + 2 * b) & 0xFFu) << (8 * b);
        wb |= (uint32_t)(__shfl_sync(0xFFFFFFFFu, (uint32_t)sbb, (lane & ~7) + 2 * b) & 0xFFu) << (8 * b);
    }
    for (int j0 = 0; j0 < k; j0 += 32) {
        // lane i looks up pair j0 + i's tile and row (tile -1: invalid expert id)
        int dtile = -1, drow = 0;
        if (j0 + lane < k) {
            const int dst = pair_dest[(int64_t)tok * k + j0 + lane];
            if (dst >= 0) {
                dtile = dst / nmax;
                drow = dst - dtile * nmax;
            }
        }
        const int jn = min(32, k - j0);
        for (int j = 0; j < jn; ++j) {
            const int tile = __shfl_sync(0xFFFFFFFFu, dtile, j);
            const int row = __shfl_sync(0xFFFFFFFFu, drow, j);
            if (tile < 0) continue;  // warp-uniform
            uint8_t* tbase = tiles + (int64_t)tile * KT * bb;
            if (ja < nchunk) {
                uint8_t* blk = tbase + (int64_t)(ja >> 3) * bb;
                *reinterpret_cast<uint4*>(blk + mxt::code_offset(row, (ja & 7) * 16)) = ca;
                if ((ja & 7) == 0) *reinterpret_cast<uint32_t*>(blk + mxt::scale_offset(nmax, row, 0)) = wa;
            }
            if (jb < nchunk) {
                uint8_t* blk = tbase + (int64_t)(jb >> 3) * bb;
                *reinterpret_cast<uint4*>(blk + mxt::code_offset(row, (jb & 7) * 16)) = cb;
                if ((jb & 7) == 0) *reinterpret_cast<uint32_t*>(blk + mxt::scale_offset(nmax, row, 0)) = wb;
            }
        }
    }
}

// Items are strided over a grid of up to four waves of the CTAs that fit on
// the GPU at once.
__global__ void __launch_bounds__(kPqWarps * 32)
permute_quant_mx_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ pair_dest, int k, int H,
                        int nmax, int T, uint8_t* __restrict__ tiles) {
    pdl_sync();
    const int64_t items = (int64_t)T * (H / 1024 + (H % 1024 != 0));
    for (int64_t wid = (int64_t)blockIdx.x * kPqWarps + (threadIdx.x >> 5); wid < items;
         wid += (int64_t)gridDim.x * kPqWarps)
        permute_quant_mx_item(wid, x, pair_dest, k, H, nmax, tiles);
}

// CTAs of `kernel` that fit on the current GPU at once (0 on error).
template <typename K>
static int64_t resident_ctas(K kernel, int threads) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess)
        return 0;
    return (int64_t)sms * per_sm;
}

int permute_quant_mx_launch(const qmoe_dims* d, const uint16_t* x, const int32_t* pair_slot, const int32_t* offsets,
                            const int32_t* tile_start, uint8_t* tiles, cudaStream_t st) {
    if ((int64_t)d->T * d->k == 0) return QMOE_OK;
    const int64_t warps = (int64_t)d->T * (d->H / 1024 + (d->H % 1024 != 0));
    int64_t blocks = (warps + kPqWarps - 1) / kPqWarps;
    const int64_t fit = resident_ctas(permute_quant_mx_kernel, kPqWarps * 32);
    if (fit <= 0) return QMOE_ERR_CUDA;
    // up to four waves: an item's k scattered row stores are latency-bound, and more warps in flight
    // (about one item each at T=4096) beat fewer warps striding over several (41.6 -> 37.1 us at T=4096)
    if (blocks > 4 * fit) blocks = 4 * fit;
    // each pair's token-tile row, written by the routing sort beside the schedule
    const int32_t* pair_dest = tile_start + schedule_ints(d->E) + slot_ints((int64_t)d->T * d->k);
    return launch_pdl(permute_quant_mx_kernel, (unsigned)blocks, kPqWarps * 32, 0, st, x, pair_dest, d->k, d->H,
                      mxt::nmax_for(d), d->T, tiles);
}

// Permute bf16 activations into W4A16 x tiles: one warp per expert-sorted
// slot.  The row's largest magnitude picks the power of two 2^-e that moves
// it into [2^14, 2^15); every element is then written as the fp16 value
// v * 2^-e (exact for bf16 inputs in range) in 16-byte chunks of 8 elements,
// and 2^e goes to the tile's per-row tail for the GEMM epilogue.
__global__ void __launch_bounds__(kPqWarps * 32)
permute_x_f16_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ sorted_pair_ids,
                     const int32_t* __restrict__ slot_dest, int k, int H, int nmax, int64_t P, int64_t tail_off,
                     uint8_t* __restrict__ tiles) {
    pdl_sync();
    const int lane = threadIdx.x & 31;
    const int64_t slot = (int64_t)blockIdx.x * kPqWarps + (threadIdx.x >> 5);
    int tile = -1, row = 0, tok = 0;
    if (lane == 0 && slot < P) {
        const int dst = slot_dest[slot];  // -1 past the routed slots
        const int p = sorted_pair_ids[slot];
        if (dst >= 0) {
            tile = dst / nmax;
            row = dst - tile * nmax;
            tok = p / k;
        }
    }
    tile = __shfl_sync(0xFFFFFFFFu, tile, 0);
    if (tile < 0) return;
    row = __shfl_sync(0xFFFFFFFFu, row, 0);
    tok = __shfl_sync(0xFFFFFFFFu, tok, 0);
    const uint16_t* xr = x + (int64_t)tok * H;
    float amax = 0.f;
    for (int j = lane; j < H / 8; j += 32) {
        const uint4 v = *reinterpret_cast<const uint4*>(xr + 8 * j);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(u[i] << 16)), fabsf(__uint_as_float(u[i] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int e = f16_row_exponent(amax);
    const float m = exp2i(-e);
    const int64_t bb = bft::block_bytes(nmax);
    uint8_t* tbase = tiles + (int64_t)tile * (H / 64) * bb;
    for (int j = lane; j < H / 8; j += 32) {  // chunk j: K step j/8, chunk j%8 of the 128-byte row
        const uint4 v = *reinterpret_cast<const uint4*>(xr + 8 * j);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 hv = __floats2half2_rn(__uint_as_float(u[i] << 16) * m, __uint_as_float(u[i] & 0xFFFF0000u) * m);
            o[i] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        uint8_t* blk = tbase + (int64_t)(j >> 3) * bb;
        *reinterpret_cast<uint4*>(blk + row * 128 + (((j & 7) ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (lane == 0) reinterpret_cast<float*>(tiles + tail_off)[(int64_t)tile * nmax + row] = exp2i(e);
}

int permute_x_f16_launch(const qmoe_dims* d, const uint16_t* x, const int32_t* sorted, const int32_t* offsets,
                         const int32_t* tile_start, uint8_t* tiles, cudaStream_t st) {
    const int64_t P = (int64_t)d->T * d->k;
    if (P == 0) return QMOE_OK;
    const int64_t blocks = (P + kPqWarps - 1) / kPqWarps;
    return launch_pdl(permute_x_f16_kernel, (unsigned)blocks, kPqWarps * 32, 0, st, x, sorted,
                      tile_start + schedule_ints(d->E), d->k, d->H, mxt::nmax_for(d), P, bft::blocks_bytes(d, d->H),
                      tiles);
}

// rint(v / s) with the IEEE quotient, clamped to +-127, usually without a
// division: r = v * inv (inv = 1/s rounded once) is within |v/s| * 2^-23 +
// 2^-18 < 2^-16 of the exact quotient for |v / s| <= 127.5 (and the clamp
// decides everything beyond), so when r is at least 1e-4 away from a
// half-integer the correctly rounded quotient rounds to the same integer;
// the rare values nearer a tie take the IEEE division.
__device__ __forceinline__ float rint_quot_clamped(float v, float s, float inv) {
    const float r = v * inv;
    const float frac = r - floorf(r);
    const float q = (fabsf(frac - 0.5f) > 1e-4f) ? rintf(r) : rintf(__fdiv_rn(v, s));
    return fminf(fmaxf(q, -127.f), 127.f);
}

// W8A8 activation tiles.  Each row is quantised with the per-row int8 rule of
// quant_rows_int8_kernel (s = amax / 127, IEEE division, nearest-even,
// clamped to +-127) and each code is written as the fp16 value equal to it
// (exact) into the 128-byte-swizzled tile layout the W4A16 x tiles use, 8
// codes per 16-byte chunk; s goes to the per-row tail.  For every 112-row
// part of a tile and 128-element K step the tiles also record the largest L1
// norm sum |q| over the part's rows: the GEMM uses it to bound its fp32
// partial sums.
constexpr int kTqSub = 112;
constexpr int kTqMaxSteps = 128;  // K <= 16384

__device__ __forceinline__ void load8_as_float(const uint16_t* p, float (&f)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ void load8_as_float(const float* p, float (&f)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// int8 quantisation into W8A8 tiles, one warp per source row (strided over a
// grid of resident CTAs).  The row is read and quantised once, with the rule
// above, and its codes (as equal fp16 values) go to k
// token-tile rows dest[row * k + j] (-1: none) in the W8A8 tile layout, its
// scale to each row's tail.  Each row's per-128-step sum |q| is max-ed into
// its 112-row half tile's entry by global atomics; the launch zeroes those
// entries first.
//   stage 1: rows = the T token rows of bf16 x, dest = each pair's row (the
//            routing sort's per-pair rows), k = top-k: a token row is
//            quantised once for its k pairs;
//   stage 2: rows = the P slot rows of fp32 h, dest = each slot's row, k = 1.
template <typename In>
__global__ void __launch_bounds__(kPqWarps * 32)
permute_quant_int8_kernel(const In* __restrict__ x, const int32_t* __restrict__ pair_dest, int k, int K,
                          int nmax, int64_t T, int64_t tail_off, int64_t l1_off, uint8_t* __restrict__ tiles) {
    pdl_sync();
    const int lane = threadIdx.x & 31;
    const int halves = (nmax + kTqSub - 1) / kTqSub;
    const int KT = K / 128, NC = K / 8;  // 128-element steps, 8-code chunks
    const int64_t bb = bft::block_bytes(nmax);
    float* tail = reinterpret_cast<float*>(tiles + tail_off);
    int* l1g = reinterpret_cast<int*>(tiles + l1_off);
    for (int64_t tok = (int64_t)blockIdx.x * kPqWarps + (threadIdx.x >> 5); tok < T;
         tok += (int64_t)gridDim.x * kPqWarps) {
        // destinations of the first 32 pairs; a row with none (invalid ids, or a slot past the routed
        // ones) is not read
        const int dst0 = (lane < k) ? pair_dest[tok * k + lane] : -1;
        if (k <= 32 && __ballot_sync(0xFFFFFFFFu, dst0 >= 0) == 0) continue;
        const In* xr = x + tok * K;
        float amax = 0.f;
        for (int j = lane; j < NC; j += 32) {
            float f[8];
            load8_as_float(xr + 8 * j, f);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float sc = (amax == 0.f) ? 1.0f : __fdiv_rn(amax, 127.0f);
        const float inv = __frcp_rn(sc);
        for (int p0 = 0; p0 < k; p0 += 32) {
            // lane i: the token-tile row tile * nmax + row of pair p0 + i (-1: invalid expert id)
            const int dst = p0 == 0 ? dst0 : ((p0 + lane < k) ? pair_dest[tok * k + p0 + lane] : -1);
            if (dst >= 0) tail[dst] = sc;
            const int pn = min(32, k - p0);
            for (int j0 = 0; j0 < NC; j0 += 32) {  // warp-uniform trip count (the shuffles below)
                const int j = j0 + lane;
                int l1 = 0;
                uint4 code = make_uint4(0u, 0u, 0u, 0u);
                if (j < NC) {
                    float f[8];
                    load8_as_float(xr + 8 * j, f);
                    uint32_t o[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float q0 = rint_quot_clamped(f[2 * i], sc, inv);
                        const float q1 = rint_quot_clamped(f[2 * i + 1], sc, inv);
                        l1 += abs((int)q0) + abs((int)q1);
                        const __half2 hv = __floats2half2_rn(q0, q1);
                        o[i] = *reinterpret_cast<const uint32_t*>(&hv);
                    }
                    code = make_uint4(o[0], o[1], o[2], o[3]);
                }
                // lanes 0-15 hold step j0/16, lanes 16-31 step j0/16 + 1
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
                const int step = (j0 >> 4) + (lane >> 4);
                for (int q = 0; q < pn; ++q) {
                    const int d = __shfl_sync(0xFFFFFFFFu, dst, q);
                    if (d < 0) continue;  // warp-uniform
                    const int tile = d / nmax, row = d - tile * nmax;
                    if (j < NC) {
                        uint8_t* blk = tiles + ((int64_t)tile * (K / 64) + (j >> 3)) * bb;
                        *reinterpret_cast<uint4*>(blk + row * 128 + (((j & 7) ^ (row & 7)) << 4)) = code;
                    }
                    if ((lane & 15) == 0 && step < KT)
                        atomicMax(l1g + ((int64_t)tile * halves + row / kTqSub) * KT + step, l1);
                }
            }
        }
    }
}

int quant_tiles_int8_launch(const qmoe_dims* d, int64_t K, const void* x, bool from_bf16_tokens,
                            const int32_t* sorted, const int32_t* offsets, const int32_t* tile_start, uint8_t* tiles,
                            cudaStream_t st) {
    const int64_t P = (int64_t)d->T * d->k;
    if (P == 0) return QMOE_OK;
    if (K % 128 != 0 || K / 128 > kTqMaxSteps) return QMOE_ERR_UNSUPPORTED;
    const int nmax = mxt::nmax_for(d);
    const int64_t blocks = mxt::max_tiles(d, nmax) * ((nmax + kTqSub - 1) / kTqSub);
    const int64_t tail = bft::blocks_bytes(d, K);
    const int64_t l1 = tail + mxt::max_tiles(d, nmax) * nmax * 4;
    // one warp per source row: token rows (each quantised once for its k pairs), or slot rows of h
    const size_t l1_bytes = (size_t)(blocks * (K / 128) * 4);
    if (cudaMemsetAsync(tiles + l1, 0, l1_bytes, st) != cudaSuccess) return QMOE_ERR_LAUNCH;
    const int32_t* slot_dest = tile_start + schedule_ints(d->E);
    const int64_t rows = from_bf16_tokens ? (int64_t)d->T : P;
    const int64_t fit = from_bf16_tokens ? resident_ctas(permute_quant_int8_kernel<uint16_t>, kPqWarps * 32)
                                         : resident_ctas(permute_quant_int8_kernel<float>, kPqWarps * 32);
    if (fit <= 0) return QMOE_ERR_CUDA;
    const int64_t grid = std::min<int64_t>((rows + kPqWarps - 1) / kPqWarps, fit);
    if (from_bf16_tokens)
        return launch_pdl(permute_quant_int8_kernel<uint16_t>, (unsigned)grid, kPqWarps * 32, 0, st,
                          static_cast<const uint16_t*>(x), slot_dest + slot_ints(P), d->k, (int)K, nmax, rows, tail,
                          l1, tiles);
    return launch_pdl(permute_quant_int8_kernel<float>, (unsigned)grid, kPqWarps * 32, 0, st,
                      static_cast<const float*>(x), slot_dest, 1, (int)K, nmax, rows, tail, l1, tiles);
}

// W4A16 h tiles (bf16, with per-32-column group maxima) -> fp16 tiles for
// the down projection: one warp per expert-sorted slot.  The row's largest
// magnitude (the largest of its group maxima) picks the power of two 2^-e that
// moves it into [2^14, 2^15) (as for the x tiles); every bf16 value v of the
// row becomes the fp16 value v * 2^-e (exact in range) at the same place of
// the same tile layout, and 2^e goes to the output's per-row tail.
__global__ void __launch_bounds__(kPqWarps * 32)
h_to_f16_kernel(const uint8_t* __restrict__ h_tiles, const float* __restrict__ gmax,
                const int32_t* __restrict__ slot_dest, int I, int nmax, int64_t P, uint8_t* __restrict__ out,
                float* __restrict__ fac) {
    pdl_sync();
    const int lane = threadIdx.x & 31;
    const int64_t slot = (int64_t)blockIdx.x * kPqWarps + (threadIdx.x >> 5);
    int tile = -1, row = 0;
    if (lane == 0 && slot < P) {
        const int dst = slot_dest[slot];  // -1 past the routed slots
        if (dst >= 0) {
            tile = dst / nmax;
            row = dst - tile * nmax;
        }
    }
    tile = __shfl_sync(0xFFFFFFFFu, tile, 0);
    if (tile < 0) return;
    row = __shfl_sync(0xFFFFFFFFu, row, 0);
    const int NG = I / 32;
    const float* gm = gmax + ((int64_t)tile * nmax + row) * NG;
    float amax = 0.f;
    for (int g = lane; g < NG; g += 32) amax = fmaxf(amax, gm[g]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int e = f16_row_exponent(amax);
    const float m = exp2i(-e);
    const int64_t bb = bft::block_bytes(nmax);
    const int64_t base = (int64_t)tile * (I / 64) * bb + row * 128;
    for (int j = lane; j < I / 8; j += 32) {  // chunk j: K step j/8; the chunk's place is the same in both layouts
        const int64_t off = base + (int64_t)(j >> 3) * bb + (((j & 7) ^ (row & 7)) << 4);
        const uint4 v = *reinterpret_cast<const uint4*>(h_tiles + off);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 hv = __floats2half2_rn(__uint_as_float(u[i] << 16) * m, __uint_as_float(u[i] & 0xFFFF0000u) * m);
            o[i] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        *reinterpret_cast<uint4*>(out + off) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (lane == 0) fac[(int64_t)tile * nmax + row] = exp2i(e);
}

int h_to_f16_launch(const qmoe_dims* d, const uint8_t* h_tiles, const int32_t* offsets, const int32_t* tile_start,
                    uint8_t* out, cudaStream_t st) {
    const int64_t P = (int64_t)d->T * d->k;
    if (P == 0) return QMOE_OK;
    const int64_t blocks = (P + kPqWarps - 1) / kPqWarps;
    const int64_t tail = bft::blocks_bytes(d, d->I);
    return launch_pdl(h_to_f16_kernel, (unsigned)blocks, kPqWarps * 32, 0, st, h_tiles,
                      reinterpret_cast<const float*>(h_tiles + tail), tile_start + schedule_ints(d->E), d->I,
                      mxt::nmax_for(d), P, out, reinterpret_cast<float*>(out + tail));
}

int quant_mx_launch(int64_t rows, int64_t cols, const uint16_t* x, uint8_t* q, uint8_t* s, cudaStream_t st) {
    const int64_t n8 = rows * cols / 8;
    if (n8 == 0) return QMOE_OK;
    const int64_t blocks = (n8 + 255) / 256;
    return launch_pdl(quant_mx_bf16_kernel, (unsigned)blocks, 256, 0, st, reinterpret_cast<const uint4*>(x), n8,
                      reinterpret_cast<uint2*>(q), s);
}

template <typename In>
int quant_int8_launch(int64_t rows, int64_t cols, const In* x, int8_t* q, float* s, cudaStream_t st) {
    if (rows == 0) return QMOE_OK;
    return launch_pdl(quant_rows_int8_kernel<In>, (unsigned)rows, 256, 0, st, x, cols, q, s);
}
template int quant_int8_launch<uint16_t>(int64_t, int64_t, const uint16_t*, int8_t*, float*, cudaStream_t);
template int quant_int8_launch<float>(int64_t, int64_t, const float*, int8_t*, float*, cudaStream_t);

}  // namespace qmoe

extern "C" int qmoe_quant_act_mxfp8(int64_t rows, int64_t cols, const uint16_t* x_bf16, uint8_t* x_q, uint8_t* x_s,
                                    qmoe_stream_t stream) {
    using namespace qmoe;
    if (rows < 0 || cols <= 0 || cols % 32 != 0 || rows > (1ll << 31)) return QMOE_ERR_ARG;
    if (rows > 0 && (!x_bf16 || !x_q || !x_s || !aligned16(x_bf16) || !aligned16(x_q))) return QMOE_ERR_ARG;
    return quant_mx_launch(rows, cols, x_bf16, x_q, x_s, (cudaStream_t)stream);
}

extern "C" int qmoe_quant_rows_int8_bf16(int64_t rows, int64_t cols, const uint16_t* x, int8_t* q, float* s,
                                         qmoe_stream_t stream) {
    using namespace qmoe;
    if (rows < 0 || cols <= 0 || rows > (1ll << 31)) return QMOE_ERR_ARG;
    if (rows > 0 && (!x || !q || !s)) return QMOE_ERR_ARG;
    return quant_int8_launch<uint16_t>(rows, cols, x, q, s, (cudaStream_t)stream);
}

extern "C" int qmoe_quant_rows_int8_f32(int64_t rows, int64_t cols, const float* x, int8_t* q, float* s,
                                        qmoe_stream_t stream) {
    using namespace qmoe;
    if (rows < 0 || cols <= 0 || rows > (1ll << 31)) return QMOE_ERR_ARG;
    if (rows > 0 && (!x || !q || !s)) return QMOE_ERR_ARG;
    return quant_int8_launch<float>(rows, cols, x, q, s, (cudaStream_t)stream);
}
