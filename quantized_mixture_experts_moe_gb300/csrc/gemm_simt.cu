// Grouped expert GEMMs, plain SIMT tiles (all schemes).
//
// One launch covers every expert ("perf(qmoe): group prefill expert matmuls",
// description): the grid's x index enumerates (expert, 32-slot tile) pairs in
// expert order, found by a per-CTA scan of the expert offsets, and y the
// output-column tiles.  Operands are dequantised exactly to fp32 (int32 for
// W8A8) in shared memory, so this path is also the exact reference point for
// the tensor-core kernels.  Stage 1 computes the gate rows n and the up rows
// I + n of the same 64 columns and applies SwiGLU and the scheme's
// intermediate quantisation in the epilogue; stage 2 writes y rows (fp32
// sums stored as bf16).
#include "qmoe_common.cuh"
#include "gemm_simt.cuh"

namespace qmoe {

constexpr int BM = 32;  // slots per tile
constexpr int BN = 64;  // output columns per tile
constexpr int BK = 32;  // one scale block

enum { S_W4A16 = 0, S_MXFP4 = 1, S_W8A8 = 2 };

template <int SCHEME>
struct Acc {
    using T = float;
};
template <>
struct Acc<S_W8A8> {
    using T = int32_t;
};

// Finds this CTA's (expert, slot range) from the expert offsets: tile b of the
// sequence in which expert e contributes ceil(M_e / BM) tiles.  Returns false
// when b is past the last tile.
__device__ bool find_tile(const int32_t* __restrict__ offsets, int E, int b, int* e_out, int* m0, int* m1) {
    __shared__ int s_e, s_m0, s_m1;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int running = 0;
        int found = -1;
        for (int base = 0; base < E && found < 0; base += 32) {
            const int e = base + lane;
            const int cnt = e < E ? offsets[e + 1] - offsets[e] : 0;
            const int tiles = (cnt + BM - 1) / BM;
            int incl = tiles;
            for (int o = 1; o < 32; o <<= 1) {
                int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
            if (b < running + total) {
                const bool mine = (b >= running + incl - tiles) && (b < running + incl);
                const uint32_t who = __ballot_sync(0xFFFFFFFFu, mine);
                const int src = __ffs(who) - 1;
                if (lane == src) {
                    s_e = e;
                    s_m0 = offsets[e] + (b - (running + incl - tiles)) * BM;
                    s_m1 = min(s_m0 + BM, offsets[e + 1]);
                }
                found = 1;
            }
            running += total;
        }
        if (found < 0 && lane == 0) s_e = -1;
    }
    __syncthreads();
    *e_out = s_e;
    *m0 = s_m0;
    *m1 = s_m1;
    return s_e >= 0;
}

// ---- operand loaders: 4 consecutive K elements of an activation row
template <int SCHEME>
__device__ __forceinline__ void load_act4(const SimtArgs& a, int64_t row, int K, int kk, typename Acc<SCHEME>::T* o) {
    if constexpr (SCHEME == S_W4A16) {
        const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.act) + row * K + kk);
        o[0] = __uint_as_float(v.x << 16);
        o[1] = __uint_as_float(v.x & 0xFFFF0000u);
        o[2] = __uint_as_float(v.y << 16);
        o[3] = __uint_as_float(v.y & 0xFFFF0000u);
    } else if constexpr (SCHEME == S_MXFP4) {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(a.act) + row * K + kk);
        const float s = e8m0_to_float(static_cast<const uint8_t*>(a.act_s)[row * (K / 32) + kk / 32]);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = e4m3_to_float((uint8_t)(v >> (8 * i))) * s;
    } else {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(static_cast<const int8_t*>(a.act) + row * K + kk);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = (int32_t)(int8_t)(v >> (8 * i));
    }
}

// ---- NE consecutive K elements (NE = 16 or 8, from element kk) of weight row `wrow`
template <int SCHEME, int NE>
__device__ __forceinline__ void load_w(const SimtArgs& a, int64_t wrow, int K, int kk, typename Acc<SCHEME>::T* o) {
    if constexpr (SCHEME == S_W8A8) {
        const int8_t* p = static_cast<const int8_t*>(a.w) + wrow * K + kk;
        uint32_t v[NE / 4];
        if constexpr (NE == 16) {
            const uint4 t = *reinterpret_cast<const uint4*>(p);
            v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
        } else {
            const uint2 t = *reinterpret_cast<const uint2*>(p);
            v[0] = t.x; v[1] = t.y;
        }
#pragma unroll
        for (int i = 0; i < NE; ++i) o[i] = (int32_t)(int8_t)(v[i / 4] >> (8 * (i % 4)));
    } else {
        const uint8_t* p;
        if constexpr (SCHEME == S_W4A16) {
            p = static_cast<const uint8_t*>(a.w) + wrow * (K / 2) + kk / 2;
        } else {
            // tile-major pre-packed: 128x128 tiles of 8 KiB, 64 bytes per tile row
            const int64_t KT = (K + 127) / 128;
            p = static_cast<const uint8_t*>(a.w) + ((wrow / 128) * KT + kk / 128) * 8192 + (wrow & 127) * 64 +
                (kk & 127) / 2;
        }
        uint32_t v[NE / 8];
        if constexpr (NE == 16) {
            const uint2 t = *reinterpret_cast<const uint2*>(p);
            v[0] = t.x; v[1] = t.y;
        } else {
            v[0] = *reinterpret_cast<const uint32_t*>(p);
        }
        float s;
        if constexpr (SCHEME == S_W4A16)
            s = __half2float(__ushort_as_half(static_cast<const uint16_t*>(a.w_s)[wrow * (K / 32) + kk / 32]));
        else {
            // pre-packed scale atoms: (row tile, group of 4 blocks) x 512 bytes
            const int64_t kb = kk / 32, KG = (K + 127) / 128;
            const int64_t atom = (wrow / 128) * KG + kb / 4;
            const int r = (int)(wrow & 127);
            s = e8m0_to_float(static_cast<const uint8_t*>(a.w_s)[atom * 512 + 16 * (r & 31) + 4 * (r >> 5) + (kb & 3)]);
        }
#pragma unroll
        for (int i = 0; i < NE; ++i) {
            const uint32_t nib = (v[i / 8] >> (4 * (i % 8))) & 15u;  // element 2b in the low nibble of byte b
            const float q = (SCHEME == S_W4A16) ? (float)((int)nib - 8) : e2m1_to_float(nib);
            o[i] = q * s;
        }
    }
}

template <int SCHEME, int STAGE>
__global__ void __launch_bounds__(256) gemm_simt_kernel(SimtArgs a) {
    using AccT = typename Acc<SCHEME>::T;
    constexpr int NW = (STAGE == 1) ? 2 * BN : BN;  // weight rows per tile
    __shared__ AccT As[BM][BK + 1];
    __shared__ AccT Bs[NW][BK + 1];

    int e, m0, m1;
    if (!find_tile(a.offsets, a.E, blockIdx.x, &e, &m0, &m1)) return;
    const int K = (STAGE == 1) ? a.H : a.I;      // reduction length
    const int N = (STAGE == 1) ? a.I : a.H;      // output columns
    const int WR = (STAGE == 1) ? 2 * a.I : a.H; // weight rows per expert
    const int n0 = blockIdx.y * BN;
    const int tid = threadIdx.x;

    // activation row for the loader thread: slot m0 + tid/8, K part (tid%8)*4
    const int lr = tid >> 3;
    const int lslot = m0 + lr;
    const bool lvalid = lslot < m1;
    int64_t arow = 0;
    if (lvalid) arow = (STAGE == 1) ? (int64_t)(a.sorted[lslot] / a.k) : (int64_t)lslot;

    // weight row for the loader thread
    constexpr int NE = (STAGE == 1) ? 16 : 8;
    const int wr_local = (STAGE == 1) ? (tid >> 1) : (tid >> 2);
    const int wk = (STAGE == 1) ? (tid & 1) * 16 : (tid & 3) * 8;
    int ncol;
    int64_t wrow;
    if (STAGE == 1) {
        const int half = wr_local / BN;  // 0 gate, 1 up
        ncol = n0 + (wr_local % BN);
        wrow = (int64_t)e * WR + half * a.I + ncol;
    } else {
        ncol = n0 + wr_local;
        wrow = (int64_t)e * WR + ncol;
    }
    const bool wvalid = ncol < N;

    const int ty = tid >> 4, tx = tid & 15;
    AccT acc[2][2][4];  // [gate/up][row][col]
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[g][r][c] = 0;

    for (int k0 = 0; k0 < K; k0 += BK) {
        AccT av[4] = {0, 0, 0, 0};
        if (lvalid) load_act4<SCHEME>(a, arow, K, k0 + (tid & 7) * 4, av);
#pragma unroll
        for (int i = 0; i < 4; ++i) As[lr][(tid & 7) * 4 + i] = av[i];
        AccT wv[NE];
#pragma unroll
        for (int i = 0; i < NE; ++i) wv[i] = 0;
        if (wvalid) load_w<SCHEME, NE>(a, wrow, K, k0 + wk, wv);
#pragma unroll
        for (int i = 0; i < NE; ++i) Bs[wr_local][wk + i] = wv[i];
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            const AccT a0 = As[ty * 2][kk], a1 = As[ty * 2 + 1][kk];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const AccT bg = Bs[tx * 4 + c][kk];
                acc[0][0][c] += a0 * bg;
                acc[0][1][c] += a1 * bg;
                if (STAGE == 1) {
                    const AccT bu = Bs[BN + tx * 4 + c][kk];
                    acc[1][0][c] += a0 * bu;
                    acc[1][1][c] += a1 * bu;
                }
            }
        }
        __syncthreads();
    }

    const int col = n0 + tx * 4;
    const bool cvalid = col < N;  // N % 32 == 0, so 4-column groups are all in or all out
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int slot = m0 + ty * 2 + r;
        const bool rvalid = slot < m1;
        if (STAGE == 2) {
            if (!(rvalid && cvalid)) continue;
            float o[4];
            if constexpr (SCHEME == S_W8A8) {
                const float hs = static_cast<const float*>(a.act_s)[slot];
                const float* sw = static_cast<const float*>(a.w_s) + (int64_t)e * a.H;
#pragma unroll
                for (int c = 0; c < 4; ++c) o[c] = __fmul_rn(__fmul_rn((float)acc[0][r][c], hs), sw[col + c]);
                if (a.dbg_acc) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) a.dbg_acc[(int64_t)slot * a.H + col + c] = (int32_t)acc[0][r][c];
                }
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) o[c] = (float)acc[0][r][c];
            }
            uint2 ob;
            ob.x = (uint32_t)float_to_bf16_bits(o[0]) | ((uint32_t)float_to_bf16_bits(o[1]) << 16);
            ob.y = (uint32_t)float_to_bf16_bits(o[2]) | ((uint32_t)float_to_bf16_bits(o[3]) << 16);
            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + (int64_t)slot * a.H + col) = ob;
            continue;
        }
        // stage 1 epilogue: SwiGLU, then the scheme's intermediate format
        float h[4];
        if constexpr (SCHEME == S_W8A8) {
            if (rvalid && cvalid) {
                const int64_t tok = a.sorted[slot] / a.k;
                const float sa = static_cast<const float*>(a.act_s)[tok];
                const float* sw = static_cast<const float*>(a.w_s) + (int64_t)e * 2 * a.I;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float g = __fmul_rn(__fmul_rn((float)acc[0][r][c], sa), sw[col + c]);
                    const float u = __fmul_rn(__fmul_rn((float)acc[1][r][c], sa), sw[a.I + col + c]);
                    h[c] = silu_mul(g, u);
                }
                if (a.dbg_acc) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        a.dbg_acc[(int64_t)slot * 2 * a.I + col + c] = (int32_t)acc[0][r][c];
                        a.dbg_acc[(int64_t)slot * 2 * a.I + a.I + col + c] = (int32_t)acc[1][r][c];
                    }
                }
                *reinterpret_cast<float4*>(static_cast<float*>(a.out) + (int64_t)slot * a.I + col) =
                    make_float4(h[0], h[1], h[2], h[3]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) h[c] = silu_mul((float)acc[0][r][c], (float)acc[1][r][c]);
            if constexpr (SCHEME == S_W4A16) {
                if (rvalid && cvalid) {
                    uint2 o;
                    o.x = (uint32_t)float_to_bf16_bits(h[0]) | ((uint32_t)float_to_bf16_bits(h[1]) << 16);
                    o.y = (uint32_t)float_to_bf16_bits(h[2]) | ((uint32_t)float_to_bf16_bits(h[3]) << 16);
                    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + (int64_t)slot * a.I + col) = o;
                }
            } else {
                // MX quantisation along I: a 32-block is 8 lanes (tx 0..7 or 8..15)
                float amax = fmaxf(fmaxf(fabsf(h[0]), fabsf(h[1])), fmaxf(fabsf(h[2]), fabsf(h[3])));
                amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
                amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
                if (rvalid && cvalid) {
                    uint32_t codes = 0;
                    uint8_t sb = 127;
                    if (amax > 0.f) {
                        const int X = mx_block_exponent(amax);
                        const float m = exp2i(-X);
                        sb = (uint8_t)(X + 127);
                        codes = (uint32_t)e4m3x2_from_float(h[0] * m, h[1] * m) |
                                ((uint32_t)e4m3x2_from_float(h[2] * m, h[3] * m) << 16);
                    }
                    *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.out) + (int64_t)slot * a.I + col) = codes;
                    if ((tx & 7) == 0) static_cast<uint8_t*>(a.out_s)[(int64_t)slot * (a.I / 32) + col / 32] = sb;
                }
            }
        }
    }
}

template <int SCHEME, int STAGE>
int gemm_simt_launch(const SimtArgs& a, cudaStream_t st) {
    const int64_t P = (int64_t)a.T * a.k;
    if (P == 0) return QMOE_OK;
    const int N = (STAGE == 1) ? a.I : a.H;
    const int64_t max_tiles = (P + BM - 1) / BM + a.E;
    if (max_tiles > 0x7FFFFFFF) return QMOE_ERR_UNSUPPORTED;
    dim3 grid((unsigned)max_tiles, (unsigned)ceil_div(N, BN));
    if (grid.y > 65535) return QMOE_ERR_UNSUPPORTED;
    gemm_simt_kernel<SCHEME, STAGE><<<grid, 256, 0, st>>>(a);
    return launch_status();
}

int gemm_simt(int scheme, int stage, const SimtArgs& a, cudaStream_t st) {
    switch (scheme * 2 + (stage - 1)) {
        case 0: return gemm_simt_launch<S_W4A16, 1>(a, st);
        case 1: return gemm_simt_launch<S_W4A16, 2>(a, st);
        case 4: return gemm_simt_launch<S_W8A8, 1>(a, st);
        case 5: return gemm_simt_launch<S_W8A8, 2>(a, st);
    }
    return QMOE_ERR_ARG;
}

}  // namespace qmoe
