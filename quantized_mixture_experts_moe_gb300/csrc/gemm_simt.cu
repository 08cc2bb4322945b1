// Grouped W8A8 expert GEMMs, plain SIMT tiles with exact int32 accumulation.
//
// One launch covers every expert ("perf(qmoe): group prefill expert matmuls",
// description): the grid's x index enumerates (expert, 32-slot tile) pairs in
// expert order, found by a per-CTA scan of the expert offsets, and y the
// output-column tiles.  int8 x int8 products are summed in int32 ("Evaluate
// native IU4/IU8 WMMA for grouped-INT MoE prefill on gfx1151", Constraint).
// Stage 1 computes the gate rows n and the up rows I + n of the same 64
// columns and applies the dequantisation and SwiGLU in the epilogue; stage 2
// writes y rows (fp32 stored as bf16).
#include "qmoe_common.cuh"
#include "gemm_simt.cuh"

namespace qmoe {

constexpr int BM = 32;  // slots per tile
constexpr int BN = 64;  // output columns per tile
constexpr int BK = 32;  // one scale block

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

// ---- 4 consecutive K elements of an activation row
__device__ __forceinline__ void load_act4(const SimtArgs& a, int64_t row, int K, int kk, int32_t* o) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(static_cast<const int8_t*>(a.act) + row * K + kk);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = (int32_t)(int8_t)(v >> (8 * i));
}

// ---- NE consecutive K elements (NE = 16 or 8, from element kk) of weight row `wrow`
template <int NE>
__device__ __forceinline__ void load_w(const SimtArgs& a, int64_t wrow, int K, int kk, int32_t* o) {
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
}

template <int STAGE>
__global__ void __launch_bounds__(256) gemm_simt_kernel(SimtArgs a) {
    using AccT = int32_t;
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
        if (lvalid) load_act4(a, arow, K, k0 + (tid & 7) * 4, av);
#pragma unroll
        for (int i = 0; i < 4; ++i) As[lr][(tid & 7) * 4 + i] = av[i];
        AccT wv[NE];
#pragma unroll
        for (int i = 0; i < NE; ++i) wv[i] = 0;
        if (wvalid) load_w<NE>(a, wrow, K, k0 + wk, wv);
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
            const float hs = static_cast<const float*>(a.act_s)[slot];
            const float* sw = static_cast<const float*>(a.w_s) + (int64_t)e * a.H;
#pragma unroll
            for (int c = 0; c < 4; ++c) o[c] = __fmul_rn(__fmul_rn((float)acc[0][r][c], hs), sw[col + c]);
            if (a.dbg_acc) {
#pragma unroll
                for (int c = 0; c < 4; ++c) a.dbg_acc[(int64_t)slot * a.H + col + c] = (int32_t)acc[0][r][c];
            }
            uint2 ob;
            ob.x = (uint32_t)float_to_bf16_bits(o[0]) | ((uint32_t)float_to_bf16_bits(o[1]) << 16);
            ob.y = (uint32_t)float_to_bf16_bits(o[2]) | ((uint32_t)float_to_bf16_bits(o[3]) << 16);
            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + (int64_t)slot * a.H + col) = ob;
            continue;
        }
        // stage 1 epilogue: dequantisation and SwiGLU
        if (rvalid && cvalid) {
            float h[4];
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
    }
}

template <int STAGE>
int gemm_simt_launch(const SimtArgs& a, cudaStream_t st) {
    const int64_t P = (int64_t)a.T * a.k;
    if (P == 0) return QMOE_OK;
    const int N = (STAGE == 1) ? a.I : a.H;
    const int64_t max_tiles = (P + BM - 1) / BM + a.E;
    if (max_tiles > 0x7FFFFFFF) return QMOE_ERR_UNSUPPORTED;
    dim3 grid((unsigned)max_tiles, (unsigned)ceil_div(N, BN));
    if (grid.y > 65535) return QMOE_ERR_UNSUPPORTED;
    gemm_simt_kernel<STAGE><<<grid, 256, 0, st>>>(a);
    return launch_status();
}

int gemm_simt_w8a8(int stage, const SimtArgs& a, cudaStream_t st) {
    return stage == 1 ? gemm_simt_launch<1>(a, st) : gemm_simt_launch<2>(a, st);
}

}  // namespace qmoe
