// Grouped W4A16 expert GEMMs on the 5th-generation tensor cores (tcgen05,
// kind::f16 with bf16 operands, fp32 accumulation in TMEM).
//
// "perf(qmoe): group prefill expert matmuls" (description) batches symmetric
// int4 expert projections into one launch for all experts; "Evaluate native
// IU4/IU8 WMMA for grouped-INT MoE prefill on gfx1151" (Problem, Constraint)
// notes that int4 weights with bf16 activations are computed by dequantising
// to bf16 and running a bf16 dot.  This is that computation for sm_103a:
//   stage 1: h = silu(W1_gate . x) * (W1_up . x), rounded to bf16;
//   stage 2: y = W2 . h, accumulated in fp32, stored as bf16.
// The GPU dequantises each weight as q * s rounded to bf16 (the scale is
// first rounded to bf16), a relative error of at most about 2^-8 per weight.
//
// Structure (one persistent CTA per SM, 16 warps):
//   warp 0      raw weight producer: bulk copies of pre-packed int4 blocks
//               (128 rows x 64 elements of codes + their fp16 scales, 4608
//               contiguous bytes) into a raw ring, two per step (stage 1: a
//               gate block and its up partner; stage 2: two adjacent W2 row
//               tiles).
//   warp 1      activation producer: bulk copy of the step's bf16 tile rows
//               (already 128-byte swizzled, see mx_tiles.cuh).
//   warps 2-3   MMA issuers, one per weight tile (M = 128 weight rows, N =
//               tokens rounded up to 16, K = 16 per instruction).
//   warps 4-11  converters: one thread per weight row; (n - 8) * s in bf16x2
//               arithmetic into the swizzled K-major bf16 tile, then a
//               generic -> async proxy fence before publishing the slot.
//   warps 12-15 epilogue, one per TMEM lane quadrant.
// Units and tiling are those of the MXFP4 kernels (token tiles of 112 or 224
// from the routing sort's schedule, weights as the MMA's A operand).
#include "qmoe_common.cuh"
#include "mx_tiles.cuh"
#include "tc_ptx.cuh"

namespace qmoe {
namespace w4 {

constexpr int WARP_W = 0, WARP_B = 1, WARP_MMA = 2, WARP_MMA2 = 3;
constexpr int WARP_CVT0 = 4, CVT_WARPS = 8;
constexpr int WARP_EPI0 = 12, EPI_WARPS = 4;
constexpr int THREADS = (WARP_EPI0 + EPI_WARPS) * 32;
constexpr int KSTEP = 64;  // K elements per step (128-byte bf16 rows)
constexpr int MAX_E = 512;

template <int STAGE, int NMAX_>
struct Cfg {
    static constexpr int NMAX = NMAX_;
    static constexpr int AT = 2;
    static constexpr int ACC_BUFS = (AT * NMAX * 2 <= 512) ? 2 : 1;
    static constexpr int A_BYTES = AT * 128 * 128;               // bf16 tiles, 128 rows x 128 bytes each
    static constexpr int B_BYTES = ((NMAX + 7) / 8) * 1024;
    static constexpr int RAW_BYTES = AT * bft::kW4Block;
    static constexpr int RS = 3;                                  // raw ring depth
    static constexpr int SLOT_BYTES = A_BYTES + B_BYTES;
    static constexpr int S = (224 * 1024 - RS * RAW_BYTES - 8 * 1024) / SLOT_BYTES;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = A_OFF + S * A_BYTES;
    static constexpr int RAW_OFF = B_OFF + S * B_BYTES;
    static constexpr int BAR_OFF = RAW_OFF + RS * RAW_BYTES;
    static constexpr int NBAR = 2 * RS + 2 * S + 2 * ACC_BUFS;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int SCHED_OFF = MISC_OFF + 64;
    static constexpr size_t smem_bytes(int E) { return (size_t)SCHED_OFF + (size_t)(E + 1) * 4 + 1024; }
    static constexpr uint32_t ACC_COLS = AT * NMAX;
    static_assert(ACC_BUFS * ACC_COLS <= 512, "TMEM budget");
    static_assert(S >= 2 && NMAX % 16 == 0, "ring / N tile");
};
static_assert(Cfg<1, 112>::smem_bytes(MAX_E) <= 232448 && Cfg<1, 224>::smem_bytes(MAX_E) <= 232448 &&
                  Cfg<2, 112>::smem_bytes(MAX_E) <= 232448 && Cfg<2, 224>::smem_bytes(MAX_E) <= 232448,
              "shared memory per CTA");

struct Args {
    int T, k, H, I, E;
    const uint8_t* act;         // bf16 activation tiles: stage 1 x (K = H), stage 2 h (K = I)
    const uint8_t* w;           // pre-packed int4 blocks
    const int32_t* offsets;
    const int32_t* tile_start;
    uint8_t* h_tiles;           // stage 1 output (K = I)
    uint16_t* y;                // stage 2 output, bf16 slot order
    int32_t* status;
};

template <int NMAX>
__device__ __forceinline__ void decode_unit(int u, int NB, const int* tile_start, int E, const int32_t* offsets,
                                            int& e, int& m0, int& ntok, int& nb, int& t) {
    t = u / NB;
    nb = u - t * NB;
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tile_start[mid] <= t) lo = mid; else hi = mid;
    }
    e = lo;
    m0 = offsets[e] + (t - tile_start[e]) * NMAX;
    ntok = min(NMAX, offsets[e + 1] - m0);
}

__device__ __forceinline__ void set_abort(volatile int* flag, int32_t* status) {
    *flag = 1;
    atomicOr(status, QMOE_DEV_WAIT_TIMEOUT);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane) {
    int w = 1;
    if (lane == 0) w = tc::mbar_wait(bar, parity) ? 1 : 0;
    return __shfl_sync(0xFFFFFFFFu, w, 0) != 0;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Eight int4 codes (one reordered word) times a bf16x2 scale -> four bf16x2
// pairs in K order.  0x4300 | n is the bf16 value 128 + n; subtracting 136
// gives n - 8 exactly.
__device__ __forceinline__ uint4 dequant8(uint32_t w, uint32_t s2) {
    const uint32_t magic = 0x43004300u, bias = 0x43084308u;  // 128, 136 as bf16x2
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) p[j] = bf16x2_mul(bf16x2_sub(((w >> (4 * j)) & 0x000F000Fu) | magic, bias), s2);
    return make_uint4(p[0], p[1], p[2], p[3]);
}

template <int STAGE, int NMAX>
__global__ void __launch_bounds__(THREADS, 1) w4_gemm_kernel(const Args a) {
    using C = Cfg<STAGE, NMAX>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::A_OFF;
    uint8_t* sB = smem + C::B_OFF;
    uint8_t* sRaw = smem + C::RAW_OFF;
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* raw_empty = raw_full + C::RS;
    uint64_t* full = raw_empty + C::RS;
    uint64_t* empty = full + C::S;
    uint64_t* acc_full = empty + C::S;
    uint64_t* acc_empty = acc_full + C::ACC_BUFS;
    uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 8);
    int* tile_start = reinterpret_cast<int*>(smem + C::SCHED_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E;
    const int K = (STAGE == 1) ? a.H : a.I;
    const int NB = (STAGE == 1) ? a.I / 128 : a.H / 256;
    const int KT = K / KSTEP;

    for (int i = threadIdx.x; i <= E; i += blockDim.x) tile_start[i] = a.tile_start[i];
    if (threadIdx.x == 32 * WARP_MMA) {
        for (int s = 0; s < C::RS; ++s) {
            tc::mbar_init(&raw_full[s], 1);
            tc::mbar_init(&raw_empty[s], CVT_WARPS);
        }
        for (int s = 0; s < C::S; ++s) {
            tc::mbar_init(&full[s], 1 + CVT_WARPS);  // activation producer (with tx) + converters
            tc::mbar_init(&empty[s], 2);             // the two MMA issuers' commits
        }
        for (int b = 0; b < C::ACC_BUFS; ++b) {
            tc::mbar_init(&acc_full[b], 2);
            tc::mbar_init(&acc_empty[b], EPI_WARPS);
        }
        *abort_flag = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    const int total_units = tile_start[E] * NB;
    if ((int)blockIdx.x >= total_units) return;

    if (warp == WARP_MMA) {
        tc::tmem_alloc(tmem_base_smem, 512);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tm = *tmem_base_smem;

    if (warp == WARP_W) {
        // ------------------------------------------------ raw weight producer
        if (lane == 0) {
            int rs = 0;
            uint32_t phase = 0;
            const int rows_per_e = (STAGE == 1) ? 2 * a.I : a.H;
            const int64_t second = (STAGE == 1) ? (int64_t)(a.I / 128) * KT : KT;  // block distance to tile 2
            for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x) {
                int e, m0, ntok, nb, t;
                decode_unit<NMAX>(u, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t);
                const int rt0 = (STAGE == 1) ? (e * rows_per_e + nb * 128) / 128 : (e * rows_per_e + nb * 256) / 128;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(&raw_empty[rs], phase ^ 1)) { set_abort(abort_flag, a.status); break; }
                    tc::mbar_arrive_expect_tx(&raw_full[rs], C::RAW_BYTES);
                    const int64_t b0 = (int64_t)rt0 * KT + kt;
                    uint8_t* d = sRaw + rs * C::RAW_BYTES;
                    tc::bulk_load(d, a.w + b0 * bft::kW4Block, bft::kW4Block, &raw_full[rs]);
                    tc::bulk_load(d + bft::kW4Block, a.w + (b0 + second) * bft::kW4Block, bft::kW4Block,
                                  &raw_full[rs]);
                    if (++rs == C::RS) { rs = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == WARP_B) {
        // ------------------------------------------------ activation producer
        if (lane == 0) {
            int slot = 0;
            uint32_t phase = 0;
            const int64_t bb = bft::block_bytes(NMAX);
            for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x) {
                int e, m0, ntok, nb, t;
                decode_unit<NMAX>(u, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t);
                const uint32_t bytes = (uint32_t)((ntok + 15) & ~15) * 128u;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(&empty[slot], phase ^ 1)) { set_abort(abort_flag, a.status); break; }
                    tc::mbar_arrive_expect_tx(&full[slot], bytes);
                    tc::bulk_load(sB + slot * C::B_BYTES, a.act + ((int64_t)t * KT + kt) * bb, bytes, &full[slot]);
                    if (++slot == C::S) { slot = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == WARP_MMA || warp == WARP_MMA2) {
        // ------------------------------------------------ MMA issuers
        const int iss = warp - WARP_MMA;
        if (lane == 0) {
            int slot = 0, ab = 0;
            uint32_t phase = 0, pacc = 0;
            for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x) {
                int e, m0, ntok, nb, t;
                decode_unit<NMAX>(u, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t);
                const int nmma = (ntok + 15) & ~15;
                const uint32_t idesc = tc::idesc_bf16_f32(128, nmma);
                if (!tc::mbar_wait(&acc_empty[ab], pacc ^ 1)) { set_abort(abort_flag, a.status); break; }
                tc::tc_fence_after();
                const uint32_t dcol = ab * C::ACC_COLS + iss * NMAX;
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(&full[slot], phase)) { set_abort(abort_flag, a.status); ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(sA + slot * C::A_BYTES + iss * 128 * 128);
                    const uint32_t b0 = tc::smem_u32(sB + slot * C::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_f16(tm + dcol, tc::sdesc_kmajor_sw128(a0 + 32 * kk), tc::sdesc_kmajor_sw128(b0 + 32 * kk),
                                    idesc, (kt > 0 || kk > 0) ? 1u : 0u);
                    tc::mma_commit(&empty[slot]);
                    if (++slot == C::S) { slot = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit(&acc_full[ab]);
                if (++ab == C::ACC_BUFS) { ab = 0; pacc ^= 1; }
            }
        }
        __syncwarp();
    } else if (warp < WARP_EPI0) {
        // ------------------------------------------------ converters: int4 -> bf16 tiles
        const int ct = (warp - WARP_CVT0) * 32 + lane;  // 0..255
        const int tile = ct >> 7, row = ct & 127;
        int rs = 0, slot = 0;
        uint32_t rphase = 0, phase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok && !*abort_flag; u += gridDim.x) {
            for (int kt = 0; kt < KT; ++kt) {
                if (!warp_wait(&raw_full[rs], rphase, lane) || !warp_wait(&empty[slot], phase ^ 1, lane)) {
                    if (lane == 0) set_abort(abort_flag, a.status);
                    ok = false;
                    break;
                }
                const uint8_t* src = sRaw + rs * C::RAW_BYTES + tile * bft::kW4Block;
                const uint4 c0 = *reinterpret_cast<const uint4*>(src + row * 32);
                const uint4 c1 = *reinterpret_cast<const uint4*>(src + row * 32 + 16);
                const uint32_t sc = *reinterpret_cast<const uint32_t*>(src + 4096 + row * 4);
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&raw_empty[rs]);
                // fp16 scales -> bf16x2 (s, s)
                const float s0 = __half2float(__ushort_as_half((uint16_t)(sc & 0xFFFFu)));
                const float s1 = __half2float(__ushort_as_half((uint16_t)(sc >> 16)));
                const uint32_t b0 = float_to_bf16_bits(s0), b1 = float_to_bf16_bits(s1);
                const uint32_t s2a = b0 | (b0 << 16), s2b = b1 | (b1 << 16);
                const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                uint8_t* dst = sA + slot * C::A_BYTES + tile * 128 * 128 + row * 128;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8)
                    *reinterpret_cast<uint4*>(dst + ((w8 ^ (row & 7)) << 4)) = dequant8(wv[w8], w8 < 4 ? s2a : s2b);
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&full[slot]);
                if (++rs == C::RS) { rs = 0; rphase ^= 1; }
                if (++slot == C::S) { slot = 0; phase ^= 1; }
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        int ab = 0;
        uint32_t pacc = 0;
        for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x) {
            int e, m0, ntok, nb, t;
            decode_unit<NMAX>(u, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t);
            int w = 1;
            if (lane == 0) w = tc::mbar_wait_sleep(&acc_full[ab], pacc) ? 1 : 0;
            if (!__shfl_sync(0xFFFFFFFFu, w, 0)) {
                if (lane == 0) set_abort(abort_flag, a.status);
                break;
            }
            tc::tc_fence_after();
            const uint32_t dcol = ab * C::ACC_COLS;
            const int nl = q * 32 + lane;  // column within the 128-column block
            uint8_t* hblk = nullptr;
            if (STAGE == 1)
                hblk = a.h_tiles + ((int64_t)t * (a.I / KSTEP) + nb * 2 + (nl >> 6)) * bft::block_bytes(NMAX);
            for (int c0 = 0; c0 < ntok; c0 += 16) {
                uint32_t g[16], g2[16];
                tc::tmem_ld_32x32b_x16(tm + lane_addr + dcol + c0, g);
                tc::tmem_ld_32x32b_x16(tm + lane_addr + dcol + NMAX + c0, g2);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = c0 + j;
                    if (c >= ntok) break;
                    if (STAGE == 1) {
                        const float gv = __uint_as_float(g[j]);
                        const float h = __fdividef(gv, 1.0f + __expf(-gv)) * __uint_as_float(g2[j]);
                        *reinterpret_cast<uint16_t*>(hblk + bft::elem_offset(c, nl & 63)) = float_to_bf16_bits(h);
                    } else {
                        uint16_t* yr = a.y + (int64_t)(m0 + c) * a.H + 2 * nb * 128 + nl;
                        yr[0] = float_to_bf16_bits(__uint_as_float(g[j]));
                        yr[128] = float_to_bf16_bits(__uint_as_float(g2[j]));
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acc_empty[ab]);
            if (++ab == C::ACC_BUFS) { ab = 0; pacc ^= 1; }
        }
    }

    if (*abort_flag) {
        const long long t0 = clock64();
        while (clock64() - t0 < 20000000ll) { }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tm, 512);
    }
}

int num_sms_here() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

template <int STAGE, int NMAX>
static int launch_cfg(const Args& a, cudaStream_t st) {
    using C = Cfg<STAGE, NMAX>;
    if (cudaFuncSetAttribute(w4_gemm_kernel<STAGE, NMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::smem_bytes(MAX_E)) != cudaSuccess)
        return QMOE_ERR_LAUNCH;
    const int grid = num_sms_here();
    if (grid <= 0) return QMOE_ERR_CUDA;
    w4_gemm_kernel<STAGE, NMAX><<<grid, THREADS, C::smem_bytes(a.E), st>>>(a);
    return launch_status();
}

}  // namespace w4

bool w4_tc_ok(const qmoe_dims* d) { return d->H % 256 == 0 && d->I % 128 == 0 && d->E <= w4::MAX_E; }

int w4_tc_gemm1(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1, const int32_t* offsets,
                const int32_t* tile_start, uint8_t* h_tiles, int32_t* status, cudaStream_t st) {
    w4::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.act = x_tiles; a.w = w1; a.offsets = offsets; a.tile_start = tile_start; a.h_tiles = h_tiles; a.status = status;
    return mxt::nmax_for(d) == 224 ? w4::launch_cfg<1, 224>(a, st) : w4::launch_cfg<1, 112>(a, st);
}

int w4_tc_gemm2(const qmoe_dims* d, const uint8_t* h_tiles, const uint8_t* w2, const int32_t* offsets,
                const int32_t* tile_start, uint16_t* y, int32_t* status, cudaStream_t st) {
    w4::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.act = h_tiles; a.w = w2; a.offsets = offsets; a.tile_start = tile_start; a.y = y; a.status = status;
    return mxt::nmax_for(d) == 224 ? w4::launch_cfg<2, 224>(a, st) : w4::launch_cfg<2, 112>(a, st);
}

}  // namespace qmoe
