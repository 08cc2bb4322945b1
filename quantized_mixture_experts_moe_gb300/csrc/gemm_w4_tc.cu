// Grouped W4A16 expert GEMMs on the 5th-generation tensor cores (tcgen05,
// kind::f16 with fp16 operands, fp32 accumulation in TMEM).
//
// "perf(qmoe): group prefill expert matmuls" (description) batches symmetric
// int4 expert projections into one launch for all experts; "Evaluate native
// IU4/IU8 WMMA for grouped-INT MoE prefill on gfx1151" (Problem, Constraint)
// computes int4 weights with 16-bit activations by dequantising the weights
// and running a 16-bit dot.  This is that computation for sm_103a:
//   stage 1: h = silu(W1_gate . x) * (W1_up . x), rounded to bf16;
//   stage 2: y = W2 . h, accumulated in fp32, stored as bf16.
// The operands are fp16 rather than bf16 (same MMA rate): every weight
// (n - 8) * s * 2^p is one fp16 rounding (relative error <= 2^-11) of the
// exact value, with 2^p a per-row power of two chosen at pre-pack time; every
// activation row is scaled by a power of two 2^-e into [2^14, 2^15), which is
// exact for bf16 values.  The epilogue multiplies the fp32 sums by 2^(e - p).
//
// Structure (one persistent CTA per SM, 16 warps):
//   warp 0      raw weight producer: bulk copies of pre-packed int4 blocks
//               (128 rows x 64 elements of codes + their scales, 4608
//               contiguous bytes) into a raw ring, two per step (stage 1: a
//               gate block and its up partner; stage 2: two adjacent W2 row
//               tiles).
//   warp 1      activation producer: bulk copy of the step's tile rows,
//               already 128-byte swizzled (stage 1: fp16 x tiles; stage 2:
//               bf16 h tiles, converted to fp16 in place by the converters).
//   warps 2-3   MMA issuers, one per weight tile (M = 128 weight rows, N =
//               tokens rounded up to 16, K = 16 per instruction).
//   warps 4-11  converters: one thread per weight row; (n - 8) * s in f16x2
//               arithmetic into the swizzled K-major fp16 tile, then (stage 2)
//               the activation rows in place, then a generic -> async proxy
//               fence before publishing the slot.
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
constexpr int CVT_THREADS = CVT_WARPS * 32;
constexpr int KSTEP = 64;  // K elements per step (128-byte 16-bit rows)
constexpr int MAX_E = 512;
constexpr int EXP_BUFS = 2;  // stage 2: per-unit activation exponents in flight

template <int STAGE, int NMAX_>
struct Cfg {
    static constexpr int NMAX = NMAX_;
    static constexpr int AT = 2;
    static constexpr int ACC_BUFS = (AT * NMAX * 2 <= 512) ? 2 : 1;
    static constexpr int A_BYTES = AT * 128 * 128;  // two 128-row x 128-byte fp16 tiles
    static constexpr int B_BYTES = NMAX * 128;
    static constexpr int RAW_BYTES = AT * bft::kW4Block;
    static constexpr int RS = 3;  // raw ring depth
    static constexpr int SLOT_BYTES = A_BYTES + B_BYTES;
    static constexpr int S = (224 * 1024 - RS * RAW_BYTES - 8 * 1024) / SLOT_BYTES;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = A_OFF + S * A_BYTES;
    static constexpr int RAW_OFF = B_OFF + S * B_BYTES;
    static constexpr int EXP_OFF = RAW_OFF + RS * RAW_BYTES;
    static constexpr int BAR_OFF = EXP_OFF + EXP_BUFS * NMAX * 4;
    static constexpr int NBAR = 2 * RS + 3 * S + 2 * ACC_BUFS + 2 * EXP_BUFS;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int SCHED_OFF = MISC_OFF + 64;
    static constexpr size_t smem_bytes(int E) { return (size_t)SCHED_OFF + (size_t)(E + 1) * 4 + 1024; }
    static constexpr uint32_t ACC_COLS = AT * NMAX;
    static_assert(ACC_BUFS * ACC_COLS <= 512, "TMEM budget");
    static_assert(S >= 2 && NMAX % 16 == 0 && NMAX <= CVT_THREADS, "ring / N tile");
    static_assert(B_OFF % 1024 == 0 && B_BYTES % 1024 == 0, "SW128 tiles start on 1024-byte boundaries");
};
static_assert(Cfg<1, 112>::smem_bytes(MAX_E) <= 232448 && Cfg<1, 224>::smem_bytes(MAX_E) <= 232448 &&
                  Cfg<2, 112>::smem_bytes(MAX_E) <= 232448 && Cfg<2, 224>::smem_bytes(MAX_E) <= 232448,
              "shared memory per CTA");

struct Args {
    int T, k, H, I, E;
    const uint8_t* act;      // stage 1: fp16 x tiles (K = H); stage 2: bf16 h tiles (K = I)
    const float* act_tail;   // stage 1: 2^e per tile row; stage 2: |max| per tile row and 32-column group
    const uint8_t* w;        // pre-packed int4 blocks
    const float* rowfac;     // 2^-p per weight row
    const int32_t* offsets;
    const int32_t* tile_start;
    uint8_t* h_tiles;        // stage 1 output (bf16, K = I)
    float* h_tail;           // stage 1 output: |max| per tile row and 32-column group
    uint16_t* y;             // stage 2 output, bf16 slot order
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
    w = __shfl_sync(0xFFFFFFFFu, w, 0);
    __syncwarp();  // orders the other lanes' shared-memory reads after lane 0's wait
    return w != 0;
}

// Eight int4 codes (one reordered word) times an f16x2 scale -> four f16x2
// pairs in K order.  0x6400 | n is the fp16 value 1024 + n; subtracting 1032
// gives n - 8 exactly; the product is the one rounding.
__device__ __forceinline__ uint4 dequant8(uint32_t w, uint32_t s2) {
    const uint32_t magic = 0x64006400u, bias = 0x64086408u;
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t v = ((w >> (4 * j)) & 0x000F000Fu) | magic;
        asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(v) : "r"(bias));
        asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(v) : "r"(s2));
        p[j] = v;
    }
    return make_uint4(p[0], p[1], p[2], p[3]);
}

// Eight bf16 values -> eight fp16 values times 2^-e (exact for values in range).
__device__ __forceinline__ uint4 bf16x8_to_f16(uint4 v, float m) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(__uint_as_float(u[i] << 16) * m, __uint_as_float(u[i] & 0xFFFF0000u) * m);
        o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int STAGE, int NMAX>
__global__ void __launch_bounds__(THREADS, 1) w4_gemm_kernel(const Args a) {
    using C = Cfg<STAGE, NMAX>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::A_OFF;
    uint8_t* sB = smem + C::B_OFF;
    uint8_t* sRaw = smem + C::RAW_OFF;
    int* sExp = reinterpret_cast<int*>(smem + C::EXP_OFF);
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* raw_empty = raw_full + C::RS;
    uint64_t* full = raw_empty + C::RS;
    uint64_t* empty = full + C::S;
    uint64_t* bfull = empty + C::S;       // stage 2: raw bf16 activation rows landed
    uint64_t* acc_full = bfull + C::S;
    uint64_t* acc_empty = acc_full + C::ACC_BUFS;
    uint64_t* exp_full = acc_empty + C::ACC_BUFS;  // stage 2: a unit's exponents written
    uint64_t* exp_free = exp_full + EXP_BUFS;      // stage 2: ... and no longer read
    uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 8);
    int* tile_start = reinterpret_cast<int*>(smem + C::SCHED_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E;
    const int K = (STAGE == 1) ? a.H : a.I;
    const int NB = (STAGE == 1) ? a.I / 128 : a.H / 256;
    const int KT = K / KSTEP;
    const int NG = a.I / 32;  // 32-column groups of an h row

    for (int i = threadIdx.x; i <= E; i += blockDim.x) tile_start[i] = a.tile_start[i];
    if (threadIdx.x == 32 * WARP_MMA) {
        for (int s = 0; s < C::RS; ++s) {
            tc::mbar_init(&raw_full[s], 1);
            tc::mbar_init(&raw_empty[s], CVT_WARPS);
        }
        for (int s = 0; s < C::S; ++s) {
            // stage 1: the activation producer (with its bytes) + the converters;
            // stage 2: the converters only (the producer's bytes go to bfull)
            tc::mbar_init(&full[s], STAGE == 1 ? 1 + CVT_WARPS : CVT_WARPS);
            tc::mbar_init(&empty[s], 2);  // the two MMA issuers' commits
            tc::mbar_init(&bfull[s], 1);
        }
        for (int b = 0; b < C::ACC_BUFS; ++b) {
            tc::mbar_init(&acc_full[b], 2);
            tc::mbar_init(&acc_empty[b], EPI_WARPS);
        }
        for (int b = 0; b < EXP_BUFS; ++b) {
            tc::mbar_init(&exp_full[b], CVT_WARPS);
            tc::mbar_init(&exp_free[b], EPI_WARPS);
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
            const int64_t second = (STAGE == 1) ? (int64_t)(a.I / 128) * KT : KT;  // block distance to tile 2
            for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x) {
                int e, m0, ntok, nb, t;
                decode_unit<NMAX>(u, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t);
                const int64_t rt0 = (STAGE == 1) ? (int64_t)e * (2 * a.I / 128) + nb : (int64_t)e * (a.H / 128) + 2 * nb;
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(&raw_empty[rs], phase ^ 1)) { set_abort(abort_flag, a.status); ok = false; break; }
                    tc::mbar_arrive_expect_tx(&raw_full[rs], C::RAW_BYTES);
                    const int64_t b0 = rt0 * KT + kt;
                    uint8_t* d = sRaw + rs * C::RAW_BYTES;
                    tc::bulk_load(d, a.w + b0 * bft::kW4Block, bft::kW4Block, &raw_full[rs]);
                    tc::bulk_load(d + bft::kW4Block, a.w + (b0 + second) * bft::kW4Block, bft::kW4Block,
                                  &raw_full[rs]);
                    if (++rs == C::RS) { rs = 0; phase ^= 1; }
                }
                if (!ok) break;
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
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(&empty[slot], phase ^ 1)) { set_abort(abort_flag, a.status); ok = false; break; }
                    uint64_t* bar = (STAGE == 1) ? &full[slot] : &bfull[slot];
                    tc::mbar_arrive_expect_tx(bar, bytes);
                    tc::bulk_load(sB + slot * C::B_BYTES, a.act + ((int64_t)t * KT + kt) * bb, bytes, bar);
                    if (++slot == C::S) { slot = 0; phase ^= 1; }
                }
                if (!ok) break;
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
                const uint32_t idesc = tc::idesc_f16_f32(128, nmma);
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
        // ------------------------------------------------ converters
        const int ct = (warp - WARP_CVT0) * 32 + lane;  // 0..255
        const int tile = ct >> 7, row = ct & 127;
        int rs = 0, slot = 0, ui = 0;
        uint32_t rphase = 0, phase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok && !*abort_flag; u += gridDim.x, ++ui) {
            int e, m0, ntok, nb, t;
            decode_unit<NMAX>(u, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t);
            const int eb = ui & (EXP_BUFS - 1);
            const uint32_t ephase = (uint32_t)(ui / EXP_BUFS) & 1u;
            int* uexp = sExp + eb * NMAX;
            if (STAGE == 2) {
                // this unit's per-row exponents, from the h rows' group maxima
                if (!warp_wait(&exp_free[eb], ephase ^ 1, lane)) {
                    if (lane == 0) set_abort(abort_flag, a.status);
                    ok = false;
                    break;
                }
                if (ct < NMAX) {
                    float amax = 0.f;
                    if (ct < ntok) {
                        const float* tr = a.act_tail + ((int64_t)t * NMAX + ct) * NG;
                        for (int g = 0; g < NG; ++g) amax = fmaxf(amax, tr[g]);
                    }
                    uexp[ct] = f16_row_exponent(amax);
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&exp_full[eb]);
                if (!warp_wait(&exp_full[eb], ephase, lane)) {
                    if (lane == 0) set_abort(abort_flag, a.status);
                    ok = false;
                    break;
                }
            }
            const int nchunks = ((ntok + 15) & ~15) * 8;  // 16-byte activation chunks per step
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
                const uint32_t s2a = (sc & 0xFFFFu) * 0x10001u, s2b = (sc >> 16) * 0x10001u;
                const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                uint8_t* dst = sA + slot * C::A_BYTES + tile * 128 * 128 + row * 128;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8)
                    *reinterpret_cast<uint4*>(dst + ((w8 ^ (row & 7)) << 4)) = dequant8(wv[w8], w8 < 4 ? s2a : s2b);
                if (STAGE == 2) {
                    // bf16 h rows -> fp16 in place (elementwise, so the swizzle does not matter)
                    if (!warp_wait(&bfull[slot], phase, lane)) {
                        if (lane == 0) set_abort(abort_flag, a.status);
                        ok = false;
                        break;
                    }
                    uint8_t* bs = sB + slot * C::B_BYTES;
                    for (int i = ct; i < nchunks; i += CVT_THREADS) {
                        uint4* p = reinterpret_cast<uint4*>(bs + i * 16);
                        *p = bf16x8_to_f16(*p, exp2i(-uexp[i >> 3]));
                    }
                }
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
        const int nl = q * 32 + lane;  // weight row within the tile = output column within the 128-column block
        int ab = 0, ui = 0;
        uint32_t pacc = 0;
        for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x, ++ui) {
            int e, m0, ntok, nb, t;
            decode_unit<NMAX>(u, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t);
            const int eb = ui & (EXP_BUFS - 1);
            const uint32_t ephase = (uint32_t)(ui / EXP_BUFS) & 1u;
            int w = 1;
            if (lane == 0) {
                w = tc::mbar_wait_sleep(&acc_full[ab], pacc) ? 1 : 0;
                if (w && STAGE == 2) w = tc::mbar_wait(&exp_full[eb], ephase) ? 1 : 0;
            }
            w = __shfl_sync(0xFFFFFFFFu, w, 0);
            __syncwarp();
            if (!w) {
                if (lane == 0) set_abort(abort_flag, a.status);
                break;
            }
            tc::tc_fence_after();
            const uint32_t dcol = ab * C::ACC_COLS;
            float f0, f1;  // 2^-p of the two weight rows this thread's TMEM lane holds
            if (STAGE == 1) {
                const int64_t rt0 = (int64_t)e * (2 * a.I / 128) + nb;
                f0 = a.rowfac[rt0 * 128 + nl];
                f1 = a.rowfac[(rt0 + a.I / 128) * 128 + nl];
            } else {
                const int64_t rt0 = (int64_t)e * (a.H / 128) + 2 * nb;
                f0 = a.rowfac[rt0 * 128 + nl];
                f1 = a.rowfac[(rt0 + 1) * 128 + nl];
            }
            uint8_t* hblk = nullptr;
            if (STAGE == 1)
                hblk = a.h_tiles + ((int64_t)t * (a.I / KSTEP) + nb * 2 + (nl >> 6)) * bft::block_bytes(NMAX);
            const int* uexp = sExp + eb * NMAX;
            // 16 tokens per chunk, computed independently (no per-token branch, so the
            // chains overlap), then stored under the uniform predicate c < ntok
            for (int c0 = 0; c0 < ntok; c0 += 16) {
                uint32_t g[16], g2[16];
                tc::tmem_ld_32x32b_x16(tm + lane_addr + dcol + c0, g);
                tc::tmem_ld_32x32b_x16(tm + lane_addr + dcol + NMAX + c0, g2);
                // the chunk's 16 per-token factors 2^e, one per lane, broadcast below
                float fl = 0.f;
                if (lane < 16 && c0 + lane < ntok)
                    fl = (STAGE == 1) ? a.act_tail[(int64_t)t * NMAX + c0 + lane] : exp2i(uexp[c0 + lane]);
                tc::tmem_ld_wait();
                const int nv = min(16, ntok - c0);
                if (STAGE == 1) {
                    uint32_t hb[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float fx = __shfl_sync(0xFFFFFFFFu, fl, j);
                        const float gv = __uint_as_float(g[j]) * (fx * f0);
                        const float uv = __uint_as_float(g2[j]) * (fx * f1);
                        hb[j] = float_to_bf16_bits(__fdividef(gv, 1.0f + __expf(-gv)) * uv);
                    }
                    float tmax = 0.f;  // lane j < nv: |max| over this warp's 32 columns of token c0 + j
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (j < nv) *reinterpret_cast<uint16_t*>(hblk + bft::elem_offset(c0 + j, nl & 63)) = (uint16_t)hb[j];
                        const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, (hb[j] & 0x7FFFu) << 16);
                        if (lane == j) tmax = __uint_as_float(mx);
                    }
                    if (lane < nv) a.h_tail[((int64_t)t * NMAX + c0 + lane) * NG + nb * 4 + q] = tmax;
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float fx = __shfl_sync(0xFFFFFFFFu, fl, j);
                        const uint16_t v0 = float_to_bf16_bits(__uint_as_float(g[j]) * (fx * f0));
                        const uint16_t v1 = float_to_bf16_bits(__uint_as_float(g2[j]) * (fx * f1));
                        if (j < nv) {
                            uint16_t* yr = a.y + (int64_t)(m0 + c0 + j) * a.H + 2 * nb * 128 + nl;
                            yr[0] = v0;
                            yr[128] = v1;
                        }
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&acc_empty[ab]);
                if (STAGE == 2) tc::mbar_arrive(&exp_free[eb]);
            }
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
    a.act = x_tiles;
    a.act_tail = reinterpret_cast<const float*>(x_tiles + bft::blocks_bytes(d, d->H));
    a.w = w1;
    a.rowfac = reinterpret_cast<const float*>(w1 + bft::w4_blocks_bytes((int64_t)d->E * 2 * d->I, d->H));
    a.offsets = offsets; a.tile_start = tile_start;
    a.h_tiles = h_tiles;
    a.h_tail = reinterpret_cast<float*>(h_tiles + bft::blocks_bytes(d, d->I));
    a.status = status;
    return mxt::nmax_for(d) == 224 ? w4::launch_cfg<1, 224>(a, st) : w4::launch_cfg<1, 112>(a, st);
}

int w4_tc_gemm2(const qmoe_dims* d, const uint8_t* h_tiles, const uint8_t* w2, const int32_t* offsets,
                const int32_t* tile_start, uint16_t* y, int32_t* status, cudaStream_t st) {
    w4::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.act = h_tiles;
    a.act_tail = reinterpret_cast<const float*>(h_tiles + bft::blocks_bytes(d, d->I));
    a.w = w2;
    a.rowfac = reinterpret_cast<const float*>(w2 + bft::w4_blocks_bytes((int64_t)d->E * d->H, d->I));
    a.offsets = offsets; a.tile_start = tile_start; a.y = y; a.status = status;
    return mxt::nmax_for(d) == 224 ? w4::launch_cfg<2, 224>(a, st) : w4::launch_cfg<2, 112>(a, st);
}

}  // namespace qmoe
