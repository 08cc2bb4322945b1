// Grouped integer-weight expert GEMMs on the 5th-generation tensor cores:
// W8A8 and W4A8 with exact int32 sums, and W4A16 (int4 codes with per-32
// fp16 scales, dequantised on chip, fp16 activations).
//
// "Evaluate native IU4/IU8 WMMA for grouped-INT MoE prefill on gfx1151"
// (Constraint) runs W8A8 as int8 x int8 products summed in int32; "perf(qmoe):
// group prefill expert matmuls" (description) puts every expert in one launch.
// sm_103a has no integer tcgen05 MMA in this toolkit, so the products run as
// kind::f16 MMAs on fp16 operands that hold the int8 values exactly (every
// integer in [-128, 127] is an fp16), with fp32 accumulation in TMEM.  A
// product is at most 128 * 127 in magnitude, and a fp32 sum stays an exact
// integer while it is below 2^24.  The accumulator is therefore drained
// before that bound can be reached: the tile kernel records, per 128-element
// K step, the largest sum |x| over a sub-tile's rows, and the GEMM closes a
// chunk of steps whenever 128 * (the chunk's summed maxima) could pass
// 2^24 - 4096 (at most every 1024 K elements, usually far less often).  The
// epilogue splits the exact fp32 value v into hi * 2^13 + lo with |lo| <=
// 4096, adds hi to a 16-bit running sum kept in shared memory and writes lo
// back as the fp32 accumulator, on which the next chunk accumulates.  At the
// end acc = hi * 2^13 + v, the exact int32 sum, for K <= 16384
// (|hi| <= 16384 * 128 * 127 / 2^13 < 2^15).
//
//   stage 1: g = ((float)acc_g * s_x) * s_w,  u likewise,  h = silu(g) * u  (fp32)
//   stage 2: y = ((float)acc * s_h) * s_w                                 (bf16)
//
// W4A8 uses the W8A8 path with int4 codes (|q| <= 7) in place of int8: its
// partial sums stay below 2^24 for K <= 16384, so it needs no drains.  W4A16
// dequantises (n - 8) * s on chip, one fp16 rounding per weight, and sums in
// fp32 like any float GEMM.
//
// Structure (one persistent CTA per SM, 20 warps), swap-AB as in the other
// grouped GEMMs (weights are the MMA's M = 128 rows, tokens its N):
//   warp 0      weight producer: per step the raw weights of both weight
//               tiles (stage 1: a gate tile and its up partner; stage 2: two
//               adjacent W2 row tiles): W8A8 two TMA boxes of int8 rows (64
//               K elements each), W4A8 one TMA box of packed int4 rows, W4A16
//               bulk copies of pre-packed blocks; 64-byte swizzled by TMA.
//   warp 1      activation producer: bulk copies per step of the step's fp16
//               token rows, already 128-byte swizzled by the tile kernel.
//   warps 2-3   MMA issuers, one per weight tile: A (the weight tile) from
//               TMEM, B (tokens) from shared memory, N = tokens rounded to 16.
//   warps 4-11  converters: one thread per weight row; int8 / int4 / int4 x
//               scale -> fp16 pairs written straight into TMEM as the A
//               operand, so the converted weights never pass through shared
//               memory.
//   warps 12-19 epilogue: two per TMEM lane quadrant, alternate 16-token
//               column chunks; the drains (W8A8) and the final dequantisation.
#include "qmoe_common.cuh"
#include "mx_tiles.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

#include <cstring>

namespace qmoe {
namespace ig {

constexpr int WARP_W = 0, WARP_B = 1, WARP_MMA = 2;
constexpr int WARP_CVT0 = 4, CVT_WARPS = 8;
constexpr int WARP_EPI0 = 12, EPI_WARPS = 8;
constexpr int THREADS = (WARP_EPI0 + EPI_WARPS) * 32;
// Drains keep every fp32 partial sum below 2^24: a chunk of steps may add at
// most L1_BOUND * 128 (|w| <= 128 for int8 weights, sum |x| over the chunk's
// steps <= L1_BOUND for every row) on top of a remainder |lo| <= 4096.
constexpr int L1_BOUND = ((1 << 24) - 4097) / 128;
constexpr int HI_SHIFT = 13;
constexpr int MAX_E = 512;
constexpr int MAX_K = 16384;

// Per weight format:
//   W8 (int8, exact int32 sums): tokens per MMA NS = 112 (a 224-row schedule
//      tile is two of them), 128-element steps, raw int8 rows by TMA;
//   I4 (int4 codes with per-channel scales, int8 activations, exact int32
//      sums): W8 in everything but the weights, which arrive as packed int4
//      rows by TMA (one 64-byte row per 128-element step) and are widened to
//      exact fp16 integers by the converters.  |code| <= 7 keeps every partial
//      sum of a K <= 16384 dot below 2^24, so no drains are needed;
//   W4 (int4 + fp16 scales):     NS = 160 (a 224-row tile is 160 + 64, so an
//      expert with up to 160 pairs is one unit), 64-element steps in a
//      three-slot A ring (the wider accumulators leave 192 TMEM columns),
//      raw pre-packed blocks by bulk copy.
// TMEM columns: the fp32 accumulators of the two tiles (2 * NS), then the A
// ring.  Shared memory: raw ring, activation ring, and NS x 128 words staging
// the drains' high parts (W8) and the final outputs.
enum { FMT_W8 = 0, FMT_W4 = 1, FMT_I4 = 2 };

template <int FMT>
struct Cfg {
    static constexpr bool W4 = (FMT == FMT_W4);
    static constexpr bool I4 = (FMT == FMT_I4);
    static constexpr int NS = W4 ? 160 : 112;
    static constexpr int AS = W4 ? 3 : 2;         // A slots in TMEM
    static constexpr int BS = AS + 1;             // activation slots
    static constexpr int KSTEP = W4 ? 64 : 128;  // K elements per step
    static constexpr int HPS = KSTEP / 64;        // 64-element halves per step
    static constexpr int A_SLOT_COLS = KSTEP;     // two tiles x KSTEP/2 fp16 pairs
    static constexpr int HALF_RAW = W4 ? 2 * bft::kW4Block : 2 * 128 * 64;  // one 64-element half, both tiles
    static constexpr int RAW_BYTES = I4 ? HALF_RAW : HPS * HALF_RAW;  // I4: a whole step in one 64-byte row
    static constexpr int RS = (W4 || I4) ? 4 : 2;  // raw weight slots
    static constexpr int HALF_B = NS * 128;  // one 64-element half of the step's fp16 token rows
    static constexpr int B_BYTES = HPS * HALF_B;
    static constexpr int CHUNKS = NS / 16;   // 16-token column chunks of an accumulator
    static constexpr int EPI_CHUNKS = (CHUNKS + 1) / 2;  // per epilogue warp (the warp pair alternates)
    static constexpr uint32_t R_COL = 0;
    static constexpr uint32_t A_COL = 2 * NS;
    static constexpr int RAW_OFF = 0;
    static constexpr int B_OFF = (RAW_OFF + RS * RAW_BYTES + 1023) / 1024 * 1024;
    static constexpr int S_OFF = B_OFF + BS * B_BYTES;
    static constexpr int S_BYTES = NS * 128 * 4;
    static constexpr int BAR_OFF = S_OFF + S_BYTES;
    static constexpr int NBAR = 2 * RS + 2 * BS + AS + 2;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int SCHED_OFF = MISC_OFF + 64;
    static constexpr size_t smem_bytes(int E) { return (size_t)SCHED_OFF + 2 * (size_t)(E + 1) * 4 + 1024; }
    static_assert(R_COL + 2 * NS <= A_COL && A_COL + AS * A_SLOT_COLS <= 512 && NS % 16 == 0, "TMEM budget");
    static_assert(BS >= AS + 1, "a step's done barrier is not reused before the converter has waited on it");
    static_assert(B_OFF % 1024 == 0 && HALF_B % 1024 == 0, "swizzled activation tiles 1024-aligned");
    static_assert(W4 || HALF_RAW % 1024 == 0, "swizzled raw int8 / int4 tiles 1024-aligned");
    static_assert(smem_bytes(MAX_E) <= 232448, "shared memory per CTA");
};

struct Args {
    int T, k, H, I, E;
    int nmax;                 // schedule tile (16, 112 or 224 tokens)
    const uint8_t* act;       // fp16 token tiles (K = H for stage 1, I for stage 2)
    const float* act_scale;   // per tile row: s_x / s_h (W8) or the power of two 2^e (W4)
    const uint8_t* wq;        // W4: pre-packed int4 blocks (W8 weights come through the tensor map)
    const float* w_scale;     // per weight row: channel scale (W8) or 2^-p (W4)
    float* h_tail;            // W4 stage 1: |max| per tile row and 32-column group of h
    const int32_t* offsets;
    const int32_t* tile_start;
    float* h;                 // W8 stage 1 output, fp32 [P, I] in slot order
    uint8_t* h_tiles;         // W4 stage 1 output, bf16 tiles (K = I)
    uint16_t* y;              // stage 2 output, bf16 [P, H] in slot order
    const int32_t* l1max;     // per (sub-tile, step): the largest sum |x| over the sub-tile's rows
    int32_t* dbg_acc;         // optional exact sums: [P, 2I] (stage 1) or [P, H] (stage 2)
    int32_t* status;
    int weights_early;        // weight producer and converters may run before the predecessor kernel completes
};

// Unit u -> (expert e, schedule tile t, half of it, column block nb) and the
// unit's first slot m0 and token count (always > 0).  Units enumerate only
// the non-empty token halves: sub_start is the prefix over experts of their
// sub-unit counts (full tiles x halves, plus the halves the last tile fills),
// and an expert's sub-units j run over (tile j / halves, half j % halves).  So
// a static round-robin over units hands every CTA the same number of real
// units; with the empty halves in the enumeration some CTAs drew one or two
// more than others.
template <int NS>
__device__ __forceinline__ void decode_unit(int u, int NB, int halves, int nmax, const int* tile_start,
                                            const int* sub_start, int E, const int32_t* offsets, int& e, int& t,
                                            int& half, int& nb, int& m0, int& ntok, bool l2) {
    const int th = u / NB;
    nb = u - th * NB;
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sub_start[mid] <= th) lo = mid; else hi = mid;
    }
    e = lo;
    const int j = th - sub_start[e];
    const int jt = j / halves;
    half = j - jt * halves;
    t = tile_start[e] + jt;
    // l2: a role that runs before this kernel's dependent-launch wait reads
    // the routing sort's offsets from L2 (the sort completed before the launch)
    const int o0 = l2 ? __ldcg(offsets + e) : offsets[e];
    const int o1 = l2 ? __ldcg(offsets + e + 1) : offsets[e + 1];
    m0 = o0 + jt * nmax + half * NS;
    ntok = min(min(NS, nmax - half * NS), o1 - m0);
}

// sub_start[0..E]: prefix over experts of ceil-split sub-units (one warp; the
// offsets are complete: read through L2 as the schedule is).
template <int NS>
__device__ __forceinline__ void build_sub_start(const int32_t* offsets, int E, int nmax, int halves, int* sub_start,
                                                int lane) {
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        int c = 0;
        if (e < E) {
            const int cnt = __ldcg(offsets + e + 1) - __ldcg(offsets + e);
            const int full = cnt / nmax, rem = cnt - full * nmax;
            c = full * halves + (rem + NS - 1) / NS;
        }
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, c, s);
            if (lane >= s) c += v;
        }
        if (e < E) sub_start[e + 1] = carry + c;
        carry += __shfl_sync(0xFFFFFFFFu, c, 31);
    }
    if (lane == 0) sub_start[0] = 0;
}

__device__ __forceinline__ void set_abort(volatile int* flag, int32_t* status) {
    *flag = 1;
    atomicOr(status, QMOE_DEV_WAIT_TIMEOUT);
}

// The abort flag as one value for the whole warp (lane 0's read).
__device__ __forceinline__ bool warp_flag(volatile int* flag) {
    return __shfl_sync(0xFFFFFFFFu, *flag, 0) != 0;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane) {
    int w = 1;
    if (lane == 0) w = tc::mbar_wait(bar, parity) ? 1 : 0;
    w = __shfl_sync(0xFFFFFFFFu, w, 0);
    __syncwarp();
    return w != 0;
}

// Four int8 values (one word) -> two fp16 pairs holding them exactly:
// 0x6400 | (b ^ 0x80) is the fp16 1152 + b; subtracting 1152 leaves b.
__device__ __forceinline__ void i8x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = w ^ 0x80808080u;
    lo = __byte_perm(x, 0x64u, 0x4140);
    hi = __byte_perm(x, 0x64u, 0x4342);
    const uint32_t bias = 0x64806480u;
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(bias));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(bias));
}

// Eight int4 codes (one reordered word: pair j = nibbles j and j + 4) times
// an f16x2 scale -> four f16x2 pairs in K order, with one shift per word.
// Masking nibbles 0/4 (or, after the shift by 8, 2/6) into 0x6400 gives the
// fp16 values 1024 + n, from which subtracting 1032 leaves n - 8; masking
// nibbles 1/5 (3/7) in place gives 1024 + 16 n, and (1024 + 16 n) / 16 - 72
// is n - 8 in one exact fma.  The product with the scale is the one rounding.
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t s2, uint32_t* out) {
    const uint32_t magic = 0x64006400u, bias = 0x64086408u;
    const uint32_t sixteenth = 0x2C002C00u, m72 = 0xD480D480u;  // 1/16, -72
    const uint32_t w8 = w >> 8;
    uint32_t v[4] = {(w & 0x000F000Fu) | magic, (w & 0x00F000F0u) | magic, (w8 & 0x000F000Fu) | magic,
                     (w8 & 0x00F000F0u) | magic};
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(v[0]) : "r"(bias));
    asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(v[1]) : "r"(sixteenth), "r"(m72));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(v[2]) : "r"(bias));
    asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(v[3]) : "r"(sixteenth), "r"(m72));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(v[j]) : "r"(s2));
        out[j] = v[j];
    }
}

// Eight int4 codes (byte i: codes 2i, 2i+1 in its low, high nibble; stored
// n = q + 8) -> four fp16 pairs holding q exactly: the nibbles are spread
// into the low bytes of fp16 1024 + n (0x64nn) with byte permutes, then 1032
// is subtracted.
__device__ __forceinline__ void i4x8_to_f16x2(uint32_t w, uint32_t* out) {
    const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
    const uint32_t n03 = __byte_perm(lo, hi, 0x5140), n47 = __byte_perm(lo, hi, 0x7362);
    const uint32_t magic = 0x64646464u, bias = 0x64086408u;
    uint32_t v[4] = {__byte_perm(n03, magic, 0x4140), __byte_perm(n03, magic, 0x4342), __byte_perm(n47, magic, 0x4140),
                     __byte_perm(n47, magic, 0x4342)};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(v[j]) : "r"(bias));
        out[j] = v[j];
    }
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) { tc::tmem_ld_32x32b_x16(taddr, r); }
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) { tc::tmem_st_32x32b_x16(taddr, r); }

// Exact fp32 integer v -> (hi, lo) with v = hi * 2^13 + lo, lo in [-4096, 4095].
__device__ __forceinline__ void split_hi_lo(uint32_t vbits, int& hi, int& lo) {
    const int v = __float2int_rn(__uint_as_float(vbits));
    hi = (v + (1 << (HI_SHIFT - 1))) >> HI_SHIFT;
    lo = v - hi * (1 << HI_SHIFT);
}

// A unit's chunk starts (warp-uniform; every lane of the warp calls it): bit
// kt set when a new chunk, and so a drain before it, starts at step kt > 0.
// Chunks are grown greedily while the sum of the per-step L1 maxima stays
// within L1_BOUND, which bounds every partial sum of every row of the unit.
__device__ __forceinline__ void chunk_starts(const int32_t* l1, int KT, int lane, uint32_t (&starts)[4]) {
    int run = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        starts[i] = 0;
        const int v = (32 * i + lane < KT) ? l1[32 * i + lane] : 0;
        for (int k2 = 0; k2 < 32 && 32 * i + k2 < KT; ++k2) {
            const int m = __shfl_sync(0xFFFFFFFFu, v, k2);
            if (run > 0 && run + m > L1_BOUND) {
                starts[i] |= 1u << k2;
                run = 0;
            }
            run += m;
        }
    }
}

__device__ __forceinline__ bool bit_at(const uint32_t (&b)[4], int kt) {
    const uint32_t w = (kt < 32) ? b[0] : (kt < 64) ? b[1] : (kt < 96) ? b[2] : b[3];
    return kt < 128 && ((w >> (kt & 31)) & 1u);
}

template <int STAGE, int FMT>
__global__ void __launch_bounds__(THREADS, 1) int_gemm_kernel(const __grid_constant__ CUtensorMap wmap, const Args a) {
    using C = Cfg<FMT>;
    constexpr bool W4 = C::W4, I4 = C::I4;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sRaw = smem + C::RAW_OFF;
    uint8_t* sB = smem + C::B_OFF;
    uint32_t* sS = reinterpret_cast<uint32_t*>(smem + C::S_OFF);  // [token][row] packed high parts
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* raw_empty = raw_full + C::RS;
    uint64_t* b_full = raw_empty + C::RS;
    uint64_t* done = b_full + C::BS;  // step g completed (both issuers' MMAs): frees B slot g % C::BS and A slot g % C::AS
    uint64_t* a_full = done + C::BS;
    uint64_t* acc_full = a_full + C::AS;
    uint64_t* acc_empty = acc_full + 1;
    uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 8);
    int* tile_start = reinterpret_cast<int*>(smem + C::SCHED_OFF);
    int* sub_start = tile_start + (a.E + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E;
    const int K = (STAGE == 1) ? a.H : a.I;
    const int NB = (STAGE == 1) ? a.I / 128 : a.H / 256;
    const int KT = K / C::KSTEP;
    const int halves = (a.nmax + C::NS - 1) / C::NS;

    // Dependent launch: by default everything waits for the predecessor
    // kernel.  With weights_early (set by the whole-layer call, whose routing
    // sort ran two launches back) the weight producer and the converters,
    // which read only the schedule and the weights, start before that; the
    // warps that read the predecessor's output wait.
    if (!a.weights_early) pdl_wait();
    for (int i = threadIdx.x; i <= E; i += blockDim.x) tile_start[i] = __ldcg(a.tile_start + i);
    if (warp == WARP_CVT0) build_sub_start<C::NS>(a.offsets, E, a.nmax, halves, sub_start, lane);
    if (threadIdx.x == 32 * WARP_MMA) {
        for (int s = 0; s < C::RS; ++s) {
            tc::mbar_init(&raw_full[s], 1);
            tc::mbar_init(&raw_empty[s], CVT_WARPS);
        }
        for (int s = 0; s < C::BS; ++s) {
            tc::mbar_init(&b_full[s], 1);
            tc::mbar_init(&done[s], 2);  // the two issuers' commits
        }
        for (int s = 0; s < C::AS; ++s) tc::mbar_init(&a_full[s], CVT_WARPS);
        tc::mbar_init(acc_full, 2);
        tc::mbar_init(acc_empty, EPI_WARPS);
        *abort_flag = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    const int total_units = sub_start[E] * NB;
    if ((int)blockIdx.x >= total_units) {
        pdl_wait();  // the grid still completes only after its predecessor
        return;
    }

    if (warp == WARP_MMA) {
        tc::tmem_alloc(tmem_base_smem, 512);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tm = *tmem_base_smem;

    if (warp == WARP_W) {
        // ------------------------------------------------ weight producer
        if (lane == 0) {
            tc::prefetch_tensormap(&wmap);
            int rs = 0;
            uint32_t ph = 0;
            for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x) {
                int e, t, half, nb, m0, ntok;
                decode_unit<C::NS>(u, NB, halves, a.nmax, tile_start, sub_start, E, a.offsets, e, t, half, nb, m0, ntok, a.weights_early != 0);
                if (ntok <= 0) continue;
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(&raw_empty[rs], ph ^ 1)) { set_abort(abort_flag, a.status); ok = false; break; }
                    tc::mbar_arrive_expect_tx(&raw_full[rs], C::RAW_BYTES);
                    uint8_t* dst = sRaw + rs * C::RAW_BYTES;
                    if constexpr (W4) {
                        // pre-packed blocks (row tile, 64-element K block): [half hh][tile i]
                        const int KB = K / 64;
                        const int64_t rt0 = (STAGE == 1) ? (int64_t)e * (2 * a.I / 128) + nb : (int64_t)e * (a.H / 128) + 2 * nb;
                        const int64_t rt1 = (STAGE == 1) ? rt0 + a.I / 128 : rt0 + 1;
#pragma unroll
                        for (int hh = 0; hh < C::HPS; ++hh) {
                            tc::bulk_load(dst + (2 * hh) * bft::kW4Block,
                                          a.wq + (rt0 * KB + C::HPS * kt + hh) * bft::kW4Block, bft::kW4Block,
                                          &raw_full[rs]);
                            tc::bulk_load(dst + (2 * hh + 1) * bft::kW4Block,
                                          a.wq + (rt1 * KB + C::HPS * kt + hh) * bft::kW4Block, bft::kW4Block,
                                          &raw_full[rs]);
                        }
                    } else if constexpr (I4) {
                        // packed int4 rows: the step's 128 elements are 64 bytes
                        if (STAGE == 1)
                            tc::tma_load_3d(dst, &wmap, &raw_full[rs], kt * 64, nb * 128, 2 * e);
                        else
                            tc::tma_load_2d(dst, &wmap, &raw_full[rs], kt * 64, e * a.H + nb * 256);
                    } else {
#pragma unroll
                        for (int hh = 0; hh < C::HPS; ++hh) {
                            if (STAGE == 1)
                                tc::tma_load_3d(dst + hh * C::HALF_RAW, &wmap, &raw_full[rs], kt * C::KSTEP + 64 * hh,
                                                nb * 128, 2 * e);
                            else
                                tc::tma_load_2d(dst + hh * C::HALF_RAW, &wmap, &raw_full[rs], kt * C::KSTEP + 64 * hh,
                                                e * a.H + nb * 256);
                        }
                    }
                    if (++rs == C::RS) { rs = 0; ph ^= 1; }
                }
                if (!ok) break;
            }
            // every load issued: the next kernel may launch (after this CTA's own wait)
            pdl_wait();
            pdl_trigger();
        }
    } else if (warp == WARP_B) {
        // ------------------------------------------------ activation producer
        if (a.weights_early) pdl_wait();
        if (lane == 0) {
            int bs = 0;
            uint32_t ph = 0;
            const int64_t bb = (int64_t)a.nmax * 128;
            for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x) {
                int e, t, half, nb, m0, ntok;
                decode_unit<C::NS>(u, NB, halves, a.nmax, tile_start, sub_start, E, a.offsets, e, t, half, nb, m0, ntok, false);
                if (ntok <= 0) continue;
                const uint32_t bytes = (uint32_t)((ntok + 15) & ~15) * 128u;
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(&done[bs], ph ^ 1)) { set_abort(abort_flag, a.status); ok = false; break; }
                    tc::mbar_arrive_expect_tx(&b_full[bs], C::HPS * bytes);
#pragma unroll
                    for (int hh = 0; hh < C::HPS; ++hh)
                        tc::bulk_load(sB + bs * C::B_BYTES + hh * C::HALF_B,
                                      a.act + ((int64_t)t * (K / 64) + C::HPS * kt + hh) * bb + (int64_t)half * C::NS * 128, bytes,
                                      &b_full[bs]);
                    if (++bs == C::BS) { bs = 0; ph ^= 1; }
                }
                if (!ok) break;
            }
        }
    } else if (warp == WARP_MMA || warp == WARP_MMA + 1) {
        // ------------------------------------------------ MMA issuers (warp-uniform; one elected lane issues)
        if (a.weights_early) pdl_wait();
        const int iss = warp - WARP_MMA;
        int bs = 0, as = 0;
        uint32_t bph = 0, aph = 0, ev = 0;
        bool pending = false;  // an accumulator event not yet handed back by the epilogue
        for (int u = blockIdx.x; u < total_units && !warp_flag(abort_flag); u += gridDim.x) {
            int e, t, half, nb, m0, ntok;
            decode_unit<C::NS>(u, NB, halves, a.nmax, tile_start, sub_start, E, a.offsets, e, t, half, nb, m0, ntok, false);
            if (ntok <= 0) continue;
            const int nmma = (ntok + 15) & ~15;
            const uint32_t idesc = tc::idesc_f16_f32(128, nmma);
            const uint32_t dcol = tm + C::R_COL + (uint32_t)(iss * C::NS);
            uint32_t starts[4] = {0u, 0u, 0u, 0u};
            if constexpr (FMT == FMT_W8) chunk_starts(a.l1max + (int64_t)(t * halves + half) * KT, KT, lane, starts);
            bool ok = true;
            for (int kt = 0; kt < KT; ++kt) {
                if (pending) {
                    if (!warp_wait(acc_empty, (ev - 1) & 1, lane)) { ok = false; break; }
                    pending = false;
                }
                if (!warp_wait(&b_full[bs], bph, lane) || !warp_wait(&a_full[as], aph, lane)) { ok = false; break; }
                tc::tc_fence_after();
                const uint32_t b0 = tc::smem_u32(sB + bs * C::B_BYTES);
                const uint32_t a0 = tm + C::A_COL + (uint32_t)(as * C::A_SLOT_COLS + iss * (C::KSTEP / 2));
#pragma unroll
                for (int kk = 0; kk < C::KSTEP / 16; ++kk)
                    tc::mma_f16_ts_elect(dcol, a0 + 8 * kk,
                                         tc::sdesc_kmajor_sw128(b0 + (kk >> 2) * C::HALF_B + 32 * (kk & 3)), idesc,
                                         (kt > 0 || kk > 0) ? 1u : 0u);
                tc::mma_commit_elect(&done[bs]);
                if (++bs == C::BS) { bs = 0; bph ^= 1; }
                if (++as == C::AS) { as = 0; aph ^= 1; }
                if (kt == KT - 1 || bit_at(starts, kt + 1)) {
                    tc::mma_commit_elect(acc_full);
                    ++ev;
                    pending = true;
                }
            }
            if (!ok) {
                if (lane == 0) set_abort(abort_flag, a.status);
                break;
            }
        }
        __syncwarp();
    } else if (warp < WARP_EPI0) {
        // ------------------------------------------------ converters (int8 -> fp16 into TMEM)
        const int tile = (warp - WARP_CVT0) >> 2, q = warp & 3;
        const int m = q * 32 + lane;  // weight row within the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int sw = (m >> 1) & 3;  // 64-byte swizzle of the TMA box: 16-byte chunk j at j ^ sw
        int rs = 0;
        uint32_t rph = 0;
        uint32_t gs = 0;  // steps converted so far (all units): A slot gs % C::AS, done barrier gs % C::BS
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok && !*abort_flag; u += gridDim.x) {
            int e, t, half, nb, m0, ntok;
            decode_unit<C::NS>(u, NB, halves, a.nmax, tile_start, sub_start, E, a.offsets, e, t, half, nb, m0, ntok, a.weights_early != 0);
            if (ntok <= 0) continue;
            for (int kt = 0; kt < KT; ++kt, ++gs) {
                if (!warp_wait(&raw_full[rs], rph, lane)) {
                    if (lane == 0) set_abort(abort_flag, a.status);
                    ok = false;
                    break;
                }
                // KSTEP weights of this row -> KSTEP/2 fp16 pairs, 16 per TMEM store
                uint32_t o[2 * C::HPS][16];
                if constexpr (W4) {
                    uint4 cw[C::HPS][2];
                    uint32_t sc[C::HPS];
#pragma unroll
                    for (int hh = 0; hh < C::HPS; ++hh) {
                        const uint8_t* src = sRaw + rs * C::RAW_BYTES + (2 * hh + tile) * bft::kW4Block;
                        cw[hh][0] = *reinterpret_cast<const uint4*>(src + m * 32);
                        cw[hh][1] = *reinterpret_cast<const uint4*>(src + m * 32 + 16);
                        sc[hh] = *reinterpret_cast<const uint32_t*>(src + 4096 + m * 4);
                    }
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&raw_empty[rs]);
                    if (++rs == C::RS) { rs = 0; rph ^= 1; }
#pragma unroll
                    for (int hh = 0; hh < C::HPS; ++hh) {
                        const uint32_t s2a = (sc[hh] & 0xFFFFu) * 0x10001u, s2b = (sc[hh] >> 16) * 0x10001u;
                        const uint32_t wv[8] = {cw[hh][0].x, cw[hh][0].y, cw[hh][0].z, cw[hh][0].w,
                                                cw[hh][1].x, cw[hh][1].y, cw[hh][1].z, cw[hh][1].w};
#pragma unroll
                        for (int w8 = 0; w8 < 8; ++w8)
                            dequant8(wv[w8], w8 < 4 ? s2a : s2b, &o[2 * hh + (w8 >> 2)][(w8 & 3) * 4]);
                    }
                } else if constexpr (I4) {
                    // one 64-byte row: 128 int4 codes (n = q + 8), element 2i in the low nibble of byte i
                    const uint8_t* src = sRaw + rs * C::RAW_BYTES + tile * (128 * 64) + m * 64;
                    uint4 c[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) c[j] = *reinterpret_cast<const uint4*>(src + ((j ^ sw) << 4));
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&raw_empty[rs]);
                    if (++rs == C::RS) { rs = 0; rph ^= 1; }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t wv[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
#pragma unroll
                        for (int p = 0; p < 4; ++p) i4x8_to_f16x2(wv[p], &o[j][4 * p]);
                    }
                } else {
                    const uint8_t* src = sRaw + rs * C::RAW_BYTES + tile * (128 * 64) + m * 64;
                    uint4 c[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        c[j] = *reinterpret_cast<const uint4*>(src + (j >> 2) * C::HALF_RAW + (((j & 3) ^ sw) << 4));
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&raw_empty[rs]);
                    if (++rs == C::RS) { rs = 0; rph ^= 1; }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t wv[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
#pragma unroll
                        for (int p = 0; p < 4; ++p)
                            i8x4_to_f16x2(wv[p], o[j >> 1][(j & 1) * 8 + 2 * p], o[j >> 1][(j & 1) * 8 + 2 * p + 1]);
                    }
                }
                // the A slot is free once the MMAs of step gs - C::AS have completed
                if (gs >= (uint32_t)C::AS) {
                    const uint32_t j = gs - C::AS;
                    if (!warp_wait(&done[j % C::BS], (j / C::BS) & 1u, lane)) {
                        if (lane == 0) set_abort(abort_flag, a.status);
                        ok = false;
                        break;
                    }
                }
                const int as = (int)(gs % C::AS);
                const uint32_t ta = tm + lane_base + C::A_COL + (uint32_t)(as * C::A_SLOT_COLS + tile * (C::KSTEP / 2));
#pragma unroll
                for (int q4 = 0; q4 < 2 * C::HPS; ++q4) tmem_st16(ta + 16 * q4, o[q4]);
                tc::tmem_st_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&a_full[as]);
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        if (a.weights_early) pdl_wait();
        const int q = warp & 3, eh = (warp - WARP_EPI0) >> 2;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int n = q * 32 + lane;  // weight row within a tile = output column within its 128-column block
        uint32_t ev = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok && !*abort_flag; u += gridDim.x) {
            int e, t, half, nb, m0, ntok;
            decode_unit<C::NS>(u, NB, halves, a.nmax, tile_start, sub_start, E, a.offsets, e, t, half, nb, m0, ntok, false);
            if (ntok <= 0) continue;
            const float* ts = a.act_scale + (int64_t)t * a.nmax + half * C::NS;
            float ws0, ws1;  // channel scales of this thread's row in the two tiles
            int64_t col0, col1, dcol0, dcol1, ostride, dstride;
            if (STAGE == 1) {
                const int64_t wr = (int64_t)e * 2 * a.I + nb * 128 + n;
                ws0 = a.w_scale[wr];
                ws1 = a.w_scale[wr + a.I];
                col0 = nb * 128 + n;
                col1 = col0;
                ostride = a.I;
                dcol0 = col0;
                dcol1 = a.I + col0;
                dstride = 2 * (int64_t)a.I;
            } else {
                const int64_t wr = (int64_t)e * a.H + nb * 256 + n;
                ws0 = a.w_scale[wr];
                ws1 = a.w_scale[wr + 128];
                col0 = nb * 256 + n;
                col1 = col0 + 128;
                ostride = a.H;
                dcol0 = col0;
                dcol1 = col1;
                dstride = a.H;
            }
            uint32_t starts[4] = {0u, 0u, 0u, 0u};
            if constexpr (FMT == FMT_W8) chunk_starts(a.l1max + (int64_t)(t * halves + half) * KT, KT, lane, starts);
            const int nev = 1 + __popc(starts[0]) + __popc(starts[1]) + __popc(starts[2]) + __popc(starts[3]);
            // this warp's per-token activation scales (chunk i: token 16 * eh + 32 * i + lane, lanes < 16),
            // fetched before the accumulator is ready
            float fls[C::EPI_CHUNKS];
#pragma unroll
            for (int i = 0; i < C::EPI_CHUNKS; ++i) {
                const int c = 16 * eh + 32 * i + lane;
                fls[i] = (lane < 16 && c < ntok) ? ts[c] : 0.f;
            }
            bool last_final = false;
            for (int ch = 0; ch < nev; ++ch, ++ev) {
                int w = 1;
                // sleeping between polls leaves the issue slots to the converter warps on the
                // same schedulers; W8A8 drains mid-unit, so it polls more often
                if (lane == 0) w = tc::mbar_wait_sleep(acc_full, ev & 1, 4000000000ll, FMT == FMT_W8 ? 128u : 512u) ? 1 : 0;
                w = __shfl_sync(0xFFFFFFFFu, w, 0);
                __syncwarp();
                if (!w) {
                    if (lane == 0) set_abort(abort_flag, a.status);
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                if (ch < nev - 1) {
                    // drain: hi parts into the 16-bit running sums, lo back as the accumulator
                    for (int c0 = 16 * eh; c0 < ntok; c0 += 32) {
                        uint32_t g[16], v[16];
                        tmem_ld16(tm + lane_base + C::R_COL + c0, g);
                        tmem_ld16(tm + lane_base + C::R_COL + C::NS + c0, v);
                        tc::tmem_ld_wait();
                        uint32_t* sr = sS + c0 * 128 + n;
                        // the high parts so far (none before the first drain), then this chunk's added;
                        // the branch stays outside the unrolled loops so their 16 chains interleave
                        uint32_t sw[16];
                        if (ch > 0) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) sw[j] = sr[j * 128];
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) sw[j] = 0;
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            int h0, l0, h1, l1;
                            split_hi_lo(g[j], h0, l0);
                            split_hi_lo(v[j], h1, l1);
                            h0 += (int)(int16_t)(sw[j] & 0xFFFFu);
                            h1 += (int)(int16_t)(sw[j] >> 16);
                            sr[j * 128] = (uint32_t)(uint16_t)h0 | ((uint32_t)(uint16_t)h1 << 16);
                            g[j] = __float_as_uint((float)l0);
                            v[j] = __float_as_uint((float)l1);
                        }
                        tmem_st16(tm + lane_base + C::R_COL + c0, g);
                        tmem_st16(tm + lane_base + C::R_COL + C::NS + c0, v);
                    }
                    tc::tmem_st_wait();
                } else {
                    // final, first pass: the outputs into this thread's shared-memory words (where the
                    // running high parts were), so the accumulator can be handed back before the stores
#pragma unroll
                    for (int i = 0; i < C::EPI_CHUNKS; ++i) {
                        const int c0 = 16 * eh + 32 * i;
                        if (c0 >= ntok) break;
                        uint32_t g[16], v[16];
                        tmem_ld16(tm + lane_base + C::R_COL + c0, g);
                        tmem_ld16(tm + lane_base + C::R_COL + C::NS + c0, v);
                        uint32_t* sr = sS + c0 * 128 + n;
                        const float fl = fls[i];
                        tc::tmem_ld_wait();
                        // high parts from the drains (none when there were none), as floats
                        float hf0[16], hf1[16];
                        if (nev > 1) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const uint32_t w = sr[j * 128];
                                hf0[j] = (float)(int16_t)(w & 0xFFFFu);
                                hf1[j] = (float)(int16_t)(w >> 16);
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) hf0[j] = hf1[j] = 0.f;
                        }
                        if (!W4 && a.dbg_acc) {
                            const int nv = min(16, ntok - c0);
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                if (j >= nv) break;
                                const int64_t slot = m0 + c0 + j;
                                a.dbg_acc[slot * dstride + dcol0] =
                                    (int)hf0[j] * (1 << HI_SHIFT) + __float2int_rn(__uint_as_float(g[j]));
                                a.dbg_acc[slot * dstride + dcol1] =
                                    (int)hf1[j] * (1 << HI_SHIFT) + __float2int_rn(__uint_as_float(v[j]));
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            // (float) of the exact sum hi * 2^13 + v: the fma rounds the exact value once
                            const float f0 = __fmaf_rn(hf0[j], (float)(1 << HI_SHIFT), __uint_as_float(g[j]));
                            const float f1 = __fmaf_rn(hf1[j], (float)(1 << HI_SHIFT), __uint_as_float(v[j]));
                            const float fx = __shfl_sync(0xFFFFFFFFu, fl, j);
                            const float r0 = (f0 * fx) * ws0;
                            const float r1 = (f1 * fx) * ws1;
                            if (STAGE == 1) {
                                const float h = __fdividef(r0, 1.0f + __expf(-r0)) * r1;
                                sr[j * 128] = W4 ? (uint32_t)float_to_bf16_bits(h) : __float_as_uint(h);
                            } else
                                sr[j * 128] = (uint32_t)float_to_bf16_bits(r0) | ((uint32_t)float_to_bf16_bits(r1) << 16);
                        }
                    }
                    last_final = true;
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(acc_empty);
            }
            if (last_final && W4 && STAGE == 1) {
                // final, second pass (W4 stage 1): bf16 h into the h tiles, and each 32-column
                // group's largest |h| (this warp's 32 columns) into the tile tail
                const int NG = a.I / 32;
                uint8_t* hblk = a.h_tiles + ((int64_t)t * (a.I / 64) + nb * 2 + (n >> 6)) * bft::block_bytes(a.nmax);
                for (int c0 = 16 * eh; c0 < ntok; c0 += 32) {
                    const uint32_t* sr = sS + c0 * 128 + n;
                    const int nv = min(16, ntok - c0);
                    for (int j = 0; j < nv; ++j) {  // warp-uniform: every lane takes part in the reduction
                        const int row = half * C::NS + c0 + j;  // row within the schedule tile
                        const uint32_t w = sr[j * 128];
                        *reinterpret_cast<uint16_t*>(hblk + bft::elem_offset(row, n & 63)) = (uint16_t)w;
                        const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, (w & 0x7FFFu) << 16);
                        if (lane == 0) a.h_tail[((int64_t)t * a.nmax + row) * NG + nb * 4 + q] = __uint_as_float(mx);
                    }
                }
            } else if (last_final) {
                // final, second pass: shared memory -> outputs, overlapping the next unit's MMAs
                for (int c0 = 16 * eh; c0 < ntok; c0 += 32) {
                    const uint32_t* sr = sS + c0 * 128 + n;
                    const int nv = min(16, ntok - c0);
                    for (int j = 0; j < nv; ++j) {
                        const int64_t slot = m0 + c0 + j;
                        const uint32_t w = sr[j * 128];
                        if (STAGE == 1) {
                            a.h[slot * ostride + col0] = __uint_as_float(w);
                        } else {
                            a.y[slot * ostride + col0] = (uint16_t)(w & 0xFFFFu);
                            a.y[slot * ostride + col1] = (uint16_t)(w >> 16);
                        }
                    }
                }
            }
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

// Raw int8 weights viewed through a TMA map with 64-byte rows (64 K elements,
// half a step; for packed int4 weights a whole 128-element step) and the
// 64-byte swizzle.  Stage 1: {H, I, 2E} (gate rows of expert e are
// plane 2e, its up rows plane 2e+1), box {64, 128, 2}: a gate tile and its up
// partner.  Stage 2: {I, E*H}, box {64, 256}: two adjacent row tiles.
static int make_w_map(CUtensorMap* map, const void* w, const qmoe_dims* d, int stage, bool int4 = false) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return QMOE_ERR_CUDA;
    CUresult r;
    // row bytes: K int8 values, or K/2 bytes of packed int4 codes
    const cuuint64_t H = int4 ? d->H / 2 : d->H, I = int4 ? d->I / 2 : d->I;
    if (stage == 1) {
        cuuint64_t gdim[3] = {H, (cuuint64_t)d->I, (cuuint64_t)(2 * d->E)};
        cuuint64_t gstride[2] = {H, (cuuint64_t)d->I * H};
        cuuint32_t box[3] = {64, 128, 2};
        cuuint32_t estr[3] = {1, 1, 1};
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(w), gdim, gstride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t gdim[2] = {I, (cuuint64_t)d->E * (cuuint64_t)d->H};
        cuuint64_t gstride[1] = {I};
        cuuint32_t box[2] = {64, 256};
        cuuint32_t estr[2] = {1, 1};
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(w), gdim, gstride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS ? QMOE_OK : QMOE_ERR_UNSUPPORTED;
}

static int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

template <int STAGE, int FMT>
static int launch(const CUtensorMap& map, const Args& a, cudaStream_t st) {
    using C = Cfg<FMT>;
    if (cudaFuncSetAttribute(int_gemm_kernel<STAGE, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::smem_bytes(MAX_E)) != cudaSuccess)
        return QMOE_ERR_LAUNCH;
    const int grid = sm_count();
    if (grid <= 0) return QMOE_ERR_CUDA;
    Args b = a;
    b.weights_early = launch_ctx().weights_early ? 1 : 0;
    return launch_pdl(int_gemm_kernel<STAGE, FMT>, grid, THREADS, C::smem_bytes(a.E), st, map, b);
}

}  // namespace ig

bool i8_tc_ok(const qmoe_dims* d) {
    return d->H % 256 == 0 && d->I % 128 == 0 && d->H <= ig::MAX_K && d->I <= ig::MAX_K && d->E <= ig::MAX_E;
}

int i8_tc_gemm1(const qmoe_dims* d, const uint8_t* x_tiles, const int8_t* w1, const float* w1_s,
                const int32_t* offsets, const int32_t* tile_start, float* h, int32_t* dbg_acc, int32_t* status,
                cudaStream_t st) {
    CUtensorMap map;
    int rc = ig::make_w_map(&map, w1, d, 1);
    if (rc != QMOE_OK) return rc;
    ig::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.nmax = mxt::nmax_for(d);
    a.act = x_tiles;
    a.act_scale = reinterpret_cast<const float*>(x_tiles + bft::blocks_bytes(d, d->H));
    a.l1max = reinterpret_cast<const int32_t*>(x_tiles + bft::blocks_bytes(d, d->H) +
                                               mxt::max_tiles(d, a.nmax) * a.nmax * 4);
    a.w_scale = w1_s;
    a.offsets = offsets; a.tile_start = tile_start;
    a.h = h; a.dbg_acc = dbg_acc; a.status = status;
    return ig::launch<1, ig::FMT_W8>(map, a, st);
}

int i8_tc_gemm2(const qmoe_dims* d, const uint8_t* h_tiles, const int8_t* w2, const float* w2_s,
                const int32_t* offsets, const int32_t* tile_start, uint16_t* y, int32_t* dbg_acc, int32_t* status,
                cudaStream_t st) {
    CUtensorMap map;
    int rc = ig::make_w_map(&map, w2, d, 2);
    if (rc != QMOE_OK) return rc;
    ig::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.nmax = mxt::nmax_for(d);
    a.act = h_tiles;
    a.act_scale = reinterpret_cast<const float*>(h_tiles + bft::blocks_bytes(d, d->I));
    a.l1max = reinterpret_cast<const int32_t*>(h_tiles + bft::blocks_bytes(d, d->I) +
                                               mxt::max_tiles(d, a.nmax) * a.nmax * 4);
    a.w_scale = w2_s;
    a.offsets = offsets; a.tile_start = tile_start;
    a.y = y; a.dbg_acc = dbg_acc; a.status = status;
    return ig::launch<2, ig::FMT_W8>(map, a, st);
}

// ------------------------------------------------------------------ W4A8 (int4 weights, int8 activations)

int i4_tc_gemm1(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1, const float* w1_s,
                const int32_t* offsets, const int32_t* tile_start, float* h, int32_t* dbg_acc, int32_t* status,
                cudaStream_t st) {
    CUtensorMap map;
    int rc = ig::make_w_map(&map, w1, d, 1, true);
    if (rc != QMOE_OK) return rc;
    ig::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.nmax = mxt::nmax_for(d);
    a.act = x_tiles;
    a.act_scale = reinterpret_cast<const float*>(x_tiles + bft::blocks_bytes(d, d->H));
    a.w_scale = w1_s;
    a.offsets = offsets; a.tile_start = tile_start;
    a.h = h; a.dbg_acc = dbg_acc; a.status = status;
    return ig::launch<1, ig::FMT_I4>(map, a, st);
}

int i4_tc_gemm2(const qmoe_dims* d, const uint8_t* h_tiles, const uint8_t* w2, const float* w2_s,
                const int32_t* offsets, const int32_t* tile_start, uint16_t* y, int32_t* dbg_acc, int32_t* status,
                cudaStream_t st) {
    CUtensorMap map;
    int rc = ig::make_w_map(&map, w2, d, 2, true);
    if (rc != QMOE_OK) return rc;
    ig::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.nmax = mxt::nmax_for(d);
    a.act = h_tiles;
    a.act_scale = reinterpret_cast<const float*>(h_tiles + bft::blocks_bytes(d, d->I));
    a.w_scale = w2_s;
    a.offsets = offsets; a.tile_start = tile_start;
    a.y = y; a.dbg_acc = dbg_acc; a.status = status;
    return ig::launch<2, ig::FMT_I4>(map, a, st);
}

// ------------------------------------------------------------------ W4A16

bool w4_tc_ok(const qmoe_dims* d) { return d->H % 256 == 0 && d->I % 128 == 0 && d->E <= ig::MAX_E; }

int w4_tc_gemm1(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1, const int32_t* offsets,
                const int32_t* tile_start, uint8_t* h_tiles, int32_t* status, cudaStream_t st) {
    CUtensorMap map;
    memset(&map, 0, sizeof(map));  // W4 weights come by bulk copy
    ig::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.nmax = mxt::nmax_for(d);
    a.act = x_tiles;
    a.act_scale = reinterpret_cast<const float*>(x_tiles + bft::blocks_bytes(d, d->H));
    a.wq = w1;
    a.w_scale = reinterpret_cast<const float*>(w1 + bft::w4_blocks_bytes((int64_t)d->E * 2 * d->I, d->H));
    a.offsets = offsets; a.tile_start = tile_start;
    a.h_tiles = h_tiles;
    a.h_tail = reinterpret_cast<float*>(h_tiles + bft::blocks_bytes(d, d->I));
    a.status = status;
    return ig::launch<1, ig::FMT_W4>(map, a, st);
}

int w4_tc_gemm2(const qmoe_dims* d, const uint8_t* h16_tiles, const uint8_t* w2, const int32_t* offsets,
                const int32_t* tile_start, uint16_t* y, int32_t* status, cudaStream_t st) {
    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    ig::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.nmax = mxt::nmax_for(d);
    a.act = h16_tiles;
    a.act_scale = reinterpret_cast<const float*>(h16_tiles + bft::blocks_bytes(d, d->I));
    a.wq = w2;
    a.w_scale = reinterpret_cast<const float*>(w2 + bft::w4_blocks_bytes((int64_t)d->E * d->H, d->I));
    a.offsets = offsets; a.tile_start = tile_start; a.y = y; a.status = status;
    return ig::launch<2, ig::FMT_W4>(map, a, st);
}

}  // namespace qmoe
