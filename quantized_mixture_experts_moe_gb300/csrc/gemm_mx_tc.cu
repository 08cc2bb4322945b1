// Grouped MXFP4-weight x FP8-activation expert GEMMs on the 5th-generation
// tensor cores (tcgen05, block-scaled kind::mxf8f6f4, E8M0 scales).
//
// The aiter tuned grouped-fmoe page (Changes, Test Plan) runs a two-stage
// grouped a8w4 kernel with fp8 activations and MXFP4 weights; this is that
// computation written for sm_103a:
//   stage 1: h = silu(W1_gate . x) * (W1_up . x), then MX-quantised to
//            E4M3 codes + E8M0 scales per 32 columns of I;
//   stage 2: y = W2 . h, accumulated in fp32, stored as bf16.
//
// Structure (one persistent CTA per SM, 12 warps; 19 in the gathering stage-1
// form, whose 7 extra gather warps join warp 1):
//   warp 0     weight producer: per pipeline step one TMA load (a 4D box) of
//              the step's two FP4 weight tiles (stage 1: a gate tile and its
//              up partner; stage 2: two adjacent row tiles of W2) from
//              tile-major pre-packed weights -- each 128x128 tile
//              is one contiguous 8 KiB read, unpacked by the tensor map into
//              the 16-byte-aligned form the MMA reads -- plus bulk copies of
//              the matching 512-byte scale atoms.
//   warp 1     activation producer: per step two bulk copies of the step's
//              block of the stage-ready MX activation tiles (the token rows,
//              already 128-byte swizzled, and their scale atoms); or, in
//              stage 1 from token-major MX x, a gather: the 32 lanes copy each
//              routed token's 128 codes and 4 scale bytes of the step with
//              cp.async into the same swizzled slot layout.
//   warps 2-3  MMA issuers (warp 2 also owns tensor memory), one per weight
//              tile: one lane copies its scale atoms into TMEM and issues the
//              MMAs (M = 128 weight rows, N = tokens rounded up to 16, K = 32
//              per instruction), one commit per step.  Two issuers halve the
//              serial instruction stream each thread issues.
//   warps 4-11 epilogue (two warps per TMEM lane quadrant, alternating
//              16-token chunks): TMEM -> registers, then SwiGLU + MX
//              quantisation through a shared-memory transpose (stage 1) or
//              bf16 stores (stage 2).
// Every tcgen05 or TMA instruction costs the issuing thread on the order of
// a hundred cycles, so a step carries as much data per instruction as the
// hardware allows: one ring slot holds a whole step (weights, activations,
// both scale sets) behind a single full/empty barrier pair, and the ring is
// as deep as shared memory allows (3 to 6 steps with 224- to 16-token tiles).
// Two accumulator buffers in TMEM (16- and 112-token tiles) let the epilogue
// of one unit overlap the MMAs of the next; 224-token tiles have one.
//
// The weights are the A operand ("swap AB"): per-expert token counts are
// small at prefill sizes (about 80 at T = 4096), so tokens take the MMA's N
// dimension (a multiple of 16) instead of being padded to M = 128.  A work
// unit is (expert, tile of up to NMAX of its tokens, 128 output columns of h
// in stage 1 / 256 columns of y in stage 2);
// units are ordered with the column block fastest so concurrent CTAs share
// activation rows through L2, and each unit streams a disjoint slice of the
// expert's weights exactly once.
#include "qmoe_common.cuh"
#include "mx_tiles.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

#include <mutex>

namespace qmoe {

namespace mx {

// warp roles
constexpr int WARP_A = 0;                   // weight producer (TMA)
constexpr int WARP_B = 1;                   // activation producer (bulk copies of stage-ready tiles)
constexpr int WARP_MMA = 2;                 // TMEM owner + MMA issuer for weight tile 0
constexpr int WARP_MMA2 = WARP_MMA + 1;     // stage 1: second issuer (up accumulator)
constexpr int WARP_EPI0 = WARP_MMA2 + 1;    // epilogue warps
constexpr int EPI_WARPS = 8;                // two per TMEM lane quadrant, splitting the token columns
constexpr int WARP_G1 = WARP_EPI0 + EPI_WARPS;  // stage-1 gather: warps after the epilogue join warp 1
constexpr int KSTAGE = 128;                 // K elements per pipeline step (4 MMAs of K = 32)
constexpr uint32_t FP4_TILE_TX = 128 * 64;  // bytes one 128x128 FP4 tile moves (packed)

// GATHER: stage 1 gathers token-major x (its own instantiation, so the
// permuted-tile kernels keep their 12 warps and their code)
template <int STAGE, int NMAX_, bool GATHER = false>
struct Cfg {
    static constexpr int NMAX = NMAX_;
    // weight tiles per step, one per MMA issuer: stage 1 gate + up, stage 2
    // two adjacent 128-column blocks of W2; both share the step's activations
    static constexpr int AT = 2;
    static constexpr int ACC_BUFS = (AT * NMAX * 2 <= 448) ? 2 : 1;
    // L2 eviction hints on the loads (weights evict-first, activations
    // evict-last) for 16-row tiles, which the tile table picks for small
    // batches: there each expert has one tile and its weights pass once.
    // Measured on GB300 with L2 flushed: decode T=16 114.6 -> 103.2 us/step;
    // at larger tiles they were neutral to 0.5% slower.
    static constexpr bool L2_HINTS = (NMAX == 16);
    // 112- and 224-token tiles: the weight producer also asks L2 for the
    // weight tiles PF_AHEAD steps past its newest load (across units), so the
    // ring's own loads find them there.  The ring holds only 3 or 4 steps,
    // and a timing variant with 5 showed the weight stream is limited by how
    // much is in flight.  Measured on GB300 at T = 4096: stage 1 424 -> 416 us,
    // stage 2 254 -> 248 us (distances 2-6 gave 415-416 us in stage 1, 8
    // gave 417, 16 gave 438).  With 16-token tiles (6-step ring, weights
    // evict-first) it made every decode size 2-8% slower, so it is off there,
    // and so it is for units shorter than 8 steps (stage 2 of the I = 512 and
    // 256 shards: 152 -> 162 and 121 -> 125 us with it).
    // Stage 2 with 224-token tiles (T = 8192) prefers 8 steps ahead: 408 -> 395 us there.
    static constexpr bool L2_PREFETCH = (NMAX != 16);
    static constexpr int PF_AHEAD = (STAGE == 2 && NMAX == 224) ? 8 : 4;
    static constexpr int NSFB = (NMAX + 127) / 128;      // activation scale atoms per step
    static constexpr int A_BYTES = AT * 128 * 128;
    static constexpr int B_BYTES = ((NMAX + 7) / 8) * 1024;
    static constexpr int SFA_BYTES = AT * 512;
    static constexpr int SFB_BYTES = NSFB * 512;
    static constexpr int SLOT_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    // stage 1 epilogue: per epilogue warp a 16-token x 32-column transpose
    // buffer of h (rows padded to 36 floats: the 16-byte reads of 8 rows at
    // a time hit distinct banks)
    // (16-token tiles have a single chunk, so only the first four warps ever use it)
    static constexpr int EPI_ROW = 36;
    static constexpr int EPI_BYTES = (STAGE == 1) ? (NMAX == 16 ? 4 : EPI_WARPS) * 16 * EPI_ROW * 4 : 0;
    // ring depth: as many whole steps as fit in the 227 KB of shared memory
    // next to 1 KB of alignment slack, the epilogue buffer, and barriers for
    // up to 16 slots, the misc words and the schedule of up to MAX_E experts
    // Stage-1 gather warps (warp 1 and GW - 1 more): one warp copies ~6 bytes
    // a clock with cp.async, against the ~15-30 KB of token rows a 112- or
    // 224-row step needs every ~800-1400 clocks (at T = 4096, stage 1 took
    // 1005 us with one warp, 528 with four, 497 with eight).
    static constexpr int GW = (STAGE == 1 && GATHER) ? (NMAX == 16 ? 1 : 8) : 0;
    static constexpr int THREADS = (WARP_G1 + (GW > 1 ? GW - 1 : 0)) * 32;
    static constexpr int TOK_BYTES = GW * NMAX * 4;  // per gather warp: the unit's token per row
    static constexpr int FIXED_BYTES = 2 * 16 * 8 + 64 + TOK_BYTES + (512 + 1) * 4;
    static constexpr int S = (232448 - 1024 - EPI_BYTES - FIXED_BYTES) / SLOT_BYTES;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = A_OFF + S * A_BYTES;
    static constexpr int SFA_OFF = B_OFF + S * B_BYTES;
    static constexpr int SFB_OFF = SFA_OFF + S * SFA_BYTES;
    static constexpr int EPI_OFF = SFB_OFF + S * SFB_BYTES;
    static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
    static constexpr int NBAR = 2 * S + 2 * ACC_BUFS;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int TOK_OFF = MISC_OFF + 64;
    static constexpr int SCHED_OFF = TOK_OFF + TOK_BYTES;
    static constexpr size_t smem_bytes(int E) { return (size_t)SCHED_OFF + (size_t)(E + 1) * 4 + 1024; }
    // TMEM columns: accumulators, then a 2-slot ring for scale factors
    static constexpr uint32_t ACC_COLS = AT * NMAX;
    static constexpr uint32_t SF_COL = ACC_BUFS * ACC_COLS;
    // one scale-factor column block per issuer: its weight atom + the activation atoms
    static constexpr uint32_t SF_SLOT = 4 + NSFB * 4;
    static_assert(SF_COL + 2 * AT * SF_SLOT <= 512, "TMEM budget");
    static_assert(NMAX % 16 == 0 && NMAX <= 256, "N tile");
    static_assert(S >= 2 && S <= 16, "ring");
};

constexpr int MAX_E = 512;  // schedule prefix kept in shared memory
static_assert(Cfg<1, 16>::smem_bytes(MAX_E) <= 232448 && Cfg<2, 16>::smem_bytes(MAX_E) <= 232448 &&
                  Cfg<1, 112>::smem_bytes(MAX_E) <= 232448 && Cfg<1, 224>::smem_bytes(MAX_E) <= 232448 &&
                  Cfg<2, 112>::smem_bytes(MAX_E) <= 232448 && Cfg<2, 224>::smem_bytes(MAX_E) <= 232448 &&
                  Cfg<1, 16, true>::smem_bytes(MAX_E) <= 232448 && Cfg<1, 112, true>::smem_bytes(MAX_E) <= 232448 &&
                  Cfg<1, 224, true>::smem_bytes(MAX_E) <= 232448,
              "shared memory per CTA");

struct Args {
    int T, k, H, I, E;
    const uint8_t* act;         // MX activation tiles: stage 1 x (K = H), stage 2 h (K = I)
    const uint8_t* w_s;         // pre-packed weight scale atoms
    const int32_t* offsets;     // [E+1]
    const int32_t* tile_start;  // [E+1] token-tile schedule (from the routing workspace)
    uint8_t* h_tiles;           // stage 1 output: h as MX activation tiles (K = I)
    uint16_t* y;                // stage 2 output: bf16, slot order
    int32_t* status;
    int weights_early;          // the weight producer may run before the predecessor kernel completes
    const uint8_t* w;           // the pre-packed weights (for L2 prefetches; the loads go through the tensor map)
    int64_t gate_bytes;         // stage 1: bytes of one expert's gate tiles (its up tiles follow)
    // stage-1 gather (xq non-null): token-major MX x, codes [T, H] and scales
    // [T, H/32], and the routing sort's slot -> pair map (token = pair / k)
    const uint8_t* xq;
    const uint8_t* xs;
    const int32_t* sorted;
};

template <int NMAX>
__device__ __forceinline__ void decode_unit(int u, int NB, const int* tile_start, int E, const int32_t* offsets,
                                            int& e, int& m0, int& ntok, int& nb, int& t, bool l2) {
    t = u / NB;
    nb = u - t * NB;
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tile_start[mid] <= t) lo = mid; else hi = mid;
    }
    e = lo;
    // l2: a role that runs before this kernel's dependent-launch wait reads
    // the routing sort's offsets from L2 (the sort completed before the launch)
    const int o0 = l2 ? __ldcg(offsets + e) : offsets[e];
    const int o1 = l2 ? __ldcg(offsets + e + 1) : offsets[e + 1];
    m0 = o0 + (t - tile_start[e]) * NMAX;
    ntok = min(NMAX, o1 - m0);
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

// Stage-1 activation producer, gather form (warp g of C::GW, each taking an
// interleaved share of the chunks and rows).  Per step each routed
// token row of the unit's tile gets its 128 E4M3 codes (eight 16-byte
// cp.async, 8 lanes per row, so a warp instruction reads four whole 128-byte
// rows) at the swizzled position the MX tile layout gives it, and its 4 scale
// bytes at its place in the scale atom.  Rows past the tile's token count are
// left as they are: they only feed accumulator columns the epilogue never
// stores.  Every lane then makes one arrival on the slot's full barrier that
// the hardware delivers once the lane's copies have landed
// (cp.async.mbarrier.arrive.noinc; the barrier expects the weight producer
// and these 32 * GW), so no warp waits for its own copies; the MMA issuer
// orders the landed bytes before its tensor-core reads with a proxy fence
// after the barrier wait.
template <typename C, int NMAX>
__device__ __forceinline__ void gather_x(const Args& a, uint8_t* sB, uint8_t* sSFB, uint64_t* full, uint64_t* empty,
                                         int* tok_row, const int* tile_start, int total_units, int NB, int KT,
                                         volatile int* abort_flag, int lane, int g) {
    const uint64_t pol = tc::l2_evict_last();  // x rows are read by every column block of each of their experts
    const int64_t xs_row = a.H / 32;
    int slot = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total_units && !*abort_flag && ok; u += gridDim.x) {
        int e, m0, ntok, nb, t;
        decode_unit<NMAX>(u, NB, tile_start, a.E, a.offsets, e, m0, ntok, nb, t, false);
        __syncwarp();  // every lane is done with the previous unit's rows
        // a pair id outside [0, T*k) (not a routing sort's output) is not read: its row keeps stale data
        for (int r = lane; r < ntok; r += 32) {
            const int p = a.sorted[m0 + r];
            tok_row[r] = (p >= 0 && (int64_t)p < (int64_t)a.T * a.k) ? p / a.k : -1;
        }
        __syncwarp();
        for (int kt = 0; kt < KT; ++kt) {
            if (!warp_wait(&empty[slot], phase ^ 1, lane)) {
                if (lane == 0) set_abort(abort_flag, a.status);
                ok = false;
                break;
            }
            uint8_t* dB = sB + slot * C::B_BYTES;
            uint8_t* dS = sSFB + slot * C::SFB_BYTES;
            for (int i = g * 32 + lane; i < ntok * 8; i += 32 * C::GW) {
                const int r = i >> 3, c = i & 7;
                const int tok = tok_row[r];
                if (tok >= 0)
                    tc::cp_async_16_hint(dB + mxt::code_offset(r, c * 16), a.xq + (int64_t)tok * a.H + kt * 128 + c * 16,
                                         pol);
            }
            for (int r = g * 32 + lane; r < ntok; r += 32 * C::GW) {
                const int tok = tok_row[r];
                if (tok >= 0)
                    tc::cp_async_4(dS + (mxt::scale_offset(NMAX, r, 0) - NMAX * 128), a.xs + (int64_t)tok * xs_row + kt * 4);
            }
            tc::cp_async_mbar_arrive_noinc(&full[slot]);
            if (++slot == C::S) { slot = 0; phase ^= 1; }
        }
    }
    tc::cp_async_wait<0>();
}

template <int STAGE, int NMAX, bool GATHER>
__global__ void __launch_bounds__(Cfg<STAGE, NMAX, GATHER>::THREADS, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap mapW, const Args a) {
    using C = Cfg<STAGE, NMAX, GATHER>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::A_OFF;
    uint8_t* sB = smem + C::B_OFF;
    uint8_t* sSFA = smem + C::SFA_OFF;
    uint8_t* sSFB = smem + C::SFB_OFF;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* empty = full + C::S;
    uint64_t* acc_full = empty + C::S;
    uint64_t* acc_empty = acc_full + C::ACC_BUFS;
    uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 8);
    int* tile_start = reinterpret_cast<int*>(smem + C::SCHED_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E;
    const int K = (STAGE == 1) ? a.H : a.I;            // reduction length
    const int NOUT = (STAGE == 1) ? a.I : a.H;          // output columns
    const int NB = (STAGE == 1) ? NOUT / 128 : NOUT / 256;  // stage 2 units cover two column blocks
    const int KT = K / KSTAGE;

    // Dependent launch: by default everything waits for the predecessor
    // kernel.  With weights_early (set by the whole-layer call, whose routing
    // sort ran two launches back) only the warps that consume the
    // predecessor's output wait; the schedule is read and weights stream
    // before that.
    if (!a.weights_early) pdl_wait();

    // ---- token-tile schedule (computed with the routing sort)
    for (int i = threadIdx.x; i <= E; i += blockDim.x) tile_start[i] = __ldcg(a.tile_start + i);
    if (threadIdx.x == 32 * WARP_MMA) {
        for (int s = 0; s < C::S; ++s) {
            // weight producer (with tx bytes) + activation producer (its 32 lanes when it gathers)
            tc::mbar_init(&full[s], GATHER ? 1 + 32 * C::GW : 2);
            tc::mbar_init(&empty[s], C::AT);   // one commit per MMA issuer
        }
        for (int b = 0; b < C::ACC_BUFS; ++b) {
            tc::mbar_init(&acc_full[b], C::AT);
            tc::mbar_init(&acc_empty[b], EPI_WARPS);
        }
        *abort_flag = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    const int total_units = tile_start[E] * NB;
    if ((int)blockIdx.x >= total_units) {  // no work: nothing allocated yet
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

    if (warp == WARP_A) {
        // ------------------------------------------------ weight producer (TMA)
        if (lane == 0) {
            tc::prefetch_tensormap(&mapW);
            // 16-row tiles (small batches): one tile per expert, its weights streamed once
            const uint64_t pol = C::L2_HINTS ? tc::l2_evict_first() : 0ull;
            int slot = 0;
            uint32_t phase = 0;
            const int rows_per_e = (STAGE == 1) ? 2 * a.I : a.H;
            const int64_t up_tiles = (int64_t)(a.I / 128) * KT;  // gate tile -> up tile distance (stage 1)
            // L2 prefetch cursor: unit pu, step pk, its two 8 KiB weight tiles at pA, pB (+ pk * 8 KiB)
            int pu = blockIdx.x, pk = 0;
            const uint8_t* pA = nullptr;
            const uint8_t* pB = nullptr;
            auto pf_unit = [&]() {
                if (pu >= total_units) return;
                int e, m0, ntok, nb, t;
                decode_unit<NMAX>(pu, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t, a.weights_early != 0);
                if (STAGE == 1) {
                    pA = a.w + (int64_t)e * 2 * a.gate_bytes + (int64_t)nb * KT * 8192;
                    pB = pA + a.gate_bytes;
                } else {
                    pA = a.w + (int64_t)((e * rows_per_e + nb * 256) / 128) * KT * 8192;
                    pB = pA + (int64_t)KT * 8192;
                }
            };
            auto pf_step = [&]() {
                if (pu >= total_units) return;
                tc::bulk_prefetch_l2(pA + (int64_t)pk * 8192, 8192);
                tc::bulk_prefetch_l2(pB + (int64_t)pk * 8192, 8192);
                if (++pk == KT) {
                    pk = 0;
                    pu += gridDim.x;
                    pf_unit();
                }
            };
            const bool prefetch = C::L2_PREFETCH && KT >= 8;
            if (prefetch) {
                pf_unit();
                for (int i = 0; i < C::PF_AHEAD; ++i) pf_step();
            }
            for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x) {
                int e, m0, ntok, nb, t;
                decode_unit<NMAX>(u, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t, a.weights_early != 0);
                const int rt0 = (STAGE == 1) ? (e * rows_per_e + nb * 128) / 128 : (e * rows_per_e + nb * 256) / 128;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(&empty[slot], phase ^ 1)) { set_abort(abort_flag, a.status); break; }
                    tc::mbar_arrive_expect_tx(&full[slot], C::AT * (FP4_TILE_TX + 512));
                    uint8_t* dS = sSFA + slot * C::SFA_BYTES;
                    const int64_t t0 = (int64_t)rt0 * KT + kt;
                    if (STAGE == 1) {
                        // 4D view {row bytes, rows within a half, gate/up half, expert}: one box = both tiles
                        tc::tma_load_4d_hint(sA + slot * C::A_BYTES, &mapW, &full[slot], 0, (nb * KT + kt) * 128, 0, e,
                                             pol, C::L2_HINTS);
                        tc::bulk_load_hint(dS, a.w_s + t0 * 512, 512, &full[slot], pol, C::L2_HINTS);
                        tc::bulk_load_hint(dS + 512, a.w_s + (t0 + up_tiles) * 512, 512, &full[slot], pol,
                                           C::L2_HINTS);
                    } else {
                        // 4D view {row bytes, tile rows, K tile, row tile}: one box = row tiles rt0, rt0 + 1
                        tc::tma_load_4d_hint(sA + slot * C::A_BYTES, &mapW, &full[slot], 0, 0, kt, rt0, pol,
                                             C::L2_HINTS);
                        tc::bulk_load_hint(dS, a.w_s + t0 * 512, 512, &full[slot], pol, C::L2_HINTS);
                        tc::bulk_load_hint(dS + 512, a.w_s + (t0 + KT) * 512, 512, &full[slot], pol, C::L2_HINTS);
                    }
                    if (prefetch) pf_step();
                    if (++slot == C::S) { slot = 0; phase ^= 1; }
                }
            }
            // every load issued: the next kernel may launch (after this CTA's own wait)
            pdl_wait();
            pdl_trigger();
        }
    } else if (warp == WARP_B) {
        // ------------------------------------------------ activation producer (bulk copies)
        // A step's activations are one block of the MX tile layout: the
        // first nmma rows of codes (already swizzled) and the scale atoms.
        if (a.weights_early) pdl_wait();
        if constexpr (GATHER) {
            gather_x<C, NMAX>(a, sB, sSFB, full, empty, reinterpret_cast<int*>(smem + C::TOK_OFF), tile_start,
                              total_units, NB, KT, abort_flag, lane, 0);
        } else if (lane == 0) {
            const uint64_t pol = C::L2_HINTS ? tc::l2_evict_last() : 0ull;  // re-read by the expert's column blocks
            int slot = 0;
            uint32_t phase = 0;
            const int64_t bb = mxt::block_bytes(NMAX);
            for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x) {
                int e, m0, ntok, nb, t;
                decode_unit<NMAX>(u, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t, false);
                const uint32_t rows_bytes = (uint32_t)((ntok + 15) & ~15) * 128u;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(&empty[slot], phase ^ 1)) { set_abort(abort_flag, a.status); break; }
                    tc::mbar_arrive_expect_tx(&full[slot], rows_bytes + C::SFB_BYTES);
                    const uint8_t* blk = a.act + ((int64_t)t * KT + kt) * bb;
                    tc::bulk_load_hint(sB + slot * C::B_BYTES, blk, rows_bytes, &full[slot], pol, C::L2_HINTS);
                    tc::bulk_load_hint(sSFB + slot * C::SFB_BYTES, blk + NMAX * 128, C::SFB_BYTES, &full[slot], pol,
                                       C::L2_HINTS);
                    if (++slot == C::S) { slot = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == WARP_MMA || warp == WARP_MMA2) {
        // ------------------------------------------------ MMA issuers
        // Two issuers, one per accumulator (stage 1: gate rows, up rows;
        // stage 2: the unit's two column blocks): each copies its own scale
        // atoms to TMEM, issues its four MMAs per step and commits; the slot
        // frees after both commits.
        const int iss = warp - WARP_MMA;
        if (a.weights_early) pdl_wait();
        if (lane == 0 && iss < C::AT) {
            int slot = 0, sf = 0, ab = 0;
            uint32_t phase = 0, pacc = 0;
            const uint32_t sf_base = C::SF_COL + iss * 2 * C::SF_SLOT;
            for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x) {
                int e, m0, ntok, nb, t;
                decode_unit<NMAX>(u, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t, false);
                const int nmma = (ntok + 15) & ~15;
                if (!tc::mbar_wait(&acc_empty[ab], pacc ^ 1)) { set_abort(abort_flag, a.status); break; }
                tc::tc_fence_after();
                const uint32_t dcol = ab * C::ACC_COLS + iss * NMAX;
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(&full[slot], phase)) { set_abort(abort_flag, a.status); ok = false; break; }
                    tc::tc_fence_after();
                    // gathered activations were written by cp.async (generic proxy): order them before the
                    // tensor core's reads of the slot
                    if constexpr (GATHER) tc::fence_proxy_async_smem();
                    const uint32_t sfa_col = sf_base + sf * C::SF_SLOT;
                    const uint32_t sfb_col = sfa_col + 4;
                    const uint32_t sfa_addr = tc::smem_u32(sSFA + slot * C::SFA_BYTES + iss * 512);
                    const uint32_t sfb_addr = tc::smem_u32(sSFB + slot * C::SFB_BYTES);
                    tc::tmem_cp_32x128b_warpx4(tm + sfa_col, tc::smem_desc(sfa_addr, 0, 128, 0));
#pragma unroll
                    for (int t = 0; t < C::NSFB; ++t)
                        tc::tmem_cp_32x128b_warpx4(tm + sfb_col + 4 * t, tc::smem_desc(sfb_addr + 512 * t, 0, 128, 0));
                    const uint32_t a0 = tc::smem_u32(sA + slot * C::A_BYTES + iss * 128 * 128);
                    const uint32_t b0 = tc::smem_u32(sB + slot * C::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t idesc = tc::idesc_mxf8f6f4(128, nmma, 5, 0, kk, kk);
                        tc::mma_mxf8f6f4(tm + dcol, tc::sdesc_kmajor_sw128(a0 + 32 * kk),
                                         tc::sdesc_kmajor_sw128(b0 + 32 * kk), idesc, tm + sfa_col, tm + sfb_col,
                                         (kt > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(&empty[slot]);
                    if (++slot == C::S) { slot = 0; phase ^= 1; }
                    sf ^= 1;
                }
                if (!ok) break;
                tc::mma_commit(&acc_full[ab]);
                if (++ab == C::ACC_BUFS) { ab = 0; pacc ^= 1; }
            }
        }
        __syncwarp();
    } else if (warp >= WARP_G1) {
        // ------------------------------------------------ more stage-1 gather warps
        if constexpr (GATHER) {
            if (a.weights_early) pdl_wait();
            const int g = warp - WARP_G1 + 1;
            gather_x<C, NMAX>(a, sB, sSFB, full, empty, reinterpret_cast<int*>(smem + C::TOK_OFF) + g * NMAX, tile_start,
                              total_units, NB, KT, abort_flag, lane, g);
        }
    } else {
        // ------------------------------------------------ epilogue warps
        if (a.weights_early) pdl_wait();
        const int q = warp & 3;                       // TMEM lane quadrant this warp may access
        const int half = (warp - WARP_EPI0) >> 2;     // which 16-column chunks it takes
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        float* epi = reinterpret_cast<float*>(smem + C::EPI_OFF) + (warp - WARP_EPI0) * 16 * C::EPI_ROW;
        int ab = 0;
        uint32_t pacc = 0;
        for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x) {
            int e, m0, ntok, nb, t;
            decode_unit<NMAX>(u, NB, tile_start, E, a.offsets, e, m0, ntok, nb, t, false);
            int w = 1;
            if (lane == 0) w = tc::mbar_wait_sleep(&acc_full[ab], pacc) ? 1 : 0;
            if (!__shfl_sync(0xFFFFFFFFu, w, 0)) {
                if (lane == 0) set_abort(abort_flag, a.status);
                break;
            }
            tc::tc_fence_after();
            const uint32_t dcol = ab * C::ACC_COLS;
            // stage 1 writes h block (tile t, K step nb of the down projection)
            uint8_t* hblk = (STAGE == 1) ? a.h_tiles + ((int64_t)t * (a.I / 128) + nb) * mxt::block_bytes(NMAX) : nullptr;
            // Chunks of 16 tokens, alternating between the quadrant's two
            // warps; per chunk the accumulator pair (stage 1: gate, up; stage 2:
            // column blocks 2nb, 2nb + 1).
            for (int c0 = 16 * half; c0 < ntok; c0 += 32) {
                uint32_t g[16], g2[16];
                tc::tmem_ld_32x32b_x16(tm + lane_addr + dcol + c0, g);
                tc::tmem_ld_32x32b_x16(tm + lane_addr + dcol + NMAX + c0, g2);
                tc::tmem_ld_wait();
                if (STAGE == 1) {
                    // h for the chunk (lane = column of the 32-column MX block,
                    // j = token), transposed through shared memory so that each
                    // lane then holds 16 columns of one token: lanes t and t + 16
                    // share token c0 + t.  Columns past ntok are computed but
                    // not stored.
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float gv = __uint_as_float(g[j]);
                        epi[j * C::EPI_ROW + lane] = __fdividef(gv, 1.0f + __expf(-gv)) * __uint_as_float(g2[j]);
                    }
                    __syncwarp();
                    const int tok = lane & 15, hh = lane >> 4;
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 f = *reinterpret_cast<const float4*>(epi + tok * C::EPI_ROW + hh * 16 + 4 * i);
                        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
                    }
                    __syncwarp();
                    float amax = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
                    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 16));
                    uint32_t sb = 127;
                    uint4 codes = make_uint4(0u, 0u, 0u, 0u);
                    if (amax > 0.f) {
                        const int X = mx_block_exponent(amax);
                        sb = (uint32_t)(X + 127);
                        const float sc = exp2i(-X);
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            w[i] = (uint32_t)e4m3x2_from_float(v[4 * i] * sc, v[4 * i + 1] * sc) |
                                   ((uint32_t)e4m3x2_from_float(v[4 * i + 2] * sc, v[4 * i + 3] * sc) << 16);
                        codes = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    if (c0 + tok < ntok) {
                        *reinterpret_cast<uint4*>(hblk + mxt::code_offset(c0 + tok, q * 32 + hh * 16)) = codes;
                        if (hh == 0) hblk[mxt::scale_offset(NMAX, c0 + tok, q)] = (uint8_t)sb;
                    }
                } else {
                    // stage 2: token rows of y, 64 contiguous bytes per block and token
                    const int n0 = 2 * nb * 128 + q * 32 + lane;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int c = c0 + j;
                        if (c >= ntok) break;
                        uint16_t* yr = a.y + (int64_t)(m0 + c) * a.H;
                        yr[n0] = float_to_bf16_bits(__uint_as_float(g[j]));
                        yr[n0 + 128] = float_to_bf16_bits(__uint_as_float(g2[j]));
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acc_empty[ab]);
            if (++ab == C::ACC_BUFS) { ab = 0; pacc ^= 1; }
        }
    }

    // ---- wind down: on an abort, give in-flight copies time to land
    if (*abort_flag) {
        tc::cp_async_wait<0>();
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

// ------------------------------------------------------------------ host side

// Tile-major pre-packed FP4 weights viewed as 64-byte rows (128 elements),
// one 128-row box per 128x128 tile: each box is a contiguous 8 KiB read,
// unpacked by the TMA to 16-byte-aligned groups and 128-byte swizzled in
// shared memory.  With half_bytes > 0 (the gate/up weights of stage 1) the
// map is 4D, {row bytes, rows within a half, half, expert}: an expert's gate
// tiles occupy the first half_bytes of its block and the up tiles the next,
// so one 128 x 128 x 2 box brings a gate tile and its up partner.
static int make_fp4_map(CUtensorMap* map, const void* w, int64_t tiles, int64_t half_bytes, int E, int64_t KT) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return QMOE_ERR_CUDA;
    CUresult r;
    if (half_bytes > 0) {
        cuuint64_t gdim[4] = {128, (cuuint64_t)(half_bytes / 64), 2, (cuuint64_t)E};
        cuuint64_t gstride[3] = {64, (cuuint64_t)half_bytes, (cuuint64_t)(2 * half_bytes)};
        cuuint32_t box[4] = {128, 128, 2, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, const_cast<void*>(w), gdim, gstride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        // {row bytes, tile rows, K tile, row tile}: a 128 x 128 x 1 x 2 box brings row tiles rt, rt + 1
        cuuint64_t gdim[4] = {128, 128, (cuuint64_t)KT, (cuuint64_t)(tiles / KT)};
        cuuint64_t gstride[3] = {64, 8192, (cuuint64_t)(KT * 8192)};
        cuuint32_t box[4] = {128, 128, 1, 2};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, const_cast<void*>(w), gdim, gstride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS ? QMOE_OK : QMOE_ERR_UNSUPPORTED;
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

bool mx_tc_supported(const qmoe_dims* d, const void* w1, const void* w2) {
    auto a32 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; };
    const int64_t tiles1 = (int64_t)d->E * 2 * d->I / 128 * (d->H / 128);
    const int64_t tiles2 = (int64_t)d->E * d->H / 128 * (d->I / 128);
    return d->H % 256 == 0 && d->I % 128 == 0 && d->E <= MAX_E && tiles1 * 128 < (1ll << 31) &&
           tiles2 * 128 < (1ll << 31) && (!w1 || a32(w1)) && (!w2 || a32(w2));
}

template <int STAGE, int NMAX, bool GATHER = false>
static int launch_cfg(const void* w, int64_t tiles, int64_t half_bytes, const Args& a, cudaStream_t st) {
    using C = Cfg<STAGE, NMAX, GATHER>;
    CUtensorMap map;
    const int64_t KT = (STAGE == 1) ? a.H / 128 : a.I / 128;
    int rc = make_fp4_map(&map, w, tiles, half_bytes, a.E, KT);
    if (rc != QMOE_OK) return rc;
    const size_t smem = C::smem_bytes(a.E);
    if (cudaFuncSetAttribute(mx_gemm_kernel<STAGE, NMAX, GATHER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::smem_bytes(MAX_E)) != cudaSuccess)
        return QMOE_ERR_LAUNCH;
    const int grid = num_sms();
    if (grid <= 0) return QMOE_ERR_CUDA;
    return launch_pdl(mx_gemm_kernel<STAGE, NMAX, GATHER>, grid, C::THREADS, smem, st, map, a);
}

}  // namespace mx

// Token-tile size (mx_tiles.cuh): the average expert load decides, since the
// grid never syncs with the host to look at the real counts.  Up to ~100
// tokens per expert 112-token tiles with two accumulator buffers; above,
// 224-token tiles so an expert's weights are still streamed once.  Both
// stages and the permute/quantise kernel use the same tiles.
int mx_tc_gemm1(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1, const uint8_t* w1_s,
                const int32_t* offsets, const int32_t* tile_start, uint8_t* h_tiles, int32_t* status,
                cudaStream_t st) {
    mx::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.act = x_tiles; a.w_s = w1_s; a.offsets = offsets; a.tile_start = tile_start;
    a.h_tiles = h_tiles; a.status = status;
    a.weights_early = launch_ctx().weights_early ? 1 : 0;
    a.w = w1;
    a.gate_bytes = (int64_t)(d->I / 128) * (d->H / 128) * 8192;
    const int64_t KT = d->H / 128;
    const int64_t tiles = (int64_t)d->E * 2 * d->I / 128 * KT;
    const int64_t half = (int64_t)(d->I / 128) * KT * 8192;  // bytes of one expert's gate (or up) tiles
    const int nmax = mxt::nmax_for(d);
    return nmax == 224 ? mx::launch_cfg<1, 224>(w1, tiles, half, a, st)
                       : (nmax == 16 ? mx::launch_cfg<1, 16>(w1, tiles, half, a, st)
                                     : mx::launch_cfg<1, 112>(w1, tiles, half, a, st));
}

int mx_tc_gemm1_gather(const qmoe_dims* d, const uint8_t* x_q, const uint8_t* x_s, const int32_t* sorted,
                       const uint8_t* w1, const uint8_t* w1_s, const int32_t* offsets, const int32_t* tile_start,
                       uint8_t* h_tiles, int32_t* status, cudaStream_t st) {
    mx::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.act = nullptr; a.w_s = w1_s; a.offsets = offsets; a.tile_start = tile_start;
    a.h_tiles = h_tiles; a.status = status;
    a.weights_early = launch_ctx().weights_early ? 1 : 0;
    a.w = w1;
    a.gate_bytes = (int64_t)(d->I / 128) * (d->H / 128) * 8192;
    a.xq = x_q; a.xs = x_s; a.sorted = sorted;
    const int64_t KT = d->H / 128;
    const int64_t tiles = (int64_t)d->E * 2 * d->I / 128 * KT;
    const int64_t half = (int64_t)(d->I / 128) * KT * 8192;
    const int nmax = mxt::nmax_for(d);
    return nmax == 224 ? mx::launch_cfg<1, 224, true>(w1, tiles, half, a, st)
                       : (nmax == 16 ? mx::launch_cfg<1, 16, true>(w1, tiles, half, a, st)
                                     : mx::launch_cfg<1, 112, true>(w1, tiles, half, a, st));
}

int mx_tc_gemm2(const qmoe_dims* d, const uint8_t* h_tiles, const uint8_t* w2, const uint8_t* w2_s,
                const int32_t* offsets, const int32_t* tile_start, uint16_t* y, int32_t* status, cudaStream_t st) {
    mx::Args a{};
    a.T = d->T; a.k = d->k; a.H = d->H; a.I = d->I; a.E = d->E;
    a.act = h_tiles; a.w_s = w2_s; a.offsets = offsets; a.tile_start = tile_start; a.y = y; a.status = status;
    a.weights_early = launch_ctx().weights_early ? 1 : 0;
    a.w = w2;
    const int64_t tiles = (int64_t)d->E * d->H / 128 * (d->I / 128);
    const int nmax = mxt::nmax_for(d);
    return nmax == 224 ? mx::launch_cfg<2, 224>(w2, tiles, 0, a, st)
                       : (nmax == 16 ? mx::launch_cfg<2, 16>(w2, tiles, 0, a, st)
                                     : mx::launch_cfg<2, 112>(w2, tiles, 0, a, st));
}

bool mx_tc_ok(const qmoe_dims* d, const void* w1, const void* w2) { return mx::mx_tc_supported(d, w1, w2); }


}  // namespace qmoe
