// Shared device helpers of the sm_103a quantized-MoE library: storage-format
// decoding, the MX / int8 quantisation rules, host-side argument checks.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/qmoe.h"

namespace qmoe {

// ------------------------------------------------------------------ host checks

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool dims_ok(const qmoe_dims* d) {
    return d && d->T >= 0 && d->k > 0 && d->H > 0 && d->I > 0 && d->E > 0 && d->H % 32 == 0 && d->I % 32 == 0 &&
           (int64_t)d->T * d->k < (1ll << 31);
}

inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QMOE_OK : QMOE_ERR_LAUNCH;
}

inline int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// The routing workspace holds, after the per-chunk histograms, the token-tile
// schedule (E + 1 ints, padded to 256 bytes with room for 64 more), then one
// int per slot: the slot's row in the token tiles, tile * NMAX + row (-1 past
// the routed slots), then one int per pair: the pair's row (-1 for an
// invalid expert id).  schedule_ints: ints from the schedule's start to the
// per-slot rows; slot_ints: from the per-slot rows to the per-pair rows.
inline int64_t schedule_ints(int E) { return ((int64_t)(E + 1 + 64) * 4 + 255) / 256 * 64; }
inline int64_t slot_ints(int64_t P) { return (P * 4 + 255) / 256 * 64; }

// ------------------------------------------------------------------ dependent launches
//
// Every kernel of the layer is launched with programmatic stream
// serialization: it may be scheduled while its predecessor in the stream is
// still running, so its launch and prologue hide behind the predecessor's
// tail.  The kernel then calls pdl_wait() before it touches anything its
// predecessor reads or writes (griddepcontrol.wait returns once the
// predecessor grid has completed and its memory operations are visible), and
// pdl_trigger() only after that wait.  Hence when a kernel is launched, the
// kernel two places before it in the stream has completed.  The small kernels
// trigger right after their wait; the GEMMs trigger once their weight
// producer has issued its last load, so that their successor's CTAs do not
// take bandwidth from the GEMM's last units, which finish the launch.
// Launched without the attribute (or with no predecessor kernel) both are
// no-ops.

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_sync() {
    pdl_wait();
    pdl_trigger();
}

#ifndef QMOE_PDL
#define QMOE_PDL 1
#endif

// One launch of `kernel` on `st` that may overlap its predecessor's tail.
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = QMOE_PDL ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...) == cudaSuccess ? QMOE_OK : QMOE_ERR_LAUNCH;
}

// Host-thread launch context.  The whole-layer call sets weights_early while
// it launches its GEMMs: it knows that the routing sort, which writes the
// token-tile schedule and offsets, ran at least two launches earlier, so a
// GEMM may read them, and start streaming weights, before its pdl_wait().
struct LaunchCtx {
    bool weights_early = false;
};
inline LaunchCtx& launch_ctx() {
    static thread_local LaunchCtx c;
    return c;
}

// ------------------------------------------------------------------ format decoding

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// E8M0 byte -> 2^(b-127) as fp32 (b = 0 gives the subnormal 2^-127; 255 is NaN).
__device__ __forceinline__ float e8m0_to_float(uint8_t b) {
    if (b == 0) return __uint_as_float(0x00400000u);
    if (b == 255) return __uint_as_float(0x7FC00000u);
    return __uint_as_float((uint32_t)b << 23);
}

// E2M1 nibble -> value (sign bit 3; magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6).
__device__ __forceinline__ float e2m1_to_float(uint32_t c) {
    const uint32_t m = c & 7u;
    // magnitude = m/2 for m < 4 (0, .5, 1, 1.5); 2, 3, 4, 6 for m = 4..7
    float v = (m < 4u) ? 0.5f * (float)m : (float)((m & 1u) ? 3u : 2u) * (float)(1u << ((m >> 1) - 2u));
    return (c & 8u) ? -v : v;
}

// E4M3 ("fn") byte -> value via the hardware conversion to f16x2.
__device__ __forceinline__ float e4m3_to_float(uint8_t b) {
    uint32_t h2;
    uint16_t in = b;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu)));
}

// floor(log2(a)) for finite a > 0, exact (handles fp32 subnormals).
__device__ __forceinline__ int floor_log2_pos(float a) {
    uint32_t u = __float_as_uint(a);
    int ex = (int)((u >> 23) & 0xFF);
    if (ex != 0) return ex - 127;
    return (31 - __clz(u & 0x7FFFFF)) - 149;
}

// Shared exponent of an MX block with the given amax (> 0):
// X = floor(log2 amax) - 8 (8 = emax of E4M3), clamped to the E8M0 range.
__device__ __forceinline__ int mx_block_exponent(float amax) {
    int X = floor_log2_pos(amax) - 8;
    return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// Exponent e of the power of two 2^-e that moves a row with largest
// magnitude amax into [2^14, 2^15), so that every value of the row (a bf16)
// converts to fp16 exactly unless it is below 2^-24 of the fp16 range; 0 for
// an all-zero row, clamped to [-112, 113] so that 2^e and 2^-e stay normal.
__device__ __forceinline__ int f16_row_exponent(float amax) {
    if (!(amax > 0.f)) return 0;
    const int e = floor_log2_pos(amax) - 14;
    return e < -112 ? -112 : (e > 113 ? 113 : e);
}

// 2^e as fp32 for e in [-127, 127] (exact; 2^-127 is subnormal).
__device__ __forceinline__ float exp2i(int e) {
    if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
    return __uint_as_float(0x00400000u >> (-127 - e));
}

// Two fp32 values -> two E4M3 codes (nearest even, saturating to +-448);
// `lo` lands in the low byte.
__device__ __forceinline__ uint16_t e4m3x2_from_float(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

}  // namespace qmoe
