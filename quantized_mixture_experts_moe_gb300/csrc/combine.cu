// Top-k weighted combine (qmoe_combine).
//
// out[t][c] = bf16( sum_{j=0..k-1} w[t][j] * y[slot(t, j)][c] ), summed in fp32
// with j ascending from 0: the fixed order makes the result bit-reproducible
// ("perf(qmoe): group prefill expert matmuls", description: the scatter back
// keeps a deterministic order).  y rows are bf16.  Each thread owns 8
// consecutive columns of one token (16-byte loads of every y row, 16-byte
// bf16 stores).  y is read exactly once, so its loads are marked evict-first
// (it is larger than L2 at prefill sizes); the output keeps the default
// policy, since the caller reads it next.
#include "qmoe_common.cuh"

namespace qmoe {

__global__ void __launch_bounds__(128)
combine_kernel(const uint16_t* __restrict__ y, const float* __restrict__ topk_w, const int32_t* __restrict__ pair_slot,
               uint16_t* __restrict__ out, int T, int k, int H) {
    const int c8 = blockIdx.x * blockDim.x + threadIdx.x;  // column group of 8
    const int t = blockIdx.y;
    pdl_sync();
    if (c8 * 8 >= H) return;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    // ceil(k/8) groups of equal size (at most 8 pairs): a group's slots and
    // weights, then its y rows, are loaded together (independent loads in
    // flight), then summed in j order.  Equal groups keep as many loads in
    // flight in the last group as in the first (k = 10: 5 + 5, not 8 + 2).
    const int groups = (k + 7) / 8;
    const int gsz = (k + groups - 1) / groups;
    for (int j0 = 0; j0 < k; j0 += gsz) {
        int slot[8];
        float w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const bool in = j < gsz && j0 + j < k;
            slot[j] = in ? pair_slot[(int64_t)t * k + j0 + j] : -1;
            w[j] = in ? topk_w[(int64_t)t * k + j0 + j] : 0.f;
        }
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = slot[j] >= 0 ? __ldcs(reinterpret_cast<const uint4*>(y + (int64_t)slot[j] * H + c8 * 8)) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (slot[j] < 0) continue;
            const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = fmaf(w[j], __uint_as_float(u[i] << 16), acc[2 * i]);
                acc[2 * i + 1] = fmaf(w[j], __uint_as_float(u[i] & 0xFFFF0000u), acc[2 * i + 1]);
            }
        }
    }
    uint4 o;
    o.x = (uint32_t)float_to_bf16_bits(acc[0]) | ((uint32_t)float_to_bf16_bits(acc[1]) << 16);
    o.y = (uint32_t)float_to_bf16_bits(acc[2]) | ((uint32_t)float_to_bf16_bits(acc[3]) << 16);
    o.z = (uint32_t)float_to_bf16_bits(acc[4]) | ((uint32_t)float_to_bf16_bits(acc[5]) << 16);
    o.w = (uint32_t)float_to_bf16_bits(acc[6]) | ((uint32_t)float_to_bf16_bits(acc[7]) << 16);
    *reinterpret_cast<uint4*>(out + (int64_t)t * H + c8 * 8) = o;
}

int combine_launch(const qmoe_dims* d, const uint16_t* y, const float* topk_w, const int32_t* pair_slot,
                   uint16_t* out, cudaStream_t st) {
    if (d->T == 0) return QMOE_OK;
    // 128-thread CTAs: at T = 4096, H = 4096 they measured 61.6 us against
    // 63.6 us for 256 threads (finer tail of the last wave)
    dim3 grid((unsigned)ceil_div(d->H / 8, 128), (unsigned)d->T);
    return launch_pdl(combine_kernel, grid, 128, 0, st, y, topk_w, pair_slot, out, d->T, d->k, d->H);
}

}  // namespace qmoe

extern "C" int qmoe_combine(const qmoe_dims* d, const uint16_t* y, const float* topk_w, const int32_t* pair_slot,
                            uint16_t* out_bf16, qmoe_stream_t stream) {
    using namespace qmoe;
    if (!dims_ok(d)) return QMOE_ERR_ARG;
    if (d->T > 0 && (!y || !topk_w || !pair_slot || !out_bf16 || !aligned16(y) || !aligned16(out_bf16)))
        return QMOE_ERR_ARG;
    if (d->T > 65535) return QMOE_ERR_UNSUPPORTED;
    return combine_launch(d, y, topk_w, pair_slot, out_bf16, (cudaStream_t)stream);
}
