// Top-k weighted combine (qmoe_combine).
//
// out[t][c] = bf16( sum_{j=0..k-1} w[t][j] * y[slot(t, j)][c] ), summed in fp32
// with j ascending from 0: the fixed order makes the result bit-reproducible
// ("perf(qmoe): group prefill expert matmuls", description: "preserving
// deterministic scatter order").  Each thread owns 4 consecutive columns of
// one token (16-byte loads of every y row, 8-byte bf16 stores).
#include "qmoe_common.cuh"

namespace qmoe {

__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ y, const float* __restrict__ topk_w, const int32_t* __restrict__ pair_slot,
               uint16_t* __restrict__ out, int T, int k, int H) {
    const int c4 = blockIdx.x * blockDim.x + threadIdx.x;  // column group
    const int t = blockIdx.y;
    if (c4 * 4 >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int slot = pair_slot[(int64_t)t * k + j];
        if (slot < 0) continue;
        const float w = topk_w[(int64_t)t * k + j];
        const float4 v = *reinterpret_cast<const float4*>(y + (int64_t)slot * H + c4 * 4);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    uint2 o;
    o.x = (uint32_t)float_to_bf16_bits(acc.x) | ((uint32_t)float_to_bf16_bits(acc.y) << 16);
    o.y = (uint32_t)float_to_bf16_bits(acc.z) | ((uint32_t)float_to_bf16_bits(acc.w) << 16);
    *reinterpret_cast<uint2*>(out + (int64_t)t * H + c4 * 4) = o;
}

int combine_launch(const qmoe_dims* d, const float* y, const float* topk_w, const int32_t* pair_slot, uint16_t* out,
                   cudaStream_t st) {
    if (d->T == 0) return QMOE_OK;
    dim3 grid((unsigned)ceil_div(d->H / 4, 256), (unsigned)d->T);
    combine_kernel<<<grid, 256, 0, st>>>(y, topk_w, pair_slot, out, d->T, d->k, d->H);
    return launch_status();
}

}  // namespace qmoe

extern "C" int qmoe_combine(const qmoe_dims* d, const float* y, const float* topk_w, const int32_t* pair_slot,
                            uint16_t* out_bf16, qmoe_stream_t stream) {
    using namespace qmoe;
    if (!dims_ok(d)) return QMOE_ERR_ARG;
    if (d->T > 0 && (!y || !topk_w || !pair_slot || !out_bf16 || !aligned16(y) || !aligned16(out_bf16)))
        return QMOE_ERR_ARG;
    if (d->T > 65535) return QMOE_ERR_UNSUPPORTED;
    return combine_launch(d, y, topk_w, pair_slot, out_bf16, (cudaStream_t)stream);
}
