// C-ABI entry points of the grouped expert GEMMs, status strings and the
// whole-layer call.  Argument checks run on the host before any launch.
#include "qmoe_common.cuh"
#include "mx_tiles.cuh"

namespace qmoe {
size_t align_ws_bytes(int64_t P, int E);
int align_sort_launch(int64_t P, int E, const int32_t* ids, int32_t* counts, int32_t* offsets,
                      int32_t* sorted_pair_ids, int32_t* pair_slot, int32_t* dev_status, int32_t* hist,
                      int nmax, int32_t* tile_start, cudaStream_t stream);
int quant_mx_launch(int64_t rows, int64_t cols, const uint16_t* x, uint8_t* q, uint8_t* s, cudaStream_t st);
int align_sort_launches(int64_t P);
template <typename In>
int quant_int8_launch(int64_t rows, int64_t cols, const In* x, int8_t* q, float* s, cudaStream_t st);
int combine_launch(const qmoe_dims* d, const uint16_t* y, const float* topk_w, const int32_t* pair_slot,
                   uint16_t* out, cudaStream_t st);
bool mx_tc_ok(const qmoe_dims* d, const void* w1, const void* w2);
int mx_tc_gemm1(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1, const uint8_t* w1_s,
                const int32_t* offsets, const int32_t* tile_start, uint8_t* h_tiles, int32_t* status,
                cudaStream_t st);
int mx_tc_gemm1_gather(const qmoe_dims* d, const uint8_t* x_q, const uint8_t* x_s, const int32_t* sorted,
                       const uint8_t* w1, const uint8_t* w1_s, const int32_t* offsets, const int32_t* tile_start,
                       uint8_t* h_tiles, int32_t* status, cudaStream_t st);
int mx_tc_gemm2(const qmoe_dims* d, const uint8_t* h_tiles, const uint8_t* w2, const uint8_t* w2_s,
                const int32_t* offsets, const int32_t* tile_start, uint16_t* y, int32_t* status, cudaStream_t st);
int permute_quant_mx_launch(const qmoe_dims* d, const uint16_t* x, const int32_t* pair_slot, const int32_t* offsets,
                            const int32_t* tile_start, uint8_t* tiles, cudaStream_t st);
int32_t* tile_schedule_in(void* ws, const qmoe_dims* d);
int permute_x_f16_launch(const qmoe_dims* d, const uint16_t* x, const int32_t* sorted, const int32_t* offsets,
                         const int32_t* tile_start, uint8_t* tiles, cudaStream_t st);
bool w4_tc_ok(const qmoe_dims* d);
int w4_tc_gemm1(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1, const int32_t* offsets,
                const int32_t* tile_start, uint8_t* h_tiles, int32_t* status, cudaStream_t st);
int w4_tc_gemm2(const qmoe_dims* d, const uint8_t* h16_tiles, const uint8_t* w2, const int32_t* offsets,
                const int32_t* tile_start, uint16_t* y, int32_t* status, cudaStream_t st);
bool i8_tc_ok(const qmoe_dims* d);
int i8_tc_gemm1(const qmoe_dims* d, const uint8_t* x_tiles, const int8_t* w1, const float* w1_s,
                const int32_t* offsets, const int32_t* tile_start, float* h, int32_t* dbg_acc, int32_t* status,
                cudaStream_t st);
int i8_tc_gemm2(const qmoe_dims* d, const uint8_t* h_tiles, const int8_t* w2, const float* w2_s,
                const int32_t* offsets, const int32_t* tile_start, uint16_t* y, int32_t* dbg_acc, int32_t* status,
                cudaStream_t st);
int i4_tc_gemm1(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1, const float* w1_s,
                const int32_t* offsets, const int32_t* tile_start, float* h, int32_t* dbg_acc, int32_t* status,
                cudaStream_t st);
int i4_tc_gemm2(const qmoe_dims* d, const uint8_t* h_tiles, const uint8_t* w2, const float* w2_s,
                const int32_t* offsets, const int32_t* tile_start, uint16_t* y, int32_t* dbg_acc, int32_t* status,
                cudaStream_t st);
int h_to_f16_launch(const qmoe_dims* d, const uint8_t* h_tiles, const int32_t* offsets, const int32_t* tile_start,
                    uint8_t* out, cudaStream_t st);
int quant_tiles_int8_launch(const qmoe_dims* d, int64_t K, const void* x, bool from_bf16_tokens,
                            const int32_t* sorted, const int32_t* offsets, const int32_t* tile_start, uint8_t* tiles,
                            cudaStream_t st);

static int gemm_args_ok(const qmoe_dims* d, std::initializer_list<const void*> ptrs) {
    if (!dims_ok(d)) return QMOE_ERR_ARG;
    if ((int64_t)d->T * d->k == 0) return QMOE_OK;
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return QMOE_ERR_ARG;
    return QMOE_OK;
}

}  // namespace qmoe

using namespace qmoe;

extern "C" const char* qmoe_status_str(int code) {
    switch (code) {
        case QMOE_OK: return "ok";
        case QMOE_ERR_ARG: return "invalid argument (null or misaligned pointer, bad dimension, small workspace)";
        case QMOE_ERR_UNSUPPORTED: return "shape outside the kernels' limits";
        case QMOE_ERR_LAUNCH: return "kernel launch failed";
        case QMOE_ERR_CUDA: return "CUDA runtime error";
    }
    return "unknown status";
}

extern "C" const char* qmoe_version(void) { return "qmoe-gb300 0.1 (sm_103a)"; }

extern "C" size_t qmoe_mx_tiles_bytes(const qmoe_dims* d, int64_t K) {
    if (!dims_ok(d) || K <= 0 || K % 128 != 0) return 0;
    return (size_t)mxt::buffer_bytes(d, K);
}

static bool mx_ws_ok(const qmoe_dims* d, const void* ws, size_t ws_bytes) {
    return ws && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0 && ws_bytes >= qmoe_workspace_bytes(d);
}

extern "C" int qmoe_permute_quant_mxfp8(const qmoe_dims* d, const uint16_t* x_bf16, const int32_t* pair_slot,
                                        const int32_t* offsets, uint8_t* x_tiles, const void* ws, size_t ws_bytes,
                                        qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {x_bf16, pair_slot, offsets, x_tiles});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (d->H % 128 != 0) return QMOE_ERR_UNSUPPORTED;
    return permute_quant_mx_launch(d, x_bf16, pair_slot, offsets,
                                   tile_schedule_in(const_cast<void*>(ws), d), x_tiles, (cudaStream_t)stream);
}

extern "C" int qmoe_gemm1_swiglu_mxfp4(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1,
                                       const uint8_t* w1_s, const int32_t* offsets, uint8_t* h_tiles,
                                       int32_t* dev_status, void* ws, size_t ws_bytes, qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {x_tiles, w1, w1_s, offsets, h_tiles, dev_status});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (!mx_tc_ok(d, w1, nullptr)) return QMOE_ERR_UNSUPPORTED;
    return mx_tc_gemm1(d, x_tiles, w1, w1_s, offsets, tile_schedule_in(ws, d), h_tiles, dev_status,
                       (cudaStream_t)stream);
}

extern "C" int qmoe_gemm1_swiglu_mxfp4_gather(const qmoe_dims* d, const uint8_t* x_q, const uint8_t* x_s,
                                              const int32_t* sorted_pair_ids, const uint8_t* w1, const uint8_t* w1_s,
                                              const int32_t* offsets, uint8_t* h_tiles, int32_t* dev_status, void* ws,
                                              size_t ws_bytes, qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {x_q, x_s, sorted_pair_ids, w1, w1_s, offsets, h_tiles, dev_status});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (!mx_tc_ok(d, w1, nullptr)) return QMOE_ERR_UNSUPPORTED;
    return mx_tc_gemm1_gather(d, x_q, x_s, sorted_pair_ids, w1, w1_s, offsets, tile_schedule_in(ws, d), h_tiles,
                              dev_status, (cudaStream_t)stream);
}

extern "C" int qmoe_gemm2_mxfp4(const qmoe_dims* d, const uint8_t* h_tiles, const uint8_t* w2, const uint8_t* w2_s,
                                const int32_t* offsets, uint16_t* y, int32_t* dev_status, void* ws, size_t ws_bytes,
                                qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {h_tiles, w2, w2_s, offsets, y, dev_status});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (!mx_tc_ok(d, nullptr, w2)) return QMOE_ERR_UNSUPPORTED;
    return mx_tc_gemm2(d, h_tiles, w2, w2_s, offsets, tile_schedule_in(ws, d), y, dev_status, (cudaStream_t)stream);
}

// ------------------------------------------------------------------ W4A16 (bf16 tensor cores)

extern "C" size_t qmoe_w4a16_x_tiles_bytes(const qmoe_dims* d) {
    if (!dims_ok(d) || d->H % 64 != 0) return 0;
    return (size_t)bft::x_tiles_bytes(d);
}

extern "C" size_t qmoe_w4a16_h_tiles_bytes(const qmoe_dims* d) {
    if (!dims_ok(d) || d->I % 64 != 0) return 0;
    return (size_t)bft::h_tiles_bytes(d);
}

extern "C" size_t qmoe_w4a16_h16_tiles_bytes(const qmoe_dims* d) {
    if (!dims_ok(d) || d->I % 64 != 0) return 0;
    const int nmax = mxt::nmax_for(d);
    return (size_t)(bft::blocks_bytes(d, d->I) + mxt::max_tiles(d, nmax) * nmax * 4);
}

extern "C" int qmoe_w4a16_h_to_f16(const qmoe_dims* d, const uint8_t* h_tiles, const int32_t* offsets,
                                   uint8_t* h16_tiles, const void* ws, size_t ws_bytes, qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {h_tiles, offsets, h16_tiles});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (d->I % 64 != 0) return QMOE_ERR_UNSUPPORTED;
    return h_to_f16_launch(d, h_tiles, offsets, tile_schedule_in(const_cast<void*>(ws), d), h16_tiles,
                           (cudaStream_t)stream);
}

extern "C" int qmoe_permute_x_f16(const qmoe_dims* d, const uint16_t* x_bf16, const int32_t* sorted_pair_ids,
                                 const int32_t* offsets, uint8_t* x_tiles, const void* ws, size_t ws_bytes,
                                 qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {x_bf16, sorted_pair_ids, offsets, x_tiles});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (d->H % 64 != 0) return QMOE_ERR_UNSUPPORTED;
    return permute_x_f16_launch(d, x_bf16, sorted_pair_ids, offsets, tile_schedule_in(const_cast<void*>(ws), d),
                                x_tiles, (cudaStream_t)stream);
}

extern "C" int qmoe_gemm1_swiglu_w4a16(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1,
                                       const int32_t* offsets, uint8_t* h_tiles, int32_t* dev_status, void* ws,
                                       size_t ws_bytes, qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {x_tiles, w1, offsets, h_tiles, dev_status});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (!w4_tc_ok(d)) return QMOE_ERR_UNSUPPORTED;
    return w4_tc_gemm1(d, x_tiles, w1, offsets, tile_schedule_in(ws, d), h_tiles, dev_status, (cudaStream_t)stream);
}

extern "C" int qmoe_gemm2_w4a16(const qmoe_dims* d, const uint8_t* h16_tiles, const uint8_t* w2, const int32_t* offsets,
                                uint16_t* y, int32_t* dev_status, void* ws, size_t ws_bytes, qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {h16_tiles, w2, offsets, y, dev_status});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (!w4_tc_ok(d)) return QMOE_ERR_UNSUPPORTED;
    return w4_tc_gemm2(d, h16_tiles, w2, offsets, tile_schedule_in(ws, d), y, dev_status, (cudaStream_t)stream);
}

// ------------------------------------------------------------------ W8A8 (exact int32 sums on fp16 tensor cores)

extern "C" size_t qmoe_w8a8_tiles_bytes(const qmoe_dims* d, int64_t K) {
    if (!dims_ok(d) || K <= 0 || K % 128 != 0 || K > 16384) return 0;
    const int nmax = mxt::nmax_for(d);
    const int64_t tiles = mxt::max_tiles(d, nmax);
    return (size_t)(bft::blocks_bytes(d, K) + tiles * nmax * 4 + tiles * ((nmax + 111) / 112) * (K / 128) * 4);
}

extern "C" int qmoe_permute_quant_int8(const qmoe_dims* d, const uint16_t* x_bf16, const int32_t* sorted_pair_ids,
                                       const int32_t* offsets, uint8_t* x_tiles, const void* ws, size_t ws_bytes,
                                       qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {x_bf16, sorted_pair_ids, offsets, x_tiles});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (d->H % 128 != 0 || d->H > 16384) return QMOE_ERR_UNSUPPORTED;
    return quant_tiles_int8_launch(d, d->H, x_bf16, true, sorted_pair_ids, offsets,
                                   tile_schedule_in(const_cast<void*>(ws), d), x_tiles, (cudaStream_t)stream);
}

extern "C" int qmoe_quant_tiles_int8_f32(const qmoe_dims* d, const float* h_f32, const int32_t* offsets,
                                         uint8_t* h_tiles, const void* ws, size_t ws_bytes, qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {h_f32, offsets, h_tiles});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (d->I % 128 != 0 || d->I > 16384) return QMOE_ERR_UNSUPPORTED;
    return quant_tiles_int8_launch(d, d->I, h_f32, false, nullptr, offsets,
                                   tile_schedule_in(const_cast<void*>(ws), d), h_tiles, (cudaStream_t)stream);
}

extern "C" int qmoe_gemm1_swiglu_w8a8(const qmoe_dims* d, const uint8_t* x_tiles, const int8_t* w1, const float* w1_s,
                                      const int32_t* offsets, float* h, int32_t* dbg_acc, int32_t* dev_status,
                                      void* ws, size_t ws_bytes, qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {x_tiles, w1, w1_s, offsets, h, dev_status});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (dbg_acc && !aligned16(dbg_acc)) return QMOE_ERR_ARG;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (!i8_tc_ok(d)) return QMOE_ERR_UNSUPPORTED;
    return i8_tc_gemm1(d, x_tiles, w1, w1_s, offsets, tile_schedule_in(ws, d), h, dbg_acc, dev_status,
                       (cudaStream_t)stream);
}

extern "C" int qmoe_gemm2_w8a8(const qmoe_dims* d, const uint8_t* h_tiles, const int8_t* w2, const float* w2_s,
                               const int32_t* offsets, uint16_t* y, int32_t* dbg_acc, int32_t* dev_status, void* ws,
                               size_t ws_bytes, qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {h_tiles, w2, w2_s, offsets, y, dev_status});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (dbg_acc && !aligned16(dbg_acc)) return QMOE_ERR_ARG;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (!i8_tc_ok(d)) return QMOE_ERR_UNSUPPORTED;
    return i8_tc_gemm2(d, h_tiles, w2, w2_s, offsets, tile_schedule_in(ws, d), y, dbg_acc, dev_status,
                       (cudaStream_t)stream);
}

// ------------------------------------------------------------------ W4A8 (int4 weights widened to exact integers)

extern "C" int qmoe_gemm1_swiglu_w4a8(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1, const float* w1_s,
                                      const int32_t* offsets, float* h, int32_t* dbg_acc, int32_t* dev_status,
                                      void* ws, size_t ws_bytes, qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {x_tiles, w1, w1_s, offsets, h, dev_status});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (dbg_acc && !aligned16(dbg_acc)) return QMOE_ERR_ARG;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (!i8_tc_ok(d)) return QMOE_ERR_UNSUPPORTED;
    return i4_tc_gemm1(d, x_tiles, w1, w1_s, offsets, tile_schedule_in(ws, d), h, dbg_acc, dev_status,
                       (cudaStream_t)stream);
}

extern "C" int qmoe_gemm2_w4a8(const qmoe_dims* d, const uint8_t* h_tiles, const uint8_t* w2, const float* w2_s,
                               const int32_t* offsets, uint16_t* y, int32_t* dbg_acc, int32_t* dev_status, void* ws,
                               size_t ws_bytes, qmoe_stream_t stream) {
    int rc = gemm_args_ok(d, {h_tiles, w2, w2_s, offsets, y, dev_status});
    if (rc != QMOE_OK || (int64_t)d->T * d->k == 0) return rc;
    if (dbg_acc && !aligned16(dbg_acc)) return QMOE_ERR_ARG;
    if (!mx_ws_ok(d, ws, ws_bytes)) return QMOE_ERR_ARG;
    if (!i8_tc_ok(d)) return QMOE_ERR_UNSUPPORTED;
    return i4_tc_gemm2(d, h_tiles, w2, w2_s, offsets, tile_schedule_in(ws, d), y, dbg_acc, dev_status,
                       (cudaStream_t)stream);
}

// ------------------------------------------------------------------ whole layer

// Which stage-1 input the whole-layer call gives the MXFP4 GEMM.  The
// permute writes every routed row once per pair (k expanded copies of x) and
// the GEMM streams them with bulk copies; the gathering form skips that copy
// but fetches each tile's rows once per 128-column block of h with cp.async,
// a slower path per byte.  The saved copy wins with at most four column
// blocks (I <= 512), 112- or 224-row tiles and at least 64 pairs per expert
// on average.  Measured on GB300 at H 4096, E 512, top-10 (us per step,
// permuted tiles -> gather): I 256: T 1024 243.8 -> 241.6, T 4096 368.6 ->
// 337.9, T 8192 606.7 -> 546.9; I 512: T 1024 372.6 -> 382.9, T 4096 491.3 ->
// 481.7, T 8192 814.8 -> 783.2; I 1024: T 1024 635.2 -> 684.0, T 4096 768.9 ->
// 814.0, T 8192 1188.8 -> 1209.6; 16-row tiles even or slower (I 256 T 16
// 71.5 -> 71.4).
extern "C" int qmoe_mx_layer_gathers(const qmoe_dims* d) {
    if (!dims_ok(d)) return 0;
    return (mxt::nmax_for(d) != 16 && d->I <= 512 && (int64_t)d->T * d->k >= (int64_t)64 * d->E) ? 1 : 0;
}

namespace {

struct FwdLayout {
    size_t counts, offsets, sorted, slot, xq, h, ht, y, align_ws, total;
};

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

FwdLayout fwd_layout(const qmoe_dims* d, int scheme) {
    const size_t P = (size_t)d->T * d->k, H = d->H, I = d->I, E = d->E;
    FwdLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o += up256(bytes); return at; };
    L.counts = take(4 * E);
    L.offsets = take(4 * (E + 1));
    L.sorted = take(4 * P);
    L.slot = take(4 * P);
    // schemes 2 (W8A8) and 3 (W4A8) share the integer activation path
    // MXFP4: the MX x tiles, or token-major MX x (codes [T, H], then scales [T, H/32]) when stage 1 gathers
    const size_t mx_x = qmoe_mx_layer_gathers(d) ? up256((size_t)d->T * H) + (size_t)d->T * (H / 32)
                                                 : (size_t)mxt::buffer_bytes(d, d->H);
    L.xq = take(scheme == 0 ? (size_t)bft::x_tiles_bytes(d) : (scheme == 1 ? mx_x : qmoe_w8a8_tiles_bytes(d, d->H)));
    L.h = take(scheme == 0 ? (size_t)bft::h_tiles_bytes(d)
                           : (scheme == 1 ? (size_t)mxt::buffer_bytes(d, d->I) : 4 * P * I));
    L.ht = take(scheme >= 2 ? qmoe_w8a8_tiles_bytes(d, d->I) : (scheme == 0 ? qmoe_w4a16_h16_tiles_bytes(d) : 0));
    L.y = take(2 * P * H);
    L.align_ws = take(qmoe_workspace_bytes(d));
    L.total = o;
    return L;
}

}  // namespace

extern "C" int qmoe_forward_launches(const qmoe_dims* d, int scheme) {
    if (!dims_ok(d) || scheme < 0 || scheme > 3) return 0;
    int n = align_sort_launches((int64_t)d->T * d->k);  // routing sort
    if (d->T == 0) return n;
    n += 1;                                          // activation quantisation (into tiles, or token-major)
    n += 2;                                          // the two grouped GEMMs
    if (scheme != 1) n += 1;                         // W4A16 h -> fp16 rows, or the integer intermediate pass
    n += 1;                                          // combine
    return n;
}

extern "C" size_t qmoe_forward_workspace_bytes(const qmoe_dims* d, int scheme) {
    if (!dims_ok(d) || scheme < 0 || scheme > 3) return 0;
    return fwd_layout(d, scheme).total;
}

extern "C" int qmoe_moe_forward(int scheme, const qmoe_dims* d, const uint16_t* x_bf16, const int32_t* topk_ids,
                                const float* topk_w, const void* w1, const void* w1_s, const void* w2,
                                const void* w2_s, uint16_t* out_bf16, int32_t* dev_status, void* ws, size_t ws_bytes,
                                qmoe_stream_t stream) {
    if (!dims_ok(d) || scheme < 0 || scheme > 3) return QMOE_ERR_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || !dev_status) return QMOE_ERR_ARG;
    const FwdLayout L = fwd_layout(d, scheme);
    if (ws_bytes < L.total) return QMOE_ERR_ARG;
    if (d->T > 0 && (!x_bf16 || !topk_ids || !topk_w || !w1 || !w2 || !out_bf16)) return QMOE_ERR_ARG;
    if (d->T > 0 && scheme != 0 && (!w1_s || !w2_s)) return QMOE_ERR_ARG;
    char* base = static_cast<char*>(ws);
    auto at = [&](size_t off) { return static_cast<void*>(base + off); };
    int32_t* counts = (int32_t*)at(L.counts);
    int32_t* offsets = (int32_t*)at(L.offsets);
    int32_t* sorted = (int32_t*)at(L.sorted);
    int32_t* slot = (int32_t*)at(L.slot);
    void* aws = at(L.align_ws);
    const size_t aws_bytes = qmoe_workspace_bytes(d);
    int rc = qmoe_align_sort(d, topk_ids, counts, offsets, sorted, slot, dev_status, aws, aws_bytes, stream);
    if (rc != QMOE_OK) return rc;
    if (d->T == 0) return QMOE_OK;
    uint16_t* y = (uint16_t*)at(L.y);
    // Every GEMM below is launched at least two kernels after the routing
    // sort, so it may read the schedule and stream weights before its
    // predecessor completes.
    struct EarlyWeights {
        EarlyWeights() { launch_ctx().weights_early = true; }
        ~EarlyWeights() { launch_ctx().weights_early = false; }
    } early;
    if (scheme == 0) {
        rc = qmoe_permute_x_f16(d, x_bf16, sorted, offsets, (uint8_t*)at(L.xq), aws, aws_bytes, stream);
        if (rc == QMOE_OK)
            rc = qmoe_gemm1_swiglu_w4a16(d, (const uint8_t*)at(L.xq), (const uint8_t*)w1, offsets, (uint8_t*)at(L.h),
                                         dev_status, aws, aws_bytes, stream);
        if (rc == QMOE_OK)
            rc = qmoe_w4a16_h_to_f16(d, (const uint8_t*)at(L.h), offsets, (uint8_t*)at(L.ht), aws, aws_bytes, stream);
        if (rc == QMOE_OK)
            rc = qmoe_gemm2_w4a16(d, (const uint8_t*)at(L.ht), (const uint8_t*)w2, offsets, y, dev_status, aws,
                                  aws_bytes, stream);
    } else if (scheme == 1) {
        uint8_t* xq = (uint8_t*)at(L.xq);
        if (qmoe_mx_layer_gathers(d)) {
            // x quantised once per token (token-major); stage 1 gathers each routed row from it
            uint8_t* xs = xq + up256((size_t)d->T * d->H);
            rc = qmoe_quant_act_mxfp8(d->T, d->H, x_bf16, xq, xs, stream);
            if (rc == QMOE_OK)
                rc = qmoe_gemm1_swiglu_mxfp4_gather(d, xq, xs, sorted, (const uint8_t*)w1, (const uint8_t*)w1_s,
                                                    offsets, (uint8_t*)at(L.h), dev_status, aws, aws_bytes, stream);
        } else {
            rc = qmoe_permute_quant_mxfp8(d, x_bf16, slot, offsets, xq, aws, aws_bytes, stream);
            if (rc == QMOE_OK)
                rc = qmoe_gemm1_swiglu_mxfp4(d, xq, (const uint8_t*)w1, (const uint8_t*)w1_s, offsets,
                                             (uint8_t*)at(L.h), dev_status, aws, aws_bytes, stream);
        }
        if (rc == QMOE_OK)
            rc = qmoe_gemm2_mxfp4(d, (const uint8_t*)at(L.h), (const uint8_t*)w2, (const uint8_t*)w2_s, offsets, y,
                                  dev_status, aws, aws_bytes, stream);
    } else {
        rc = qmoe_permute_quant_int8(d, x_bf16, sorted, offsets, (uint8_t*)at(L.xq), aws, aws_bytes, stream);
        if (rc == QMOE_OK)
            rc = scheme == 2 ? qmoe_gemm1_swiglu_w8a8(d, (const uint8_t*)at(L.xq), (const int8_t*)w1, (const float*)w1_s,
                                                      offsets, (float*)at(L.h), nullptr, dev_status, aws, aws_bytes,
                                                      stream)
                             : qmoe_gemm1_swiglu_w4a8(d, (const uint8_t*)at(L.xq), (const uint8_t*)w1, (const float*)w1_s,
                                                      offsets, (float*)at(L.h), nullptr, dev_status, aws, aws_bytes,
                                                      stream);
        if (rc == QMOE_OK)
            rc = qmoe_quant_tiles_int8_f32(d, (const float*)at(L.h), offsets, (uint8_t*)at(L.ht), aws, aws_bytes,
                                           stream);
        if (rc == QMOE_OK)
            rc = scheme == 2 ? qmoe_gemm2_w8a8(d, (const uint8_t*)at(L.ht), (const int8_t*)w2, (const float*)w2_s,
                                               offsets, y, nullptr, dev_status, aws, aws_bytes, stream)
                             : qmoe_gemm2_w4a8(d, (const uint8_t*)at(L.ht), (const uint8_t*)w2, (const float*)w2_s,
                                               offsets, y, nullptr, dev_status, aws, aws_bytes, stream);
    }
    if (rc != QMOE_OK) return rc;
    return qmoe_combine(d, y, topk_w, slot, out_bf16, stream);
}
