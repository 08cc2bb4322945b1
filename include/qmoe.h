/*
 * qmoe.h -- C ABI of the GB300 (sm_103a) quantized Mixture-of-Experts expert
 * path: routed top-k pairs -> expert-sorted order -> grouped gate/up GEMM with
 * fused SwiGLU -> grouped down GEMM over packed low-bit expert weights ->
 * top-k-weighted combine in a fixed order.
 *
 * Sources the operations follow:
 *   [hip-ep]  "perf(qmoe): group prefill expert matmuls" -- description:
 *             grouped expert projections over symmetric int4 weights, one
 *             launch for all experts, deterministic scatter order.
 *   [gfx1151] "Evaluate native IU4/IU8 WMMA for grouped-INT MoE prefill on
 *             gfx1151" -- Problem (dequantise-then-dot for W4A16, decode is
 *             GEMV-like), Constraint (int8 x int8 -> int32 needs quantised
 *             activations: W8A8).
 *   [aiter]   the tuned grouped-fmoe config page for an MXFP4 model on
 *             gfx1250 -- Changes (fp8 activations, MXFP4 weights, two-stage
 *             grouped kernel), Test Plan (stage1/stage2 tiles, rel L2 check,
 *             K tiles larger than inter_dim excluded).
 *
 * Notation: T tokens, k = top_k, P = T*k routed pairs (pair p = t*k + j),
 * H hidden size, I intermediate size, E experts.  A "slot" is a position in
 * expert-sorted order; slot-ordered buffers hold one row per valid pair.
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers unless stated otherwise.  The
 *     caller owns every buffer, including the workspace; the library never
 *     allocates, frees or synchronises.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *   - Host-side checks run before any launch: a NULL pointer, a dimension
 *     <= 0 (T may be 0), H or I not a multiple of 32, or a pointer not
 *     16-byte aligned returns QMOE_ERR_ARG; shapes beyond the kernels'
 *     limits return QMOE_ERR_UNSUPPORTED; a failed launch returns
 *     QMOE_ERR_LAUNCH.  Nothing is launched after an error.
 *   - Device-side errors never trap: a routing id outside [0, E) sets bit
 *     QMOE_DEV_BAD_EXPERT_ID of *dev_status (which the caller zeroes before
 *     the first call and reads after synchronising); that pair then takes no
 *     slot and contributes nothing to the output.  A tensor-core kernel whose
 *     pipeline wait exceeds its time limit sets QMOE_DEV_WAIT_TIMEOUT, stops
 *     and releases its resources; its outputs are then undefined.
 *   - Calls on different streams are independent when they use different
 *     output and workspace buffers.
 *
 * Storage formats (K = the reduction axis, always contiguous):
 *   bf16      uint16 bit patterns.
 *   int4      W [rows, K/2] bytes; element 2i in the low nibble of byte i,
 *             2i+1 in the high nibble; stored n = q + 8, value (n - 8) * s;
 *             scales fp16 [rows, K/32].  The W4A16 GEMMs take codes and
 *             scales pre-packed together (qmoe_prepack_int4_weights).
 *   E2M1      same nibble order; OCP MX element encoding; scales E8M0
 *             (value 2^(b-127)), one per 32 K elements.  The MXFP4 GEMMs take
 *             weights and scales pre-packed (qmoe_prepack_fp4_weights,
 *             qmoe_prepack_mx_scales).
 *   E4M3      OCP "fn" fp8 (max 448, no infinities).
 *   int8      W int8 [rows, K], fp32 scale per output row.
 * Weight tensors: W1 [E, 2I, H] (rows 0..I-1 gate, I..2I-1 up), W2 [E, H, I].
 */
#ifndef QMOE_H
#define QMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* qmoe_stream_t;

typedef enum {
    QMOE_OK = 0,
    QMOE_ERR_ARG = -1,
    QMOE_ERR_UNSUPPORTED = -2,
    QMOE_ERR_LAUNCH = -3,
    QMOE_ERR_CUDA = -4
} qmoe_status;

/* Bits of the device status word. */
enum { QMOE_DEV_BAD_EXPERT_ID = 1, QMOE_DEV_WAIT_TIMEOUT = 2 };

typedef struct {
    int32_t T, k, H, I, E;
} qmoe_dims;

/* Human-readable name of a qmoe_status code (static string). */
const char* qmoe_status_str(int code);

/* Library version string (static). */
const char* qmoe_version(void);

/* ---------------------------------------------------------------- token-tile table
 *
 * Every call below cuts each expert's slots into token tiles of NMAX = 16, 112
 * or 224 rows (the activation tile layouts, the tile schedule qmoe_align_sort
 * writes, the GEMMs' work units).  Without rules NMAX is 224 when T*k > 96*E,
 * else 112.  A tuned table (the aiter tuned grouped-fmoe page, Changes: one
 * configuration row per model shape and token bucket) replaces that choice:
 *
 * qmoe_tile_rule -- matches dims with H, I, E, k equal to the rule's (0 = any)
 *   and t_min <= T <= t_max; nmax is 16, 112 or 224 (16 shrinks each
 *   pipeline slot of the MXFP4 GEMMs, so small batches keep more weight
 *   loads in flight).
 * qmoe_set_tile_rules -- replaces the table with rules[0..n) (n = 0 clears it);
 *   the first matching rule wins.  QMOE_ERR_ARG for a bad rule (table
 *   unchanged).  Host state shared by the process: set it before sizing
 *   buffers and workspaces for a shape, and not while calls for that shape are
 *   in flight, since every size and schedule of the shape follows NMAX.
 * qmoe_tile_nmax -- the NMAX the library uses for *d. */
typedef struct {
    int32_t H, I, E, k;
    int64_t t_min, t_max;
    int32_t nmax;
    int32_t reserved;
} qmoe_tile_rule;
int qmoe_set_tile_rules(const qmoe_tile_rule* rules, int n);
int qmoe_tile_nmax(const qmoe_dims* d);

/* ---------------------------------------------------------------- routing
 *
 * Bytes of device workspace the routing and GEMM calls need for dims *d
 * (scratch for per-chunk histograms, the GEMM tile schedule and each slot's
 * row in the token tiles). */
size_t qmoe_workspace_bytes(const qmoe_dims* d);

/* qmoe_align_sort -- expert-sorted permutation of the routed pairs.
 * [hip-ep] description (all experts grouped into one launch, the scatter
 * back kept in a deterministic order); [aiter] Changes (two-stage grouped
 * kernel over sorted tokens).
 *
 * in   topk_ids        int32 [T, k], expert id of pair p = t*k + j
 * out  counts          int32 [E], pairs routed to each expert
 * out  offsets         int32 [E+1], exclusive prefix sum of counts;
 *                      offsets[E] = number of valid pairs
 * out  sorted_pair_ids int32 [P]; slot s -> pair id, ascending p within an
 *                      expert (a stable sort); slots >= offsets[E] hold -1
 * out  pair_slot       int32 [P]; pair id -> slot, -1 for an invalid id
 * i/o  dev_status      int32 [1]; bit QMOE_DEV_BAD_EXPERT_ID is OR-ed in
 * ws   workspace of qmoe_workspace_bytes(d) bytes, 256-byte aligned; besides
 *      scratch it receives the token-tile schedule and each slot's token-tile
 *      row, which the permute, intermediate and GEMM calls read
 * The result is bit-identical run to run (no atomics decide an order). */
int qmoe_align_sort(const qmoe_dims* d, const int32_t* topk_ids, int32_t* counts, int32_t* offsets,
                    int32_t* sorted_pair_ids, int32_t* pair_slot, int32_t* dev_status, void* ws,
                    size_t ws_bytes, qmoe_stream_t stream);

/* qmoe_align_sort_static_scratch -- the same sort as qmoe_align_sort, for
 * callers that cannot allocate device memory.  The source pages have no
 * counterpart to this call; it exists for integrations where cudaMalloc is
 * not available when tokens are routed: a host framework that owns every
 * device allocation through its own pool, a plugin that may not allocate
 * after start-up, or a latency path where allocating is forbidden.
 *
 * The caller still passes every input and output (same meaning and layout as
 * qmoe_align_sort); the histogram scratch is a fixed array of
 * QMOE_STATIC_SCRATCH_BYTES inside the library, present on every GPU that
 * loads the library until the process exits.  No cudaMalloc, cudaFree or
 * other allocating call is made.
 *
 * Limits: E <= 4096 and ceil(T*k / 2048) * E * 4 <= QMOE_STATIC_SCRATCH_BYTES
 * (for example T*k <= 81920 with E = 512 uses 80 KiB); larger shapes return
 * QMOE_ERR_UNSUPPORTED before any launch -- use qmoe_align_sort with a
 * workspace for them.
 *
 * The first call on a device looks up the array's device address on the
 * current device (kept once it succeeds; a failed lookup returns
 * QMOE_ERR_CUDA and is tried again on the next call).  With lazy module
 * loading (the CUDA default) that lookup is also what loads the library's
 * device code onto the GPU and places the array there, so the first call is
 * not itself free of allocation: make it once per device at start-up, before
 * any region that must not allocate and before any stream capture.  Later
 * calls allocate nothing.  Every call on a device shares the one array and it keeps the last
 * call's contents; nothing in it needs to start at zero (each call rewrites
 * all it reads).  Calls whose executions overlap on the GPU (different
 * streams, or different host threads) race on the array: serialise them. */
#define QMOE_STATIC_SCRATCH_BYTES (1u << 20)
int qmoe_align_sort_static_scratch(const qmoe_dims* d, const int32_t* topk_ids, int32_t* counts, int32_t* offsets,
                                   int32_t* sorted_pair_ids, int32_t* pair_slot, int32_t* dev_status,
                                   qmoe_stream_t stream);

/* ---------------------------------------------------------------- activation quantisation
 *
 * qmoe_quant_act_mxfp8 -- bf16 rows to E4M3 codes with one E8M0 scale per 32
 * consecutive columns (the fp8 activations of [aiter] Changes).  Per block:
 * X = 2^(floor(log2 amax) - 8), code = nearest-even E4M3 of v / X saturated
 * to +-448; amax = 0 gives scale byte 127 and zero codes (OCP MX v1.0).
 * in x_bf16 [rows, cols]; out x_q uint8 [rows, cols], x_s uint8 [rows, cols/32].
 * cols must be a multiple of 32. */
int qmoe_quant_act_mxfp8(int64_t rows, int64_t cols, const uint16_t* x_bf16, uint8_t* x_q, uint8_t* x_s,
                         qmoe_stream_t stream);

/* MX activation tiles -- the layout in which the MXFP4 GEMMs take their
 * activations (x for stage 1, h for stage 2).  The valid slots of each expert
 * are cut into token tiles of NMAX rows (NMAX = qmoe_tile_nmax(d), see the
 * token-tile table; tile_start = prefix over experts of ceil(count / NMAX),
 * kept by qmoe_align_sort in its workspace).  For reduction length K the buffer holds,
 * per (tile t, K step kt of 128), a block of NMAX*128 + ceil(NMAX/128)*512
 * bytes at ((t * K/128) + kt) * that size:
 *   row r's 128 E4M3 codes at r*128, 16-byte chunk c at ((c ^ (r % 8)) * 16);
 *   then the E8M0 scales, row r / block b (0..3 of the step) at
 *   NMAX*128 + (r/128)*512 + 16*(r%32) + 4*((r%128)/32) + b.
 * Rows past a tile's token count are unspecified.
 *
 * qmoe_mx_tiles_bytes -- bytes of such a buffer for dims *d and length K. */
size_t qmoe_mx_tiles_bytes(const qmoe_dims* d, int64_t K);

/* qmoe_permute_quant_mxfp8 -- the expert-sorted permutation of the routed
 * activations and their MX quantisation (rule of qmoe_quant_act_mxfp8) in one
 * pass: for every pair p = t*k + j with pair_slot[p] >= 0 (the inverse
 * permutation from qmoe_align_sort), slot pair_slot[p] of its expert gets the
 * codes of token t, written as MX activation tiles with K = H.  Each token
 * row is read and quantised once and written to its k slots.
 * ws = the workspace qmoe_align_sort filled for this routing; the kernel
 * reads each pair's token-tile row from it (pair_slot and offsets must be
 * that call's outputs). */
int qmoe_permute_quant_mxfp8(const qmoe_dims* d, const uint16_t* x_bf16, const int32_t* pair_slot,
                             const int32_t* offsets, uint8_t* x_tiles, const void* ws, size_t ws_bytes,
                             qmoe_stream_t stream);

/* W4A16 activation tiles -- the layout in which the W4A16 GEMMs take their
 * activations: the token tiles of the MX layout above (same NMAX and
 * tile_start), per (tile t, K step kt of 64 elements) one block of NMAX*128
 * bytes at ((t * K/64) + kt) * NMAX*128, row r's 64 16-bit values at r*128
 * with 16-byte chunk c at ((c ^ (r % 8)) * 16); after the blocks a per-row
 * tail of fp32 values.  Two kinds:
 *   x tiles (K = H, stage-1 input): fp16 values v * 2^-e_r, where 2^-e_r is
 *     the power of two that moves the row's largest |v| into [2^14, 2^15)
 *     (e_r = 0 for a zero row; exact for bf16 inputs); tail: 2^e_r at
 *     (t*NMAX + r).  qmoe_w4a16_x_tiles_bytes(d) bytes.
 *   h tiles (K = I, stage-1 output / stage-2 input): bf16 values; tail: the
 *     largest |h| of each 32-column group at ((t*NMAX + r) * I/32 + g).
 *     qmoe_w4a16_h_tiles_bytes(d) bytes.
 * Rows past a tile's token count are unspecified. */
size_t qmoe_w4a16_x_tiles_bytes(const qmoe_dims* d);
size_t qmoe_w4a16_h_tiles_bytes(const qmoe_dims* d);

/* h16 tiles (K = I, stage-2 input): the x-tile form of h -- fp16 values
 * h * 2^-e_r with e_r chosen from the row's largest |h| as for x tiles, tail
 * 2^e_r at (t*NMAX + r).  qmoe_w4a16_h16_tiles_bytes(d) bytes (0 unless
 * I % 64 == 0).
 * qmoe_w4a16_h_to_f16 -- h tiles (from qmoe_gemm1_swiglu_w4a16) -> h16 tiles,
 * exactly for rows whose values stay within fp16's range after the scaling,
 * reading the group maxima of the h tail.  The input is not modified.  ws =
 * the workspace qmoe_align_sort filled for this routing. */
size_t qmoe_w4a16_h16_tiles_bytes(const qmoe_dims* d);
int qmoe_w4a16_h_to_f16(const qmoe_dims* d, const uint8_t* h_tiles, const int32_t* offsets, uint8_t* h16_tiles,
                        const void* ws, size_t ws_bytes, qmoe_stream_t stream);

/* qmoe_permute_x_f16 -- the expert-sorted permutation of the routed bf16
 * activations, written as W4A16 x tiles: slot s of expert e gets row
 * sorted_pair_ids[s] / k of x_bf16 [T, H] ([hip-ep] description: one grouped
 * launch over all experts' routed tokens).  H % 64 == 0.  ws = the workspace
 * qmoe_align_sort filled for this routing. */
int qmoe_permute_x_f16(const qmoe_dims* d, const uint16_t* x_bf16, const int32_t* sorted_pair_ids,
                       const int32_t* offsets, uint8_t* x_tiles, const void* ws, size_t ws_bytes,
                       qmoe_stream_t stream);

/* qmoe_quant_rows_int8_{bf16,f32} -- per-row symmetric int8 quantisation,
 * the activation-quantised W8A8 scheme of [gfx1151] Constraint: s = amax/127
 * (1 when amax = 0), q = clamp(rint(v / s), -127, 127), all in fp32.
 * in x [rows, cols] (bf16 bits or fp32); out q int8 [rows, cols], s fp32 [rows]. */
int qmoe_quant_rows_int8_bf16(int64_t rows, int64_t cols, const uint16_t* x, int8_t* q, float* s,
                              qmoe_stream_t stream);
int qmoe_quant_rows_int8_f32(int64_t rows, int64_t cols, const float* x, int8_t* q, float* s,
                             qmoe_stream_t stream);

/* W8A8 activation tiles -- the layout in which the W8A8 GEMMs take their
 * activations: the blocks of the W4A16 tiles above (same NMAX, tile_start,
 * 128-byte rows of 64 fp16 values, chunk swizzle), each value the fp16 equal
 * to an int8 code (exact); then a per-row tail of one fp32 scale s at
 * (t*NMAX + r); then, for each 112-row part h of a tile (ceil(NMAX/112)
 * parts; a 16-row tile is one short part) and each 128-element K step j, the
 * int32 max over the part's rows of sum |code| over the step, at
 * ((t*ceil(NMAX/112) + h) * K/128 + j): the GEMMs
 * bound their partial sums with it.  Rows past a tile's token count are
 * unspecified.
 * qmoe_w8a8_tiles_bytes -- bytes of such a buffer for dims *d and length K
 * (K % 128 == 0 and K <= 16384; 0 otherwise). */
size_t qmoe_w8a8_tiles_bytes(const qmoe_dims* d, int64_t K);

/* qmoe_permute_quant_int8 -- the expert-sorted permutation of the routed
 * activations and their per-token int8 quantisation (the rule of
 * qmoe_quant_rows_int8_bf16 applied to each token row of x_bf16 [T, H]) in
 * one pass: slot s gets the codes of token sorted_pair_ids[s] / k and its
 * scale, written as W8A8 tiles with K = H ([gfx1151] Constraint: W8A8 needs
 * quantised activations).  Each token row is read and quantised once and
 * written to its k slots.  H % 128 == 0, H <= 16384.  ws = the workspace
 * qmoe_align_sort filled for this routing; the kernel reads each pair's
 * token-tile row from it (sorted_pair_ids and offsets must be that call's
 * outputs). */
int qmoe_permute_quant_int8(const qmoe_dims* d, const uint16_t* x_bf16, const int32_t* sorted_pair_ids,
                            const int32_t* offsets, uint8_t* x_tiles, const void* ws, size_t ws_bytes,
                            qmoe_stream_t stream);

/* qmoe_quant_tiles_int8_f32 -- the W8A8 intermediate quantisation: each slot
 * row of h_f32 [P, I] (slot order, from qmoe_gemm1_swiglu_w8a8) quantised
 * with the rule of qmoe_quant_rows_int8_f32 and written as W8A8 tiles with
 * K = I.  I % 128 == 0, I <= 16384.  ws as above. */
int qmoe_quant_tiles_int8_f32(const qmoe_dims* d, const float* h_f32, const int32_t* offsets, uint8_t* h_tiles,
                              const void* ws, size_t ws_bytes, qmoe_stream_t stream);

/* ---------------------------------------------------------------- weight preparation
 *
 * qmoe_prepack_mx_scales -- one-time rearrangement of E8M0 weight scales
 * [rows, K/32] (row-major, one byte per 32 K elements) into the order the
 * block-scaled tensor-core MMA consumes: 512-byte atoms, one per (128-row
 * tile, group of 4 scale blocks), group index fastest; inside an atom, row r
 * (0..127) and block b (0..3) at byte 16*(r%32) + 4*(r/32) + b.  Padding rows
 * and blocks hold 127 (scale 1).  The MXFP4 GEMMs take their weight scales in
 * this form.  Output size: qmoe_mx_scales_packed_bytes(rows, K) bytes,
 * 16-byte aligned.  No counterpart on the pages: it is a storage-order
 * choice for this hardware, like any weight repacking at load time. */
size_t qmoe_mx_scales_packed_bytes(int64_t rows, int64_t K);
int qmoe_prepack_mx_scales(int64_t rows, int64_t K, const uint8_t* s_rowmajor, uint8_t* s_packed, qmoe_stream_t stream);

/* qmoe_prepack_fp4_weights -- one-time rearrangement of packed 4-bit weights
 * [rows, K/2 bytes] (element 2i in the low nibble of byte i) into tile-major
 * order: every 128-row x 128-element tile becomes one contiguous 8 KiB block,
 * tile (rt, kt) at (rt * ceil(K/128) + kt) * 8192, tile row r at r * 64 in it,
 * nibble order unchanged; padding is zero.  The MXFP4 GEMMs take their E2M1
 * weights in this form (a tile is then one contiguous read from HBM).
 * Output size: qmoe_fp4_weights_packed_bytes(rows, K), 32-byte aligned.  No
 * counterpart on the pages (a storage-order choice, made at load time). */
size_t qmoe_fp4_weights_packed_bytes(int64_t rows, int64_t K);
int qmoe_prepack_fp4_weights(int64_t rows, int64_t K, const uint8_t* w_rowmajor, uint8_t* w_packed,
                             qmoe_stream_t stream);

/* qmoe_prepack_int4_weights -- one-time rearrangement of symmetric int4
 * weights (codes [rows, K/2] bytes, nibble order as above, n = q + 8) and
 * their fp16 scales [rows, K/32] into the blocks the W4A16 GEMMs read: per
 * (128-row tile rt, 64-element K step kt) one 4608-byte block at
 * (rt * ceil(K/64) + kt) * 4608 holding row r's 32 code bytes at r*32 and
 * then, at 4096 + r*4, its two scales of the step as fp16(s * 2^p_r), where
 * 2^p_r is the power of two that moves the row's largest |s| into
 * [2^10, 2^11) (p_r = 0 for an all-zero row).  After all blocks, one fp32
 * 2^-p_r per row, ceil(rows/128)*128 of them.  Inside each 32-bit code word
 * (8 elements) the nibbles are reordered so that nibble j holds element 2j
 * and nibble 4+j element 2j+1 (j = 0..3).  Padding codes are 8 (value 0),
 * padding scales 0, padding rows' factors 1.  K % 32 == 0; packed 16-byte
 * aligned, codes 4-byte aligned.  Output size:
 * qmoe_int4_weights_packed_bytes(rows, K).  No counterpart on the pages (a
 * storage-order choice, made at load time). */
size_t qmoe_int4_weights_packed_bytes(int64_t rows, int64_t K);
int qmoe_prepack_int4_weights(int64_t rows, int64_t K, const uint8_t* w_rowmajor, const uint16_t* s_fp16,
                              uint8_t* packed, qmoe_stream_t stream);

/* ---------------------------------------------------------------- stage 1: gate/up + SwiGLU
 *
 * For every expert e and slot s in [offsets[e], offsets[e+1]), with
 * a = the activation row of token sorted_pair_ids[s] / k:
 *   g[n] = W1[e][n] . a,  u[n] = W1[e][I+n] . a,  h[s][n] = silu(g[n]) * u[n]
 * for n < I, silu(v) = v / (1 + exp(-v)); then h is quantised per scheme.
 * [hip-ep] description (grouped projections, all experts in one launch);
 * [aiter] Changes/Test Plan (stage 1 of the grouped a8w4 kernel).
 * Only slots < offsets[E] are written.
 *
 * W4A16 (tensor cores, fp16 MMAs; needs H % 256 == 0, I % 128 == 0,
 *        E <= 512): x_tiles = qmoe_permute_x_f16 output (K = H); w1 =
 *        qmoe_prepack_int4_weights of the int4 [E*2I, H/2] codes and their
 *        fp16 [E*2I, H/32] scales.  Each weight is dequantised on chip
 *        ([gfx1151] Problem: dequantise, then a 16-bit dot) to
 *        fp16((n - 8) * s * 2^p_r), one rounding of relative size <= 2^-11;
 *        products are summed in fp32 and the sums scaled back by
 *        2^(e_r - p_r), exactly; out h_tiles: h rounded to bf16 (nearest
 *        even), stored as W4A16 h tiles.  ws = the workspace that
 *        qmoe_align_sort filled for this routing. */
int qmoe_gemm1_swiglu_w4a16(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1, const int32_t* offsets,
                            uint8_t* h_tiles, int32_t* dev_status, void* ws, size_t ws_bytes, qmoe_stream_t stream);

/* MXFP4 x FP8 (tensor cores; needs H % 256 == 0, I % 128 == 0, E <= 512):
 *        x_tiles = qmoe_permute_quant_mxfp8 output (MX activation tiles, K = H);
 *        w1 = qmoe_prepack_fp4_weights of the E2M1 [E*2I, H/2] bytes (32-byte
 *        aligned); w1_s = qmoe_prepack_mx_scales of the E8M0 [E*2I, H/32] scales;
 *        out h_tiles: the fp32 h quantised with the rule of
 *        qmoe_quant_act_mxfp8 along I, stored as MX activation tiles (K = I),
 *        qmoe_mx_tiles_bytes(d, I) bytes.  ws = the workspace that
 *        qmoe_align_sort filled for this routing (it holds the tile schedule). */
int qmoe_gemm1_swiglu_mxfp4(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1, const uint8_t* w1_s,
                            const int32_t* offsets, uint8_t* h_tiles, int32_t* dev_status, void* ws,
                            size_t ws_bytes, qmoe_stream_t stream);

/* MXFP4 x FP8, gathering form: the same stage 1 (same weights, output, rules
 *        and limits) reading the activations token-major instead of from
 *        permuted tiles, as x plus the routing sort's order.  x_q uint8 [T, H]
 *        and x_s uint8 [T, H/32] = qmoe_quant_act_mxfp8 of x_bf16 [T, H]
 *        (16-byte aligned); sorted_pair_ids = the qmoe_align_sort output for
 *        this routing.  Row r of expert e's slots (slot offsets[e] + r) takes
 *        token sorted_pair_ids[offsets[e] + r] / k (an entry outside [0, T*k)
 *        is not read, and that row's output is undefined); the kernel copies that
 *        token's codes and scales into each pipeline step, so no expanded copy
 *        of x is written.  The result equals qmoe_gemm1_swiglu_mxfp4 on the
 *        qmoe_permute_quant_mxfp8 tiles of the same x, bit for bit ([aiter]
 *        Changes: fp8 activations into the stage-1 grouped GEMM). */
int qmoe_gemm1_swiglu_mxfp4_gather(const qmoe_dims* d, const uint8_t* x_q, const uint8_t* x_s,
                                   const int32_t* sorted_pair_ids, const uint8_t* w1, const uint8_t* w1_s,
                                   const int32_t* offsets, uint8_t* h_tiles, int32_t* dev_status, void* ws,
                                   size_t ws_bytes, qmoe_stream_t stream);

/* qmoe_mx_layer_gathers -- 1 if qmoe_moe_forward runs MXFP4 stage 1 in the
 *        gathering form for these dims (qmoe_quant_act_mxfp8, then
 *        qmoe_gemm1_swiglu_mxfp4_gather), 0 if through qmoe_permute_quant_mxfp8
 *        and qmoe_gemm1_swiglu_mxfp4; 0 for invalid dims.  Host only.  The two
 *        give the same bits; the choice is by speed: the gathering form when
 *        the token tile has 112 or 224 rows, I <= 512 and T*k >= 64*E. */
int qmoe_mx_layer_gathers(const qmoe_dims* d);

/* qmoe_forward_launches -- how many kernels one qmoe_moe_forward call with
 *        these dims and scheme launches (0 for invalid arguments).  Host only.
 *        The routing sort is one launch up to 2048 pairs and two above; then
 *        the activation quantisation, the two GEMMs, the W4A16 / integer
 *        intermediate pass, and the combine. */
int qmoe_forward_launches(const qmoe_dims* d, int scheme);

/* W8A8 (tensor cores; needs H % 256 == 0, I % 128 == 0, H and I <= 16384,
 *        E <= 512): x_tiles = qmoe_permute_quant_int8 output (K = H);
 *        w1 int8 [E, 2I, H] (row-major, as given; 16-byte aligned);
 *        w1_s fp32 [E, 2I].  The int8 x int8 products are summed exactly in
 *        int32 ([gfx1151] Constraint): the tensor cores take the codes as
 *        exact fp16 values and accumulate in fp32, and the epilogue carries
 *        the sum on in integers whenever the tiles' step maxima say a fp32
 *        partial sum could otherwise reach 2^24.  g = ((float)acc * s_x) *
 *        w1_s[e][n] in fp32, likewise u; out h fp32 [P, I] in slot order;
 *        dbg_acc (nullable, 16-byte aligned) int32 [P, 2I] receives the exact
 *        gate/up sums. */
int qmoe_gemm1_swiglu_w8a8(const qmoe_dims* d, const uint8_t* x_tiles, const int8_t* w1, const float* w1_s,
                           const int32_t* offsets, float* h, int32_t* dbg_acc, int32_t* dev_status, void* ws,
                           size_t ws_bytes, qmoe_stream_t stream);

/* W4A8 ([gfx1151] Constraint: int4 weights widened to 8-bit integers before
 *        the integer MMA, with int8 activations).  As W8A8 in every argument
 *        and rule except the weights: w1 holds int4 codes q in [-7, 7] as
 *        bytes [E, 2I, H/2] (byte i of a row: code 2i in the low nibble, code
 *        2i+1 in the high nibble, stored n = q + 8; 16-byte aligned), with
 *        one fp32 scale per output channel in w1_s [E, 2I].  The codes are
 *        widened on chip to exact fp16 integers; |q| <= 7 keeps every fp32
 *        partial sum below 2^24 for H, I <= 16384, so the sums are exact with
 *        no carry passes.  dbg_acc as for W8A8. */
int qmoe_gemm1_swiglu_w4a8(const qmoe_dims* d, const uint8_t* x_tiles, const uint8_t* w1, const float* w1_s,
                           const int32_t* offsets, float* h, int32_t* dbg_acc, int32_t* dev_status, void* ws,
                           size_t ws_bytes, qmoe_stream_t stream);

/* ---------------------------------------------------------------- stage 2: down projection
 *
 * y[s][c] = W2[e][c] . hq[s] for c < H, slots of expert e as above, summed
 * in fp32 and stored as bf16 (round to nearest even) [P, H] in slot order.  [aiter] Test Plan ("stage2 tiles"; K tiles larger
 * than inter_dim read out of bounds, so the kernels never let a K tile pass
 * the end of I).
 *
 * W4A16: h16_tiles from qmoe_w4a16_h_to_f16 (h rows already scaled into
 *        fp16 by powers of two); w2 = qmoe_prepack_int4_weights of the int4
 *        [E*H, I/2] codes and fp16 [E*H, I/32] scales, dequantised on chip as
 *        in stage 1; fp16 MMAs, fp32 sums scaled back by 2^(e_r - p_r); ws as
 *        for stage 1. */
int qmoe_gemm2_w4a16(const qmoe_dims* d, const uint8_t* h16_tiles, const uint8_t* w2, const int32_t* offsets,
                     uint16_t* y, int32_t* dev_status, void* ws, size_t ws_bytes, qmoe_stream_t stream);

/* MXFP4 x FP8: h_tiles from qmoe_gemm1_swiglu_mxfp4; w2 = qmoe_prepack_fp4_weights
 *        of the E2M1 [E*H, I/2] bytes; w2_s = qmoe_prepack_mx_scales of the
 *        E8M0 [E*H, I/32] scales; ws as for stage 1. */
int qmoe_gemm2_mxfp4(const qmoe_dims* d, const uint8_t* h_tiles, const uint8_t* w2, const uint8_t* w2_s,
                     const int32_t* offsets, uint16_t* y, int32_t* dev_status, void* ws, size_t ws_bytes,
                     qmoe_stream_t stream);

/* W8A8: h_tiles = qmoe_quant_tiles_int8_f32 output (K = I); w2 int8
 *        [E, H, I]; w2_s fp32 [E, H]; y = ((float)acc * s_h) * w2_s[e][c]
 *        with acc the exact int32 sum (as for stage 1); dbg_acc (nullable,
 *        16-byte aligned) int32 [P, H].  ws as for stage 1. */
int qmoe_gemm2_w8a8(const qmoe_dims* d, const uint8_t* h_tiles, const int8_t* w2, const float* w2_s,
                    const int32_t* offsets, uint16_t* y, int32_t* dbg_acc, int32_t* dev_status, void* ws,
                    size_t ws_bytes, qmoe_stream_t stream);

/* W4A8: as W8A8 stage 2 with w2 int4 codes [E, H, I/2] (layout of stage 1)
 *        and w2_s fp32 [E, H]. */
int qmoe_gemm2_w4a8(const qmoe_dims* d, const uint8_t* h_tiles, const uint8_t* w2, const float* w2_s,
                    const int32_t* offsets, uint16_t* y, int32_t* dbg_acc, int32_t* dev_status, void* ws,
                    size_t ws_bytes, qmoe_stream_t stream);

/* ---------------------------------------------------------------- combine
 *
 * qmoe_combine -- out[t][c] = bf16( sum_{j=0..k-1} topk_w[t][j] * y[pair_slot[t*k+j]][c] ),
 * summed in fp32 with j ascending from 0 (a fixed order, so the result is
 * reproducible bit for bit: [hip-ep] description, "deterministic scatter
 * order").  Pairs with pair_slot = -1 contribute nothing.
 * in y bf16 [P, H] (slot order), topk_w fp32 [T, k], pair_slot int32 [P];
 * out out_bf16 [T, H]. */
int qmoe_combine(const qmoe_dims* d, const uint16_t* y, const float* topk_w, const int32_t* pair_slot,
                 uint16_t* out_bf16, qmoe_stream_t stream);

/* ---------------------------------------------------------------- whole layer
 *
 * One call for the whole path: routing, activation quantisation (MXFP4,
 * W8A8, W4A8), stage 1, intermediate quantisation (W8A8, W4A8), stage 2 and
 * combine, all launched in order on `stream`.  scheme: 0 = W4A16, 1 = MXFP4
 * x FP8, 2 = W8A8, 3 = W4A8.  Weights and scales as for the per-stage calls (MXFP4 weights
 * and scales pre-packed; W4A16 weights pre-packed with their scales, so
 * w1_s and w2_s are ignored and may be NULL for scheme 0).  All
 * intermediates live in the caller's workspace of
 * qmoe_forward_workspace_bytes(d, scheme) bytes (256-byte aligned).
 * dev_status as for qmoe_align_sort. */
size_t qmoe_forward_workspace_bytes(const qmoe_dims* d, int scheme);
int qmoe_moe_forward(int scheme, const qmoe_dims* d, const uint16_t* x_bf16, const int32_t* topk_ids,
                     const float* topk_w, const void* w1, const void* w1_s, const void* w2, const void* w2_s,
                     uint16_t* out_bf16, int32_t* dev_status, void* ws, size_t ws_bytes, qmoe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QMOE_H */
