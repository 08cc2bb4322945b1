/*
 * CPU oracle for the quantized Mixture-of-Experts expert path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library; the only thing the two
 * have in common is the seeded input generator that feeds both.
 *
 * What it computes (per token t, top-k pairs j = 0..k-1, e = id[t, j]):
 *
 *     out[t] = sum_j  w[t, j] * W2_e . Q_h( silu(W1g_e . a_t) * (W1u_e . a_t) )
 *
 * where a_t is the token's activation as the scheme sees it, W1g_e / W1u_e are
 * rows 0..I-1 / I..2I-1 of expert e's dequantised gate/up matrix, and Q_h is
 * the scheme's quantisation of the intermediate.  This is the plain definition
 * of a routed top-k MoE layer with SwiGLU experts: grouping the expert matmuls
 * ("perf(qmoe): group prefill expert matmuls", description) and sorting pairs
 * by expert only reorder that work, and the page asks that the scatter back
 * keep a deterministic order.
 *
 * Arithmetic: every dot product is accumulated in double, weights are
 * dequantised exactly, and out is returned in double.  Where a float value
 * decides an integer code (activation and intermediate quantisation), the
 * decision is taken in fp32 exactly as the CUDA kernels take it; W8A8 integer
 * dots are exact (int64, checked to fit int32) and their dequantisation is
 * done in fp32 in the order ((float)acc * s_a) * s_w.  Compiled with
 * -ffp-contract=off so results agree across x86-64 and aarch64.
 *
 * Formats (all K-contiguous, K = the reduction axis):
 *   int4     byte i of a row holds elements 2i (low nibble) and 2i+1 (high
 *            nibble); stored n = q + 8, value (n - 8) * s, one fp16 s per 32
 *            consecutive K elements.  "Symmetric int4" (the hip-ep page,
 *            description) fixes no zero point.
 *   E2M1     sign bit 3, exponent bits 2..1, mantissa bit 0; values
 *            0, .5, 1, 1.5, 2, 3, 4, 6 and negatives; same nibble order.
 *   E8M0     byte b -> 2^(b - 127); 255 is NaN.  One scale per 32 along K.
 *   E4M3     "fn" variant: bias 7, no infinities, S.1111.111 is NaN, max 448.
 *   MX quant per block of 32: X = 2^(floor(log2 amax) - 8), codes are the
 *            round-to-nearest-even of v / X, saturated to +-448; amax == 0
 *            gives scale byte 127 and zero codes (OCP MX v1.0 conversion).
 *   int8     per row: s = amax / 127 (fp32; 1 when amax == 0),
 *            q = clamp(rint(v / s), -127, 127) in fp32.
 *
 * W4A8 (the gfx1151 page, Constraint: int4 weights widened to 8-bit integers
 * before an integer MMA, with 8-bit activations): weights are int4 codes in
 * the int4 byte layout above with one fp32 scale per output channel (a scale
 * inside the K sum would break the integer dot), activations and the
 * intermediate are int8 per row, and everything after the weight decode is
 * the W8A8 arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { SCHEME_W4A16 = 0, SCHEME_MXFP4 = 1, SCHEME_W8A8 = 2, SCHEME_W4A8 = 3 };

/* schemes whose dots are exact integer sums of int8-range codes */
static int integer_scheme(int scheme) { return scheme == SCHEME_W8A8 || scheme == SCHEME_W4A8; }

/* ------------------------------------------------------------ decoders */

double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_fp16_to_double(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + f, e - 25);
    return s ? -v : v;
}

double oracle_int4_to_double(uint8_t n) { return (double)((int)(n & 15) - 8); }

double oracle_e2m1_to_double(uint8_t c) {
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

double oracle_e8m0_to_double(uint8_t b) { return b == 255 ? NAN : ldexp(1.0, (int)b - 127); }

double oracle_e4m3_to_double(uint8_t b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9); /* m/8 * 2^-6 */
    else
        v = ldexp(8.0 + m, e - 10); /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* ------------------------------------------------------------ encoders */

/* Nearest e4m3 (ties to even), saturating to +-448.  The sign of a value
 * that rounds to zero is kept (IEEE behaviour). */
uint8_t oracle_e4m3_from_double_sat(double v) {
    if (isnan(v)) return 0x7F;
    uint8_t s = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return s | 0x7E;
    if (a == 0.0) return s;
    int ex;
    frexp(a, &ex);      /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;     /* floor(log2 a) */
    if (E < -6) E = -6; /* subnormal range shares the 2^-9 quantum */
    double n = nearbyint(ldexp(a, 3 - E)); /* a / 2^(E-3), exact; RNE */
    /* Normal codes are ((E+7) << 3) + (n - 8) for n in [8, 16]; for E = -6
     * the same expression gives the subnormal codes n = 0..7. */
    int code = ((E + 7) << 3) + (int)n - 8;
    return s | (uint8_t)code;
}

/* float -> bfloat16 bits, round to nearest even. */
uint16_t oracle_float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* ------------------------------------------------------------ quantisers */

/* MX quantisation of n (multiple of 32) fp32 values into e4m3 codes and one
 * E8M0 scale per 32. */
void oracle_mx_quant(const float* v, int64_t n, uint8_t* q, uint8_t* s) {
    for (int64_t b = 0; b < n / 32; ++b) {
        const float* vb = v + 32 * b;
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs((double)vb[i]));
        if (amax == 0.0) {
            s[b] = 127;
            memset(q + 32 * b, 0, 32);
            continue;
        }
        int ex;
        frexp(amax, &ex);
        int X = (ex - 1) - 8; /* floor(log2 amax) - emax(e4m3) */
        if (X < -127) X = -127;
        if (X > 127) X = 127;
        s[b] = (uint8_t)(X + 127);
        for (int i = 0; i < 32; ++i) q[32 * b + i] = oracle_e4m3_from_double_sat(ldexp((double)vb[i], -X));
    }
}

/* Per-row symmetric int8 quantisation in fp32. */
void oracle_int8_quant(const float* v, int64_t rows, int64_t n, int8_t* q, float* s) {
    for (int64_t r = 0; r < rows; ++r) {
        const float* vr = v + r * n;
        float amax = 0.0f;
        for (int64_t i = 0; i < n; ++i) {
            float a = fabsf(vr[i]);
            if (a > amax) amax = a;
        }
        float sc = (amax == 0.0f) ? 1.0f : amax / 127.0f;
        for (int64_t i = 0; i < n; ++i) {
            float t = rintf(vr[i] / sc);
            if (t > 127.0f) t = 127.0f;
            if (t < -127.0f) t = -127.0f;
            q[r * n + i] = (int8_t)t;
        }
        s[r] = sc;
    }
}

/* Activation quantisation of bf16 rows as the scheme's first step:
 * MXFP4 -> e4m3 codes + E8M0 per 32; W8A8 -> int8 + fp32 per row. */
int oracle_quant_act(int scheme, int64_t rows, int64_t cols, const uint16_t* x, uint8_t* q, void* s) {
    float* buf = (float*)malloc(sizeof(float) * cols);
    if (!buf) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t i = 0; i < cols; ++i) buf[i] = (float)oracle_bf16_to_double(x[r * cols + i]);
        if (scheme == SCHEME_MXFP4)
            oracle_mx_quant(buf, cols, q + r * cols, (uint8_t*)s + r * (cols / 32));
        else if (integer_scheme(scheme))
            oracle_int8_quant(buf, 1, cols, (int8_t*)q + r * cols, (float*)s + r);
        else {
            free(buf);
            return -2;
        }
    }
    free(buf);
    return 0;
}

/* ------------------------------------------------------------ align / sort */

/* Expert-sorted order of the P = T*k routed pairs (pair p = t*k + j):
 * counts[e], offsets[e] (exclusive prefix sum, offsets[E] = number of valid
 * pairs), sorted_pair_ids[s] (ascending p within each expert: a stable
 * counting sort) and pair_slot[p], its inverse.  Ids outside [0, E) take no
 * slot (pair_slot = -1) and are counted in the return value. */
int64_t oracle_align_sort(int64_t P, int E, const int32_t* ids, int32_t* counts, int32_t* offsets,
                          int32_t* sorted_pair_ids, int32_t* pair_slot) {
    int64_t invalid = 0;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < P; ++p) {
        int e = ids[p];
        if (e < 0 || e >= E)
            ++invalid;
        else
            ++counts[e];
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (E > 0 ? E : 1));
    for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int64_t p = 0; p < P; ++p) {
        int e = ids[p];
        if (e < 0 || e >= E) {
            pair_slot[p] = -1;
            continue;
        }
        int32_t s = cursor[e]++;
        sorted_pair_ids[s] = (int32_t)p;
        pair_slot[p] = s;
    }
    for (int64_t s = offsets[E]; s < P; ++s) sorted_pair_ids[s] = -1;
    free(cursor);
    return invalid;
}

/* ------------------------------------------------------------ weights */

typedef struct {
    int scheme;
    int H, I, E;
    const void* w1;
    const void* w1s;
    const void* w2;
    const void* w2s;
} model_t;

/* Dequantise row `row` of expert e of a [E, R, K] weight into out[K]
 * (W4A16 and MXFP4 only). */
static void dequant_row(int scheme, const uint8_t* w, const void* ws, int64_t R, int64_t K, int e, int64_t row,
                        double* out) {
    const uint8_t* wr = w + ((int64_t)e * R + row) * (K / 2);
    int64_t sbase = ((int64_t)e * R + row) * (K / 32);
    for (int64_t kk = 0; kk < K; ++kk) {
        uint8_t byte = wr[kk / 2];
        uint8_t nib = (kk & 1) ? (byte >> 4) : (byte & 15);
        double v, sc;
        if (scheme == SCHEME_W4A16) {
            v = oracle_int4_to_double(nib);
            sc = oracle_fp16_to_double(((const uint16_t*)ws)[sbase + kk / 32]);
        } else {
            v = oracle_e2m1_to_double(nib);
            sc = oracle_e8m0_to_double(((const uint8_t*)ws)[sbase + kk / 32]);
        }
        out[kk] = v * sc;
    }
}

/* Integer codes of row `row` of expert e of a [E, R, K] weight (W8A8: int8
 * as stored; W4A8: int4 nibbles n -> n - 8) into out[K]. */
static void int_row(int scheme, const void* w, int64_t R, int64_t K, int e, int64_t row, int8_t* out) {
    if (scheme == SCHEME_W8A8) {
        memcpy(out, (const int8_t*)w + ((int64_t)e * R + row) * K, (size_t)K);
        return;
    }
    const uint8_t* wr = (const uint8_t*)w + ((int64_t)e * R + row) * (K / 2);
    for (int64_t kk = 0; kk < K; ++kk) {
        uint8_t code = (uint8_t)((wr[kk / 2] >> (4 * (kk % 2))) & 15);
        out[kk] = (int8_t)((int)oracle_int4_to_double(code));
    }
}

static double dot(const double* a, const double* b, int64_t n) {
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) acc += a[i] * b[i];
    return acc;
}

static int64_t idot8(const int8_t* a, const int8_t* b, int64_t n) {
    int64_t acc = 0;
    for (int64_t i = 0; i < n; ++i) acc += (int64_t)a[i] * (int64_t)b[i];
    return acc;
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* ------------------------------------------------------------ stage 2 */

/* Intermediate row in its quantised form, dequantised to double for the
 * down projection (W4A16, MXFP4), or kept as int8 + scale (W8A8). */
typedef struct {
    double* hd;      /* [I] */
    const int8_t* hq8;
    float hs8;
} hrow_t;

/* Down projection of one intermediate row through expert e: y[c], c < H. */
static int down_row(const model_t* m, int e, const hrow_t* h, double* wrow, double* y, int32_t* acc_out) {
    int H = m->H, I = m->I;
    int err = 0;
    int8_t* wr = integer_scheme(m->scheme) ? (int8_t*)malloc((size_t)I) : NULL;
    for (int c = 0; c < H; ++c) {
        if (integer_scheme(m->scheme)) {
            int_row(m->scheme, m->w2, H, I, e, c, wr);
            int64_t acc = idot8(h->hq8, wr, I);
            if (acc > INT32_MAX || acc < INT32_MIN) err = 1;
            if (acc_out) acc_out[c] = (int32_t)acc;
            float sw = ((const float*)m->w2s)[(int64_t)e * H + c];
            float yv = ((float)acc * h->hs8) * sw;
            y[c] = (double)yv;
        } else {
            dequant_row(m->scheme, (const uint8_t*)m->w2, m->w2s, H, I, e, c, wrow);
            y[c] = dot(h->hd, wrow, I);
        }
    }
    free(wr);
    return err;
}

/* The down projection on its own, for rows that already hold quantised
 * intermediates: row r goes through expert experts[r].
 *   W4A16: h bf16 bits [rows, I]
 *   MXFP4: h e4m3 [rows, I], h_s E8M0 [rows, I/32]
 *   W8A8, W4A8: h int8 [rows, I], h_s fp32 [rows]
 * y is double [rows, H]; acc2 (W8A8, W4A8; nullable) int32 [rows, H]. */
int oracle_stage2(int scheme, int64_t rows, int H, int I, int E, const int32_t* experts, const void* h,
                  const void* h_s, const void* w2, const void* w2s, double* y, int32_t* acc2) {
    model_t m = {scheme, H, I, E, NULL, NULL, w2, w2s};
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t r = 0; r < rows; ++r) {
        double* hd = (double*)malloc(sizeof(double) * I);
        double* wrow = (double*)malloc(sizeof(double) * I);
        hrow_t hr = {hd, NULL, 0.0f};
        int e = experts[r];
        if (e < 0 || e >= E) {
            err |= 2;
        } else {
            if (scheme == SCHEME_W4A16) {
                for (int i = 0; i < I; ++i) hd[i] = oracle_bf16_to_double(((const uint16_t*)h)[r * I + i]);
            } else if (scheme == SCHEME_MXFP4) {
                for (int i = 0; i < I; ++i)
                    hd[i] = oracle_e4m3_to_double(((const uint8_t*)h)[r * I + i]) *
                            oracle_e8m0_to_double(((const uint8_t*)h_s)[r * (I / 32) + i / 32]);
            } else {
                hr.hq8 = (const int8_t*)h + r * I;
                hr.hs8 = ((const float*)h_s)[r];
            }
            err |= down_row(&m, e, &hr, wrow, y + r * H, acc2 ? acc2 + r * H : NULL);
        }
        free(hd);
        free(wrow);
    }
    return err ? -err : 0;
}

/* ------------------------------------------------------------ forward */

/* Full forward for the tokens in tok_list (all T tokens when tok_list is
 * NULL; ntok must then be T).  Index i below runs over the listed tokens.
 *   x      bf16 bits [T, H]; topk_ids int32 [T, k]; topk_w fp32 [T, k]
 *   W4A16: w1 int4 [E, 2I, H/2], w1s fp16 [E, 2I, H/32]; w2 [E, H, I/2], w2s [E, H, I/32]
 *   MXFP4: same with E2M1 bytes and E8M0 scales
 *   W8A8:  w1 int8 [E, 2I, H], w1s fp32 [E, 2I]; w2 int8 [E, H, I], w2s fp32 [E, H]
 *   W4A8:  as W8A8 with int4 bytes w1 [E, 2I, H/2] and w2 [E, H, I/2]
 * Outputs: out double [ntok, H].  Debug outputs (each nullable), row i*k + j:
 *   dbg_h    fp32 [ntok*k, I]  intermediate before Q_h
 *   dbg_hq   Q_h codes [ntok*k, I] (bf16 bits for W4A16, e4m3, int8)
 *   dbg_hs   Q_h scales (E8M0 [ntok*k, I/32] or fp32 [ntok*k])
 *   dbg_acc1 int32 [ntok*k, 2I] (W8A8, W4A8 gate/up accumulators)
 *   dbg_y    double [ntok*k, H] down projection before the weighted sum
 * Pairs whose id is outside [0, E) contribute nothing; the return value is
 * minus the number of such pairs (0 when all are valid), or -2^30 when an
 * integer dot does not fit int32. */
int64_t oracle_moe_forward(int scheme, int64_t T, int k, int H, int I, int E, const uint16_t* x,
                           const int32_t* topk_ids, const float* topk_w, const void* w1, const void* w1s,
                           const void* w2, const void* w2s, int64_t ntok, const int64_t* tok_list, double* out,
                           float* dbg_h, void* dbg_hq, void* dbg_hs, int32_t* dbg_acc1, double* dbg_y) {
    model_t m = {scheme, H, I, E, w1, w1s, w2, w2s};
    int64_t invalid = 0;
    int overflow = 0;
    if (!tok_list && ntok != T) return -(1 << 30) - 1;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : invalid) reduction(| : overflow)
    for (int64_t i = 0; i < ntok; ++i) {
        int64_t t = tok_list ? tok_list[i] : i;
        double* a = (double*)malloc(sizeof(double) * H);
        double* wrow = (double*)malloc(sizeof(double) * (H > I ? H : I));
        double* y = (double*)malloc(sizeof(double) * H);
        float* xf = (float*)malloc(sizeof(float) * H);
        float* h32 = (float*)malloc(sizeof(float) * I);
        double* hd = (double*)malloc(sizeof(double) * I);
        uint8_t* q8 = (uint8_t*)malloc(H > I ? H : I);
        uint8_t* s8 = (uint8_t*)malloc((H > I ? H : I) / 32 + 1);
        int8_t* hq8 = (int8_t*)malloc(I);
        int8_t* wg = (int8_t*)malloc(H);
        int8_t* wu = (int8_t*)malloc(H);
        float sa = 1.0f;

        /* the token's activation as the scheme consumes it */
        for (int c = 0; c < H; ++c) xf[c] = (float)oracle_bf16_to_double(x[t * H + c]);
        if (scheme == SCHEME_MXFP4) {
            oracle_mx_quant(xf, H, q8, s8);
            for (int c = 0; c < H; ++c) a[c] = oracle_e4m3_to_double(q8[c]) * oracle_e8m0_to_double(s8[c / 32]);
        } else if (integer_scheme(scheme)) {
            oracle_int8_quant(xf, 1, H, (int8_t*)q8, &sa);
        } else {
            for (int c = 0; c < H; ++c) a[c] = (double)xf[c];
        }

        double* o = out + i * H;
        for (int c = 0; c < H; ++c) o[c] = 0.0;

        for (int j = 0; j < k; ++j) {
            int e = topk_ids[t * k + j];
            int64_t row = i * k + j;
            if (e < 0 || e >= E) {
                ++invalid;
                continue;
            }
            /* gate/up projection and SwiGLU, h[n] for n < I */
            for (int n = 0; n < I; ++n) {
                double g, u;
                if (integer_scheme(scheme)) {
                    int_row(scheme, w1, 2 * I, H, e, n, wg);
                    int_row(scheme, w1, 2 * I, H, e, I + n, wu);
                    int64_t ag = idot8((const int8_t*)q8, wg, H);
                    int64_t au = idot8((const int8_t*)q8, wu, H);
                    if (ag > INT32_MAX || ag < INT32_MIN || au > INT32_MAX || au < INT32_MIN) overflow = 1;
                    if (dbg_acc1) {
                        dbg_acc1[row * 2 * I + n] = (int32_t)ag;
                        dbg_acc1[row * 2 * I + I + n] = (int32_t)au;
                    }
                    const float* sw = (const float*)w1s + (int64_t)e * 2 * I;
                    float gf = ((float)ag * sa) * sw[n];
                    float uf = ((float)au * sa) * sw[I + n];
                    g = (double)gf;
                    u = (double)uf;
                } else {
                    dequant_row(scheme, (const uint8_t*)w1, w1s, 2 * I, H, e, n, wrow);
                    g = dot(a, wrow, H);
                    dequant_row(scheme, (const uint8_t*)w1, w1s, 2 * I, H, e, I + n, wrow);
                    u = dot(a, wrow, H);
                }
                h32[n] = (float)(silu(g) * u);
            }
            if (dbg_h) memcpy(dbg_h + row * I, h32, sizeof(float) * I);

            /* Q_h, then the down projection on the quantised intermediate */
            hrow_t hr = {hd, NULL, 0.0f};
            if (scheme == SCHEME_W4A16) {
                for (int n = 0; n < I; ++n) {
                    uint16_t b = oracle_float_to_bf16(h32[n]);
                    hd[n] = oracle_bf16_to_double(b);
                    if (dbg_hq) ((uint16_t*)dbg_hq)[row * I + n] = b;
                }
            } else if (scheme == SCHEME_MXFP4) {
                oracle_mx_quant(h32, I, q8, s8);
                for (int n = 0; n < I; ++n) hd[n] = oracle_e4m3_to_double(q8[n]) * oracle_e8m0_to_double(s8[n / 32]);
                if (dbg_hq) memcpy((uint8_t*)dbg_hq + row * I, q8, I);
                if (dbg_hs) memcpy((uint8_t*)dbg_hs + row * (I / 32), s8, I / 32);
            } else {
                float hs;
                oracle_int8_quant(h32, 1, I, hq8, &hs);
                hr.hq8 = hq8;
                hr.hs8 = hs;
                if (dbg_hq) memcpy((int8_t*)dbg_hq + row * I, hq8, I);
                if (dbg_hs) ((float*)dbg_hs)[row] = hs;
            }
            overflow |= down_row(&m, e, &hr, wrow, y, NULL);
            if (dbg_y) memcpy(dbg_y + row * H, y, sizeof(double) * H);

            /* top-k weighted sum, j ascending */
            double wt = (double)topk_w[t * k + j];
            for (int c = 0; c < H; ++c) o[c] += wt * y[c];
        }
        free(a);
        free(wrow);
        free(y);
        free(xf);
        free(h32);
        free(hd);
        free(q8);
        free(s8);
        free(hq8);
        free(wg);
        free(wu);
    }
    if (overflow) return -(1 << 30);
    return -invalid;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* The top-k weighted sum on its own: out[t][c] = sum_j w[t][j] * y[slot][c],
 * slot = pair_slot[t*k + j] (skipped when -1), j ascending, in double.
 * y fp32 [rows, H]; out double [T, H]. */
void oracle_combine(int64_t T, int k, int H, const float* y, const float* topk_w, const int32_t* pair_slot,
                    double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int c = 0; c < H; ++c) out[t * H + c] = 0.0;
        for (int j = 0; j < k; ++j) {
            int32_t s = pair_slot[t * k + j];
            if (s < 0) continue;
            double w = (double)topk_w[t * k + j];
            for (int c = 0; c < H; ++c) out[t * H + c] += w * (double)y[(int64_t)s * H + c];
        }
    }
}
