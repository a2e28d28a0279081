/*
 * CPU oracle for the FMPQ W4Ax path -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg load this
 * library. The product (the CUDA library under bit_quantized_gemm_fmpq_gb300/csrc) shares
 * no code, header, table or constant with it, and never calls it.
 *
 * What it computes, step by step, in the order the method states it:
 *   1. gather-permute the channels, Xp[m, j] = X[m, perm[j]]        (COMET news article,
 *      section 1 "outlier distribution": channel reordering gathers the outliers)
 *   2. split the K channels into blocks of 128                        (same section)
 *   3. per token and block: absmax, fp16 scale, round-half-even quantization to INT8 for
 *      outlier blocks and INT4 for the rest                          (same section; the
 *      "dynamic precision" sentence), symmetric ranges [-127,127] / [-7,7]
 *   4. INT4 weights, per output channel and block, quantized the same way offline
 *   5. exact integer partial sums per block P[m,n,b]                 (COMET abstract:
 *      W4A4/W4A8 mixed-precision matrix multiplication)
 *   6. scale-and-sum epilogue Y[m,n] = sum_b sx[m,b] * sw[n,b] * P[m,n,b]  (QUIK explainer,
 *      section "kernel fusion": dequantization applied in the GEMM epilogue)
 *
 * Readings where the pages are silent (each listed with its reason in the design notes):
 *   - symmetric absmax quantization; INT4 range [-7,7], INT8 range [-127,127]
 *   - scale s = fp16_rne( fp32(absmax) / fp32(qmax) ); a zero scale quantizes the block to 0
 *   - q = clamp( rne_f32( fp32(x) / fp32(s) ), -qmax, qmax ) with IEEE fp32 division
 *   - packed activation layout (an encoding, not arithmetic of the method): one byte per
 *     code holding an E4M3 number equal to part of |q| times 2^-9 (INT8 codes use two
 *     planes, |q| mod 16 and the rest), planes block after block, 16-byte chunks of each
 *     128-byte row rotated by XOR with the row index mod 8 (see "Packed activation format")
 *
 * Floating point here is IEEE fp32 where the method decides an integer (the kernel's
 * precision), and fp64 or exact int128 fixed point for the epilogue reference.
 * Build with -O2 -fno-fast-math -ffp-contract=off.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BLOCK 128

/* ------------------------------------------------------------------------------------
 * IEEE 754 binary16 <-> binary32, written from the format's definition (value based).
 * ------------------------------------------------------------------------------------ */

/* binary16 bits -> value.  normal: (1024 + f) * 2^(e - 25); subnormal: f * 2^-24. */
float oracle_f16_to_f32(uint16_t h) {
    unsigned sign = (h >> 15) & 1u, e = (h >> 10) & 31u, f = h & 1023u;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024u + f), (int)e - 25);
    return (float)(sign ? -v : v);
}

/* round a non-negative double that is an exact multiple of 1/2 ... to an integer, ties to even
 * (used on values r = |x| / quantum, which are exact in double) */
static double round_half_even_d(double r) {
    double fl = floor(r);
    double d = r - fl;
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* value -> binary16 bits, round to nearest, ties to even (NaN -> 0x7e00). */
static uint16_t f64_to_f16(double x) {
    if (isnan(x)) return 0x7e00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a >= 65520.0) return sign | 0x7c00;           /* 65504 + half an ulp (16): overflow */
    if (a == 0.0) return sign;
    /* quantum of the binade that contains a (subnormal binades share 2^-24) */
    int e2;
    frexp(a, &e2);                                      /* a = m * 2^e2, m in [0.5, 1) */
    int ex = e2 - 1;                                    /* floor(log2 a) */
    double quantum = (ex < -14) ? ldexp(1.0, -24) : ldexp(1.0, ex - 10);
    double n = round_half_even_d(a / quantum);          /* exact division by a power of 2 */
    double v = n * quantum;                             /* the rounded value */
    if (v >= 65520.0) return sign | 0x7c00;
    if (v < ldexp(1.0, -14)) {                          /* subnormal (or zero) */
        return sign | (uint16_t)(v / ldexp(1.0, -24));
    }
    frexp(v, &e2);
    ex = e2 - 1;
    unsigned frac = (unsigned)(v / ldexp(1.0, ex - 10)) - 1024u;
    unsigned expf = (unsigned)(ex + 15);
    if (expf >= 31) return sign | 0x7c00;
    return sign | (uint16_t)((expf << 10) | frac);
}

uint16_t oracle_f32_to_f16(float x) { return f64_to_f16((double)x); }

void oracle_f32_to_f16_array(const float* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(x[i]);
}

void oracle_f16_to_f32_array(const uint16_t* h, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f32(h[i]);
}

/* ------------------------------------------------------------------------------------
 * Quantization of one block of 128 values (steps 3-4 above).
 * ------------------------------------------------------------------------------------ */

/* round-half-even of an fp32 value to an integer (|v| well below 2^23 here) */
static int32_t rne_f32_to_int(float v) {
    float fl = floorf(v);
    float d = v - fl;                                   /* exact: fl and v share the binade */
    int32_t i = (int32_t)fl;
    if (d > 0.5f) return i + 1;
    if (d < 0.5f) return i;
    return (i % 2 == 0) ? i : i + 1;
}

/* Quantize 128 fp16 values xs (already permuted) with range [-qmax, qmax].
 * Writes q[128] and returns the fp16 scale bits. */
static uint16_t quantize_block(const uint16_t* xs, int qmax, int8_t* q) {
    float absmax = 0.0f;
    for (int j = 0; j < ORACLE_BLOCK; ++j) {
        float v = fabsf(oracle_f16_to_f32(xs[j]));
        if (v > absmax) absmax = v;
    }
    float s32 = absmax / (float)qmax;                   /* IEEE fp32 division */
    uint16_t s16 = oracle_f32_to_f16(s32);
    float s = oracle_f16_to_f32(s16);
    for (int j = 0; j < ORACLE_BLOCK; ++j) {
        if (s == 0.0f) { q[j] = 0; continue; }
        float r = oracle_f16_to_f32(xs[j]) / s;          /* IEEE fp32 division */
        int32_t v = rne_f32_to_int(r);
        if (v > qmax) v = qmax;
        if (v < -qmax) v = -qmax;
        q[j] = (int8_t)v;
    }
    return s16;
}

/* ------------------------------------------------------------------------------------
 * Packed activation format: operand-ready code planes.
 *
 * Every code is stored as one byte holding the E4M3 number (FP8: 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal) equal to a part of
 * the code's magnitude times 2^-9, with bit 7 = the sign bit of the fp16 input (so a
 * negative input whose code is 0 gives -0, numerically 0).
 *   INT4 block: one plane, part = |q|                       (0..7)
 *   INT8 block: two planes, part = |q| mod 16               (0..15)  [the "low" plane]
 *                           part = |q| - (|q| mod 16)       (0..112) [the "high" plane]
 * The parts of a code sum to |q|. Planes are stored block after block (plane offset of
 * block b = number of planes of the blocks before it); a plane is [M][128] bytes; in row m
 * the 16-byte chunk holding channels 16c..16c+15 sits at chunk position c XOR (m mod 8).
 * ------------------------------------------------------------------------------------ */

/* Value of an E4M3 byte, from the format's definition (0x7F/0xFF are NaN). */
double oracle_e4m3_value(uint8_t b) {
    int sign = (b >> 7) & 1, e = (b >> 3) & 15, f = b & 7;
    double v;
    if (e == 15 && f == 7) return NAN;
    if (e == 0)
        v = ldexp((double)f / 8.0, -6);
    else
        v = ldexp(1.0 + (double)f / 8.0, e - 7);
    return sign ? -v : v;
}

/* The non-negative E4M3 byte whose value is exactly n * 2^-9 (found by search over the
 * encodings), or -1 if no encoding has that value. */
static int e4m3_of_multiple(int n) {
    const double target = ldexp((double)n, -9);
    for (int b = 0; b < 128; ++b) {
        const double v = oracle_e4m3_value((uint8_t)b);
        if (!isnan(v) && v == target) return b;
    }
    return -1;
}

static unsigned mag(int8_t q) { return (unsigned)(q < 0 ? -q : q); }

/* part of |q| stored in plane `plane` of a block */
static unsigned code_part(int8_t q, int is_int8, int plane) {
    const unsigned a = mag(q);
    if (!is_int8) return a;
    return plane == 0 ? a % 16u : a - a % 16u;
}

/* byte position of channel c in row m of a plane */
static int64_t plane_pos(int m, int c) {
    return (int64_t)((((c / 16) ^ (m % 8)) * 16) + c % 16);
}

static int num_planes(const uint8_t* mask, int b) { return mask[b] ? 2 : 1; }

/* Plane offset of block b: planes of the blocks before it. */
int64_t oracle_plane_offset(const uint8_t* mask, int b) {
    int64_t off = 0;
    for (int i = 0; i < b; ++i) off += num_planes(mask, i);
    return off;
}

int64_t oracle_packed_a_bytes(const uint8_t* mask, int K, int M) {
    return oracle_plane_offset(mask, K / ORACLE_BLOCK) * (int64_t)M * ORACLE_BLOCK;
}

/* Write the codes q[128] of token m, block b into its plane(s); xs[128] are the block's
 * fp16 inputs (for the sign bit). */
static void pack_block_row(const int8_t* q, const uint16_t* xs, int is_int8, uint8_t* A_packed, int64_t plane0,
                           int M, int m) {
    for (int p = 0; p < (is_int8 ? 2 : 1); ++p) {
        uint8_t* row = A_packed + (plane0 + p) * (int64_t)M * ORACLE_BLOCK + (int64_t)m * ORACLE_BLOCK;
        for (int c = 0; c < ORACLE_BLOCK; ++c) {
            const int e = e4m3_of_multiple((int)code_part(q[c], is_int8, p));
            row[plane_pos(m, c)] = (uint8_t)(((xs[c] >> 15) << 7) | (unsigned)e);
        }
    }
}

/* Read the codes of token m, block b back from its plane(s): the parts' values sum to
 * |q| * 2^-9; the sign is bit 7 of the first plane. */
static void unpack_block_row(const uint8_t* A_packed, int is_int8, int64_t plane0, int M, int m, int8_t* q) {
    for (int c = 0; c < ORACLE_BLOCK; ++c) {
        double v = 0.0;
        unsigned sign = 0;
        for (int p = 0; p < (is_int8 ? 2 : 1); ++p) {
            const uint8_t byte =
                A_packed[(plane0 + p) * (int64_t)M * ORACLE_BLOCK + (int64_t)m * ORACLE_BLOCK + plane_pos(m, c)];
            v += fabs(oracle_e4m3_value(byte));
            if (p == 0) sign = byte >> 7;
        }
        const int a = (int)ldexp(v, 9);
        q[c] = (int8_t)(sign ? -a : a);
    }
}

/* Activations: X fp16 bits [M][ldx] -> packed A, a_scales [nb][M] (fp16 bits) and, if
 * Aq != NULL, the integer codes Aq [M][K] in permuted channel order. Returns 0 on success. */
int oracle_quantize_activations(const uint16_t* X, int64_t ldx, int M, int K,
                                const int32_t* perm, const uint8_t* mask,
                                uint8_t* A_packed, uint16_t* a_scales, int8_t* Aq) {
    if (K % ORACLE_BLOCK) return -1;
    const int nb = K / ORACLE_BLOCK;
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)nb);
    if (!off) return -2;
    for (int b = 0; b < nb; ++b) off[b] = oracle_plane_offset(mask, b);
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m) {
        uint16_t xs[ORACLE_BLOCK];
        int8_t q[ORACLE_BLOCK];
        for (int b = 0; b < nb; ++b) {
            /* step 1: gather-permute this block's channels */
            for (int j = 0; j < ORACLE_BLOCK; ++j)
                xs[j] = X[(int64_t)m * ldx + perm[b * ORACLE_BLOCK + j]];
            /* steps 2-3: per-block scale and codes */
            const int qmax = mask[b] ? 127 : 7;
            a_scales[(int64_t)b * M + m] = quantize_block(xs, qmax, q);
            if (Aq)
                for (int j = 0; j < ORACLE_BLOCK; ++j) Aq[(int64_t)m * K + b * ORACLE_BLOCK + j] = q[j];
            /* pack */
            pack_block_row(q, xs, mask[b] != 0, A_packed, off[b], M, m);
        }
    }
    free(off);
    return 0;
}

/* Decode the packed activation buffer back to codes Aq [M][K]. */
int oracle_unpack_activations(const uint8_t* A_packed, const uint8_t* mask, int M, int K, int8_t* Aq) {
    if (K % ORACLE_BLOCK) return -1;
    const int nb = K / ORACLE_BLOCK;
    for (int b = 0; b < nb; ++b) {
        const int64_t plane0 = oracle_plane_offset(mask, b);
        for (int m = 0; m < M; ++m)
            unpack_block_row(A_packed, mask[b] != 0, plane0, M, m, Aq + (int64_t)m * K + b * ORACLE_BLOCK);
    }
    return 0;
}

/* Weights (offline): W fp16 bits [N][ldw] -> codes Wq [N][K] in permuted channel order
 * (INT4 range [-7,7] everywhere) and w_scales [nb][N] (fp16 bits). The same channel
 * permutation is applied to W so the products pair up (QUIK explainer, step 1: the
 * weight matrix is reordered together with the outlier columns). */
int oracle_quantize_weights(const uint16_t* W, int64_t ldw, int N, int K, const int32_t* perm,
                            int8_t* Wq, uint16_t* w_scales) {
    if (K % ORACLE_BLOCK) return -1;
    const int nb = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        uint16_t xs[ORACLE_BLOCK];
        for (int b = 0; b < nb; ++b) {
            for (int j = 0; j < ORACLE_BLOCK; ++j) xs[j] = W[(int64_t)n * ldw + perm[b * ORACLE_BLOCK + j]];
            w_scales[(int64_t)b * N + n] = quantize_block(xs, 7, Wq + (int64_t)n * K + b * ORACLE_BLOCK);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------------------
 * Integer partial sums and the epilogue (steps 5-6).
 * ------------------------------------------------------------------------------------ */

/* P[m][n][b] = sum_{j in block b} Aq[m][j] * Wq[n][j], exact (int64 accumulate). */
void oracle_partials(const int8_t* Aq, const int8_t* Wq, int M, int N, int K, int32_t* P) {
    const int nb = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n)
            for (int b = 0; b < nb; ++b) {
                int64_t acc = 0;
                for (int j = b * ORACLE_BLOCK; j < (b + 1) * ORACLE_BLOCK; ++j)
                    acc += (int64_t)Aq[(int64_t)m * K + j] * (int64_t)Wq[(int64_t)n * K + j];
                P[((int64_t)m * N + n) * nb + b] = (int32_t)acc;
            }
}

/* The zero-extension form (COMET news article, section 3: unsigned extension of the 4-bit
 * weight, compensated through the scale path): with u = q_w + 8 in [1, 15],
 *   P = sum_j q_x * u  -  8 * sum_j q_x,
 * the correction depending only on (m, b). */
void oracle_partials_zero_ext(const int8_t* Aq, const int8_t* Wq, int M, int N, int K, int32_t* P) {
    const int nb = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int b = 0; b < nb; ++b) {
            int64_t sx = 0;
            for (int j = b * ORACLE_BLOCK; j < (b + 1) * ORACLE_BLOCK; ++j) sx += Aq[(int64_t)m * K + j];
            for (int n = 0; n < N; ++n) {
                int64_t acc = 0;
                for (int j = b * ORACLE_BLOCK; j < (b + 1) * ORACLE_BLOCK; ++j) {
                    int64_t u = (int64_t)Wq[(int64_t)n * K + j] + 8;   /* zero-extended code */
                    acc += (int64_t)Aq[(int64_t)m * K + j] * u;
                }
                P[((int64_t)m * N + n) * nb + b] = (int32_t)(acc - 8 * sx);
            }
        }
}

/* Y[m][n] = sum_b sx[b][m] * sw[b][n] * P[m][n][b], accumulated in fp64 in block order.
 * Each term is exact in fp64 (11 + 11 + 17 significant bits); only the sum rounds. */
void oracle_epilogue_f64(const int32_t* P, const uint16_t* a_scales, const uint16_t* w_scales,
                         int M, int N, int nb, double* Y) {
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int b = 0; b < nb; ++b) {
                double sx = oracle_f16_to_f32(a_scales[(int64_t)b * M + m]);
                double sw = oracle_f16_to_f32(w_scales[(int64_t)b * N + n]);
                acc += sx * sw * (double)P[((int64_t)m * N + n) * nb + b];
            }
            Y[(int64_t)m * N + n] = acc;
        }
}

/* fp16 value as integer * 2^(e + 24), e + 24 >= 0 (so the unit is 2^-24) */
static void f16_fixed(uint16_t h, int64_t* mant, int* shift) {
    unsigned sign = (h >> 15) & 1u, e = (h >> 10) & 31u, f = h & 1023u;
    int64_t m;
    int sh;
    if (e == 0) { m = f; sh = 0; }                      /* f * 2^-24 */
    else { m = 1024 + f; sh = (int)e - 1; }             /* (1024+f) * 2^(e-25) = m * 2^-24 * 2^(e-1) */
    *mant = sign ? -m : m;
    *shift = sh;
}

/* The same sum evaluated exactly: every term is an integer multiple of 2^-48, summed in a
 * signed 128-bit accumulator, then rounded once to the nearest double. */
void oracle_epilogue_exact(const int32_t* P, const uint16_t* a_scales, const uint16_t* w_scales,
                           int M, int N, int nb, double* Y) {
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            __int128 acc = 0;
            for (int b = 0; b < nb; ++b) {
                int64_t mx, mw;
                int shx, shw;
                f16_fixed(a_scales[(int64_t)b * M + m], &mx, &shx);
                f16_fixed(w_scales[(int64_t)b * N + n], &mw, &shw);
                __int128 t = (__int128)mx * (__int128)mw * (__int128)P[((int64_t)m * N + n) * nb + b];
                acc += t << (shx + shw);
            }
            Y[(int64_t)m * N + n] = ldexp((double)acc, -48);
        }
}

/* Sampled reference for large shapes: for S output positions (ms[s], ns[s]) compute the
 * per-block partials P[s][b] (exact) and Y[s] (fp64, block order) from the codes and scales. */
void oracle_gemm_sample(const int8_t* Aq, const int8_t* Wq, const uint16_t* a_scales,
                        const uint16_t* w_scales, int M, int N, int K, int S,
                        const int32_t* ms, const int32_t* ns, int32_t* P, double* Y) {
    const int nb = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int s = 0; s < S; ++s) {
        const int m = ms[s], n = ns[s];
        double acc = 0.0;
        for (int b = 0; b < nb; ++b) {
            int64_t p = 0;
            for (int j = b * ORACLE_BLOCK; j < (b + 1) * ORACLE_BLOCK; ++j)
                p += (int64_t)Aq[(int64_t)m * K + j] * (int64_t)Wq[(int64_t)n * K + j];
            if (P) P[(int64_t)s * nb + b] = (int32_t)p;
            double sx = oracle_f16_to_f32(a_scales[(int64_t)b * M + m]);
            double sw = oracle_f16_to_f32(w_scales[(int64_t)b * N + n]);
            acc += sx * sw * (double)p;
        }
        Y[s] = acc;
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------------------
 * Offline layout derivation from calibration activations.
 *
 * COMET news article, section 1: the activation outliers concentrate in about 10% of the
 * channels, and a channel permutation gathers them into the same 128-channel blocks, which
 * take 8-bit codes. QUIK explainer, "第一步: 识别与重排": the outlier columns are identified
 * offline on a calibration set and moved to the end of the matrix. Readings (the pages give
 * no formula): the statistic is the channel's absolute maximum over the calibration tokens;
 * channels rank by it, larger first, equal values by lower channel index; the first 128*n8
 * ranked channels fill the last n8 blocks in rank order, the others fill the first blocks in
 * ascending channel order; n8 for an outlier fraction f is ceil(round(f*K) / 128), round
 * taking halves away from zero.
 * ------------------------------------------------------------------------------------ */

/* out[c] = max over the T rows of X [T][K] of |X[t][c]|, as fp16 bits (sign cleared). */
void oracle_channel_absmax(const uint16_t* X, int64_t T, int K, uint16_t* out) {
    for (int c = 0; c < K; ++c) {
        uint16_t m = 0;
        for (int64_t t = 0; t < T; ++t) {
            const uint16_t v = (uint16_t)(X[t * K + c] & 0x7FFFu);
            if (v > m) m = v;
        }
        out[c] = m;
    }
}

typedef struct {
    uint32_t stat;
    int32_t channel;
} ranked_channel;

static int ranked_before(const void* pa, const void* pb) {
    const ranked_channel* a = (const ranked_channel*)pa;
    const ranked_channel* b = (const ranked_channel*)pb;
    if (a->stat != b->stat) return a->stat > b->stat ? -1 : 1;   /* larger statistic first */
    return a->channel < b->channel ? -1 : (a->channel > b->channel ? 1 : 0);
}

/* perm [K], mask [K/128] from the per-channel statistics stat [K]; returns 0, or -1 for bad
 * arguments. */
int oracle_plan_layout(int K, const uint32_t* stat, int n8, int32_t* perm, uint8_t* mask) {
    const int nb = K / 128;
    if (K <= 0 || K % 128 != 0 || n8 < 0 || n8 > nb) return -1;
    ranked_channel* r = (ranked_channel*)malloc(sizeof(ranked_channel) * (size_t)K);
    uint8_t* in_int8 = (uint8_t*)calloc((size_t)K, 1);
    if (r == NULL || in_int8 == NULL) {
        free(r);
        free(in_int8);
        return -1;
    }
    for (int c = 0; c < K; ++c) {
        r[c].stat = stat[c];
        r[c].channel = c;
    }
    qsort(r, (size_t)K, sizeof(ranked_channel), ranked_before);
    const int n_top = 128 * n8;
    for (int i = 0; i < n_top; ++i) in_int8[r[i].channel] = 1;
    int j = 0;
    for (int c = 0; c < K; ++c)
        if (!in_int8[c]) perm[j++] = c;
    for (int i = 0; i < n_top; ++i) perm[j++] = r[i].channel;
    for (int b = 0; b < nb; ++b) mask[b] = (uint8_t)(b >= nb - n8);
    free(r);
    free(in_int8);
    return 0;
}

/* ------------------------------------------------------------------------------------
 * Choosing the number of INT8 blocks by an error budget (COMET news article, section 1: the
 * outlier channels, about 10% of them, are gathered into blocks that keep INT8 precision so
 * that quantization error stays small; QUIK explainer, "第一步: 识别与重排": the outlier columns
 * are identified offline on calibration data). The pages fix no error measure or budget; the
 * reading taken: the error of a layout on calibration tokens is the largest, over the tokens,
 * relative Euclidean error ||x - xhat|| / ||x|| of the token's dequantized codes xhat = q * s
 * (0 for an all-zero token), and the planner takes the smallest n8 whose error is within eps.
 * ------------------------------------------------------------------------------------ */

/* x * 2^24 for a finite fp16 x: an integer (|x| = mant * 2^(max(e,1) - 25)). */
static int64_t f16_times_2p24(uint16_t h) {
    const unsigned e = (h >> 10) & 31u, f = h & 1023u;
    const int64_t mant = e ? 1024 + (int64_t)f : (int64_t)f;
    const int64_t v = mant << (e ? e - 1 : 0);
    return (h & 0x8000u) ? -v : v;
}

/* err = max over the T calibration tokens (fp16 [T][K], input channel order) of
 * sqrt(||x - xhat||^2 / ||x||^2) under the layout (perm, mask). Both squared norms are exact
 * integers in units of 2^-48 (x and q*s are integer multiples of 2^-24), converted once to
 * fp64; the ratio is one fp64 division and one square root. */
int oracle_layout_error(const uint16_t* Xc, int64_t T, int K, const int32_t* perm, const uint8_t* mask, double* err) {
    if (K <= 0 || K % ORACLE_BLOCK != 0) return -1;
    const int nb = K / ORACLE_BLOCK;
    double worst = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t* x = Xc + t * K;
        unsigned __int128 num = 0, den = 0;
        for (int b = 0; b < nb; ++b) {
            uint16_t xs[ORACLE_BLOCK];
            int8_t q[ORACLE_BLOCK];
            for (int j = 0; j < ORACLE_BLOCK; ++j) xs[j] = x[perm[b * ORACLE_BLOCK + j]];
            const uint16_t s16 = quantize_block(xs, mask[b] ? 127 : 7, q);
            const int64_t ns = f16_times_2p24(s16);
            for (int j = 0; j < ORACLE_BLOCK; ++j) {
                const int64_t nx = f16_times_2p24(xs[j]);
                const int64_t nd = nx - (int64_t)q[j] * ns;
                num += (unsigned __int128)((__int128)nd * nd);
                den += (unsigned __int128)((__int128)nx * nx);
            }
        }
        const double e = den != 0 ? sqrt((double)num / (double)den) : 0.0;
        if (e > worst) worst = e;
    }
    *err = worst;
    return 0;
}

/* The smallest n8 in [0, K/128] whose planned layout (oracle_plan_layout with that n8) has an
 * error within eps on the calibration tokens; when none has, n8 = K/128 (every block INT8).
 * Writes that layout, n8 and its error. */
int oracle_plan_layout_budget(int K, const uint32_t* stat, const uint16_t* Xc, int64_t T, double eps, int32_t* n8_out,
                              double* err_out, int32_t* perm, uint8_t* mask) {
    if (K <= 0 || K % ORACLE_BLOCK != 0) return -1;
    const int nb = K / ORACLE_BLOCK;
    for (int n8 = 0;; ++n8) {
        double e = 0.0;
        if (oracle_plan_layout(K, stat, n8, perm, mask) != 0 || oracle_layout_error(Xc, T, K, perm, mask, &e) != 0)
            return -1;
        if (e <= eps || n8 == nb) {
            *n8_out = n8;
            *err_out = e;
            return 0;
        }
    }
}

/* ------------------------------------------------------------------------------------
 * RMSNorm fused into the quantizer (QServe explainer, "运行时设计": the activation
 * quantization of the QKV projection and the first FFN layer is fused into the layer norm
 * before them; the LLaMA family's layer norm is RMSNorm, y = x / sqrt(mean(x^2) + eps) * gamma).
 * The sum of squares T is the exact real sum of the squared fp16 inputs, rounded once to
 * fp32 (round to nearest, ties to even): it does not depend on any summation order. Every
 * later step is one IEEE fp32 operation, so the normalized fp16 values are exact functions of
 * the input. The quantizer above then takes y as its input.
 * ------------------------------------------------------------------------------------ */

/* A finite fp16 value is n * 2^-24 for an integer n (|n| < 2^40), so its square is n^2 * 2^-48:
 * an integer count of 2^-48 below 2^80, and a row of at most 32768 of them stays below 2^95. */
static unsigned __int128 f16_square_fixed48(uint16_t h) {
    const unsigned e = (h >> 10) & 31u, f = h & 1023u;
    const uint64_t mant = e ? (1024u + f) : f;           /* |x| = mant * 2^(max(e,1) - 25) */
    const unsigned shift = 2u * (e ? e : 1u) - 2u;       /* x^2 = mant^2 * 2^(shift - 48) */
    return (unsigned __int128)(mant * mant) << shift;
}

/* Round v * 2^-48 (v an exact non-negative integer) to the nearest fp32, ties to even. */
static float fixed48_to_f32(unsigned __int128 v) {
    if (v == 0) return 0.0f;
    int bits = 0;
    for (unsigned __int128 t = v; t != 0; t >>= 1) ++bits;
    if (bits <= 24) return ldexpf((float)(uint64_t)v, -48);  /* exact */
    const int drop = bits - 24;
    uint64_t q = (uint64_t)(v >> drop);                       /* the top 24 bits */
    const unsigned __int128 rem = v - ((unsigned __int128)q << drop);
    const unsigned __int128 half = (unsigned __int128)1 << (drop - 1);
    if (rem > half || (rem == half && (q & 1u))) ++q;         /* q may become 2^24: still exact */
    return ldexpf((float)q, drop - 48);
}

/* T[m] = the exact sum of X[m][c]^2 over the K channels, rounded once to fp32. */
void oracle_rmsnorm_sumsq(const uint16_t* X, int64_t ldx, int M, int K, float* T) {
    for (int m = 0; m < M; ++m) {
        unsigned __int128 acc = 0;
        for (int c = 0; c < K; ++c) acc += f16_square_fixed48(X[(int64_t)m * ldx + c]);
        T[m] = fixed48_to_f32(acc);
    }
}

/* Y [M][K] (input channel order) = RMSNorm of X [M][ldx] with gamma [K] (input order):
 * r = 1 / sqrt(T / K + eps), y = fp16_rn((fp32(x) * r) * fp32(gamma)), each an IEEE fp32 step. */
void oracle_rmsnorm(const uint16_t* X, int64_t ldx, int M, int K, const uint16_t* gamma, float eps, uint16_t* Y) {
    for (int m = 0; m < M; ++m) {
        float t;
        oracle_rmsnorm_sumsq(X + (int64_t)m * ldx, ldx, 1, K, &t);
        const float ms = t / (float)K;
        const float r = 1.0f / sqrtf(ms + eps);
        const uint16_t* x = X + (int64_t)m * ldx;
        for (int c = 0; c < K; ++c)
            Y[(int64_t)m * K + c] = oracle_f32_to_f16((oracle_f16_to_f32(x[c]) * r) * oracle_f16_to_f32(gamma[c]));
    }
}

/* ------------------------------------------------------------------------------------
 * SwiGLU fused into the quantizer (QServe explainer, "运行时设计": the activation quantization
 * of the second FFN layer is fused into the activation kernel before it; the LLaMA FFN's
 * activation is SwiGLU, h = silu(g) * u with silu(g) = g / (1 + e^-g), g and u the gate and up
 * projections' outputs). The page gives no precision; the reading taken: h is the real value
 * g * u / (1 + e^-g) rounded once to fp16 (ties to even). Here it is evaluated in fp64: g * u
 * is exact, exp and the division err by a few 2^-53, far below fp16's rounding step, so the
 * result is the correctly rounded value unless the exact one lies within ~2^-50 (relative) of
 * an fp16 rounding boundary. A zero result keeps the IEEE sign of g * u.
 * ------------------------------------------------------------------------------------ */
void oracle_swiglu(const uint16_t* G, const uint16_t* U, int64_t n, uint16_t* H) {
    for (int64_t i = 0; i < n; ++i) {
        const double g = (double)oracle_f16_to_f32(G[i]);
        const double u = (double)oracle_f16_to_f32(U[i]);
        H[i] = f64_to_f16((g * u) / (1.0 + exp(-g)));
    }
}

/* ====================================================================================
 * Quantization variants the pages describe beside FMPQ.
 * ==================================================================================== */

/* Order key of fp16 bits that follows the value order (-0 sorts below +0; no NaN inputs). */
static unsigned f16_order_key(uint16_t h) { return (h & 0x8000u) ? (unsigned)(uint16_t)~h : (unsigned)(h | 0x8000u); }

/* round-half-even of the exact rational a / b, b > 0 (integers) */
static int rne_div(int a, int b) {
    int q = a / b, r = a % b;                 /* C truncates toward zero */
    if (r < 0) { q -= 1; r += b; }            /* floor division: 0 <= r < b */
    if (2 * r > b) return q + 1;
    if (2 * r == b) return (q % 2 == 0) ? q : q + 1;
    return q;
}

/* ---- QUIK asymmetric activations (QUIK explainer, "反量化背后的数学": activations take a
 * scale and a zero point, weights a scale only; the zero point's contribution z * sum(w)
 * needs only the weights' sum, computed offline).
 *
 * Reading, per token and 128-channel block (every block 4-bit; QUIK's outliers stay fp16):
 *   z = the block's smallest input (value order, -0 below +0), stored as fp16
 *   s = fp16_rne( fp32( fp32(max) - fp32(z) ) / 15 )             IEEE fp32 operations
 *   q = clamp( rne( fp32( fp32(x) - fp32(z) ) / fp32(s) ), 0, 15 ),  q = 0 when s == 0
 * so x ~ s * q + z. Codes are packed like INT4 codes (one plane, byte = E4M3 of q * 2^-9)
 * with the sign bit clear. */
static void quantize_block_asym(const uint16_t* xs, int8_t* q, uint16_t* s_bits, uint16_t* z_bits) {
    uint16_t lo = xs[0], hi = xs[0];
    for (int j = 1; j < ORACLE_BLOCK; ++j) {
        if (f16_order_key(xs[j]) < f16_order_key(lo)) lo = xs[j];
        if (f16_order_key(xs[j]) > f16_order_key(hi)) hi = xs[j];
    }
    const float z = oracle_f16_to_f32(lo);
    const float d = oracle_f16_to_f32(hi) - z;             /* IEEE fp32 subtraction */
    const float s32 = d / 15.0f;                            /* IEEE fp32 division */
    const uint16_t s16 = oracle_f32_to_f16(s32);
    const float s = oracle_f16_to_f32(s16);
    for (int j = 0; j < ORACLE_BLOCK; ++j) {
        if (s == 0.0f) { q[j] = 0; continue; }
        const float t = (oracle_f16_to_f32(xs[j]) - z) / s;
        int32_t v = rne_f32_to_int(t);
        if (v > 15) v = 15;
        if (v < 0) v = 0;
        q[j] = (int8_t)v;
    }
    *s_bits = s16;
    *z_bits = lo;
}

/* X fp16 [M][ldx] -> packed codes (every block one plane), a_scales and a_zeros [nb][M]
 * (fp16 bits) and, if Aq != NULL, the codes Aq [M][K] (0..15, permuted channel order). */
int oracle_quantize_activations_asym(const uint16_t* X, int64_t ldx, int M, int K, const int32_t* perm,
                                     uint8_t* A_packed, uint16_t* a_scales, uint16_t* a_zeros, int8_t* Aq) {
    if (K % ORACLE_BLOCK) return -1;
    const int nb = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m) {
        uint16_t xs[ORACLE_BLOCK];
        int8_t q[ORACLE_BLOCK];
        for (int b = 0; b < nb; ++b) {
            for (int j = 0; j < ORACLE_BLOCK; ++j) xs[j] = X[(int64_t)m * ldx + perm[b * ORACLE_BLOCK + j]];
            quantize_block_asym(xs, q, &a_scales[(int64_t)b * M + m], &a_zeros[(int64_t)b * M + m]);
            uint8_t* row = A_packed + (int64_t)b * M * ORACLE_BLOCK + (int64_t)m * ORACLE_BLOCK;
            for (int c = 0; c < ORACLE_BLOCK; ++c) row[plane_pos(m, c)] = (uint8_t)e4m3_of_multiple(q[c]);
            if (Aq)
                for (int j = 0; j < ORACLE_BLOCK; ++j) Aq[(int64_t)m * K + b * ORACLE_BLOCK + j] = q[j];
        }
    }
    return 0;
}

/* Offline weight sums for the zero-point term: wsum[b][n] = sw[b][n] * sum_{j in b} Wq[n][j]
 * (the block's dequantized weights summed; exact in fp32: 11-bit scale times |sum| <= 896). */
void oracle_weight_sums(const int8_t* Wq, const uint16_t* w_scales, int N, int K, float* wsum) {
    const int nb = K / ORACLE_BLOCK;
    for (int n = 0; n < N; ++n)
        for (int b = 0; b < nb; ++b) {
            int64_t t = 0;
            for (int j = b * ORACLE_BLOCK; j < (b + 1) * ORACLE_BLOCK; ++j) t += Wq[(int64_t)n * K + j];
            wsum[(int64_t)b * N + n] = (float)((double)oracle_f16_to_f32(w_scales[(int64_t)b * N + n]) * (double)t);
        }
}

/* Y[m][n] = sum_b ( sx[b][m] * sw[b][n] * P[m][n][b] + z[b][m] * wsum[b][n] ), fp64 in block
 * order; P are the integer sums of the unsigned activation codes times the weight codes. */
void oracle_epilogue_asym_f64(const int32_t* P, const uint16_t* a_scales, const uint16_t* a_zeros,
                              const uint16_t* w_scales, const float* wsum, int M, int N, int nb, double* Y) {
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int b = 0; b < nb; ++b) {
                const double sx = oracle_f16_to_f32(a_scales[(int64_t)b * M + m]);
                const double z = oracle_f16_to_f32(a_zeros[(int64_t)b * M + m]);
                const double sw = oracle_f16_to_f32(w_scales[(int64_t)b * N + n]);
                acc += sx * sw * (double)P[((int64_t)m * N + n) * nb + b] + z * (double)wsum[(int64_t)b * N + n];
            }
            Y[(int64_t)m * N + n] = acc;
        }
}

/* ---- QoQ progressive group quantization (QServe explainer, "渐进式分组量化"): the weights are
 * first quantized per output channel to symmetric INT8, then each group of those INT8 values
 * to asymmetric UINT4. The INT8 range is narrowed to [-119, 119] (the protective range) so
 * that the dequantized (q4 - z2) * s2 never leaves the INT8 range.
 *
 * Reading (the page gives no formulas):
 *   s1[n] = fp16_rne( fp32(absmax of row n) / 119 )               IEEE fp32 division
 *   q8    = clamp( rne_f32( fp32(w) / fp32(s1) ), -119, 119 )      q8 = 0 when s1 == 0
 *   per group g of 128 channels (the permuted order's blocks), the range [mn, mx] of its q8
 *   extended to include 0 (mn = min(min q8, 0), mx = max(max q8, 0)), so that the zero point
 *   is a code:
 *   s2 = max(1, ceil((mx - mn) / 15))  the smallest integer scale spanning the range in 15 steps
 *   z2 = clamp( rne(-mn / s2), 0, 15 ) integer zero point
 *   q4 = clamp( rne(q8 / s2) + z2, 0, 15 )                        (rne of exact rationals)
 * Dequantized weight: s1 * s2 * (q4 - z2). Every quotient here is an exact rational, rounded
 * half to even. With |q8| <= 119 the scale is at most ceil(238 / 15) = 16, and a code's
 * dequantized value is within s2 / 2 <= 8 of q8 or clipped toward 0, so it stays in
 * [-127, 127]. */
void oracle_qoq_group(const int8_t* q8, int* s2_out, int* z2_out, uint8_t* q4) {
    int mn = 0, mx = 0;                       /* the range always includes 0 */
    for (int j = 0; j < ORACLE_BLOCK; ++j) {
        if (q8[j] < mn) mn = q8[j];
        if (q8[j] > mx) mx = q8[j];
    }
    int s2 = (mx - mn + 14) / 15;             /* ceil, mx - mn >= 0 */
    if (s2 < 1) s2 = 1;
    int z2 = rne_div(-mn, s2);
    if (z2 < 0) z2 = 0;
    if (z2 > 15) z2 = 15;
    for (int j = 0; j < ORACLE_BLOCK; ++j) {
        int v = rne_div(q8[j], s2) + z2;
        if (v < 0) v = 0;
        if (v > 15) v = 15;
        q4[j] = (uint8_t)v;
    }
    *s2_out = s2;
    *z2_out = z2;
}

/* Batch form for tests: G groups of 128 INT8 values. */
void oracle_qoq_group_batch(const int8_t* q8, int G, int32_t* s2, int32_t* z2, uint8_t* q4) {
    for (int g = 0; g < G; ++g) {
        int a, c;
        oracle_qoq_group(q8 + (int64_t)g * ORACLE_BLOCK, &a, &c, q4 + (int64_t)g * ORACLE_BLOCK);
        s2[g] = a;
        z2[g] = c;
    }
}

/* W fp16 [N][ldw] -> q8 [N][K] and q4 [N][K] (permuted channel order), s1 [N] (fp16 bits),
 * s2 and z2 [nb][N]. */
int oracle_qoq_quantize_weights(const uint16_t* W, int64_t ldw, int N, int K, const int32_t* perm, int8_t* q8,
                                uint8_t* q4, uint16_t* s1, uint8_t* s2, uint8_t* z2) {
    if (K % ORACLE_BLOCK) return -1;
    const int nb = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        float absmax = 0.0f;
        for (int c = 0; c < K; ++c) {
            const float v = fabsf(oracle_f16_to_f32(W[(int64_t)n * ldw + c]));
            if (v > absmax) absmax = v;
        }
        const uint16_t sb = oracle_f32_to_f16(absmax / 119.0f);
        const float s = oracle_f16_to_f32(sb);
        s1[n] = sb;
        int8_t* r8 = q8 + (int64_t)n * K;
        for (int j = 0; j < K; ++j) {
            if (s == 0.0f) { r8[j] = 0; continue; }
            int32_t v = rne_f32_to_int(oracle_f16_to_f32(W[(int64_t)n * ldw + perm[j]]) / s);
            if (v > 119) v = 119;
            if (v < -119) v = -119;
            r8[j] = (int8_t)v;
        }
        for (int b = 0; b < nb; ++b) {
            int a, c;
            oracle_qoq_group(r8 + b * ORACLE_BLOCK, &a, &c, q4 + (int64_t)n * K + b * ORACLE_BLOCK);
            s2[(int64_t)b * N + n] = (uint8_t)a;
            z2[(int64_t)b * N + n] = (uint8_t)c;
        }
    }
    return 0;
}

/* QoQ activations (QServe explainer, "运行时设计": every GEMM takes W4A8 inputs): per-token
 * symmetric INT8, s = fp16_rne(fp32(absmax of the row) / 127), q = clamp(rne_f32(x / s), ±127),
 * every block packed as an INT8 block (two planes); a_sums[b][m] = sum of the block's codes
 * (the term the group zero point multiplies). */
int oracle_qoq_quantize_activations(const uint16_t* X, int64_t ldx, int M, int K, const int32_t* perm,
                                    uint8_t* A_packed, uint16_t* a_scales, int32_t* a_sums, int8_t* Aq) {
    if (K % ORACLE_BLOCK) return -1;
    const int nb = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m) {
        float absmax = 0.0f;
        for (int c = 0; c < K; ++c) {
            const float v = fabsf(oracle_f16_to_f32(X[(int64_t)m * ldx + c]));
            if (v > absmax) absmax = v;
        }
        const uint16_t sb = oracle_f32_to_f16(absmax / 127.0f);
        const float s = oracle_f16_to_f32(sb);
        a_scales[m] = sb;
        uint16_t xs[ORACLE_BLOCK];
        int8_t q[ORACLE_BLOCK];
        for (int b = 0; b < nb; ++b) {
            int32_t sum = 0;
            for (int j = 0; j < ORACLE_BLOCK; ++j) {
                xs[j] = X[(int64_t)m * ldx + perm[b * ORACLE_BLOCK + j]];
                int32_t v = 0;
                if (s != 0.0f) {
                    v = rne_f32_to_int(oracle_f16_to_f32(xs[j]) / s);
                    if (v > 127) v = 127;
                    if (v < -127) v = -127;
                }
                q[j] = (int8_t)v;
                sum += v;
            }
            a_sums[(int64_t)b * M + m] = sum;
            pack_block_row(q, xs, 1, A_packed, 2 * (int64_t)b, M, m);
            if (Aq)
                for (int j = 0; j < ORACLE_BLOCK; ++j) Aq[(int64_t)m * K + b * ORACLE_BLOCK + j] = q[j];
        }
    }
    return 0;
}

/* Y[m][n] = sum_b sx[m] * s1[n] * s2[b][n] * ( P[m][n][b] - z2[b][n] * a_sums[b][m] ), fp64 in
 * block order, P = exact sums of the INT8 activation codes times the UINT4 codes q4 (the zero
 * point subtracted after the multiplication, as the QServe explainer's "W4A8逐组快速反量化" does). */
void oracle_epilogue_qoq_f64(const int32_t* P, const uint16_t* a_scales, const int32_t* a_sums, const uint16_t* s1,
                             const uint8_t* s2, const uint8_t* z2, int M, int N, int nb, double* Y) {
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int b = 0; b < nb; ++b) {
                const int64_t g = (int64_t)b * N + n;
                const int64_t pz = (int64_t)P[((int64_t)m * N + n) * nb + b] - (int64_t)z2[g] * a_sums[(int64_t)b * M + m];
                acc += (double)s2[g] * (double)pz;
            }
            Y[(int64_t)m * N + n] = (double)oracle_f16_to_f32(a_scales[m]) * (double)oracle_f16_to_f32(s1[n]) * acc;
        }
}

/* Sampled outputs of the two variants for large shapes, (ms[s], ns[s]) positions: exact partial
 * sums P[s][b] and Y[s] by the variant's formula above (fp64, block order). */
void oracle_gemm_sample_asym(const int8_t* Aq, const int8_t* Wq, const uint16_t* a_scales, const uint16_t* a_zeros,
                             const uint16_t* w_scales, const float* wsum, int M, int N, int K, int S,
                             const int32_t* ms, const int32_t* ns, int32_t* P, double* Y) {
    const int nb = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int s = 0; s < S; ++s) {
        const int m = ms[s], n = ns[s];
        double acc = 0.0;
        for (int b = 0; b < nb; ++b) {
            int64_t p = 0;
            for (int j = b * ORACLE_BLOCK; j < (b + 1) * ORACLE_BLOCK; ++j)
                p += (int64_t)Aq[(int64_t)m * K + j] * (int64_t)Wq[(int64_t)n * K + j];
            if (P) P[(int64_t)s * nb + b] = (int32_t)p;
            const double sx = oracle_f16_to_f32(a_scales[(int64_t)b * M + m]);
            const double z = oracle_f16_to_f32(a_zeros[(int64_t)b * M + m]);
            const double sw = oracle_f16_to_f32(w_scales[(int64_t)b * N + n]);
            acc += sx * sw * (double)p + z * (double)wsum[(int64_t)b * N + n];
        }
        Y[s] = acc;
    }
}

void oracle_gemm_sample_qoq(const int8_t* Aq, const uint8_t* q4, const uint16_t* a_scales, const int32_t* a_sums,
                            const uint16_t* s1, const uint8_t* s2, const uint8_t* z2, int M, int N, int K, int S,
                            const int32_t* ms, const int32_t* ns, int32_t* P, double* Y) {
    const int nb = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int s = 0; s < S; ++s) {
        const int m = ms[s], n = ns[s];
        double acc = 0.0;
        for (int b = 0; b < nb; ++b) {
            int64_t p = 0;
            for (int j = b * ORACLE_BLOCK; j < (b + 1) * ORACLE_BLOCK; ++j)
                p += (int64_t)Aq[(int64_t)m * K + j] * (int64_t)q4[(int64_t)n * K + j];
            if (P) P[(int64_t)s * nb + b] = (int32_t)p;
            const int64_t g = (int64_t)b * N + n;
            acc += (double)s2[g] * (double)(p - (int64_t)z2[g] * a_sums[(int64_t)b * M + m]);
        }
        Y[s] = (double)oracle_f16_to_f32(a_scales[m]) * (double)oracle_f16_to_f32(s1[n]) * acc;
    }
}
