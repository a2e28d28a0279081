// FMPQ activation quantizer and offline weight packing (sm_103a).
//
// Activation quantizer: one fused pass per token row -- gather-permute (QUIK explainer,
// "kernel fusion": one kernel reads the input, computes the statistics, quantizes and
// splits in a single pass), per-(token, 128-channel block) absmax, fp16 scale, exact
// round-half-even quantization to INT8 (outlier blocks) or INT4 (the rest; COMET news
// article, section 1), and encoding into the operand-ready code planes documented in fmpq.h.
//
// Design: persistent CTAs (one per SM, two for short rows) stream whole rows into shared
// memory with bulk copies (a dedicated producer warp, several stages), take each lane's
// gather offsets from a table staged once in shared memory, gather from the staged rows, and
// write the code planes with coalesced stores (each half-warp writes one 128-byte plane row).
// Other modes of the same kernel: RMSNorm fused in front (norm warps compute each row's
// factor ahead of the quantizing warps), QUIK asymmetric codes with zero points, and QoQ
// per-token INT8 codes with block code sums.
#include <cuda_fp16.h>

#include "fmpq_device.cuh"
#include "fmpq_internal.h"

namespace fmpq {
namespace {

// ---------------------------------------------------------------------------------
// Weight quantization (offline packing): per-lane quantization of 4 values of one block
// (the warp covers the block's 128 channels, 4 per lane). Returns the 4 sign-magnitude bytes (byte i = element i) and,
// through *scale_bits, the block's fp16 scale.
//
// Scale: s = fp16_rne(fp32(absmax) / qmax) with IEEE division.
// Codes: q = clamp(rne(x / s), -qmax, qmax), where rne(x/s) is the round-half-even of the
// exact quotient. For fp16 x and s the exact quotient is never within 3e-5 of a
// half-integer unless it is one, so this equals rounding the fp32 IEEE quotient; it is
// computed as a reciprocal multiply (error < 2e-5) whose few near-half cases (|frac| >
// 0.4999) are resolved with the exact remainder x - q*s (one FMA, exact here).
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t quantize4(const uint16_t (&h)[4], int qmax, uint16_t* scale_bits) {
    uint32_t a = max(max(h[0] & 0x7FFFu, h[1] & 0x7FFFu), max(h[2] & 0x7FFFu, h[3] & 0x7FFFu));
    a = __reduce_max_sync(0xFFFFFFFFu, a);
    const float amax = __half2float(__ushort_as_half(static_cast<unsigned short>(a)));
    const __half s16 = __float2half_rn(__fdiv_rn(amax, static_cast<float>(qmax)));
    *scale_bits = __half_as_ushort(s16);
    const float s = __half2float(s16);
    if (s == 0.0f) return 0u;  // warp-uniform

    const float inv = __frcp_rn(s);
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer (RNE)
    float ax[4], r[4];
    uint32_t mag[4];
    bool near_half = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x = __half2float(__ushort_as_half(h[i]));
        ax[i] = fabsf(x);
        const float t = __fmul_rn(ax[i], inv) + kMagic;
        r[i] = t - kMagic;                                   // rint(|x| * inv), exact
        mag[i] = __float_as_uint(t) & 0x3FFu;
        const float f = __fmul_rn(ax[i], inv) - r[i];
        near_half |= (fabsf(f) > 0.4999f);
    }
    if (__any_sync(0xFFFFFFFFu, near_half)) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float e = fmaf(-r[i], s, ax[i]);           // exact remainder |x| - r*s
            const float e2 = e + e;
            if (e2 > s) {
                mag[i] += 1;
            } else if (e2 < -s) {
                mag[i] -= 1;
            } else if ((e2 == s || e2 == -s) && (mag[i] & 1u)) {
                mag[i] = (e2 > 0.0f) ? mag[i] + 1 : mag[i] - 1;  // tie: to even
            }
        }
    }
    if (s < 6.103515625e-05f) {  // subnormal scale: rounding can overshoot qmax (warp-uniform)
#pragma unroll
        for (int i = 0; i < 4; ++i) mag[i] = min(mag[i], static_cast<uint32_t>(qmax));
    }
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t sign = ((h[i] & 0x8000u) && mag[i]) ? 0x80u : 0u;
        v |= (mag[i] | sign) << (8 * i);
    }
    return v;
}

// INT4 packing of a warp's 4-code groups: lanes 2g and 2g+1 hold channels 8g..8g+3 and
// 8g+4..8g+7 as sign-magnitude bytes v; the packed word is v_even | rotl(v_odd, 4)
// (magnitudes 4..7 move to bits 4-6 and their signs to bit 3 of the next byte).
// Valid in even lanes.
__device__ __forceinline__ uint32_t pack_int4_pair(uint32_t v, int lane) {
    const uint32_t mine = (lane & 1) ? __funnelshift_l(v, v, 4) : v;
    return mine | __shfl_xor_sync(0xFFFFFFFFu, mine, 1);
}

// ---------------------------------------------------------------------------------
// Activation quantizer.
//
// A warp quantizes two blocks of one token at a time: lanes 0-15 one block, lanes 16-31
// another, 8 channels per lane. Warp w of the W compute warps owns blocks w, w + W, w + 2W,
// ... for every token, so its gather offsets are the same for every row: they are staged
// once in a shared-memory table. Rows of X are streamed into a shared-memory ring by a
// producer warp (bulk copies); the gather reads them from there.
//
// Output: operand-ready code planes (layout in fmpq.h). A code's byte is sign<<7 | the
// E4M3 encoding of part * 2^-9: INT4 part = |q|; INT8 low part = |q| & 15 (the same bits),
// INT8 high part = |q| & 0x70, whose E4M3 encoding is looked up in an 8-entry table.
// The sign bit is the sign bit of the fp16 input.
// ---------------------------------------------------------------------------------
// Compute warps W: per round the half-warps of warp w take blocks w + 2Wj and w + W + 2Wj. The
// launch picks the largest W in [16, 28] with nb a multiple of 2W (every warp the same number of
// rounds), else 16; the fused-norm kernel uses 16 compute warps and 8 norm warps, the per-token
// INT8 kernel 24 compute warps and 4 absmax warps.
constexpr int kQWarpsMin = 16, kQWarpsMax = 28;
constexpr int kQNormWarps = 8;                     // fused RMSNorm: warps computing the rows' norms
constexpr int kQTokWarps = 4;                      // per-token INT8: warps taking the rows' absmax
constexpr int kQMaxThreads = (kQWarpsMax + 1) * 32;   // >= (16 + 1 + 8) * 32 and (24 + 1 + 4) * 32
constexpr int kQSmemBudget = 200 * 1024;
enum : int { kQSym = 0, kQNorm = 1, kQAsym = 2, kQTok = 3 };   // quantizer modes

struct QuantParams {
    const uint16_t* X;
    int64_t ldx;
    int64_t M;
    int K, nb, stages;
    int Kin;                // staged row width: the channels a layout may select from (>= K)
    int iters;              // rounds per compute warp: ceil(nb / (2 * cwarps))
    int cwarps;             // compute warps (the producer is warp cwarps, statistic warps follow)
    int rwarps;             // row-statistic warps (fused RMSNorm: 8; per-token INT8 absmax: 4)
    const uint16_t* perm;
    const uint8_t* mask;
    const int32_t* poff;
    uint8_t* A;
    uint16_t* scales;
    int32_t* status;
    const uint16_t* gamma_perm;   // fused RMSNorm: gamma in the permuted channel order
    float eps;
    uint16_t* zeros;              // QUIK asymmetric: zero points [nb][M]
    int32_t* sums;                // QoQ per-token INT8: sums of each block's codes [nb][M]
    // QUIK input split: X_out[m][j] = X[m][split_cols[j]] (fp16, 0 outside the row's width)
    const int32_t* split_cols;
    int n_split;                  // a multiple of 8; 0 = no split
    uint16_t* X_out;
};

// Outlier columns cols[0..n) of one row into out[0..n): lane l takes columns 8l..8l+7 of every
// 256, read through load(c) for 0 <= c < width (0 otherwise), one 16-byte store per 8 columns.
template <typename Load>
__device__ __forceinline__ void split_row(const int32_t* cols, int n, uint16_t* out, int lane, int width, Load load) {
    for (int j0 = 8 * lane; j0 < n; j0 += 256) {
        const int4 c0 = __ldg(reinterpret_cast<const int4*>(cols + j0));
        const int4 c1 = __ldg(reinterpret_cast<const int4*>(cols + j0 + 4));
        const int c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint32_t h[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) h[k] = (c[k] >= 0 && c[k] < width) ? static_cast<uint32_t>(load(c[k])) : 0u;
        *reinterpret_cast<uint4*>(out + j0) =
            make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
    }
}

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Byte 0 of four floats -> one word (a magnitude r sits in the low mantissa byte of
// r + 1.5 * 2^23).
__device__ __forceinline__ uint32_t low_bytes4(float a, float b, float c, float d) {
    const uint32_t ab = __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x0040);
    const uint32_t cd = __byte_perm(__float_as_uint(c), __float_as_uint(d), 0x0040);
    return __byte_perm(ab, cd, 0x5410);
}

// INT8 high plane from the sign-magnitude code bytes w: byte = sign | E4M3(16h * 2^-9),
// h = bits 4-6 of the magnitude. E4M3 of h * 2^-5 for h = 0..7:
// 0x00 0x10 0x18 0x1C 0x20 0x22 0x24 0x26.
__device__ __forceinline__ uint32_t high_plane(uint32_t w) {
    const uint32_t hw = (w >> 4) & 0x07070707u;           // h per byte
    const uint32_t nib = hw | (hw >> 4);                   // nibbles h0 h1 . h2 ...
    const uint32_t sel = __byte_perm(nib, 0u, 0x0020);     // selector nibbles h0 h1 h2 h3
    return __byte_perm(0x1C181000u, 0x26242220u, sel) | (w & 0x80808080u);
}

// Order key of two fp16 values (one per half of the word): a 16-bit key per half that orders
// like the values, -0 below +0 (negative: all bits flipped; positive: the sign bit set).
__device__ __forceinline__ uint32_t f16x2_order_keys(uint32_t x) {
    return x ^ (0x80008000u | (((x >> 15) & 0x00010001u) * 0x7FFFu));
}
__device__ __forceinline__ uint32_t f16_from_order_key(uint32_t k) { return (k ^ ((k & 0x8000u) ? 0x8000u : 0xFFFFu)) & 0xFFFFu; }

// One QUIK-asymmetric block step of a half-warp (8 values per lane in h2): zero point, scale,
// codes in [0, 15], stores. The quotient (x - z) / s is approximated by a product with the
// reciprocal (error below 2^-17 for quotients up to 16); where that lands within 2^-16 of a
// half-integer the warp recomputes its quotients with IEEE division, so the rounding is that
// of the IEEE fp32 quotient.
template <typename Params>
__device__ __forceinline__ void quantize_asym_step(const Params& p, const uint32_t (&h2)[4], bool valid, int b, int64_t m,
                                                   uint32_t chunk_off, int sub, uint32_t hmask, const int32_t* s_poff) {
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t key = f16x2_order_keys(h2[k]);
        kmin = __vminu2(kmin, key);
        kmax = __vmaxu2(kmax, key);
    }
    kmin = __reduce_min_sync(hmask, min(kmin & 0xFFFFu, kmin >> 16));
    kmax = __reduce_max_sync(hmask, max(kmax & 0xFFFFu, kmax >> 16));
    const uint32_t zbits = f16_from_order_key(kmin);
    const float z = __half2float(__ushort_as_half(static_cast<unsigned short>(zbits)));
    const float mx = __half2float(__ushort_as_half(static_cast<unsigned short>(f16_from_order_key(kmax))));
    const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, z), 15.0f));
    const float sc = __half2float(s16);
    const float inv = sc > 0.0f ? rcp_approx(sc) : 0.0f;
    constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23: adding it rounds to an integer (RNE)
    float d[8], tm[8];
    bool near_half = false;
    // two channels per instruction (fma.rn.f32x2: the IEEE fma in each half)
    const float2 inv2 = make_float2(inv, inv), mg2 = make_float2(kMagic, kMagic);
    const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2[k]));
        const float2 d2 = make_float2(__fsub_rn(f.x, z), __fsub_rn(f.y, z));
        const float2 t2 = dev::ffma2(d2, inv2, mg2);
        const float2 f2 = dev::ffma2(d2, inv2, dev::ffma2(t2, neg1, mg2));   // (x - z) * inv - rounded
        d[2 * k] = d2.x;
        d[2 * k + 1] = d2.y;
        tm[2 * k] = t2.x;
        tm[2 * k + 1] = t2.y;
        near_half |= fmaxf(fabsf(f2.x), fabsf(f2.y)) >= 0.5f - 1.52587890625e-05f;   // 2^-16
    }
    if (__any_sync(0xFFFFFFFFu, near_half && sc > 0.0f)) {
        if (sc > 0.0f) {
#pragma unroll
            for (int k = 0; k < 8; ++k) tm[k] = __fadd_rn(__fdiv_rn(d[k], sc), kMagic);
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) tm[k] = sc > 0.0f ? fminf(tm[k], kMagic + 15.0f) : kMagic;
    const uint32_t w0 = low_bytes4(tm[0], tm[1], tm[2], tm[3]);
    const uint32_t w1 = low_bytes4(tm[4], tm[5], tm[6], tm[7]);
    if (valid) {
        uint8_t* dst = p.A + (static_cast<int64_t>(s_poff[b]) * p.M + m) * kBlock + chunk_off;
        *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
        if (sub == 0) {
            p.scales[static_cast<int64_t>(b) * p.M + m] = __half_as_ushort(s16);
            p.zeros[static_cast<int64_t>(b) * p.M + m] = static_cast<uint16_t>(zbits);
        }
    }
}

// One block step of the symmetric quantizer for a warp: each half-warp holds 8 fp16 values
// per lane (h2: half2 words) of one 128-channel block b of token m. It takes the block's absmax
// (kTok: the row's absmax tok_amax instead), the fp16 scale, the codes rne(|x| / s) and their
// operand-ready bytes, and writes them to the block's plane(s) (first plane poff_b of planes of M
// rows) and the scale (kTok: the sum of the block's codes) when `valid`. Both half-warps call it
// together: it votes across the warp.
template <bool kTok>
__device__ __forceinline__ void quantize_codes_step(const uint32_t (&h2)[4], bool valid, bool is8, int b, int64_t m,
                                                    uint32_t chunk_off, int sub, uint32_t hmask, int32_t poff_b,
                                                    uint8_t* A, int64_t M, uint16_t* scales, int32_t* sums,
                                                    float tok_amax) {
    // absmax of the half-warp's 128 values
    uint32_t ab[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) ab[k] = h2[k] & 0x7FFF7FFFu;
    const __half2 m01 = __hmax2(*reinterpret_cast<const __half2*>(&ab[0]),
                                *reinterpret_cast<const __half2*>(&ab[1]));
    const __half2 m23 = __hmax2(*reinterpret_cast<const __half2*>(&ab[2]),
                                *reinterpret_cast<const __half2*>(&ab[3]));
    const __half2 mx = __hmax2(m01, m23);
    const __half lm = __hmax(__low2half(mx), __high2half(mx));
    const uint32_t amax_bits = __reduce_max_sync(hmask, static_cast<uint32_t>(__half_as_ushort(lm)));
    // scale: fp16(fp32(absmax) * fp32(1/qmax)) equals fp16(fp32(absmax) / qmax)
    // for every finite fp16 absmax and qmax in {7, 127}; per-token INT8 takes the
    // row's absmax instead of the block's
    const float amax = kTok ? tok_amax : __half2float(__ushort_as_half(static_cast<unsigned short>(amax_bits)));
    const float qm = is8 ? 127.0f : 7.0f;
    const __half s16 = __float2half_rn(__fmul_rn(amax, is8 ? (1.0f / 127.0f) : (1.0f / 7.0f)));
    const float sc = __half2float(s16);
    const float inv = sc > 0.0f ? rcp_approx(sc) : 0.0f;

    // codes: rne(|x| / s). tm = fma(|x|, inv, 1.5 * 2^23) rounds |x| * inv
    // (relative error < 2^-22) to an integer held in tm's low mantissa bits;
    // quotients within 1e-4 of a half-integer are settled with the exact
    // remainder |x| - r*s (the exact quotient of two fp16 values is never
    // within 3e-5 of a half-integer unless it is one)
    constexpr float kMagic = 12582912.0f;
    float ax[8], tm[8];
    bool near_half = false;
    // two channels per instruction: fma.rn.f32x2 is the IEEE fma in each half; the
    // fractional part of |x| * inv is |x| * inv - (tm - kMagic), with tm - kMagic exact
    const float2 inv2 = make_float2(inv, inv), mg2 = make_float2(kMagic, kMagic);
    const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 a2 = __half22float2(*reinterpret_cast<const __half2*>(&ab[k]));
        const float2 t2 = dev::ffma2(a2, inv2, mg2);
        const float2 f2 = dev::ffma2(a2, inv2, dev::ffma2(t2, neg1, mg2));
        ax[2 * k] = a2.x;
        ax[2 * k + 1] = a2.y;
        tm[2 * k] = t2.x;
        tm[2 * k + 1] = t2.y;
        near_half |= fmaxf(fabsf(f2.x), fabsf(f2.y)) > 0.4999f;
    }
    if (__any_sync(0xFFFFFFFFu, near_half) && sc > 0.0f) {
        // (a zero scale keeps every code 0: its lanes skip the correction)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float r = tm[k] - kMagic;
            const float e = fmaf(-r, sc, ax[k]);   // exact remainder |x| - r*s
            const float e2 = e + e;
            if (e2 > sc) r += 1.0f;
            else if (e2 < -sc) r -= 1.0f;
            else if ((e2 == sc || e2 == -sc) && (static_cast<int>(r) & 1)) r += (e2 > 0.0f) ? 1.0f : -1.0f;  // tie: to even
            tm[k] = r + kMagic;
        }
    }
    if (__any_sync(0xFFFFFFFFu, sc > 0.0f && sc < 6.103515625e-05f)) {
        // subnormal scale: the quotient can round past qmax
#pragma unroll
        for (int k = 0; k < 8; ++k) tm[k] = fminf(tm[k], qm + kMagic);
    }
    uint32_t w0 = low_bytes4(tm[0], tm[1], tm[2], tm[3]);
    uint32_t w1 = low_bytes4(tm[4], tm[5], tm[6], tm[7]);
    // sign bits of the inputs (bit 15 of each half) into bit 7 of each byte
    w0 |= __byte_perm(h2[0], h2[1], 0x7531) & 0x80808080u;
    w1 |= __byte_perm(h2[2], h2[3], 0x7531) & 0x80808080u;

    if (valid) {
        uint8_t* dst = A + (static_cast<int64_t>(poff_b) * M + m) * kBlock + chunk_off;
        if (!is8) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
        } else {
            *reinterpret_cast<uint2*>(dst) = make_uint2(w0 & 0x8F8F8F8Fu, w1 & 0x8F8F8F8Fu);
            *reinterpret_cast<uint2*>(dst + M * kBlock) = make_uint2(high_plane(w0), high_plane(w1));
        }
        if constexpr (kTok) {
            // the sum of the block's signed codes: magnitudes (bits 0-6) times +-1
            // from the sign bits, four bytes per dp4a
            auto sum4 = [](uint32_t w) {
                const uint32_t pm = 0x01010101u | (((w >> 7) & 0x01010101u) * 0xFEu);
                return __dp4a(static_cast<int>(w & 0x7F7F7F7Fu), static_cast<int>(pm), 0);
            };
            const int t = __reduce_add_sync(hmask, sum4(w0) + sum4(w1));
            if (sub == 0) sums[static_cast<int64_t>(b) * M + m] = t;
        } else {
            if (sub == 0) scales[static_cast<int64_t>(b) * M + m] = __half_as_ushort(s16);
        }
    }
}

// Shared memory: [S] rows of X | gather offsets [iters][16 warps][32 lanes] (8 byte offsets of
// 16 bits per lane and block pair) | plane offset per block | full / empty barriers per stage.
__host__ __device__ inline size_t quant_gtab_offset(int K, int S) { return (2ull * K * S + 15) & ~15ull; }
__host__ __device__ inline size_t quant_poff_offset(int K, int S, int tab_entries) {
    return quant_gtab_offset(K, S) + static_cast<size_t>(tab_entries) * 32 * 16;   // entries: iters * cwarps
}
__host__ __device__ inline size_t quant_chunk_offset(int K, int S, int iters, int nb) {
    return quant_poff_offset(K, S, iters) + ((4ull * nb + 15) & ~15ull);
}
// Row-statistic scratch per stage: the per-token INT8 kernel keeps one fp32 absmax per chunk,
// the fused RMSNorm kernel one exact (lo, hi) pair of 64-bit sums per norm warp.
__host__ __device__ inline size_t quant_stat_bytes(int S, int nb) {
    const size_t chunks = 4ull * S * nb, pairs = 16ull * S * kQNormWarps;
    return chunks > pairs ? chunks : pairs;
}
__host__ __device__ inline size_t quant_bars_offset(int K, int S, int iters, int nb) {
    return quant_chunk_offset(K, S, iters, nb) + ((quant_stat_bytes(S, nb) + 4ull * S + 15) & ~15ull);
}

// Exact sum of squares of fp16 values. A finite fp16 x is mant * 2^(max(e,1) - 25) (e the
// exponent field, mant < 2^11), so x^2 = mant^2 * 2^(sh - 48) with sh = 2 max(e,1) - 2 in
// [0, 58]: an integer number of 2^-48 units. Squares with sh < 32 go to `lo` (units 2^-48),
// the others to `hi` (units 2^-16); a lane adds at most 128 squares, so neither overflows.
__device__ __forceinline__ void add_square_exact(uint32_t h, uint64_t& lo, uint64_t& hi) {
    const uint32_t e = (h >> 10) & 31u;
    const uint32_t mant = (h & 1023u) | (e ? 1024u : 0u);
    const uint32_t sh = e ? 2u * e - 2u : 0u;
    const uint32_t sq = mant * mant;
    const bool big = sh >= 32u;
    const uint64_t t = static_cast<uint64_t>(sq) << (big ? sh - 32u : sh);
    lo += big ? 0ull : t;
    hi += big ? t : 0ull;
}

// Carry lo's bits above 2^32 into hi: afterwards the sum is hi * 2^32 + lo, lo < 2^32.
__device__ __forceinline__ void carry_exact(uint64_t& lo, uint64_t& hi) {
    hi += lo >> 32;
    lo &= 0xFFFFFFFFull;
}

// (hi * 2^32 + lo) * 2^-48 rounded once to fp32 (nearest, ties to even); lo < 2^32. When the
// sum needs more than 64 bits, lo only matters as a sticky bit far below the rounding position.
__device__ __forceinline__ float exact_to_f32(uint64_t lo, uint64_t hi) {
    if ((hi >> 32) == 0) return __fmul_rn(__ull2float_rn((hi << 32) | lo), 3.5527136788005009e-15f);   // 2^-48
    return __fmul_rn(__ull2float_rn(hi | (lo != 0 ? 1ull : 0ull)), 1.52587890625e-05f);                // 2^-16
}

// kNorm: the quantized values are RMSNorm(x) = fp16_rn((fp32(x) * r) * fp32(gamma)) with
// r = 1 / sqrt(T / K + eps) (IEEE divisions and square root), where T is the row's exact sum of
// squares rounded once to fp32 (integer accumulation, so it does not depend on the order).
// kQAsym (QUIK explainer, "反量化背后的数学": asymmetric activations): every block 4-bit with a
// zero point z = the block's smallest input (value order, -0 below +0) and
// s = fp16_rn((fp32(max) - fp32(z)) / 15); q = clamp(rne(fp32(fp32(x) - fp32(z)) / fp32(s)), 0, 15)
// with IEEE fp32 operations; codes in one plane with the sign bit clear.
// kQTok (QServe explainer, "运行时设计": W4A8 GEMMs take per-token INT8 activations): the row's
// absmax (computed by the norm warps ahead of the quantizing warps) gives one scale per token,
// s = fp16_rn(fp32(absmax) / 127); every block INT8; the sum of each block's codes is written too.
// kTwo: the 16-warp instantiation that two CTAs share an SM with (registers bounded for it).
template <int kMode, bool kTwo = false>
__global__ void __launch_bounds__(kTwo ? (kQWarpsMin + 1) * 32 : kQMaxThreads, kTwo ? 2 : 1) quantize_kernel(QuantParams p) {
    constexpr bool kNorm = kMode == kQNorm;
    constexpr bool kRowWarps = kMode == kQNorm || kMode == kQTok;   // a per-row statistic comes first
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int K = p.K, Kr = p.Kin, nb = p.nb, S = p.stages;
    uint16_t* rows_s = reinterpret_cast<uint16_t*>(smem_raw);                                // [S][Kin]
    uint4* gtab = reinterpret_cast<uint4*>(smem_raw + quant_gtab_offset(Kr, S));              // [iters][W][32]
    int32_t* s_poff = reinterpret_cast<int32_t*>(smem_raw + quant_poff_offset(Kr, S, p.iters * p.cwarps)); // [nb]
    float* chunk_s = reinterpret_cast<float*>(smem_raw + quant_chunk_offset(Kr, S, p.iters * p.cwarps, nb));  // [S][nb]
    uint64_t* wsum_s = reinterpret_cast<uint64_t*>(chunk_s);                                     // [S][8][2] (norm)
    float* r_s = chunk_s + quant_stat_bytes(S, nb) / 4;                                            // [S]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + quant_bars_offset(Kr, S, p.iters * p.cwarps, nb));
    uint64_t* full = bars;            // [S] the row has landed
    uint64_t* empty = bars + S;       // [S] every reader is done with the row
    uint64_t* nsync = bars + 2 * S;   // [S] fused RMSNorm: both norm warps' chunk sums are in place
    uint64_t* rready = bars + 3 * S;  // [S] fused RMSNorm: the row's factor r is in r_s
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a GEMM launched as this grid's programmatic dependent may start its prologue and weight
    // stream now; it waits for this grid's completion before reading the codes
    dev::pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            dev::mbar_init(&full[s], 1);
            dev::mbar_init(&empty[s], p.cwarps + (kRowWarps ? p.rwarps : 0) + (p.n_split > 0 ? 1 : 0));
            dev::mbar_init(&nsync[s], p.rwarps);
            dev::mbar_init(&rready[s], 1);
        }
        abort_flag = 0;
        dev::fence_barrier_init();
    }
    for (int b = threadIdx.x; b < nb; b += blockDim.x) s_poff[b] = p.poff[b];
    __syncthreads();

    const uint32_t row_bytes = static_cast<uint32_t>(Kr) * 2u;
    const int W = p.cwarps;
    if (warp == W) {
        // ---------------- producer: rows of X into the stage ring
        if (lane == 0) {
            int64_t i = 0;
            for (int64_t m = blockIdx.x; m < p.M; m += gridDim.x, ++i) {
                const int s = static_cast<int>(i % S);
                const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
                if (!dev::mbar_wait(&empty[s], ph ^ 1u, &abort_flag)) {
                    abort_flag = 1;
                    break;
                }
                dev::mbar_arrive_expect_tx(&full[s], row_bytes);
                dev::bulk_g2s(rows_s + static_cast<size_t>(s) * Kr, p.X + m * p.ldx, row_bytes, &full[s]);
            }
            // drain: every stage's latest copy must have landed before the CTA exits
            const int64_t issued = i;
            for (int s = 0; s < S; ++s) {
                if (issued <= s) break;
                const int64_t last = s + ((issued - 1 - s) / S) * S;
                dev::mbar_wait(&full[s], static_cast<uint32_t>((last / S) & 1), nullptr);
            }
        }
        __syncwarp();
    } else if (warp > W + p.rwarps) {
        // ---------------- split warp (QUIK explainer, "核融合": the one pass over the input also
        // extracts the outlier part): each staged row's outlier columns, copied out in fp16
        int64_t i = 0;
        bool ok = true;
        for (int64_t m = blockIdx.x; m < p.M; m += gridDim.x, ++i) {
            const int s = static_cast<int>(i % S);
            ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&full[s], static_cast<uint32_t>((i / S) & 1), &abort_flag));
            if (!ok) break;
            const uint16_t* row = rows_s + static_cast<size_t>(s) * Kr;
            split_row(p.split_cols, p.n_split, p.X_out + m * p.n_split, lane, Kr, [&](int c) { return row[c]; });
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(&empty[s]);
        }
        if (!ok && lane == 0) abort_flag = 1;
    } else if (warp > W) {
        // ---------------- row-statistic warps, ahead of the quantizing warps. Warp w takes the
        // chunk pairs w, w + rwarps, ... (each half-warp one 128-channel chunk). Fused RMSNorm:
        // the exact sum of squares of the row (integer accumulation, order-free), rounded once to
        // fp32 by warp 0, then r. Per-token INT8: the chunk maxima, then the row's absmax.
        if constexpr (kNorm) {
            const int nw = warp - W - 1;
            const int half = lane >> 4, sub16 = lane & 15;
            int64_t i = 0;
            bool ok = true;
            for (int64_t m = blockIdx.x; m < p.M; m += gridDim.x, ++i) {
                const int s = static_cast<int>(i % S);
                const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
                ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&full[s], ph, &abort_flag));
                if (!ok) break;
                const uint8_t* row = reinterpret_cast<const uint8_t*>(rows_s + static_cast<size_t>(s) * Kr);
                uint64_t lo = 0, hi = 0;
                for (int q = nw; 2 * q < nb; q += p.rwarps) {
                    const int b = 2 * q + half;
                    if (b < nb) {
                        const uint4 v = *reinterpret_cast<const uint4*>(row + (b * kBlock + sub16 * 8) * 2);
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            add_square_exact(w4[k] & 0xFFFFu, lo, hi);
                            add_square_exact(w4[k] >> 16, lo, hi);
                        }
                    }
                }
                carry_exact(lo, hi);
#pragma unroll
                for (int st = 16; st >= 1; st >>= 1) {
                    lo += __shfl_xor_sync(0xFFFFFFFFu, lo, st);
                    hi += __shfl_xor_sync(0xFFFFFFFFu, hi, st);
                }
                uint64_t* ws = wsum_s + static_cast<size_t>(s) * (2 * kQNormWarps);
                if (lane == 0) {
                    ws[2 * nw] = lo;
                    ws[2 * nw + 1] = hi;
                }
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(&nsync[s]);
                if (nw == 0) {
                    ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&nsync[s], ph, &abort_flag));
                    if (!ok) break;
                    uint64_t tl = lane < p.rwarps ? ws[2 * lane] : 0ull;
                    uint64_t th = lane < p.rwarps ? ws[2 * lane + 1] : 0ull;
#pragma unroll
                    for (int st = 4; st >= 1; st >>= 1) {   // rwarps <= 8
                        tl += __shfl_xor_sync(0xFFFFFFFFu, tl, st);
                        th += __shfl_xor_sync(0xFFFFFFFFu, th, st);
                    }
                    if (lane == 0) {
                        carry_exact(tl, th);
                        const float t = exact_to_f32(tl, th);
                        // r = 1 / sqrt(T / K + eps), IEEE fp32 division, addition and square root
                        r_s[s] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(t, static_cast<float>(K)), p.eps)));
                        dev::mbar_arrive(&rready[s]);
                    }
                }
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(&empty[s]);
            }
            if (!ok && lane == 0) abort_flag = 1;
        } else if constexpr (kRowWarps) {
            const int nw = warp - W - 1;
            const int half = lane >> 4, sub16 = lane & 15;
            const uint32_t hm = half ? 0xFFFF0000u : 0x0000FFFFu;
            int64_t i = 0;
            bool ok = true;
            for (int64_t m = blockIdx.x; m < p.M; m += gridDim.x, ++i) {
                const int s = static_cast<int>(i % S);
                const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
                ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&full[s], ph, &abort_flag));
                if (!ok) break;
                const uint8_t* row = reinterpret_cast<const uint8_t*>(rows_s + static_cast<size_t>(s) * Kr);
                float* cs = chunk_s + static_cast<size_t>(s) * nb;
                for (int q = nw; 2 * q < nb; q += p.rwarps) {
                    const int b = 2 * q + half;
                    float acc = 0.0f;
                    if (b < nb) {
                        const uint4 v = *reinterpret_cast<const uint4*>(row + (b * kBlock + sub16 * 8) * 2);
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                        // the chunk's absmax (fp16 magnitudes order like their bit patterns)
                        uint32_t m2 = 0;
#pragma unroll
                        for (int k = 0; k < 4; ++k) m2 = __vmaxu2(m2, w4[k] & 0x7FFF7FFFu);
                        acc = __half2float(__ushort_as_half(static_cast<unsigned short>(max(m2 & 0xFFFFu, m2 >> 16))));
                    }
#pragma unroll
                    for (int st = 8; st >= 1; st >>= 1) acc = fmaxf(acc, __shfl_xor_sync(hm, acc, st));
                    if (b < nb && sub16 == 0) cs[b] = acc;
                }
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(&nsync[s]);
                if (nw == 0) {
                    ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&nsync[s], ph, &abort_flag));
                    if (!ok) break;
                    float t = 0.0f;
                    for (int b = lane; b < nb; b += 32) t = fmaxf(t, cs[b]);
#pragma unroll
                    for (int st = 16; st >= 1; st >>= 1) t = fmaxf(t, __shfl_xor_sync(0xFFFFFFFFu, t, st));
                    if (lane == 0) {
                        r_s[s] = t;   // the row's absmax
                        dev::mbar_arrive(&rready[s]);
                    }
                }
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(&empty[s]);
            }
            if (!ok && lane == 0) abort_flag = 1;
        }
    } else {
        // ---------------- compute warps
        const bool upper = lane >= 16;
        const int sub = lane & 15;                          // 8-channel group inside the block
        const uint32_t hmask = upper ? 0xFFFF0000u : 0x0000FFFFu;
        // per iteration j: this lane's block, its gather byte offsets (in shared memory, so the
        // loop over j stays compact), precision and validity bits
        uint4* my_goff = gtab + warp * 32 + lane;          // entry j at my_goff[j * W * 32]
        uint32_t is8_bits = 0, valid_bits = 0;
        for (int j = 0; j < p.iters; ++j) {
            const int b = warp + 2 * W * j + (upper ? W : 0);
            const bool valid = b < nb;
            uint4 g = make_uint4(0, 0, 0, 0);
            if (valid) {
                const uint4 pr = *reinterpret_cast<const uint4*>(p.perm + b * kBlock + sub * 8);
                // channel index -> byte offset inside the row (indices < 32768)
                g = make_uint4(pr.x << 1, pr.y << 1, pr.z << 1, pr.w << 1);
                if (p.mask[b]) is8_bits |= 1u << j;
                valid_bits |= 1u << j;
            }
            my_goff[j * W * 32] = g;
        }
        __syncwarp();
        const int iters = (nb - warp + 2 * W - 1) / (2 * W);   // rounds with a valid lower block

        int64_t i = 0;
        bool ok = true;
        for (int64_t m = blockIdx.x; m < p.M; m += gridDim.x, ++i) {
            const int s = static_cast<int>(i % S);
            const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
            ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&full[s], ph, &abort_flag));   // every lane waits
            if (!ok) break;
            const uint8_t* row = reinterpret_cast<const uint8_t*>(rows_s + static_cast<size_t>(s) * Kr);
            const uint32_t chunk_off = ((static_cast<uint32_t>(sub >> 1) ^ static_cast<uint32_t>(m & 7)) << 4) +
                                       static_cast<uint32_t>(sub & 1) * 8u;
            float r_norm = 1.0f;
            if constexpr (kRowWarps) {
                ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&rready[s], ph, &abort_flag));   // the row's statistic
                if (!ok) break;
                r_norm = r_s[s];
            }
            if constexpr (kMode == kQTok) {
                if (warp == 0 && lane == 0)
                    p.scales[m] = __half_as_ushort(__float2half_rn(__fmul_rn(r_norm, 1.0f / 127.0f)));
            }
#pragma unroll 2   // two block steps in flight: 108 against 123 us at 4096 x 28672 (unrolled 1 or 4)
            for (int j = 0; j < iters; ++j) {                // warp-uniform bound
                const bool valid = (valid_bits >> j) & 1u;
                const bool is8 = (is8_bits >> j) & 1u;
                // gather 8 fp16 values, paired into half2 words
                const uint4 g = my_goff[j * W * 32];
                uint32_t h2[4];
                {
                    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t lo = *reinterpret_cast<const uint16_t*>(row + (gw[k] & 0xFFFFu));
                        const uint32_t hi = *reinterpret_cast<const uint16_t*>(row + (gw[k] >> 16));
                        h2[k] = __byte_perm(lo, hi, 0x5410);
                    }
                }
                if constexpr (kMode == kQAsym) {
                    quantize_asym_step(p, h2, valid, warp + 2 * W * j + (upper ? W : 0), m, chunk_off, sub, hmask,
                                       s_poff);
                    continue;
                }
                if constexpr (kNorm) {
                    // normalize: y = fp16_rn((x * r) * gamma), gamma of the lane's 8 permuted channels
                    const int bn = warp + 2 * W * j + (upper ? W : 0);
                    const uint4 gv = valid ? __ldg(reinterpret_cast<const uint4*>(p.gamma_perm + bn * kBlock + sub * 8))
                                           : make_uint4(0u, 0u, 0u, 0u);
                    const uint32_t gw4[4] = {gv.x, gv.y, gv.z, gv.w};
                    const float2 r2 = make_float2(r_norm, r_norm);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&h2[k]));
                        const float2 g = __half22float2(*reinterpret_cast<const __half2*>(&gw4[k]));
                        const __half2 y = __float22half2_rn(dev::fmul2(dev::fmul2(x, r2), g));   // (x * r) * g, each rounded
                        h2[k] = *reinterpret_cast<const uint32_t*>(&y);
                    }
                }
                {
                    const int bb = warp + 2 * W * j + (upper ? W : 0);
                    quantize_codes_step<kMode == kQTok>(h2, valid, is8, bb, m, chunk_off, sub, hmask,
                                                        valid ? s_poff[bb] : 0, p.A, p.M, p.scales, p.sums, r_norm);
                }
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(&empty[s]);
        }
        if (!ok && lane == 0) abort_flag = 1;
    }
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) dev::report(p.status, dev::kStatusTimeout);
}

// ---------------------------------------------------------------------------------
// Few tokens: one warp per (token, block pair) straight from X, the channels gathered through
// the permutation with plain loads (the row stays in L1/L2 across the row's warps). The
// row-pipelined kernel gives each CTA whole rows, so with fewer tokens than SMs most SMs idle
// and each row's copy latency is exposed; this form spreads a token's blocks over the GPU.
// Same code step as the row kernel, so the codes and scales are identical.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quantize_direct_kernel(QuantParams p) {
    dev::pdl_launch_dependents();   // as in quantize_kernel
    const int lane = threadIdx.x & 31;
    const bool upper = lane >= 16;
    const int sub = lane & 15;
    const uint32_t hmask = upper ? 0xFFFF0000u : 0x0000FFFFu;
    const int pairs = (p.nb + 1) / 2;
    const int per_token = pairs + (p.n_split + 255) / 256;   // block pairs, then split chunks of 256 columns
    const int64_t items = p.M * per_token;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t item = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); item < items;
         item += warps) {   // warp-uniform
        const int64_t m = item / per_token;
        const int r = static_cast<int>(item % per_token);
        if (r >= pairs) {
            // QUIK input split: this token's outlier columns j .. j + 255
            const int j = 256 * (r - pairs);
            const uint16_t* row = p.X + m * p.ldx;
            split_row(p.split_cols + j, min(256, p.n_split - j), p.X_out + m * p.n_split + j, lane, p.Kin,
                      [&](int c) { return __ldg(row + c); });
            continue;
        }
        const int b = 2 * r + (upper ? 1 : 0);
        const bool valid = b < p.nb;
        uint32_t h2[4] = {0u, 0u, 0u, 0u};
        bool is8 = false;
        int32_t poff_b = 0;
        if (valid) {
            // channels b*128 + 8*sub .. + 7 of the permuted order
            const uint4 pv = __ldg(reinterpret_cast<const uint4*>(p.perm + static_cast<int64_t>(b) * kBlock + sub * 8));
            const uint16_t* row = p.X + m * p.ldx;
            const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                h2[k] = static_cast<uint32_t>(__ldg(row + (pw[k] & 0xFFFFu))) |
                        (static_cast<uint32_t>(__ldg(row + (pw[k] >> 16))) << 16);
            is8 = __ldg(p.mask + b) != 0;
            poff_b = __ldg(p.poff + b);
        }
        const uint32_t chunk_off = ((static_cast<uint32_t>(sub >> 1) ^ static_cast<uint32_t>(m & 7)) << 4) +
                                   static_cast<uint32_t>(sub & 1) * 8u;
        quantize_codes_step<false>(h2, valid, is8, b, m, chunk_off, sub, hmask, poff_b, p.A, p.M, p.scales, nullptr,
                                   0.0f);
    }
}

// ---------------------------------------------------------------------------------
// SwiGLU fused with the quantizer (QServe explainer, "运行时设计": the activation quantization of
// the second FFN layer is fused into the activation kernel): h = fp16_rn(g * u / (1 + e^-g)),
// then the symmetric quantizer on h. The gate and up outputs arrive in the layout's permuted
// channel order (the projections' output channels are permuted offline, like the weights), so
// a warp reads its two blocks of a token with coalesced 16-byte loads: no staging, no gather.
// One warp per (token, block pair), 8 channels per lane, grid-stride over the pairs.
// ---------------------------------------------------------------------------------
struct SwigluParams {
    const uint16_t* G;
    const uint16_t* U;
    int64_t ldg, ldu, M;
    int nb;
    const uint8_t* mask;
    const int32_t* poff;
    uint8_t* A;
    uint16_t* scales;
};

// Float-float arithmetic (a value is hi + lo, |lo| <= ulp(hi) / 2): error-free sums and
// products (Knuth's two-sum, Dekker's fast two-sum, the fma product), used to settle the
// rounding of SwiGLU values that lie near an fp16 rounding boundary.
struct FF {
    float hi, lo;
};
__device__ __forceinline__ FF ff_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return FF{s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ FF ff_fast_two_sum(float a, float b) {   // |a| >= |b|
    const float s = __fadd_rn(a, b);
    return FF{s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ FF ff_mul(FF x, FF y) {
    const float p = __fmul_rn(x.hi, y.hi);
    const float e = fmaf(x.hi, y.hi, -p);
    return ff_fast_two_sum(p, e + (x.hi * y.lo + x.lo * y.hi));
}
__device__ __forceinline__ FF ff_add(FF x, FF y) {
    const FF s = ff_two_sum(x.hi, y.hi);
    return ff_fast_two_sum(s.hi, s.lo + (x.lo + y.lo));
}

// e^x for -25 <= x <= 88 in float-float, relative error below 2^-34: x = k ln2 + r with
// |r| <= ln2 / 2 (Cody-Waite: ln2 split into a 15-bit head, so k * head is exact for |k| < 512,
// and a tail), e^r by its Taylor series to r^11 / 11! (truncation below 2^-40) in Horner form,
// then the exact scaling by 2^k.
__device__ __forceinline__ FF ff_exp(float x) {
    constexpr double kLn2 = 0.69314718055994530942;
    constexpr float kLn2Hi = 0.693145751953125f;                              // 15 significant bits
    constexpr float kLn2Lo = static_cast<float>(kLn2 - 0.693145751953125);
    const float k = rintf(x * 1.44269504088896341f);
    const float rh = fmaf(-k, kLn2Hi, x);                                      // exact
    const FF t{__fmul_rn(k, kLn2Lo), fmaf(k, kLn2Lo, -__fmul_rn(k, kLn2Lo))};
    FF r = ff_two_sum(rh, -t.hi);
    r = ff_fast_two_sum(r.hi, __fsub_rn(r.lo, t.lo));
    // 1 / n! for n = 11 .. 0 as float-float (head rounded from the double, tail the rest)
    constexpr double kInvFact[12] = {1.0, 1.0, 0.5, 1.0 / 6, 1.0 / 24, 1.0 / 120, 1.0 / 720, 1.0 / 5040,
                                     1.0 / 40320, 1.0 / 362880, 1.0 / 3628800, 1.0 / 39916800};
    FF p{static_cast<float>(kInvFact[11]), static_cast<float>(kInvFact[11] - static_cast<float>(kInvFact[11]))};
#pragma unroll
    for (int n = 10; n >= 0; --n) {
        const FF c{static_cast<float>(kInvFact[n]), static_cast<float>(kInvFact[n] - static_cast<float>(kInvFact[n]))};
        p = ff_add(ff_mul(p, r), c);
    }
    const int ki = static_cast<int>(k);
    return FF{ldexpf(p.hi, ki), ldexpf(p.lo, ki)};
}

// h for two channels (half2 words g2, u2), h = fp16_rn(g u / (1 + e^-g)) (a zero result keeps
// the IEEE sign of g u). The fp32 value v = g u / (1 + e^-g) errs by at most 5 * 2^-24 (relative;
// expf and the division within 2 ulp each, two roundings), so h = fp16_rn(v) unless the roundings
// of |v| (1 - 2^-21) and |v| (1 + 2^-21) differ (for normal fp16 results tested on v's dropped
// mantissa bits first). Then the exact value lies on one side of the
// rounding boundary m between those two candidates, and the side is the sign of
// |g u| - m (1 + e^-g): an exact sum plus m e^-g in float-float. The rare case that even this
// leaves undecided (|T| below 2^-30 m e^-g) is computed in fp64.
// The rare path (about 0.15% of the values), kept out of line so that the hot loop stays compact:
// h1 < h2 are the candidate magnitudes, a = |g u|, e = expf(-g).
__device__ __noinline__ uint16_t swiglu_settle(float g, float u, float a, float e, uint16_t h1, uint16_t h2) {
    // the boundary between the candidates (exact in fp32; 65520 when h2 is the overflow)
    const float f1 = __half2float(__ushort_as_half(h1));
    const float f2 = h2 == 0x7C00u ? 65536.0f : __half2float(__ushort_as_half(h2));
    const float m = 0.5f * (f1 + f2);
    const float x = -g;
    const FF E = x < -25.0f ? FF{e, 0.0f} : ff_exp(fminf(x, 88.0f));
    const FF mE = ff_mul(FF{m, 0.0f}, E);
    const FF t = ff_add(ff_two_sum(a, -m), FF{-mE.hi, -mE.lo});   // |g u| - m (1 + e^-g)
    const float tv = t.hi != 0.0f ? t.hi : t.lo;
    if (fabsf(tv) > 9.3132257461547852e-10f * m * E.hi) return tv > 0.0f ? h2 : h1;   // 2^-30
    const double gd = static_cast<double>(g);
    return __half_as_ushort(__double2half(fabs(gd * static_cast<double>(u)) / (1.0 + exp(-gd))));
}

__device__ __forceinline__ uint16_t swiglu_f16(float g, float u) {
    const float gu = __fmul_rn(g, u);                     // exact: fp16 x fp16
    const float a = fabsf(gu);
    const float e = expf(-g);
    const float v = __fdividef(a, __fadd_rn(1.0f, e));
    const uint16_t sign = (__float_as_uint(gu) >> 16) & 0x8000u;
    // For v in fp16's normal range the rounding drops v's 13 low mantissa bits: v is far from a
    // rounding boundary when they are more than 8 units (> 5 * 2^-24 relative) away from 0x1000.
    const int low = static_cast<int>(__float_as_uint(v) & 0x1FFFu) - 0x1000;
    if (v >= 6.103515625e-05f && (low > 8 || low < -8)) return __half_as_ushort(__float2half_rn(v)) | sign;
    const uint16_t h1 = __half_as_ushort(__float2half_rn(__fmul_rn(v, 1.0f - 4.76837158203125e-07f)));
    const uint16_t h2 = __half_as_ushort(__float2half_rn(__fmul_rn(v, 1.0f + 4.76837158203125e-07f)));
    return (h1 == h2 ? h1 : swiglu_settle(g, u, a, e, h1, h2)) | sign;
}

__device__ __forceinline__ uint32_t swiglu_f16x2(uint32_t g2, uint32_t u2) {
    const float2 g = __half22float2(*reinterpret_cast<const __half2*>(&g2));
    const float2 u = __half22float2(*reinterpret_cast<const __half2*>(&u2));
    return static_cast<uint32_t>(swiglu_f16(g.x, u.x)) | (static_cast<uint32_t>(swiglu_f16(g.y, u.y)) << 16);
}

__global__ void __launch_bounds__(256) swiglu_quantize_kernel(SwigluParams p) {
    const int lane = threadIdx.x & 31;
    const bool upper = lane >= 16;
    const int sub = lane & 15;
    const uint32_t hmask = upper ? 0xFFFF0000u : 0x0000FFFFu;
    const int pairs = (p.nb + 1) / 2;
    const int64_t items = p.M * pairs;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t item = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); item < items;
         item += warps) {   // warp-uniform
        const int64_t m = item / pairs;
        const int b = 2 * static_cast<int>(item % pairs) + (upper ? 1 : 0);
        const bool valid = b < p.nb;
        uint32_t h2[4] = {0u, 0u, 0u, 0u};
        bool is8 = false;
        int32_t poff_b = 0;
        if (valid) {
            const int64_t c = static_cast<int64_t>(b) * kBlock + sub * 8;
            const uint4 g = __ldg(reinterpret_cast<const uint4*>(p.G + m * p.ldg + c));
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(p.U + m * p.ldu + c));
            h2[0] = swiglu_f16x2(g.x, u.x);
            h2[1] = swiglu_f16x2(g.y, u.y);
            h2[2] = swiglu_f16x2(g.z, u.z);
            h2[3] = swiglu_f16x2(g.w, u.w);
            is8 = __ldg(p.mask + b) != 0;
            poff_b = __ldg(p.poff + b);
        }
        const uint32_t chunk_off = ((static_cast<uint32_t>(sub >> 1) ^ static_cast<uint32_t>(m & 7)) << 4) +
                                   static_cast<uint32_t>(sub & 1) * 8u;
        quantize_codes_step<false>(h2, valid, is8, b, m, chunk_off, sub, hmask, poff_b, p.A, p.M, p.scales, nullptr,
                                   0.0f);
    }
}

// ---------------------------------------------------------------------------------
// Offline weight packing: one warp per (output channel n, block b). Same scale and
// rounding rule as the activations with qmax = 7. Output layout (implementation-defined):
// rows grouped by 256; group g, block b occupies 16 KB at ((g*nb + b) * 16384), row r of
// the group at + r*64, in the INT4 word format of the packed activations. Rows past N
// (padding up to a multiple of 256) are written as zero codes.
// ---------------------------------------------------------------------------------
struct PackParams {
    const uint16_t* W;
    int64_t ldw;
    int64_t N, Npad;
    int K, nb;
    const uint16_t* perm;
    uint8_t* Wp;
    uint16_t* scales;
};

__global__ void __launch_bounds__(256) pack_weights_kernel(PackParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t task = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (task >= p.Npad * p.nb) return;  // warp-uniform
    const int64_t n = task / p.nb;
    const int b = static_cast<int>(task % p.nb);
    uint32_t v = 0;
    uint16_t sbits = 0;
    if (n < p.N) {
        uint16_t h[4];
        const int j0 = b * kBlock + lane * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = p.W[n * p.ldw + p.perm[j0 + i]];
        v = quantize4(h, 7, &sbits);
    }
    const uint32_t word = pack_int4_pair(v, lane);
    uint8_t* dst = p.Wp + ((n / kTileN) * p.nb + b) * 16384 + (n % kTileN) * 64;
    if ((lane & 1) == 0) reinterpret_cast<uint32_t*>(dst)[lane >> 1] = word;
    if (lane == 0 && n < p.N) p.scales[static_cast<int64_t>(b) * p.N + n] = sbits;
}

// ---------------------------------------------------------------------------------
// QoQ progressive group quantization (QServe explainer, "渐进式分组量化"), offline: one warp per
// output channel n.
//   s1 = fp16_rn(fp32(absmax of the row) / 119); q8 = clamp(rne(fp32(w) / fp32(s1)), -119, 119)
//   (IEEE division; the protective range keeps the dequantized group codes inside INT8);
//   per block b (the group): the range of its q8 extended to include 0, [mn, mx];
//   s2 = max(1, ceil((mx - mn) / 15)), z2 = clamp(rne(-mn / s2), 0, 15),
//   q4 = clamp(rne(q8 / s2) + z2, 0, 15) (exact rationals, ties to even).
// Codes are packed as unsigned nibbles in the packed-weight tile layout: byte j of a word holds
// code j in bits 0-3 and code 4 + j in bits 4-7. The row's absmax is over its K channels (the
// layout selects all of them).
// ---------------------------------------------------------------------------------
__device__ __forceinline__ int rne_div_int(int a, int b) {   // b > 0
    int q = a / b, r = a % b;
    if (r < 0) {
        q -= 1;
        r += b;
    }
    if (2 * r > b || (2 * r == b && (q & 1))) ++q;
    return q;
}

struct QoqPackParams {
    const uint16_t* W;
    int64_t ldw;
    int64_t N, Npad;
    int K, nb;
    const uint16_t* perm;
    uint8_t* Wp;
    uint16_t* s1;
    uint8_t* s2;
    uint8_t* z2;
};

__global__ void __launch_bounds__(256) qoq_pack_weights_kernel(QoqPackParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t n = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (n >= p.Npad) return;   // warp-uniform
    float s1f = 0.0f;
    if (n < p.N) {
        uint32_t m = 0;
        const uint16_t* row = p.W + n * p.ldw;
        for (int c = lane; c < p.K; c += 32) m = max(m, static_cast<uint32_t>(row[c] & 0x7FFFu));
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        const __half sb = __float2half_rn(__fdiv_rn(__half2float(__ushort_as_half(static_cast<unsigned short>(m))), 119.0f));
        s1f = __half2float(sb);
        if (lane == 0) p.s1[n] = __half_as_ushort(sb);
    }
    for (int b = 0; b < p.nb; ++b) {
        uint32_t v = 0;   // this lane's 4 codes, one per byte
        if (n < p.N) {
            int q8[4];
            int lo = 0, hi = 0;   // the range includes 0
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float w = __half2float(__ushort_as_half(p.W[n * p.ldw + p.perm[b * kBlock + lane * 4 + i]]));
                int q = s1f > 0.0f ? __float2int_rn(__fdiv_rn(w, s1f)) : 0;   // round half to even
                q = min(119, max(-119, q));
                q8[i] = q;
                lo = min(lo, q);
                hi = max(hi, q);
            }
            lo = __reduce_min_sync(0xFFFFFFFFu, lo);
            hi = __reduce_max_sync(0xFFFFFFFFu, hi);
            const int s2 = max(1, (hi - lo + 14) / 15);
            const int z2 = min(15, max(0, rne_div_int(-lo, s2)));
#pragma unroll
            for (int i = 0; i < 4; ++i) v |= static_cast<uint32_t>(min(15, max(0, rne_div_int(q8[i], s2) + z2))) << (8 * i);
            if (lane == 0) {
                p.s2[static_cast<int64_t>(b) * p.N + n] = static_cast<uint8_t>(s2);
                p.z2[static_cast<int64_t>(b) * p.N + n] = static_cast<uint8_t>(z2);
            }
        }
        // lanes 2g, 2g+1 hold channels 8g..8g+3 and 8g+4..8g+7
        const uint32_t mine = (lane & 1) ? (v << 4) : v;
        const uint32_t word = mine | __shfl_xor_sync(0xFFFFFFFFu, mine, 1);
        uint8_t* dst = p.Wp + ((n / kTileN) * p.nb + b) * 16384 + (n % kTileN) * 64;
        if ((lane & 1) == 0) reinterpret_cast<uint32_t*>(dst)[lane >> 1] = word;
    }
}

// Offline weight sums for the QUIK zero-point term: wsum[b][n] = w_scale[b][n] * (sum of the
// block's codes), one thread per (n, b), from the packed sign-magnitude words.
__global__ void weight_sums_kernel(const uint8_t* Wp, const uint16_t* w_scales, int64_t N, int nb, float* wsum) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= N * nb) return;
    const int b = static_cast<int>(t / N);
    const int64_t n = t % N;
    const uint32_t* row = reinterpret_cast<const uint32_t*>(Wp + ((n / kTileN) * nb + b) * 16384 + (n % kTileN) * 64);
    auto sum4 = [](uint32_t x) {   // four sign-magnitude bytes: magnitude bits 0-2, sign bit 7
        const uint32_t pm = 0x01010101u | (((x >> 7) & 0x01010101u) * 0xFEu);
        return __dp4a(static_cast<int>(x & 0x07070707u), static_cast<int>(pm), 0);
    };
    int sum = 0;
#pragma unroll
    for (int g = 0; g < 16; ++g) {
        const uint32_t w = row[g];
        sum += sum4(w & 0x87878787u) + sum4(__funnelshift_r(w, w, 4) & 0x87878787u);
    }
    wsum[t] = __half2float(__ushort_as_half(w_scales[t])) * static_cast<float>(sum);   // exact
}

// Debug decode of the packed weights to int8 codes [N][K] (permuted channel order);
// unsigned_codes: the QoQ nibble format.
__global__ void unpack_weights_kernel(const uint8_t* Wp, int64_t N, int K, int nb, int8_t* Wq, bool unsigned_codes) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // one word
    const int64_t words_per_row = K / 8;
    if (t >= N * words_per_row) return;
    const int64_t n = t / words_per_row;
    const int wi = static_cast<int>(t % words_per_row);
    const int b = wi / 16, g = wi % 16;
    const uint32_t w =
        *reinterpret_cast<const uint32_t*>(Wp + ((n / kTileN) * nb + b) * 16384 + (n % kTileN) * 64 + g * 4);
    int8_t* out = Wq + n * K + b * kBlock + g * 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t byte = (w >> (8 * j)) & 0xFFu;
        if (unsigned_codes) {
            out[j] = static_cast<int8_t>(byte & 15u);
            out[4 + j] = static_cast<int8_t>(byte >> 4);
            continue;
        }
        const uint32_t next = (w >> (8 * ((j + 1) & 3))) & 0xFFu;
        const int lo = byte & 7, hi = (byte >> 4) & 7;
        out[j] = static_cast<int8_t>((byte & 0x80u) ? -lo : lo);
        out[4 + j] = static_cast<int8_t>((next & 0x08u) ? -hi : hi);
    }
}

}  // namespace

cudaError_t launch_quantize(const fmpq_layout& L, const void* X, int64_t ldx, int64_t M, void* A, void* scales,
                            cudaStream_t stream, const void* gamma_perm, float eps, int mode, void* aux,
                            const QuantSplit* split) {
    const int K = L.K, Kin = L.K_in;
    if (gamma_perm != nullptr) mode = kQNorm;
    const bool row_warps = mode == kQNorm || mode == kQTok;
    // the per-token absmax is cheap: 4 statistic warps keep ahead, leaving room for 24 quantizing warps
    const int rwarps = mode == kQNorm ? kQNormWarps : mode == kQTok ? kQTokWarps : 0;
    const int swarps = split != nullptr && split->n > 0 ? 1 : 0;   // the split warp
    int cw = kQWarpsMin;
    if (mode == kQTok)
        cw = kQMaxThreads / 32 - 1 - kQTokWarps - swarps;
    else if (!row_warps)
        for (int w = kQWarpsMax - swarps; w > kQWarpsMin; --w)
            if (L.nb % (2 * w) == 0) {
                cw = w;
                break;
            }
    const int iters = (L.nb + 2 * cw - 1) / (2 * cw);
    const size_t fixed = static_cast<size_t>(iters) * cw * 32 * 16 + ((4ull * L.nb + 15) & ~15ull) +
                         ((quant_stat_bytes(8, L.nb) + 4ull * 8 + 15) & ~15ull) + 32 * 16 + 1024;
    auto stages_for = [&](size_t budget) {
        const int st = budget > fixed ? static_cast<int>((budget - fixed) / (2ull * Kin)) : 0;
        return st > 8 ? 8 : st;
    };
    // Short rows: two CTAs per SM (16 compute warps each) when each still gets 3+ row stages in
    // half the budget and both fit; the warps of the second CTA hide the first one's latencies.
    int per_sm = 1;
    int stages = stages_for(kQSmemBudget);
    if (mode == kQSym && cw == kQWarpsMin && !swarps && stages_for(kQSmemBudget / 2) >= 3) {
        const int st2 = stages_for(kQSmemBudget / 2);
        const size_t smem2 = quant_bars_offset(Kin, st2, iters * cw, L.nb) + 8ull * (4 * st2);
        int blocks = 0;
        if (ensure_smem_limit(reinterpret_cast<const void*>(quantize_kernel<kQSym, true>), kQSmemBudget + 16 * 1024) ==
                cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, quantize_kernel<kQSym, true>, (cw + 1) * 32, smem2) ==
                cudaSuccess &&
            blocks >= 2) {
            per_sm = 2;
            stages = st2;
        }
        cudaGetLastError();   // a failed query leaves no sticky error behind
    }
    stages = stages < 1 ? 1 : stages;
    const size_t smem = quant_bars_offset(Kin, stages, iters * cw, L.nb) + 8ull * (4 * stages);
    for (auto fn : {quantize_kernel<kQSym>, quantize_kernel<kQNorm>, quantize_kernel<kQAsym>, quantize_kernel<kQTok>}) {
        const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(fn), kQSmemBudget + 16 * 1024);
        if (e != cudaSuccess) return e;
    }
    QuantParams p;
    p.X = static_cast<const uint16_t*>(X);
    p.ldx = ldx;
    p.M = M;
    p.K = K;
    p.Kin = Kin;
    p.nb = L.nb;
    p.stages = stages;
    p.iters = iters;
    p.cwarps = cw;
    p.rwarps = rwarps;
    p.perm = L.d_perm16;
    p.mask = L.d_mask;
    p.poff = L.d_poff;
    p.A = static_cast<uint8_t*>(A);
    p.scales = static_cast<uint16_t*>(scales);
    p.status = L.d_status;
    p.gamma_perm = static_cast<const uint16_t*>(gamma_perm);
    p.eps = eps;
    p.zeros = mode == kQAsym ? static_cast<uint16_t*>(aux) : nullptr;
    p.sums = mode == kQTok ? static_cast<int32_t*>(aux) : nullptr;
    p.split_cols = swarps ? split->cols : nullptr;
    p.n_split = swarps ? split->n : 0;
    p.X_out = swarps ? static_cast<uint16_t*>(split->X_out) : nullptr;
    if (mode == kQSym && M < L.num_sms) {
        // fewer tokens than SMs: a warp per (token, block pair) instead of a CTA per row
        const int64_t items = M * ((L.nb + 1) / 2 + (p.n_split + 255) / 256);
        const int64_t ctas_needed = (items + 7) / 8;                       // 8 warps per CTA
        const int64_t ctas_max = static_cast<int64_t>(L.num_sms) * 8;
        quantize_direct_kernel<<<static_cast<unsigned>(ctas_needed < ctas_max ? ctas_needed : ctas_max), 256, 0,
                                 stream>>>(p);
        return cudaGetLastError();
    }
    const int64_t ctas = static_cast<int64_t>(L.num_sms) * per_sm;
    const unsigned grid = static_cast<unsigned>(M < ctas ? M : ctas);
    const unsigned threads = static_cast<unsigned>((cw + 1 + rwarps + swarps) * 32);
    switch (mode) {
        case kQNorm: quantize_kernel<kQNorm><<<grid, threads, smem, stream>>>(p); break;
        case kQAsym: quantize_kernel<kQAsym><<<grid, threads, smem, stream>>>(p); break;
        case kQTok: quantize_kernel<kQTok><<<grid, threads, smem, stream>>>(p); break;
        default:
            if (per_sm == 2)
                quantize_kernel<kQSym, true><<<grid, threads, smem, stream>>>(p);
            else
                quantize_kernel<kQSym><<<grid, threads, smem, stream>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_swiglu_quantize(const fmpq_layout& L, const void* G, int64_t ldg, const void* U, int64_t ldu,
                                   int64_t M, void* A, void* scales, cudaStream_t stream) {
    SwigluParams p;
    p.G = static_cast<const uint16_t*>(G);
    p.U = static_cast<const uint16_t*>(U);
    p.ldg = ldg;
    p.ldu = ldu;
    p.M = M;
    p.nb = L.nb;
    p.mask = L.d_mask;
    p.poff = L.d_poff;
    p.A = static_cast<uint8_t*>(A);
    p.scales = static_cast<uint16_t*>(scales);
    const int64_t items = M * ((L.nb + 1) / 2);
    const int64_t ctas_needed = (items + 7) / 8;                       // 8 warps per CTA
    const int64_t ctas_max = static_cast<int64_t>(L.num_sms) * 8;      // up to 64 warps per SM
    const unsigned grid = static_cast<unsigned>(ctas_needed < ctas_max ? ctas_needed : ctas_max);
    swiglu_quantize_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_pack_weights(const fmpq_layout& L, const void* W, int64_t ldw, int64_t N, void* Wp,
                                void* scales, cudaStream_t stream) {
    PackParams p;
    p.W = static_cast<const uint16_t*>(W);
    p.ldw = ldw;
    p.N = N;
    p.Npad = (N + kTileN - 1) / kTileN * kTileN;
    p.K = L.K;
    p.nb = L.nb;
    p.perm = L.d_perm16;
    p.Wp = static_cast<uint8_t*>(Wp);
    p.scales = static_cast<uint16_t*>(scales);
    const int64_t warps = p.Npad * p.nb;
    const int64_t blocks = (warps * 32 + 255) / 256;
    pack_weights_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_unpack_weights(const fmpq_layout& L, const void* Wp, int64_t N, int8_t* Wq, cudaStream_t stream,
                                  bool unsigned_codes) {
    const int64_t words = N * (L.K / 8);
    const int64_t blocks = (words + 255) / 256;
    unpack_weights_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<const uint8_t*>(Wp), N,
                                                                             L.K, L.nb, Wq, unsigned_codes);
    return cudaGetLastError();
}

cudaError_t launch_qoq_pack_weights(const fmpq_layout& L, const void* W, int64_t ldw, int64_t N, void* Wp,
                                    void* s1, uint8_t* s2, uint8_t* z2, cudaStream_t stream) {
    QoqPackParams p;
    p.W = static_cast<const uint16_t*>(W);
    p.ldw = ldw;
    p.N = N;
    p.Npad = (N + kTileN - 1) / kTileN * kTileN;
    p.K = L.K;
    p.nb = L.nb;
    p.perm = L.d_perm16;
    p.Wp = static_cast<uint8_t*>(Wp);
    p.s1 = static_cast<uint16_t*>(s1);
    p.s2 = s2;
    p.z2 = z2;
    const int64_t blocks = (p.Npad * 32 + 255) / 256;
    qoq_pack_weights_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_weight_sums(const fmpq_layout& L, const void* Wp, const void* w_scales, int64_t N, float* wsum,
                               cudaStream_t stream) {
    const int64_t threads = N * L.nb;
    weight_sums_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(
        static_cast<const uint8_t*>(Wp), static_cast<const uint16_t*>(w_scales), N, L.nb, wsum);
    return cudaGetLastError();
}

}  // namespace fmpq
