// Offline layout derivation from calibration activations (sm_103a).
//
// The outliers of the activations sit in a small set of channels (about 10% in COMET news
// article, section 1), and a permutation gathers them into the same 128-channel blocks,
// which then take INT8 codes. QUIK explainer, "第一步: 识别与重排": the outlier columns are
// found offline on calibration data and moved to the end. The channel statistic is the
// absolute maximum over the calibration tokens (the same statistic the quantizer scales by).
//
//   channel_absmax_kernel  HBM-bound column reduction: every CTA reads a 2048-channel strip of
//                          a slice of the tokens with 16-byte loads (8 channels per thread) and
//                          folds its maxima into the output with one atomicMax per channel.
//   plan_layout            host: rank the channels, fill the last n8 blocks with the top ones.
//   plan_layout_budget     host: the fewest INT8 blocks whose layout keeps the calibration
//                          tokens' relative quantization error within a budget.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <numeric>
#include <vector>

#include "../../include/fmpq.h"
#include "fmpq_internal.h"

namespace fmpq {
namespace {

constexpr int kCalThreads = 256;
constexpr int kCalCols = kCalThreads * 8;   // channels per CTA strip

// out[c] = max over rows [r0, r1) of |X[r][c]| as fp16 bits (sign cleared; for finite values
// the bit pattern orders like the magnitude). out is zeroed before the launch.
__global__ void __launch_bounds__(kCalThreads) channel_absmax_kernel(const uint16_t* X, int64_t ldx, int64_t T, int K,
                                                                    int64_t rows_per_cta, uint32_t* out) {
    const int c0 = blockIdx.x * kCalCols + threadIdx.x * 8;
    if (c0 >= K) return;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_cta;
    const int64_t r1 = min(T, r0 + rows_per_cta);
    uint32_t m01 = 0, m23 = 0, m45 = 0, m67 = 0;   // two channels per word, 16 bits each
    const uint16_t* p = X + r0 * ldx + c0;
    int64_t r = r0;
    // four rows in flight per thread
    for (; r + 4 <= r1; r += 4, p += 4 * ldx) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = __ldg(reinterpret_cast<const uint4*>(p + k * ldx));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            m01 = __vmaxu2(m01, v[k].x & 0x7FFF7FFFu);
            m23 = __vmaxu2(m23, v[k].y & 0x7FFF7FFFu);
            m45 = __vmaxu2(m45, v[k].z & 0x7FFF7FFFu);
            m67 = __vmaxu2(m67, v[k].w & 0x7FFF7FFFu);
        }
    }
    for (; r < r1; ++r, p += ldx) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        m01 = __vmaxu2(m01, v.x & 0x7FFF7FFFu);
        m23 = __vmaxu2(m23, v.y & 0x7FFF7FFFu);
        m45 = __vmaxu2(m45, v.z & 0x7FFF7FFFu);
        m67 = __vmaxu2(m67, v.w & 0x7FFF7FFFu);
    }
    const uint32_t m[4] = {m01, m23, m45, m67};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (m[k] & 0xFFFFu) atomicMax(out + c0 + 2 * k, m[k] & 0xFFFFu);
        if (m[k] >> 16) atomicMax(out + c0 + 2 * k + 1, m[k] >> 16);
    }
}

}  // namespace

cudaError_t launch_channel_absmax(const void* X, int64_t ldx, int64_t T, int K, uint32_t* out, int num_sms,
                                  cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(out, 0, static_cast<size_t>(K) * sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
    const int gx = (K + kCalCols - 1) / kCalCols;
    // about four CTAs per SM in total, at least 16 rows per CTA
    int64_t gy = (static_cast<int64_t>(num_sms) * 4 + gx - 1) / gx;
    gy = std::max<int64_t>(1, std::min<int64_t>(gy, (T + 15) / 16));
    const int64_t rows = (T + gy - 1) / gy;
    gy = (T + rows - 1) / rows;
    channel_absmax_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), kCalThreads, 0, stream>>>(
        static_cast<const uint16_t*>(X), ldx, T, K, rows, out);
    return cudaGetLastError();
}

void plan_layout(int K, const uint32_t* absmax, int n8, int32_t* perm, uint8_t* mask) {
    const int nb = K / kBlock;
    std::vector<int32_t> rank(K);
    std::iota(rank.begin(), rank.end(), 0);
    // larger statistic first; equal statistics keep ascending channel order
    std::stable_sort(rank.begin(), rank.end(), [&](int32_t a, int32_t b) { return absmax[a] > absmax[b]; });
    const int n_top = n8 * kBlock;
    std::vector<uint8_t> top(K, 0);
    for (int i = 0; i < n_top; ++i) top[rank[i]] = 1;
    int j = 0;
    for (int c = 0; c < K; ++c)
        if (!top[c]) perm[j++] = c;              // INT4 blocks: the other channels, in order
    for (int i = 0; i < n_top; ++i) perm[j++] = rank[i];   // the last n8 blocks, by rank
    for (int b = 0; b < nb; ++b) mask[b] = b >= nb - n8 ? 1 : 0;
}

namespace {

// x * 2^24 for a finite fp16 bit pattern: |x| = mant * 2^(max(e,1) - 25), so x * 2^24 is the
// integer mant * 2^(max(e,1) - 1), below 2^40.
int64_t fp16_fixed24(uint16_t h) {
    const int e = (h >> 10) & 31;
    const int64_t mant = (h & 1023) + (e != 0 ? 1024 : 0);
    const int64_t v = mant << (e > 0 ? e - 1 : 0);
    return (h & 0x8000u) != 0 ? -v : v;
}

float fp16_value(uint16_t h) {
    __half_raw r;
    r.x = h;
    return __half2float(__half(r));
}

}  // namespace

double layout_error(int K, const uint16_t* Xc, int64_t T, int64_t ldx, const int32_t* perm, const uint8_t* mask) {
    const int nb = K / kBlock;
    double worst = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t* row = Xc + t * ldx;
        unsigned __int128 err2 = 0, norm2 = 0;   // exact, in units of 2^-48
        for (int b = 0; b < nb; ++b) {
            const int32_t* ch = perm + static_cast<int64_t>(b) * kBlock;
            // the activation quantizer's rule: s = fp16_rn(fp32(absmax) / qmax),
            // q = clamp(rne(fp32(x) / fp32(s)), -qmax, qmax), q = 0 for a zero scale
            uint16_t amax = 0;
            for (int j = 0; j < kBlock; ++j) amax = std::max<uint16_t>(amax, row[ch[j]] & 0x7FFFu);
            const int qmax = mask[b] ? 127 : 7;
            const __half_raw s16 = __half(__float2half_rn(fp16_value(amax) / static_cast<float>(qmax)));
            const float s = fp16_value(s16.x);
            const int64_t s24 = fp16_fixed24(s16.x);
            for (int j = 0; j < kBlock; ++j) {
                const uint16_t h = row[ch[j]];
                int64_t q = 0;
                if (s != 0.0f) {
                    q = static_cast<int64_t>(std::nearbyint(fp16_value(h) / s));
                    q = std::min<int64_t>(qmax, std::max<int64_t>(-qmax, q));
                }
                const int64_t x24 = fp16_fixed24(h);
                const int64_t d24 = x24 - q * s24;   // x - q*s, exact
                err2 += static_cast<unsigned __int128>(static_cast<__int128>(d24) * d24);
                norm2 += static_cast<unsigned __int128>(static_cast<__int128>(x24) * x24);
            }
        }
        if (norm2 != 0) worst = std::max(worst, std::sqrt(static_cast<double>(err2) / static_cast<double>(norm2)));
    }
    return worst;
}

int plan_layout_budget(int K, const uint32_t* absmax, const uint16_t* Xc, int64_t T, int64_t ldx, double eps,
                       double* err, int32_t* perm, uint8_t* mask) {
    const int nb = K / kBlock;
    for (int n8 = 0;; ++n8) {
        plan_layout(K, absmax, n8, perm, mask);
        *err = layout_error(K, Xc, T, ldx, perm, mask);
        if (*err <= eps || n8 == nb) return n8;
    }
}

}  // namespace fmpq
