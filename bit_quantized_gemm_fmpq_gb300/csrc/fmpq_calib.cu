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
#include <algorithm>
#include <cstdint>
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

}  // namespace fmpq
