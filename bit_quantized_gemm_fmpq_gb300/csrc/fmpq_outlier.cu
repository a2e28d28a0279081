// Tensor-core side products of the quantization variants.
//
// The FP16 outlier path of an outlier split (QUIK explainer, "第二步: 前向传播"): the input's
// outlier columns are multiplied in FP16 by the unquantized outlier weights, and the FP16 result
// is added to the output of the INT4 path (the base columns, fmpq_layout_create_select +
// w4ax_gemm).
//
//   outlier_gather_kernel  X[:, cols] -> a dense fp16 [M][n_out] operand (one element per thread);
//                          skipped when the quantizer already split the columns off
//   outlier_gemm_kernel    Y[m][n] = fp16(Y[m][n] + fp16(sum_j X_out[m][j] * W_out[n][j])) on the
//                          tensor cores (tcgen05.mma kind::f16, FP32 accumulators in TMEM); one
//                          persistent CTA per SM walks a contiguous n-major range of 128 x 128
//                          output tiles:
//     warp 0       TMA producer: the W_out panel (128 rows x n_out, kept while consecutive tiles
//                  share it, for n_out <= 256) and the X_out boxes per 64-channel chunk
//                  (128-byte swizzle, a 6-stage ring; W_out boxes join the ring when the panel
//                  does not fit)
//     warp 1       TMEM allocation and the single-thread MMA issuer (M = 128, N = 128, K = 16),
//                  two accumulators so the next tile's MMAs overlap this tile's epilogue
//     warps 2-5    epilogue: TMEM lane quarter warp % 4, one output row per thread; rounds the
//                  FP32 product to fp16 into a staging tile that one thread adds to Y with a TMA
//                  reduce-add (the merge, done at the L2)
//   The product is bound by the copy engine's rate for X_out, which every tile re-reads from the
//   L2; the resident panel removes W_out's share.
//
// The QUIK zero-point term (QUIK explainer, "反量化背后的数学": the zero point's contribution is
// z times the sum of the weights, which is computed offline): yz[m][n] = sum_b z[b][m] *
// ws[b][n] in FP32, the same kernel with its FP32 rows stored straight from the epilogue
// (outlier_gemm_kernel<true>), on fp16 operands that zero_operands_kernel lays out so that the
// products are exact (the zero points, and a scaled two-term split of ws). The variant GEMM
// starts its accumulators from yz instead of one FP32 pass per block.
//
// Nothing is allocated: the tensor maps live in kernel parameter space.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fmpq_device.cuh"
#include "fmpq_internal.h"

namespace fmpq {
namespace {

__global__ void outlier_gather_kernel(const uint16_t* X, int64_t ldx, int64_t M, const int32_t* cols, int n_out,
                                      uint16_t* out) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n_out) return;
    const int32_t c = cols[j];
    const bool in_row = c >= 0 && c < ldx;   // an out-of-range index reads as 0
    for (int64_t m = blockIdx.y; m < M; m += gridDim.y) out[m * n_out + j] = in_row ? X[m * ldx + c] : uint16_t(0);
}

constexpr int kOThreads = 192;
constexpr int kOTileM = 128, kOTileN = 128, kOChunk = 64;   // kOChunk fp16 = one 128-byte swizzle row
constexpr int kOMaxStages = 7;
constexpr int kOBox = kOTileM * kOChunk * 2;   // one 128-row x 64-channel fp16 box (16 KB)
constexpr uint32_t kOTmemCols = 256;  // two 128-column FP32 accumulators

struct __align__(1024) OSmem {
    // 14 boxes of 128 rows x 64 channels (swizzled). The merged product uses the first 10 for its
    // operands and the last 4 as two fp16 staging tiles (two boxes of 64 columns each); the
    // stored product (no staging) uses all 14 for operands.
    uint8_t box[14][kOBox];
    uint64_t full[kOMaxStages], empty[kOMaxStages];
    uint64_t w_full, w_free;      // panel landed / every MMA reading the panel finished
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t kOSmemBytes = sizeof(OSmem) + 1024;
static_assert(kOSmemBytes <= 227 * 1024, "outlier GEMM shared memory above the per-CTA limit");

// Tiles run n-major (consecutive tiles share W_out's 128 rows) and each CTA takes a contiguous
// range of them, so with a resident panel a CTA loads W_out once or twice in all.
struct OTiles {
    int mtiles;
    int64_t t0, t1;
    __device__ int mt(int64_t t) const { return static_cast<int>(t % mtiles); }
    __device__ int nt(int64_t t) const { return static_cast<int>(t / mtiles); }
};

// kStore = false: the FP16 outlier product, merged into the fp16 Y with a TMA reduce-add.
// kStore = true: the FP32 product, times colscale[n] and (when given) rowscale[m], stored to
// yz [m_rows][ldz] (the zero-point terms of the quantization variants).
template <bool kStore>
__global__ void __launch_bounds__(kOThreads, 1)
    outlier_gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_y, int n_out, int n_cols, int mtiles, int64_t tiles,
                        float* yz, int64_t ldz, int m_rows, const float* colscale, const float* rowscale,
                        int32_t* status) {
    constexpr int kElems = kOChunk;   // K elements per 128-byte box row
    constexpr uint32_t kIdesc = dev::idesc_f16_f32(kOTileM, kOTileN);
    // W_out chunks kept resident across tiles (n_out <= 256, or 448 for the stored product) and
    // the operand boxes there are
    constexpr int kPanel = kStore ? 7 : 4;
    constexpr int kBoxes = kStore ? 14 : 10;
    extern __shared__ uint8_t smem_raw[];
    OSmem& s = *reinterpret_cast<OSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const OTiles tl{mtiles, static_cast<int64_t>(blockIdx.x) * tiles / gridDim.x,
                    static_cast<int64_t>(blockIdx.x + 1) * tiles / gridDim.x};
    const int chunks = (n_out + kElems - 1) / kElems;
    const bool panel = chunks <= kPanel;
    // panel: W_out chunk c in box c, ring stage st's X_out in box kPanel + st (6 or 7 stages);
    // otherwise stage st holds X_out in box 2 st and W_out in box 2 st + 1 (5 or 7 stages)
    const int S = panel ? kBoxes - kPanel : kBoxes / 2;
    auto xbox = [&](int st) { return s.box[panel ? kPanel + st : 2 * st]; };
    auto wbox = [&](int st, int c) { return s.box[panel ? c : 2 * st + 1]; };
    auto ybox = [&](int buf, int half) { return s.box[10 + 2 * buf + half]; };
    auto yboxes = [&](int nt) { return n_cols - nt * kOTileN > 64 ? 2 : 1; };   // a box wholly past N is skipped
    volatile int* abort_flag = &s.abort_flag;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kOMaxStages; ++i) {
            dev::mbar_init(&s.full[i], 1);
            dev::mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            dev::mbar_init(&s.acc_full[i], 1);
            dev::mbar_init(&s.acc_empty[i], 4);   // one arrival per epilogue warp
        }
        dev::mbar_init(&s.w_full, 1);
        dev::mbar_init(&s.w_free, 1);
        dev::mbar_init(&s.mma_done, 1);
        s.abort_flag = 0;
        dev::fence_barrier_init();
    }
    if (warp == 1) dev::tmem_alloc(&s.tmem_base, kOTmemCols);
    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    auto fail = [&]() {
        *abort_flag = 1;
        dev::report(status, dev::kStatusTimeout);
    };

    if (warp == 0) {
        // ---------------- TMA producer: the W_out panel when a tile starts a new one, and the
        // X_out (+ W_out) boxes per 64-channel chunk
        if (lane == 0) {
            int64_t gx = 0;   // chunks issued (ring position)
            int loads = 0;    // panels issued
            int cur_nt = -1;
            bool ok = true;
            for (int64_t t = tl.t0; t < tl.t1 && ok; ++t) {
                const int m0 = tl.mt(t) * kOTileM, nt = tl.nt(t), n0 = nt * kOTileN;
                if (panel && nt != cur_nt) {
                    // the previous panel's last MMAs must have finished reading it
                    if (loads > 0 && !dev::mbar_wait(&s.w_free, static_cast<uint32_t>((loads - 1) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    dev::mbar_arrive_expect_tx(&s.w_full, chunks * kOBox);
                    for (int c = 0; c < chunks; ++c) dev::tma_load_2d(wbox(0, c), &tm_w, c * kElems, n0, &s.w_full);
                    ++loads;
                    cur_nt = nt;
                }
                for (int c = 0; c < chunks; ++c, ++gx) {
                    const int st = static_cast<int>(gx % S);
                    if (!dev::mbar_wait(&s.empty[st], static_cast<uint32_t>((gx / S) & 1) ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    dev::mbar_arrive_expect_tx(&s.full[st], panel ? kOBox : 2 * kOBox);
                    dev::tma_load_2d(xbox(st), &tm_x, c * kElems, m0, &s.full[st]);
                    if (!panel) dev::tma_load_2d(wbox(st, c), &tm_w, c * kElems, n0, &s.full[st]);
                }
            }
            if (!ok) fail();
            // drain: every load issued lands before the CTA exits
            for (int64_t k = gx - 1; k >= 0 && k >= gx - S; --k)
                dev::mbar_wait(&s.full[k % S], static_cast<uint32_t>((k / S) & 1), nullptr);
            if (loads > 0) dev::mbar_wait(&s.w_full, static_cast<uint32_t>((loads - 1) & 1), nullptr);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer: accumulator i % 2 for this CTA's tile i
        if (lane == 0) {
            int64_t gx = 0;
            int loads = 0;
            int cur_nt = -1;
            int64_t i = 0;
            bool ok = true;
            for (int64_t t = tl.t0; t < tl.t1 && ok; ++t, ++i) {
                const int nt = tl.nt(t), ab = static_cast<int>(i & 1);
                if (!dev::mbar_wait(&s.acc_empty[ab], static_cast<uint32_t>((i >> 1) & 1) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if (panel && nt != cur_nt) {
                    if (!dev::mbar_wait(&s.w_full, static_cast<uint32_t>(loads & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    ++loads;
                    cur_nt = nt;
                }
                dev::tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(ab) * kOTileN;
                for (int c = 0; c < chunks; ++c, ++gx) {
                    const int st = static_cast<int>(gx % S);
                    if (!dev::mbar_wait(&s.full[st], static_cast<uint32_t>((gx / S) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    dev::tc_fence_after();
                    const uint64_t ad = dev::sdesc_k_sw128(dev::smem_u32(xbox(st)));
                    const uint64_t bd = dev::sdesc_k_sw128(dev::smem_u32(wbox(st, c)));
#pragma unroll
                    for (int k = 0; k < 4; ++k) {   // 32 bytes of K per MMA: +2 in the address field
                        dev::mma_f16(d, ad + 2 * k, bd + 2 * k, kIdesc, (c > 0 || k > 0) ? 1u : 0u);
                    }
                    dev::mma_commit(&s.empty[st]);
                }
                if (!ok) break;
                dev::mma_commit(&s.acc_full[ab]);
                // the panel retires after the last tile that reads it
                if (panel && (t + 1 == tl.t1 || tl.nt(t + 1) != nt)) dev::mma_commit(&s.w_free);
            }
            if (!ok) fail();
            dev::mma_commit(&s.mma_done);   // every MMA issued completes before mma_done
            dev::mbar_wait(&s.mma_done, 0, nullptr);   // and before TMEM is released
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: thread owns tile row r (TMEM lane r). The FP32 product is
        // rounded to fp16 (the FP16 outlier result) into a staging tile, which one thread adds to Y
        // with a TMA reduce-add (the merge, done at the L2: Y = fp16(Y + product)).
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const bool storer = warp == 2 && lane == 0;
        int64_t i = 0;
        for (int64_t t = tl.t0; t < tl.t1; ++t, ++i) {
            const int mt = tl.mt(t), nt = tl.nt(t), ab = static_cast<int>(i & 1);
            const int nyb = yboxes(nt);
            bool ok = dev::mbar_wait(&s.acc_full[ab], static_cast<uint32_t>((i >> 1) & 1), abort_flag);
            ok = __all_sync(0xFFFFFFFFu, ok) && !*abort_flag;
            if (!ok && lane == 0) fail();
            // staging tile ab is free: the storer saw the reduce of tile i - 2 finish reading it.
            // The barrier also makes the decision to stop the same in all four warps.
            if (dev::named_bar_sync_or(1, 128, !ok)) break;
            dev::tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(ab) * kOTileN;
            if constexpr (kStore) {
                // FP32 rows straight to yz: thread r writes 512 contiguous bytes of its row
                const int row = mt * kOTileM + r;
                const float rs = (rowscale != nullptr && row < m_rows) ? __ldg(rowscale + row) : 1.0f;
#pragma unroll 1
                for (int c = 0; c < 2 * nyb; ++c) {
                    uint32_t d0[16], d1[16];
                    dev::tmem_ld16(taddr + 32 * c, d0);
                    dev::tmem_ld16(taddr + 32 * c + 16, d1);
                    dev::tmem_ld_wait16(d0);
                    dev::tmem_ld_wait16(d1);
                    if (row < m_rows) {
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            const int col = nt * kOTileN + 32 * c + 4 * g;
                            const uint32_t* dg = g < 4 ? d0 + 4 * g : d1 + 4 * (g - 4);
                            if (col + 4 <= n_cols) {
                                const float4 cs = __ldg(reinterpret_cast<const float4*>(colscale + col));
                                *reinterpret_cast<float4*>(yz + static_cast<int64_t>(row) * ldz + col) =
                                    make_float4(__uint_as_float(dg[0]) * cs.x * rs, __uint_as_float(dg[1]) * cs.y * rs,
                                                __uint_as_float(dg[2]) * cs.z * rs, __uint_as_float(dg[3]) * cs.w * rs);
                            }
                        }
                    }
                }
                dev::tc_fence_before();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(&s.acc_empty[ab]);
            } else {
#pragma unroll 1
                for (int c = 0; c < 2 * nyb; ++c) {   // 32 columns at a time
                    uint32_t d0[16], d1[16];
                    dev::tmem_ld16(taddr + 32 * c, d0);
                    dev::tmem_ld16(taddr + 32 * c + 16, d1);
                    dev::tmem_ld_wait16(d0);
                    dev::tmem_ld_wait16(d1);
                    uint8_t* box = ybox(ab, c >> 1);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        // 16-byte chunk (c % 2) * 4 + j of row r sits at chunk position (that ^ r % 8)
                        const uint32_t pos = (static_cast<uint32_t>((c & 1) * 4 + j) ^ static_cast<uint32_t>(r & 7)) << 4;
                        const uint32_t* dj = j < 2 ? d0 + 8 * j : d1 + 8 * (j - 2);
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __half2 h = __floats2half2_rn(__uint_as_float(dj[2 * e]), __uint_as_float(dj[2 * e + 1]));
                            w[e] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                        *reinterpret_cast<uint4*>(box + r * 128 + pos) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                dev::tc_fence_before();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(&s.acc_empty[ab]);   // the accumulator is free again
                dev::fence_proxy_async_smem();   // the reduce reads what these threads wrote
                dev::named_bar_sync(2, 128);
                if (storer) {
                    dev::tma_reduce_add_2d(&tm_y, nt * kOTileN, mt * kOTileM, ybox(ab, 0));
                    if (nyb == 2) dev::tma_reduce_add_2d(&tm_y, nt * kOTileN + 64, mt * kOTileM, ybox(ab, 1));
                    dev::bulk_commit_group();
                    dev::bulk_wait_group_read1();   // tile i - 1's reduce has read its staging tile
                }
                __syncwarp();
            }
        }
        if (!kStore && storer) dev::bulk_wait_group0();   // every reduce performed before the CTA exits
        __syncwarp();
    }
    dev::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        dev::tc_fence_after();
        dev::tmem_dealloc(tmem, kOTmemCols);
    }
}

// A 2-D fp16 tensor [rows][cols] with row stride ld (elements), read in boxes of 64 x box_rows
// with the 128-byte swizzle.
bool make_map(EncodeTiledFn enc, CUtensorMap* map, const void* base, int64_t cols, int64_t rows, int64_t ld,
              uint32_t box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// QUIK zero-point term operands, fp16, K' = 2 nbp (nbp = nb rounded up to 32), one warp per row:
//   Zp[m][j] = z[j mod nbp][m]                              (the fp16 zero points)
//   Wp[n][j] = hi_b for j = b < nbp, lo_b for j = nbp + b     (0 for block indices >= nb)
// with hi_b = fp16_rn(2^e_n ws[b][n]), lo_b = fp16_rn(2^e_n ws[b][n] - hi_b), e_n putting the
// column's largest |ws| in [2^14, 2^15), colscale[n] = 2^-e_n. hi + lo hold 22 significant bits
// (w_sums = fp16 scale x code sum has at most 21), so z * hi + z * lo is z * ws exactly in FP32,
// except for terms below 2^-18 of their column's largest, whose lo part is an fp16 subnormal
// (error below 2^-40 of the column's largest term).
__global__ void zero_operands_kernel(const uint16_t* a_zeros, const float* w_sums, int64_t M, int64_t N, int nb,
                                     int nbp, uint16_t* Zp, uint16_t* Wp, float* colscale) {
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;   // warp-uniform
    const int lane = threadIdx.x & 31;
    const int kp = 2 * nbp;
    if (r < M) {
        uint16_t* row = Zp + r * kp;
        for (int b = lane; b < nbp; b += 32) {
            const uint16_t z = b < nb ? a_zeros[static_cast<int64_t>(b) * M + r] : uint16_t(0);
            row[b] = z;
            row[nbp + b] = z;
        }
    } else if (r < M + N) {
        const int64_t n = r - M;
        float mx = 0.0f;
        for (int b = lane; b < nb; b += 32) mx = fmaxf(mx, fabsf(w_sums[static_cast<int64_t>(b) * N + n]));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        int x = 0;
        if (mx > 0.0f) frexpf(mx, &x);          // mx = f 2^x, f in [0.5, 1)
        const int e = mx > 0.0f ? min(15 - x, 100) : 0;
        if (lane == 0) colscale[n] = ldexpf(1.0f, -e);
        uint16_t* row = Wp + n * kp;
        for (int b = lane; b < nbp; b += 32) {
            const float v = b < nb ? ldexpf(w_sums[static_cast<int64_t>(b) * N + n], e) : 0.0f;
            const __half h = __float2half_rn(v);
            const __half l = __float2half_rn(__fsub_rn(v, __half2float(h)));
            row[b] = __half_as_ushort(h);
            row[nbp + b] = __half_as_ushort(l);
        }
    }
}

// QoQ zero-point term (QServe explainer, "W4A8逐组快速反量化": the group zero point is subtracted
// after the multiplication). Per block b the term is -s1[n] s2[b][n] z2[b][n] * sx[m] sums[b][m];
// s1[n] and sx[m] leave the sum over b, which is an integer sum T[m][n] = sum_b sums[b][m] c[b][n]
// with c = s2 z2 <= 240. The operands split each code sum into 128 hi + lo (both exact in fp16,
// as is c), so every product is exact in FP32:
//   Zp[m][j] = 128 hi(sums[b][m]) for j = b < nbp, lo(sums[b][m]) for j = nbp + b
//   Wp[n][j] = c[b][n] for both halves,  colscale[n] = -s1[n],  rowscale[m] = sx[m].
__global__ void qoq_zero_operands_kernel(const int32_t* a_sums, const uint16_t* a_scales, const uint16_t* ch_scales,
                                         const uint8_t* grp_scales, const uint8_t* grp_zeros, int64_t M, int64_t N,
                                         int nb, int nbp, uint16_t* Zp, uint16_t* Wp, float* colscale,
                                         float* rowscale) {
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;   // warp-uniform
    const int lane = threadIdx.x & 31;
    const int kp = 2 * nbp;
    if (r < M) {
        uint16_t* row = Zp + r * kp;
        for (int b = lane; b < nbp; b += 32) {
            const int32_t v = b < nb ? a_sums[static_cast<int64_t>(b) * M + r] : 0;
            const int32_t hi = v >> 7;   // floor(v / 128); lo = v - 128 hi in [0, 128)
            row[b] = __half_as_ushort(__float2half_rn(static_cast<float>(hi * 128)));
            row[nbp + b] = __half_as_ushort(__float2half_rn(static_cast<float>(v - hi * 128)));
        }
        if (lane == 0) rowscale[r] = __half2float(__ushort_as_half(a_scales[r]));
    } else if (r < M + N) {
        const int64_t n = r - M;
        uint16_t* row = Wp + n * kp;
        for (int b = lane; b < nbp; b += 32) {
            const int64_t i = static_cast<int64_t>(b) * N + n;
            const uint16_t c = b < nb ? __half_as_ushort(__float2half_rn(static_cast<float>(
                                            static_cast<int>(grp_scales[i]) * static_cast<int>(grp_zeros[i]))))
                                      : uint16_t(0);
            row[b] = c;
            row[nbp + b] = c;
        }
        if (lane == 0) colscale[n] = -__half2float(__ushort_as_half(ch_scales[n]));
    }
}

int zero_nbp(int nb) { return (nb + 31) / 32 * 32; }
size_t align1k(size_t x) { return (x + 1023) & ~size_t(1023); }

}  // namespace

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

cudaError_t launch_outlier_gemm(const void* X, int64_t ldx, int64_t M, const int32_t* cols, int n_out,
                                const void* W_out, int64_t ldw_out, int64_t N, void* X_out, void* Y, int64_t ldy,
                                int num_sms, int32_t* status, cudaStream_t stream, bool* maps_ok) {
    *maps_ok = true;
    const EncodeTiledFn enc = encode_tiled();
    CUtensorMap tm_x, tm_w, tm_y;
    if (enc == nullptr || !make_map(enc, &tm_x, X_out, n_out, M, n_out, kOTileM) ||
        !make_map(enc, &tm_w, W_out, n_out, N, ldw_out, kOTileN) || !make_map(enc, &tm_y, Y, N, M, ldy, kOTileM)) {
        *maps_ok = false;
        return cudaSuccess;
    }
    cudaError_t e;
    if (X != nullptr) {   // otherwise X_out already holds the outlier columns (split by the quantizer)
        const unsigned gy = static_cast<unsigned>(M < 65535 ? M : 65535);
        outlier_gather_kernel<<<dim3(static_cast<unsigned>((n_out + 255) / 256), gy), 256, 0, stream>>>(
            static_cast<const uint16_t*>(X), ldx, M, cols, n_out, static_cast<uint16_t*>(X_out));
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    e = ensure_smem_limit(reinterpret_cast<const void*>(outlier_gemm_kernel<false>), static_cast<int>(kOSmemBytes));
    if (e != cudaSuccess) return e;
    const int64_t mtiles = (M + kOTileM - 1) / kOTileM, tiles = mtiles * ((N + kOTileN - 1) / kOTileN);
    const int64_t grid = tiles < num_sms ? tiles : (num_sms > 0 ? num_sms : 1);
    outlier_gemm_kernel<false><<<static_cast<unsigned>(grid), kOThreads, kOSmemBytes, stream>>>(
        tm_x, tm_w, tm_y, n_out, static_cast<int>(N), static_cast<int>(mtiles), tiles, nullptr, 0,
        static_cast<int>(M), nullptr, nullptr, status);
    return cudaGetLastError();
}

size_t zero_term_bytes(const fmpq_layout& L, int64_t M, int64_t N) {
    const size_t kp = 2 * static_cast<size_t>(zero_nbp(L.nb));
    return align1k(static_cast<size_t>(M) * N * 4) + align1k(static_cast<size_t>(M) * kp * 2) +
           align1k(static_cast<size_t>(N) * kp * 2) + align1k(static_cast<size_t>(N) * 4) +
           align1k(static_cast<size_t>(M) * 4);
}

cudaError_t launch_zero_term(const fmpq_layout& L, const GemmArgs& a, void* ws, cudaStream_t stream, bool* maps_ok) {
    const int64_t M = a.M, N = a.N;
    const bool qoq = a.zero_kind == kZeroQoq;
    *maps_ok = true;
    const int nbp = zero_nbp(L.nb), kp = 2 * nbp;
    uint8_t* base = static_cast<uint8_t*>(ws);
    float* yz = reinterpret_cast<float*>(base);
    base += align1k(static_cast<size_t>(M) * N * 4);
    uint16_t* zp = reinterpret_cast<uint16_t*>(base);
    base += align1k(static_cast<size_t>(M) * kp * 2);
    uint16_t* wp = reinterpret_cast<uint16_t*>(base);
    base += align1k(static_cast<size_t>(N) * kp * 2);
    float* colscale = reinterpret_cast<float*>(base);
    base += align1k(static_cast<size_t>(N) * 4);
    float* rowscale = reinterpret_cast<float*>(base);
    const EncodeTiledFn enc = encode_tiled();
    CUtensorMap tm_x, tm_w;
    if (enc == nullptr || !make_map(enc, &tm_x, zp, kp, M, kp, kOTileM) || !make_map(enc, &tm_w, wp, kp, N, kp, kOTileN)) {
        *maps_ok = false;
        return cudaSuccess;
    }
    const int64_t warps = M + N;
    if (qoq)
        qoq_zero_operands_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(
            a.a_sums, static_cast<const uint16_t*>(a.a_scales), static_cast<const uint16_t*>(a.ch_scales),
            a.grp_scales, a.grp_zeros, M, N, L.nb, nbp, zp, wp, colscale, rowscale);
    else
        zero_operands_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(
            static_cast<const uint16_t*>(a.a_zeros), a.w_sums, M, N, L.nb, nbp, zp, wp, colscale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = ensure_smem_limit(reinterpret_cast<const void*>(outlier_gemm_kernel<true>), static_cast<int>(kOSmemBytes));
    if (e != cudaSuccess) return e;
    const int64_t mtiles = (M + kOTileM - 1) / kOTileM, tiles = mtiles * ((N + kOTileN - 1) / kOTileN);
    const int64_t grid = tiles < L.num_sms ? tiles : (L.num_sms > 0 ? L.num_sms : 1);
    outlier_gemm_kernel<true><<<static_cast<unsigned>(grid), kOThreads, kOSmemBytes, stream>>>(
        tm_x, tm_w, tm_x, kp, static_cast<int>(N), static_cast<int>(mtiles), tiles, yz, N, static_cast<int>(M),
        colscale, qoq ? rowscale : nullptr, L.d_status);
    return cudaGetLastError();
}

}  // namespace fmpq
