// The FP16 outlier path of an outlier split (QUIK explainer, "第二步: 前向传播"): the input's
// outlier columns are multiplied in FP16 by the unquantized outlier weights and the result is
// added to the output of the INT4 path (the base columns, fmpq_layout_create_select +
// w4ax_gemm).
//
//   outlier_gather_kernel  X[:, cols] -> a dense fp16 [M][n_out] operand (one element per thread)
//   outlier_gemm_kernel    Y[m][n] += sum_j X_out[m][j] * W_out[n][j] on the tensor cores
//                          (tcgen05.mma kind::f16, FP32 accumulator in TMEM), one 128 x 128
//                          output tile per CTA:
//     warp 0       TMA producer: the tile's Y (read-modify-write) and, per 64-channel chunk of
//                  the outlier columns, the X_out and W_out boxes (128-byte swizzle), 2 stages
//     warp 1       TMEM allocation and the single-thread MMA issuer (M = 128, N = 128, K = 16)
//     warps 2-5    epilogue: TMEM lane quarter warp % 4, one output row per thread; adds the
//                  FP32 accumulator to Y in shared memory and stores the tile with TMA
// The product is HBM-bound on Y's read and write (n_out is small); two CTAs share an SM.
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
constexpr int kOStages = 2;
constexpr uint32_t kOTmemCols = 128;
constexpr uint32_t kOIdesc = dev::idesc_f16_f32(kOTileM, kOTileN);

struct __align__(1024) OSmem {
    uint8_t a[kOStages][kOTileM * kOChunk * 2];   // X_out box: 128 rows x 64 channels (swizzled)
    uint8_t b[kOStages][kOTileN * kOChunk * 2];   // W_out box: 128 rows x 64 channels (swizzled)
    uint8_t y[2][kOTileM * 64 * 2];               // Y tile as two boxes of 64 columns (swizzled)
    uint64_t full[kOStages], empty[kOStages];
    uint64_t y_full, mma_done;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t kOSmemBytes = sizeof(OSmem) + 1024;

__global__ void __launch_bounds__(kOThreads, 2)
    outlier_gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_y, int n_out, int n_cols, int32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    OSmem& s = *reinterpret_cast<OSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kOTileM, n0 = blockIdx.y * kOTileN;
    const int yboxes = n_cols - n0 > 64 ? 2 : 1;   // a Y box wholly past N is neither loaded nor stored
    const int chunks = (n_out + kOChunk - 1) / kOChunk;
    volatile int* abort_flag = &s.abort_flag;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kOStages; ++i) {
            dev::mbar_init(&s.full[i], 1);
            dev::mbar_init(&s.empty[i], 1);
        }
        dev::mbar_init(&s.y_full, 1);
        dev::mbar_init(&s.mma_done, 1);
        s.abort_flag = 0;
        dev::fence_barrier_init();
    }
    if (warp == 1) dev::tmem_alloc(&s.tmem_base, kOTmemCols);
    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    const uint32_t tmem = s.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // the tile's Y first: the epilogue adds to it
            dev::mbar_arrive_expect_tx(&s.y_full, yboxes * kOTileM * 64 * 2);
            dev::tma_load_2d(s.y[0], &tm_y, n0, m0, &s.y_full);
            if (yboxes == 2) dev::tma_load_2d(s.y[1], &tm_y, n0 + 64, m0, &s.y_full);
            int kc = 0;
            for (; kc < chunks; ++kc) {
                const int st = kc % kOStages;
                if (!dev::mbar_wait(&s.empty[st], ((kc / kOStages) & 1) ^ 1, abort_flag)) {
                    *abort_flag = 1;
                    dev::report(status, dev::kStatusTimeout);
                    break;
                }
                dev::mbar_arrive_expect_tx(&s.full[st], (kOTileM + kOTileN) * kOChunk * 2);
                dev::tma_load_2d(s.a[st], &tm_x, kc * kOChunk, m0, &s.full[st]);
                dev::tma_load_2d(s.b[st], &tm_w, kc * kOChunk, n0, &s.full[st]);
            }
            // drain: every load issued lands before the CTA exits
            for (int k = kc - 1; k >= 0 && k >= kc - kOStages; --k)
                dev::mbar_wait(&s.full[k % kOStages], (k / kOStages) & 1, nullptr);
            dev::mbar_wait(&s.y_full, 0, nullptr);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            for (int kc = 0; kc < chunks; ++kc) {
                const int st = kc % kOStages;
                if (!dev::mbar_wait(&s.full[st], (kc / kOStages) & 1, abort_flag)) {
                    *abort_flag = 1;
                    dev::report(status, dev::kStatusTimeout);
                    break;
                }
                dev::tc_fence_after();
                const uint64_t ad = dev::sdesc_k_sw128(dev::smem_u32(s.a[st]));
                const uint64_t bd = dev::sdesc_k_sw128(dev::smem_u32(s.b[st]));
#pragma unroll
                for (int k = 0; k < kOChunk / 16; ++k)   // 32 bytes of K per MMA: +2 in the address field
                    dev::mma_f16(tmem, ad + 2 * k, bd + 2 * k, kOIdesc, (kc > 0 || k > 0) ? 1u : 0u);
                dev::mma_commit(&s.empty[st]);
            }
            dev::mma_commit(&s.mma_done);   // every MMA issued completes before mma_done
            dev::mbar_wait(&s.mma_done, 0, nullptr);   // and before TMEM is released
        }
        __syncwarp();
    } else {
        // epilogue: thread owns tile row r (TMEM lane r); columns in chunks of 32
        const int q = warp & 3;
        const int r = 32 * q + lane;
        bool ok = dev::mbar_wait(&s.mma_done, 0, abort_flag) && dev::mbar_wait(&s.y_full, 0, abort_flag);
        ok = __all_sync(0xFFFFFFFFu, ok) && !*abort_flag;
        if (ok) {
            dev::tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16);
#pragma unroll 1
            for (int c = 0; c < 4 * yboxes; ++c) {   // 16 columns at a time
                uint32_t d[16];
                dev::tmem_ld16(taddr + 16 * c, d);
                dev::tmem_ld_wait16(d);
                uint8_t* box = s.y[c >> 2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    // 16-byte chunk (c % 4) * 2 + j of row r sits at chunk position (that ^ r % 8)
                    const uint32_t pos = ((static_cast<uint32_t>((c & 3) * 2 + j) ^ static_cast<uint32_t>(r & 7)) << 4);
                    uint4* yp = reinterpret_cast<uint4*>(box + r * 128 + pos);
                    uint4 v = *yp;
                    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 old = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                        const __half2 nv = __floats2half2_rn(old.x + __uint_as_float(d[8 * j + 2 * e]),
                                                             old.y + __uint_as_float(d[8 * j + 2 * e + 1]));
                        w[e] = *reinterpret_cast<const uint32_t*>(&nv);
                    }
                    *yp = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            dev::fence_proxy_async_smem();   // the TMA store reads what these threads wrote
        } else if (lane == 0) {
            *abort_flag = 1;
            dev::report(status, dev::kStatusTimeout);
        }
        dev::named_bar_sync(1, 128);
        if (warp == 2 && lane == 0 && !*abort_flag) {
            dev::tma_store_2d(&tm_y, n0, m0, s.y[0]);
            if (yboxes == 2) dev::tma_store_2d(&tm_y, n0 + 64, m0, s.y[1]);
            dev::bulk_commit_group();
            dev::bulk_wait_group_read0();   // shared memory stays valid until the store has read it
        }
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
                                int32_t* status, cudaStream_t stream, bool* maps_ok) {
    *maps_ok = true;
    const EncodeTiledFn enc = encode_tiled();
    CUtensorMap tm_x, tm_w, tm_y;
    if (enc == nullptr || !make_map(enc, &tm_x, X_out, n_out, M, n_out, kOTileM) ||
        !make_map(enc, &tm_w, W_out, n_out, N, ldw_out, kOTileN) || !make_map(enc, &tm_y, Y, N, M, ldy, kOTileM)) {
        *maps_ok = false;
        return cudaSuccess;
    }
    const unsigned gy = static_cast<unsigned>(M < 65535 ? M : 65535);
    outlier_gather_kernel<<<dim3(static_cast<unsigned>((n_out + 255) / 256), gy), 256, 0, stream>>>(
        static_cast<const uint16_t*>(X), ldx, M, cols, n_out, static_cast<uint16_t*>(X_out));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = ensure_smem_limit(reinterpret_cast<const void*>(outlier_gemm_kernel), static_cast<int>(kOSmemBytes));
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>((M + kOTileM - 1) / kOTileM), static_cast<unsigned>((N + kOTileN - 1) / kOTileN));
    outlier_gemm_kernel<<<grid, kOThreads, kOSmemBytes, stream>>>(tm_x, tm_w, tm_y, n_out, static_cast<int>(N), status);
    return cudaGetLastError();
}

}  // namespace fmpq
