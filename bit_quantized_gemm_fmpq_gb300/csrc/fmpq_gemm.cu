// FMPQ W4Ax GEMM for sm_103a (GB300).
//
// Y[m][n] = sum_b a_scale[b][m] * w_scale[b][n] * P[m][n][b],  P = exact per-block integer
// dot products of the INT4/INT8 activation codes with the INT4 weight codes (COMET
// abstract: W4A4/W4A8 mixed-precision GEMM with a software pipeline hiding load and
// conversion; QUIK explainer, "kernel fusion": dequantization in the GEMM epilogue).
//
// GB300 mapping (sm_103a has no integer tcgen05 MMA):
//   * Codes are exact E4M3 tensor-core operands. The activation quantizer already writes
//     them that way (one byte per code, value part * 2^-9, rows pre-swizzled), so a
//     128-row activation tile is one bulk copy straight into the operand ring. An INT8
//     block has two planes (|q| mod 16 and the rest) that accumulate into the same TMEM
//     tile, so every block ends in one FP32 tile P * 2^-18 (exact: |P| < 2^17).
//   * INT4 weights stay 4-bit in HBM: converter warps turn each packed word into 8
//     operand bytes with a mask and a rotate (the sign-magnitude byte s0000mmm is the E4M3
//     value (-1)^s * m * 2^-9) -- the restructured storage format that makes 4-bit ->
//     8-bit conversion a couple of instructions (COMET news article, section 3).
//   * tcgen05.mma kind::f8f6f4 (M=128, N=256, K=32) with the accumulator in TMEM,
//     double-buffered so the MMA of the next block overlaps the epilogue of this one.
//   * Per block the epilogue warps read the tile (tcgen05.ld) and accumulate
//     acc += (w_scale[n] * a_scale[m] * 2^18) * D in FP32 registers (packed f32x2 math).
//
// Warp roles (512 threads, one CTA per SM, persistent over tiles):
//   warp 0       TMA producer: activation code planes and the packed weight tile per block
//   warp 1       tcgen05 MMA issuer (one thread) + TMEM owner
//   warps 2-7    converters: packed weight codes -> 128B-swizzled K-major E4M3 tile
//   warps 8-15   epilogue: per-block FP32 scale-and-sum, fp16 output (or split-K partials)
#include <cuda_fp16.h>

#include "fmpq_device.cuh"
#include "fmpq_internal.h"

namespace fmpq {
namespace {

constexpr int kThreads = 512;
constexpr int kStages = 3;    // per-block stage: activation planes + packed weights
constexpr int kCvStages = 2;  // converted weight tiles
constexpr int kConvWarps = 6;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr uint32_t kTmemCols = 512;  // two 128 x 256 FP32 accumulators
constexpr uint32_t kIdesc = dev::idesc_e4m3_f32(128, 256);

struct __align__(1024) Smem {
    uint8_t opA[kStages][2][128 * 128];  // activation code planes (operand-ready, swizzled)
    uint8_t cvB[kCvStages][256 * 128];   // E4M3 weight operand (256 rows x 128 K), swizzled
    uint8_t pkW[kStages][256 * 64];      // packed weight codes
    float sw[2][256];                    // per-block weight scales (fp32) for the epilogue
    uint64_t st_full[kStages], st_empty[kStages];
    uint64_t cv_full[kCvStages], cv_empty[kCvStages];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int fixup_last;
};

struct Params {
    const uint8_t* A;
    const uint16_t* a_scales;
    const uint8_t* W;
    const uint16_t* w_scales;
    uint16_t* Y;
    int64_t ldy;
    int M, N, nb;
    const uint8_t* mask;
    const int32_t* poff;   // first code plane of each block
    int32_t* status;
    // tiles: the kernel covers m-tiles [mt0, mt0 + mtiles) x n-tiles [nt0, nt0 + ntiles)
    int mt0, mtiles, nt0, ntiles;
    int splits;            // K splits per tile (1 = none)
    float* ws_partial;     // [tiles][splits][128][256] FP32 partial sums (splits > 1)
    int32_t* ws_count;     // [tiles] arrival counters (zero between calls)
    // partial-sum export
    int32_t* P;
    int pm0, pmcount, pn0, pncount;
};

__device__ __forceinline__ uint32_t lo4(uint32_t w) { return w & 0x87878787u; }
__device__ __forceinline__ uint32_t hi4(uint32_t w) { return __funnelshift_r(w, w, 4) & 0x87878787u; }

// Work unit u -> (tile, split). Tiles are ordered m-fastest so the CTAs running together
// share weight panels in L2.
struct Unit {
    int mt, nt, tile, split, b0, b1;
};
__device__ __forceinline__ Unit unit_of(const Params& p, int u) {
    Unit r;
    r.tile = u / p.splits;
    r.split = u % p.splits;
    r.mt = p.mt0 + r.tile % p.mtiles;
    r.nt = p.nt0 + r.tile / p.mtiles;
    r.b0 = static_cast<int>((static_cast<int64_t>(r.split) * p.nb) / p.splits);
    r.b1 = static_cast<int>((static_cast<int64_t>(r.split + 1) * p.nb) / p.splits);
    return r;
}

// ---------------------------------------------------------------- TMA producer (warp 0)
__device__ __forceinline__ void producer_role(const Params& p, Smem& s, int lane, volatile int* abort_flag) {
    const int num_units = p.mtiles * p.ntiles * p.splits;
    if (lane == 0) {
        uint32_t it = 0;
        bool ok = true;
        const int64_t plane_bytes = static_cast<int64_t>(p.M) * kBlock;
        for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
            const Unit t = unit_of(p, u);
            const int m0 = t.mt * kTileM;
            const uint32_t abytes = static_cast<uint32_t>(min(kTileM, p.M - m0)) * kBlock;
            for (int b = t.b0; b < t.b1; ++b, ++it) {
                const int st = it % kStages;
                if (!dev::mbar_wait(&s.st_empty[st], ((it / kStages) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int planes = p.mask[b] ? 2 : 1;
                dev::mbar_arrive_expect_tx(&s.st_full[st], abytes * planes + 256 * 64);
                const uint8_t* a0 = p.A + static_cast<int64_t>(p.poff[b]) * plane_bytes + static_cast<int64_t>(m0) * kBlock;
                dev::bulk_g2s(s.opA[st][0], a0, abytes, &s.st_full[st]);
                if (planes == 2) dev::bulk_g2s(s.opA[st][1], a0 + plane_bytes, abytes, &s.st_full[st]);
                dev::bulk_g2s(s.pkW[st], p.W + (static_cast<int64_t>(t.nt) * p.nb + b) * (256 * 64), 256 * 64,
                              &s.st_full[st]);
            }
        }
        if (!ok) {
            *abort_flag = 1;
            dev::report(p.status, dev::kStatusTimeout);
        }
        // drain copies in flight
        for (int st = 0; st < kStages; ++st) {
            if (it <= static_cast<uint32_t>(st)) break;
            const uint32_t last = st + ((it - 1 - st) / kStages) * kStages;
            dev::mbar_wait(&s.st_full[st], (last / kStages) & 1, nullptr);
        }
    }
}

// ---------------------------------------------------------------- MMA issuer (warp 1)
__device__ __forceinline__ void mma_role(const Params& p, Smem& s, int lane, uint32_t tmem, volatile int* abort_flag) {
    const int num_units = p.mtiles * p.ntiles * p.splits;
    if (lane == 0) {
        uint32_t it = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
            const Unit t = unit_of(p, u);
            for (int b = t.b0; b < t.b1; ++b, ++it) {
                const int st = it % kStages;
                const int cs = it % kCvStages;
                const int ab = it & 1;
                if (!dev::mbar_wait(&s.st_full[st], (it / kStages) & 1, abort_flag) ||
                    !dev::mbar_wait(&s.cv_full[cs], (it / kCvStages) & 1, abort_flag) ||
                    !dev::mbar_wait(&s.acc_empty[ab], ((it >> 1) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                dev::tc_fence_after();
                const uint64_t bd = dev::sdesc_k_sw128(dev::smem_u32(s.cvB[cs]));
                const uint32_t d = tmem + static_cast<uint32_t>(ab) * 256u;
                const int planes = p.mask[b] ? 2 : 1;
                for (int pl = 0; pl < planes; ++pl) {
                    const uint64_t ad = dev::sdesc_k_sw128(dev::smem_u32(s.opA[st][pl]));
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dev::mma_e4m3(d, ad + 2 * k, bd + 2 * k, kIdesc, (pl > 0 || k > 0) ? 1u : 0u);
                }
                dev::mma_commit(&s.st_empty[st]);
                dev::mma_commit(&s.cv_empty[cs]);
                dev::mma_commit(&s.acc_full[ab]);
            }
        }
        if (!ok) {
            *abort_flag = 1;
            dev::report(p.status, dev::kStatusTimeout);
        }
        // every MMA issued must finish before TMEM is released
        dev::mma_commit(&s.mma_done);
        dev::mbar_wait(&s.mma_done, 0, nullptr);
    }
}

// ---------------------------------------------------------------- converters (warps 2-7)
// The weight tile is 256 rows x 8 chunks (8 packed bytes in, 16 operand bytes out). Thread
// ct converts items ct + 192k: item i is row i/8, chunk i%8. Since 192 = 24 rows, the
// chunk and the row's swizzle phase (row mod 8) are the same for every k, so each item's
// source and destination are the thread's base offsets plus constants.
__device__ __forceinline__ void converter_role(const Params& p, Smem& s, int warp, int lane, volatile int* abort_flag) {
    const int num_units = p.mtiles * p.ntiles * p.splits;
    const int ct = (warp - 2) * 32 + lane;
    const int r0 = ct >> 3, c = ct & 7;
    const uint32_t src0 = static_cast<uint32_t>(r0 * 64 + c * 8);
    const uint32_t dst0 = static_cast<uint32_t>(r0 * 128 + ((c ^ (r0 & 7)) << 4));
    constexpr int kFull = (256 * 8) / kConvThreads;                      // 10 items for every thread
    const bool extra = ct + kFull * kConvThreads < 256 * 8;              // an 11th for the first 128
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
        const Unit t = unit_of(p, u);
        for (int b = t.b0; b < t.b1; ++b, ++it) {
            const int st = it % kStages;
            const int cs = it % kCvStages;
            if (lane == 0)
                ok = dev::mbar_wait(&s.st_full[st], (it / kStages) & 1, abort_flag) &&
                     dev::mbar_wait(&s.cv_empty[cs], ((it / kCvStages) & 1) ^ 1, abort_flag);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            const uint8_t* src = s.pkW[st] + src0;
            uint8_t* dst = s.cvB[cs] + dst0;
#pragma unroll
            for (int k0 = 0; k0 < kFull; k0 += 5) {
                uint2 w[5];
#pragma unroll
                for (int k = 0; k < 5; ++k) w[k] = *reinterpret_cast<const uint2*>(src + (k0 + k) * 24 * 64);
#pragma unroll
                for (int k = 0; k < 5; ++k)
                    *reinterpret_cast<uint4*>(dst + (k0 + k) * 24 * 128) =
                        make_uint4(lo4(w[k].x), hi4(w[k].x), lo4(w[k].y), hi4(w[k].y));
            }
            if (extra) {
                const uint2 w = *reinterpret_cast<const uint2*>(src + kFull * 24 * 64);
                *reinterpret_cast<uint4*>(dst + kFull * 24 * 128) = make_uint4(lo4(w.x), hi4(w.x), lo4(w.y), hi4(w.y));
            }
            dev::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(&s.cv_full[cs]);
        }
    }
    if (!ok && lane == 0) {
        *abort_flag = 1;
        dev::report(p.status, dev::kStatusTimeout);
    }
}

// ---------------------------------------------------------------- epilogue (warps 8-15)
template <bool kPartials>
__device__ __forceinline__ void epilogue_role(const Params& p, Smem& s, int warp, int lane, uint32_t tmem,
                                              volatile int* abort_flag) {
    const int num_units = p.mtiles * p.ntiles * p.splits;
    // ======================= epilogue
    const int ew = warp - 8;           // 0..7
    const int q = warp & 3;            // TMEM lane quarter of this warp
    const int h = ew >> 2;             // column half: 0 -> cols 0..127, 1 -> 128..255
    const int et = ew * 32 + lane;     // 0..255
    uint32_t v = 0, bstep = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        const Unit t = unit_of(p, u);
        const int m0 = t.mt * kTileM, n0 = t.nt * kTileN;
        const int row = m0 + q * 32 + lane;
        const bool row_ok = row < p.M;
        float2 acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.f, 0.f);
        // prefetch scales of the first block
        const int ncol = n0 + et;
        float sw_next = (t.b0 < t.b1 && ncol < p.N) ? __half2float(__ushort_as_half(p.w_scales[static_cast<int64_t>(t.b0) * p.N + ncol])) : 0.f;
        float sx_next = (t.b0 < t.b1 && row_ok) ? __half2float(__ushort_as_half(p.a_scales[static_cast<int64_t>(t.b0) * p.M + row])) : 0.f;
        for (int b = t.b0; b < t.b1; ++b, ++bstep, ++v) {
            const float sw_cur = sw_next, sx_cur = sx_next;
            if (b + 1 < t.b1) {
                sw_next = (ncol < p.N) ? __half2float(__ushort_as_half(p.w_scales[static_cast<int64_t>(b + 1) * p.N + ncol])) : 0.f;
                sx_next = row_ok ? __half2float(__ushort_as_half(p.a_scales[static_cast<int64_t>(b + 1) * p.M + row])) : 0.f;
            }
            float* swb = s.sw[bstep & 1];
            swb[et] = sw_cur;
            dev::named_bar_sync(1, kEpiThreads);
            const int ab = v & 1;
            if (ok) {
                if (lane == 0) ok = dev::mbar_wait(&s.acc_full[ab], (v >> 1) & 1, abort_flag);
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            }
            if (ok) {
                dev::tc_fence_after();
                const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + ab * 256u + h * 128u;
                if constexpr (!kPartials) {
                    // 2^18 undoes the operand encoding (both operands carry 2^-9)
                    const float sxp = sx_cur * 262144.0f;
                    const float2 sx2 = make_float2(sxp, sxp);
#pragma unroll
                    for (int chunk = 0; chunk < 4; ++chunk) {
                        uint32_t d[32];
                        dev::tmem_ld32(taddr + chunk * 32, d);
                        dev::tmem_ld_wait();
                        const float4* sw4 = reinterpret_cast<const float4*>(swb + h * 128 + chunk * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 w4 = sw4[j];
                            const float2 c01 = dev::fmul2(make_float2(w4.x, w4.y), sx2);
                            const float2 c23 = dev::fmul2(make_float2(w4.z, w4.w), sx2);
                            float2& a01 = acc[chunk * 16 + 2 * j];
                            float2& a23 = acc[chunk * 16 + 2 * j + 1];
                            a01 = dev::ffma2(make_float2(__uint_as_float(d[4 * j]), __uint_as_float(d[4 * j + 1])), c01, a01);
                            a23 = dev::ffma2(make_float2(__uint_as_float(d[4 * j + 2]), __uint_as_float(d[4 * j + 3])), c23, a23);
                        }
                    }
                } else {
                    // export exact partial sums of the requested window
#pragma unroll 1
                    for (int chunk = 0; chunk < 4; ++chunk) {
                        uint32_t d[32];
                        dev::tmem_ld32(taddr + chunk * 32, d);
                        dev::tmem_ld_wait();
                        if (row_ok && row >= p.pm0 && row < p.pm0 + p.pmcount) {
                            for (int j = 0; j < 32; ++j) {
                                const int n = n0 + h * 128 + chunk * 32 + j;
                                if (n < p.pn0 || n >= p.pn0 + p.pncount || n >= p.N) continue;
                                p.P[(static_cast<int64_t>(row - p.pm0) * p.pncount + (n - p.pn0)) * p.nb + b] =
                                    __float2int_rn(__uint_as_float(d[j]) * 262144.0f);
                            }
                        }
                    }
                }
                dev::tc_fence_before();
            }
            __syncwarp();
            if (lane == 0 && ok) dev::mbar_arrive(&s.acc_empty[ab]);
        }
        if constexpr (!kPartials) {
            const int cbase = n0 + h * 128;
            if (p.splits == 1) {
                if (row_ok) {
                    uint16_t* yrow = p.Y + static_cast<int64_t>(row) * p.ldy;
#pragma unroll
                    for (int c8 = 0; c8 < 16; ++c8) {
                        const int col = cbase + c8 * 8;
                        if (col < p.N) {
                            uint4 o;
                            __half2 h0 = __floats2half2_rn(acc[c8 * 4 + 0].x, acc[c8 * 4 + 0].y);
                            __half2 h1 = __floats2half2_rn(acc[c8 * 4 + 1].x, acc[c8 * 4 + 1].y);
                            __half2 h2 = __floats2half2_rn(acc[c8 * 4 + 2].x, acc[c8 * 4 + 2].y);
                            __half2 h3 = __floats2half2_rn(acc[c8 * 4 + 3].x, acc[c8 * 4 + 3].y);
                            o.x = *reinterpret_cast<uint32_t*>(&h0);
                            o.y = *reinterpret_cast<uint32_t*>(&h1);
                            o.z = *reinterpret_cast<uint32_t*>(&h2);
                            o.w = *reinterpret_cast<uint32_t*>(&h3);
                            *reinterpret_cast<uint4*>(yrow + col) = o;
                        }
                    }
                }
            } else {
                // split-K: publish this split's FP32 partial; the last split to arrive sums
                // all of them in split order (deterministic) and writes Y.
                float* part = p.ws_partial +
                              ((static_cast<int64_t>(t.tile) * p.splits + t.split) * kTileM + q * 32 + lane) * kTileN + h * 128;
                if (row_ok) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        __stcg(reinterpret_cast<float4*>(part) + i, make_float4(acc[2 * i].x, acc[2 * i].y, acc[2 * i + 1].x, acc[2 * i + 1].y));
                }
                __threadfence();
                dev::named_bar_sync(1, kEpiThreads);
                if (et == 0) {
                    const int prev = atomicAdd(p.ws_count + t.tile, 1);
                    const int last = (prev == p.splits - 1);
                    if (last) p.ws_count[t.tile] = 0;  // reusable for the next call
                    s.fixup_last = last;
                }
                dev::named_bar_sync(1, kEpiThreads);
                if (s.fixup_last) {
                    // every split (this one included) is in the workspace: sum in split order
                    __threadfence();
#pragma unroll
                    for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.f, 0.f);
                    if (row_ok) {
                        for (int sp = 0; sp < p.splits; ++sp) {
                            const float* o = p.ws_partial +
                                             ((static_cast<int64_t>(t.tile) * p.splits + sp) * kTileM + q * 32 + lane) * kTileN + h * 128;
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const float4 f = __ldcg(reinterpret_cast<const float4*>(o) + i);
                                acc[2 * i].x += f.x;
                                acc[2 * i].y += f.y;
                                acc[2 * i + 1].x += f.z;
                                acc[2 * i + 1].y += f.w;
                            }
                        }
                    }
                    if (row_ok) {
                        uint16_t* yrow = p.Y + static_cast<int64_t>(row) * p.ldy;
#pragma unroll
                        for (int c8 = 0; c8 < 16; ++c8) {
                            const int col = cbase + c8 * 8;
                            if (col < p.N) {
                                uint4 o;
                                __half2 h0 = __floats2half2_rn(acc[c8 * 4 + 0].x, acc[c8 * 4 + 0].y);
                                __half2 h1 = __floats2half2_rn(acc[c8 * 4 + 1].x, acc[c8 * 4 + 1].y);
                                __half2 h2 = __floats2half2_rn(acc[c8 * 4 + 2].x, acc[c8 * 4 + 2].y);
                                __half2 h3 = __floats2half2_rn(acc[c8 * 4 + 3].x, acc[c8 * 4 + 3].y);
                                o.x = *reinterpret_cast<uint32_t*>(&h0);
                                o.y = *reinterpret_cast<uint32_t*>(&h1);
                                o.z = *reinterpret_cast<uint32_t*>(&h2);
                                o.w = *reinterpret_cast<uint32_t*>(&h3);
                                *reinterpret_cast<uint4*>(yrow + col) = o;
                            }
                        }
                    }
                }
            }
        }
    }
    if (!ok && lane == 0) {
        *abort_flag = 1;
        dev::report(p.status, dev::kStatusTimeout);
    }
}

template <bool kPartials>
__global__ void __launch_bounds__(kThreads, 1) w4ax_gemm_kernel(const Params p) {
    extern __shared__ uint8_t smem_raw[];
    Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            dev::mbar_init(&s.st_full[i], 1);
            dev::mbar_init(&s.st_empty[i], 1);
        }
        for (int i = 0; i < kCvStages; ++i) {
            dev::mbar_init(&s.cv_full[i], kConvWarps);
            dev::mbar_init(&s.cv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            dev::mbar_init(&s.acc_full[i], 1);
            dev::mbar_init(&s.acc_empty[i], kEpiWarps);
        }
        dev::mbar_init(&s.mma_done, 1);
        s.abort_flag = 0;
        dev::fence_barrier_init();
    }
    if (warp == 1) dev::tmem_alloc(&s.tmem_base, kTmemCols);
    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int* abort_flag = &s.abort_flag;

    if (warp < 8) {
        dev::setmaxnreg_dec<64>();
        if (warp == 0)
            producer_role(p, s, lane, abort_flag);
        else if (warp == 1)
            mma_role(p, s, lane, tmem, abort_flag);
        else
            converter_role(p, s, warp, lane, abort_flag);
    } else {
        dev::setmaxnreg_inc<192>();
        epilogue_role<kPartials>(p, s, warp, lane, tmem, abort_flag);
    }

    dev::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        dev::tc_fence_after();
        dev::tmem_dealloc(tmem, kTmemCols);
    }
}


constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

int choose_splits(const fmpq_layout& L, int64_t tiles) {
    if (tiles * 2 > L.num_sms) return 1;
    int s = static_cast<int>(L.num_sms / tiles);
    if (s > L.nb) s = L.nb;
    if (s > 16) s = 16;
    return s < 1 ? 1 : s;
}

}  // namespace

size_t gemm_workspace_bytes(const fmpq_layout& L, int64_t M, int64_t N) {
    const int64_t tiles = ((M + kTileM - 1) / kTileM) * ((N + kTileN - 1) / kTileN);
    const int splits = choose_splits(L, tiles);
    if (splits == 1) return 0;
    return static_cast<size_t>(tiles) * splits * kTileM * kTileN * sizeof(float) + static_cast<size_t>(tiles) * 4 + 16;
}

cudaError_t launch_gemm(const fmpq_layout& L, const GemmArgs& a, cudaStream_t stream) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(w4ax_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(w4ax_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    Params p{};
    p.A = static_cast<const uint8_t*>(a.A);
    p.a_scales = static_cast<const uint16_t*>(a.a_scales);
    p.W = static_cast<const uint8_t*>(a.W);
    p.w_scales = static_cast<const uint16_t*>(a.w_scales);
    p.Y = static_cast<uint16_t*>(a.Y);
    p.ldy = a.ldy;
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.N);
    p.nb = L.nb;
    p.mask = L.d_mask;
    p.poff = L.d_poff;
    p.status = L.d_status;
    const bool partials = a.P != nullptr;
    if (partials) {
        p.mt0 = static_cast<int>(a.pm0 / kTileM);
        p.mtiles = static_cast<int>((a.pm0 + a.pmcount - 1) / kTileM) - p.mt0 + 1;
        p.nt0 = static_cast<int>(a.pn0 / kTileN);
        p.ntiles = static_cast<int>((a.pn0 + a.pncount - 1) / kTileN) - p.nt0 + 1;
        p.splits = 1;
        p.P = a.P;
        p.pm0 = static_cast<int>(a.pm0);
        p.pmcount = static_cast<int>(a.pmcount);
        p.pn0 = static_cast<int>(a.pn0);
        p.pncount = static_cast<int>(a.pncount);
    } else {
        p.mt0 = 0;
        p.mtiles = static_cast<int>((a.M + kTileM - 1) / kTileM);
        p.nt0 = 0;
        p.ntiles = static_cast<int>((a.N + kTileN - 1) / kTileN);
        p.splits = choose_splits(L, static_cast<int64_t>(p.mtiles) * p.ntiles);
        if (p.splits > 1) {
            const int64_t tiles = static_cast<int64_t>(p.mtiles) * p.ntiles;
            p.ws_partial = static_cast<float*>(a.workspace);
            p.ws_count = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a.workspace) +
                                                    static_cast<size_t>(tiles) * p.splits * kTileM * kTileN * sizeof(float));
        }
    }
    const int64_t units = static_cast<int64_t>(p.mtiles) * p.ntiles * p.splits;
    const int grid = static_cast<int>(units < L.num_sms ? units : L.num_sms);
    if (partials)
        w4ax_gemm_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(p);
    else
        w4ax_gemm_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace fmpq
