// FMPQ W4Ax GEMM for few tokens (M <= 128, the decode shapes) on sm_103a.
//
// Same result as the main GEMM: Y[m][n] = sum_b a_scale[b][m] * w_scale[b][n] * P[m][n][b],
// P = exact per-block integer dot products (COMET abstract: mixed W4A4/W4A8 GEMM; QUIK
// explainer, "kernel fusion": dequantization in the GEMM epilogue). With few tokens the
// weights are the only large operand and the GEMM is bound by reading them from HBM, so
// the roles of the operands are swapped:
//   * the tensor core's M side is the output channels: a pair of CTAs covers 256 weight
//     rows (128 per CTA), converted from the 4-bit packed tile exactly as in the main GEMM;
//   * its N side is the tokens, T = 16, 32, 64 or 128 (M rounded up), each CTA holding T/2
//     rows of every activation code plane in shared memory;
//   * an accumulator is 128 lanes x T columns of TMEM, so 4-8 of them are in flight and
//     the per-block FP32 epilogue is 128 x T scale-and-adds per CTA;
//   * two groups of converter warps take alternate blocks, so that converting the weights
//     keeps up with streaming them;
//   * few output tiles: K is split across pairs (deterministic split-K).
//
// Warp roles (512 threads, one CTA per SM, clusters of two, persistent over units):
//   warp 0       weight producer: this CTA's 128 rows (8 KB) of each packed weight tile
//   warp 1       even CTA: tcgen05 pair-MMA issuer; odd CTA: forwards operand readiness
//   warps 2-5    converter group 0 (even blocks);  warps 12-15  converter group 1 (odd blocks)
//   warp 6       activation producer: this CTA's T/2 token rows of each block's plane(s)
//   warps 8-11   epilogue: TMEM lane quarter warp % 4, one output channel per thread
#include <cuda_fp16.h>

#include "fmpq_device.cuh"
#include "fmpq_internal.h"

namespace fmpq {
namespace {

constexpr int kSThreads = 512;
constexpr int kSCvStages = 4;  // converted weight tiles (two per converter group)
constexpr int kSScStages = 4;  // per-block scales staged for the epilogue
constexpr int kSBSlots = 8;    // activation plane slots (an INT4 block takes one, INT8 two)
constexpr int kSBlk = 16;      // per-block readiness / release barriers (ring over blocks)
constexpr int kSConvWarps = 4; // warps per converter group
constexpr int kSEpiWarps = 4;
constexpr uint32_t kSTmemCols = 512;

// Accumulators of T columns in flight (TMEM holds 512 columns; at most 8 are used).
template <int kT>
__host__ __device__ constexpr int acc_slots() { return (512 / kT) < 8 ? (512 / kT) : 8; }

// Packed weight stages (8 KB bulk copies). Every weight byte comes from HBM once, so the
// stream runs at (bytes in flight) / (HBM latency): the ring takes the shared memory the
// activation slots leave (T/2 rows each), about 80-128 KB in flight per SM.
template <int kT>
__host__ __device__ constexpr int w_stages() { return kT <= 32 ? 16 : kT == 64 ? 14 : 10; }

struct SScaleSlot {
    float sw[128];  // weight scales of this CTA's 128 output channels
    float sx[128];  // activation scales of the T tokens, times 2^18 (operand encoding)
};

template <int kT>
struct __align__(1024) SSmem {
    uint8_t cvA[kSCvStages][128 * 128];     // E4M3 weight operand: this CTA's 128 rows x 128 K
    uint8_t opB[kSBSlots][(kT / 2) * 128];  // activation code planes: T/2 token rows x 128 K
    uint8_t pkW[w_stages<kT>()][128 * 64];  // packed weight codes of this CTA's 128 rows
    SScaleSlot sc[kSScStages];
    int32_t poff[kMaxBlocks];               // first code plane of each block
    uint8_t mask[kMaxBlocks];               // 1 = INT8 block (two planes)
    uint32_t maskw[kMaxBlocks / 32];        // the same, one bit per block
    // blk_full[b % kSBlk]: block b's operands are in place in this CTA (activation rows by
    //   bulk copy, converted weights by one converter group). In the even CTA it also
    //   collects the odd CTA's forwarded readiness and the release of the accumulator the
    //   block writes (the epilogue warps of both CTAs).
    // blk_empty[b % kSBlk]: block b's MMAs are done; committed by the even CTA to both.
    uint64_t blk_full[kSBlk], blk_empty[kSBlk];
    uint64_t w_full[w_stages<kT>()], w_empty[w_stages<kT>()];
    uint64_t sc_full[kSScStages], sc_empty[kSScStages];
    uint64_t acc_full[8];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int fixup_last;
};

struct SParams {
    const uint8_t* A;
    const uint16_t* a_scales;
    const uint8_t* W;
    const uint16_t* w_scales;
    uint16_t* Y;
    int64_t ldy;
    int M, N, nb;
    const uint8_t* mask;
    const int32_t* poff;
    int32_t* status;
    int ntiles;            // 256-channel output tiles
    int splits;            // K splits per tile (1 = none)
    float* ws_partial;     // [ntiles][splits][256][T] FP32 partial sums (splits > 1)
    int32_t* ws_count;     // [ntiles][2] arrival counters per CTA half (zero between calls)
    // partial-sum export (debug): P[m - pm0][n - pn0][b] for the window, instead of Y
    int32_t* P;
    int pm0, pmcount, pn0, pncount;
};

__device__ __forceinline__ uint32_t lo4s(uint32_t w) { return w & 0x87878787u; }
__device__ __forceinline__ uint32_t hi4s(uint32_t w) { return __funnelshift_r(w, w, 4) & 0x87878787u; }

// Unit u: output tile nt, K split `split` = blocks [b0, b0 + n).
struct SUnit {
    int nt, split, b0, n;
    __device__ __forceinline__ int block(int i) const { return b0 + i; }
};
__device__ __forceinline__ SUnit sunit_of(const SParams& p, int u) {
    SUnit r;
    r.nt = u / p.splits;
    r.split = u % p.splits;
    r.b0 = static_cast<int>((static_cast<int64_t>(r.split) * p.nb) / p.splits);
    r.n = static_cast<int>((static_cast<int64_t>(r.split + 1) * p.nb) / p.splits) - r.b0;
    return r;
}

__device__ __forceinline__ void sfail(const SParams& p, volatile int* abort_flag) {
    *abort_flag = 1;
    dev::report(p.status, dev::kStatusTimeout);
}

// ---------------------------------------------------------------- weight producer (warp 0)
template <int kT>
__device__ __forceinline__ void s_weight_producer(const SParams& p, SSmem<kT>& s, uint32_t rank, int lane,
                                                  volatile int* abort_flag) {
    constexpr int kSWStages = w_stages<kT>();
    const int num_units = p.ntiles * p.splits;
    uint32_t wc = 0;
    bool ok = true;
    for (int u = blockIdx.x >> 1; ok && u < num_units; u += gridDim.x >> 1) {
        const SUnit t = sunit_of(p, u);
        for (int i = 0; i < t.n; ++i, ++wc) {
            const int b = t.block(i);
            const int ws = wc % kSWStages;
            ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&s.w_empty[ws], ((wc / kSWStages) & 1) ^ 1, abort_flag));
            if (!ok) break;
            if (lane == 0) {
                dev::mbar_arrive_expect_tx(&s.w_full[ws], 128 * 64);
                dev::bulk_g2s(s.pkW[ws], p.W + (static_cast<int64_t>(t.nt) * p.nb + b) * (256 * 64) + rank * (128 * 64),
                              128 * 64, &s.w_full[ws]);
            }
            __syncwarp();
        }
    }
    if (!ok && lane == 0) sfail(p, abort_flag);
    if (lane == 0) {
        for (int ws = 0; ws < kSWStages; ++ws) {   // drain copies in flight
            if (wc <= static_cast<uint32_t>(ws)) break;
            const uint32_t last = ws + ((wc - 1 - ws) / kSWStages) * kSWStages;
            dev::mbar_wait(&s.w_full[ws], (last / kSWStages) & 1, nullptr);
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------- activation producer (warp 6)
// This CTA's T/2 token rows [rank*T/2, rank*T/2 + T/2) of each block's plane(s): one bulk copy
// of the rows below M (the quantizer's row swizzle, row mod 8, matches the tile's since T/2 is
// a multiple of 8). Rows at or past M are never written and stay zero.
template <int kT>
__device__ __forceinline__ void s_activation_producer(const SParams& p, SSmem<kT>& s, uint32_t rank, int lane,
                                                      volatile int* abort_flag) {
    const int num_units = p.ntiles * p.splits;
    uint32_t pc = 0, it = 0;
    int32_t slot_block[kSBSlots];
#pragma unroll
    for (int i = 0; i < kSBSlots; ++i) slot_block[i] = -1;
    bool ok = true;
    const int64_t plane_bytes = static_cast<int64_t>(p.M) * kBlock;
    const int r0 = static_cast<int>(rank) * (kT / 2);
    const uint32_t abytes = static_cast<uint32_t>(max(0, min(kT / 2, p.M - r0))) * kBlock;
    for (int u = blockIdx.x >> 1; ok && u < num_units; u += gridDim.x >> 1) {
        const SUnit t = sunit_of(p, u);
        for (int i = 0; ok && i < t.n; ++i, ++it) {
            const int b = t.block(i);
            const int planes = s.mask[b] ? 2 : 1;
            for (int pl = 0; ok && pl < planes; ++pl) {
                const int sl = (pc + pl) % kSBSlots;
                int32_t last = -1;
#pragma unroll
                for (int i = 0; i < kSBSlots; ++i)
                    if (i == sl) last = slot_block[i];
                if (last >= 0)
                    ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&s.blk_empty[last % kSBlk],
                                                                (static_cast<uint32_t>(last) / kSBlk) & 1, abort_flag));
            }
            if (!ok) break;
            uint64_t* bar = &s.blk_full[it % kSBlk];
            if (lane == 0) dev::mbar_arrive_expect_tx(bar, abytes * planes);
            const uint8_t* a0 = p.A + static_cast<int64_t>(s.poff[b]) * plane_bytes + static_cast<int64_t>(r0) * kBlock;
            for (int pl = 0; pl < planes; ++pl, ++pc) {
                const int sl = pc % kSBSlots;
#pragma unroll
                for (int i = 0; i < kSBSlots; ++i)
                    if (i == sl) slot_block[i] = static_cast<int32_t>(it);
                if (lane == 0 && abytes > 0) dev::bulk_g2s(s.opB[sl], a0 + pl * plane_bytes, abytes, bar);
            }
            __syncwarp();
        }
    }
    if (!ok && lane == 0) sfail(p, abort_flag);
    if (lane == 0) {
        for (uint32_t k = 0; k < kSBlk && k < it; ++k) {   // drain: the last blocks' copies
            const uint32_t b = it - 1 - k;
            dev::mbar_wait(&s.blk_full[b % kSBlk], (b / kSBlk) & 1, nullptr);
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------- MMA issuer / forwarder (warp 1)
template <int kT>
__device__ __forceinline__ void s_mma_role(const SParams& p, SSmem<kT>& s, uint32_t rank, int lane, uint32_t tmem,
                                           volatile int* abort_flag) {
    constexpr int kAcc = acc_slots<kT>();
    constexpr uint32_t kIdesc = dev::idesc_e4m3_f32(256, kT);
    const int num_units = p.ntiles * p.splits;
    uint32_t it = 0, pc = 0;
    bool ok = true;
    const uint32_t leader_blk_full = dev::mapa(&s.blk_full[0], 0);
    for (int u = blockIdx.x >> 1; ok && u < num_units; u += gridDim.x >> 1) {
        const SUnit t = sunit_of(p, u);
        for (int i = 0; ok && i < t.n; ++i, ++it) {
            const int planes = 1 + static_cast<int>((s.maskw[t.block(i) >> 5] >> (t.block(i) & 31)) & 1u);
            ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&s.blk_full[it % kSBlk], (it / kSBlk) & 1, abort_flag));
            if (!ok) break;
            if (rank != 0) {
                if (lane == 0) dev::mbar_arrive_remote(leader_blk_full + static_cast<uint32_t>(it % kSBlk) * 8u);
                __syncwarp();
                pc += planes;
                continue;
            }
            const int ab = static_cast<int>(it % kAcc);
            if (lane == 0) {
                dev::tc_fence_after();
                const uint64_t ad = dev::sdesc_k_sw128(dev::smem_u32(s.cvA[it % kSCvStages]));
                const uint32_t d = tmem + static_cast<uint32_t>(ab * kT);
                for (int pl = 0; pl < planes; ++pl) {
                    const uint64_t bd = dev::sdesc_k_sw128(dev::smem_u32(s.opB[(pc + pl) % kSBSlots]));
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dev::mma_e4m3_pair(d, ad + 2 * k, bd + 2 * k, kIdesc, (pl > 0 || k > 0) ? 1u : 0u);
                }
                dev::mma_commit_pair(&s.blk_empty[it % kSBlk]);
                dev::mma_commit_pair(&s.acc_full[ab]);
            }
            __syncwarp();
            pc += planes;
        }
    }
    if (!ok && lane == 0) sfail(p, abort_flag);
    if (rank == 0 && lane == 0) {
        dev::mma_commit_pair(&s.mma_done);   // every MMA issued finishes before TMEM is released
        dev::mbar_wait(&s.mma_done, 0, nullptr);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- converters (warps 2-5, 12-15)
// Group g converts the blocks it with it % 2 == g (packed codes -> 128B-swizzled E4M3 tile, the
// same mapping as the main GEMM's converters) and stages their scales: weight scale of this
// CTA's output channel ct and, for ct < T, the activation scale of token ct (times 2^18).
template <int kT>
__device__ __forceinline__ void s_converter_role(const SParams& p, SSmem<kT>& s, uint32_t rank, int group, int ct,
                                                 int lane, volatile int* abort_flag) {
    const int num_units = p.ntiles * p.splits;
    const int r0 = ct >> 2, c4 = ct & 3;
    const uint32_t phase = static_cast<uint32_t>(r0 & 7);
    const uint32_t src0 = static_cast<uint32_t>(r0 * 64 + c4 * 16);
    const uint32_t dstA = static_cast<uint32_t>(r0 * 128) + (((2u * c4) ^ phase) << 4);
    const uint32_t dstB = static_cast<uint32_t>(r0 * 128) + (((2u * c4 + 1u) ^ phase) << 4);
    constexpr int kSWStages = w_stages<kT>();
    constexpr int kPieces = 4;     // 512 pieces of 16 bytes over 128 threads
    constexpr int kRowStep = 32;   // rows between a thread's pieces
    bool ok = true;
    uint32_t it = 0;
    for (int u = blockIdx.x >> 1; ok && u < num_units; u += gridDim.x >> 1) {
        const SUnit t = sunit_of(p, u);
        const int n = t.nt * kTileN + static_cast<int>(rank) * 128 + ct;
        for (int i = 0; i < t.n; ++i, ++it) {
            if (static_cast<int>(it & 1u) != group) continue;
            const int b = t.block(i);
            const uint16_t swv = (n < p.N) ? __ldg(p.w_scales + static_cast<int64_t>(b) * p.N + n) : uint16_t(0);
            const uint16_t sxv = (ct < kT && ct < p.M) ? __ldg(p.a_scales + static_cast<int64_t>(b) * p.M + ct) : uint16_t(0);
            const int ws = it % kSWStages, cs = it % kSCvStages, ss = it % kSScStages;
            ok = dev::mbar_wait(&s.w_full[ws], (it / kSWStages) & 1, abort_flag) &&
                 dev::mbar_wait(&s.sc_empty[ss], ((it / kSScStages) & 1) ^ 1, abort_flag);
            if (ok && it >= static_cast<uint32_t>(kSCvStages)) {   // converted slot: MMAs of block it - 4 done
                const uint32_t prev = it - kSCvStages;
                ok = dev::mbar_wait(&s.blk_empty[prev % kSBlk], (prev / kSBlk) & 1, abort_flag);
            }
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            const uint8_t* src = s.pkW[ws] + src0;
            uint8_t* dst = s.cvA[cs];
            uint4 w[kPieces];
#pragma unroll
            for (int k = 0; k < kPieces; ++k) w[k] = *reinterpret_cast<const uint4*>(src + k * kRowStep * 64);
#pragma unroll
            for (int k = 0; k < kPieces; ++k) {
                const uint4 v = w[k];
                *reinterpret_cast<uint4*>(dst + dstA + k * kRowStep * 128) = make_uint4(lo4s(v.x), hi4s(v.x), lo4s(v.y), hi4s(v.y));
                *reinterpret_cast<uint4*>(dst + dstB + k * kRowStep * 128) = make_uint4(lo4s(v.z), hi4s(v.z), lo4s(v.w), hi4s(v.w));
            }
            s.sc[ss].sw[ct] = __half2float(__ushort_as_half(swv));
            if (ct < kT) s.sc[ss].sx[ct] = __half2float(__ushort_as_half(sxv)) * 262144.0f;
            dev::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                dev::mbar_arrive(&s.w_empty[ws]);
                dev::mbar_arrive(&s.blk_full[it % kSBlk]);
                dev::mbar_arrive(&s.sc_full[ss]);
            }
        }
    }
    if (!ok && lane == 0) sfail(p, abort_flag);
}

// ---------------------------------------------------------------- epilogue (warps 8-11)
// Warp q holds TMEM lanes 32q..32q+31: thread `lane` owns output channel
// n0 + rank*128 + 32q + lane and accumulates its T token columns (32x32b loads, 16 columns
// at a time, the next load in flight during the math of the current one).
template <int kT, bool kPartials>
__device__ __forceinline__ void s_epilogue_role(const SParams& p, SSmem<kT>& s, uint32_t rank, int q, int lane,
                                                uint32_t tmem, volatile int* abort_flag) {
    constexpr int kAcc = acc_slots<kT>();
    constexpr int kChunks = kT / 16;
    const int num_units = p.ntiles * p.splits;
    const int lrow = 32 * q + lane;                       // this CTA's row (output channel)
    const int et = q * 32 + lane;                         // 0..127
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t leader_blk_full = dev::mapa(&s.blk_full[0], 0);
    const int mvalid = min(p.M, kT);
    uint32_t v = 0;
    bool ok = true;
    for (int u = blockIdx.x >> 1; u < num_units; u += gridDim.x >> 1) {
        const SUnit t = sunit_of(p, u);
        const int n = t.nt * kTileN + static_cast<int>(rank) * 128 + lrow;
        float2 acc[kT / 2];
#pragma unroll
        for (int j = 0; j < kT / 2; ++j) acc[j] = make_float2(0.f, 0.f);
        for (int i = 0; i < t.n; ++i, ++v) {
            const int ab = static_cast<int>(v % kAcc), ss = v % kSScStages;
            if (ok) {
                ok = dev::mbar_wait(&s.sc_full[ss], (v / kSScStages) & 1, abort_flag) &&
                     dev::mbar_wait(&s.acc_full[ab], (v / kAcc) & 1, abort_flag);
                ok = __all_sync(0xFFFFFFFFu, ok);
            }
            if (ok && kPartials) {
                // export the exact partial sums of block t.block(i) for the window: column j of
                // the accumulator is token j, P = D * 2^18 (operand encoding)
                dev::tc_fence_after();
                const int b = t.block(i);
                const uint32_t taddr = tmem + lane_addr + static_cast<uint32_t>(ab * kT);
                const bool n_in = n < p.N && n >= p.pn0 && n < p.pn0 + p.pncount;
#pragma unroll 1
                for (int c = 0; c < kChunks; ++c) {
                    uint32_t d[16];
                    dev::tmem_ld16(taddr + c * 16, d);
                    dev::tmem_ld_wait16(d);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = 16 * c + j;
                        if (n_in && m < p.M && m >= p.pm0 && m < p.pm0 + p.pmcount)
                            p.P[(static_cast<int64_t>(m - p.pm0) * p.pncount + (n - p.pn0)) * p.nb + b] =
                                __float2int_rn(__uint_as_float(d[j]) * 262144.0f);
                    }
                }
                dev::tc_fence_before();
            } else if (ok) {
                dev::tc_fence_after();
                const SScaleSlot& sl = s.sc[ss];
                const float swr = sl.sw[lrow];
                const float2 sw2 = make_float2(swr, swr);
                const uint32_t taddr = tmem + lane_addr + static_cast<uint32_t>(ab * kT);
                uint32_t d0[16], d1[16];
                dev::tmem_ld16(taddr, d0);
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    uint32_t (&dc)[16] = (c & 1) ? d1 : d0;
                    uint32_t (&dn)[16] = (c & 1) ? d0 : d1;
                    dev::tmem_ld_wait16(dc);
                    if (c + 1 < kChunks) dev::tmem_ld16(taddr + (c + 1) * 16, dn);
                    const float4* sxv = reinterpret_cast<const float4*>(sl.sx + 16 * c);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 x = sxv[i];   // same address in every lane: one broadcast
                        const float2 c0 = dev::fmul2(sw2, make_float2(x.x, x.y));
                        const float2 c1 = dev::fmul2(sw2, make_float2(x.z, x.w));
                        const int j = 8 * c + 2 * i;
                        acc[j] = dev::ffma2(make_float2(__uint_as_float(dc[4 * i]), __uint_as_float(dc[4 * i + 1])), c0, acc[j]);
                        acc[j + 1] = dev::ffma2(make_float2(__uint_as_float(dc[4 * i + 2]), __uint_as_float(dc[4 * i + 3])), c1, acc[j + 1]);
                    }
                }
                dev::tc_fence_before();
            }
            __syncwarp();
            if (lane == 0 && ok) {
                // accumulator ab is free for block v + kAcc, whose MMAs the even CTA issues
                dev::mbar_arrive_remote(leader_blk_full + static_cast<uint32_t>((v + kAcc) % kSBlk) * 8u);
                dev::mbar_arrive(&s.sc_empty[ss]);
            }
        }
        auto store = [&]() {
            if (n >= p.N) return;
#pragma unroll
            for (int j = 0; j < kT / 2; ++j) {
                if (2 * j < mvalid) p.Y[static_cast<int64_t>(2 * j) * p.ldy + n] = __half_as_ushort(__float2half_rn(acc[j].x));
                if (2 * j + 1 < mvalid) p.Y[static_cast<int64_t>(2 * j + 1) * p.ldy + n] = __half_as_ushort(__float2half_rn(acc[j].y));
            }
        };
        if constexpr (kPartials) {
            continue;   // the window's partial sums are written; no output
        }
        if (p.splits == 1) {
            store();
        } else {
            // split-K: publish this split's partial (this CTA's 128 channels x T); the last
            // split to arrive sums all of them in split order (deterministic)
            const int hrow = static_cast<int>(rank) * 128 + lrow;
            float* mine = p.ws_partial + ((static_cast<int64_t>(t.nt) * p.splits + t.split) * 256 + hrow) * kT;
#pragma unroll
            for (int j = 0; j < kT / 2; j += 2)
                __stcg(reinterpret_cast<float4*>(mine + 2 * j), make_float4(acc[j].x, acc[j].y, acc[j + 1].x, acc[j + 1].y));
            __threadfence();
            dev::named_bar_sync(1, kSEpiWarps * 32);
            if (et == 0) {
                int32_t* cnt = p.ws_count + t.nt * 2 + rank;
                const int prev = atomicAdd(cnt, 1);
                const int last = (prev == p.splits - 1);
                if (last) *cnt = 0;   // reusable for the next call
                s.fixup_last = last;
            }
            dev::named_bar_sync(1, kSEpiWarps * 32);
            if (s.fixup_last) {
                __threadfence();
#pragma unroll
                for (int j = 0; j < kT / 2; ++j) acc[j] = make_float2(0.f, 0.f);
                for (int sp = 0; sp < p.splits; ++sp) {
                    const float* o = p.ws_partial + ((static_cast<int64_t>(t.nt) * p.splits + sp) * 256 + hrow) * kT;
#pragma unroll
                    for (int j = 0; j < kT / 2; j += 2) {
                        const float4 f = __ldcg(reinterpret_cast<const float4*>(o + 2 * j));
                        acc[j].x += f.x;
                        acc[j].y += f.y;
                        acc[j + 1].x += f.z;
                        acc[j + 1].y += f.w;
                    }
                }
                store();
            }
            dev::named_bar_sync(1, kSEpiWarps * 32);   // fixup_last is read before the next unit rewrites it
        }
    }
    if (!ok && lane == 0) sfail(p, abort_flag);
}

template <int kT, bool kPartials>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kSThreads, 1) w4ax_gemm_small_kernel(const SParams p) {
    extern __shared__ uint8_t smem_raw[];
    SSmem<kT>& s = *reinterpret_cast<SSmem<kT>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int kAcc = acc_slots<kT>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = dev::cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSBlk; ++i) {
            // activation producer (expect-tx) + one converter group; in the even CTA also the
            // odd CTA's forward and the epilogue warps of both CTAs (accumulator released)
            dev::mbar_init(&s.blk_full[i], 1 + kSConvWarps + (rank == 0 ? 1 + 2 * kSEpiWarps : 0));
            dev::mbar_init(&s.blk_empty[i], 1);
        }
        for (int i = 0; i < w_stages<kT>(); ++i) {
            dev::mbar_init(&s.w_full[i], 1);
            dev::mbar_init(&s.w_empty[i], kSConvWarps);
        }
        for (int i = 0; i < kSScStages; ++i) {
            dev::mbar_init(&s.sc_full[i], kSConvWarps);
            dev::mbar_init(&s.sc_empty[i], kSEpiWarps);
        }
        for (int i = 0; i < kAcc; ++i) dev::mbar_init(&s.acc_full[i], 1);
        dev::mbar_init(&s.mma_done, 1);
        s.abort_flag = 0;
        if (rank == 0) {
            // the first kAcc blocks find their accumulators free
            for (int i = 0; i < kAcc; ++i)
                for (int k = 0; k < 2 * kSEpiWarps; ++k) dev::mbar_arrive(&s.blk_full[i]);
        }
        dev::fence_barrier_init();
    }
    for (int b = threadIdx.x; b < p.nb; b += kSThreads) {
        s.mask[b] = p.mask[b];
        s.poff[b] = p.poff[b];
    }
    if (warp < kMaxBlocks / 32) {
        const int b = warp * 32 + lane;
        const uint32_t bits = __ballot_sync(0xFFFFFFFFu, b < p.nb && p.mask[b] != 0);
        if (lane == 0) s.maskw[warp] = bits;
    }
    // token rows at or past M are never copied: they must read as zero codes
    for (int i = threadIdx.x; i < kSBSlots * (kT / 2) * 128 / 16; i += kSThreads)
        reinterpret_cast<uint4*>(&s.opB[0][0])[i] = make_uint4(0u, 0u, 0u, 0u);
    dev::fence_proxy_async_smem();
    if (warp == 1) dev::tmem_alloc_pair(&s.tmem_base, kSTmemCols);
    dev::tc_fence_before();
    __syncthreads();
    dev::cluster_sync();
    dev::tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int* abort_flag = &s.abort_flag;

    if (warp < 8) {
        dev::setmaxnreg_dec<64>();
        if (warp == 0) {
            s_weight_producer<kT>(p, s, rank, lane, abort_flag);
        } else if (warp == 1) {
            s_mma_role<kT>(p, s, rank, lane, tmem, abort_flag);
        } else if (warp >= 2 && warp < 2 + kSConvWarps) {
            s_converter_role<kT>(p, s, rank, 0, (warp - 2) * 32 + lane, lane, abort_flag);
        } else if (warp == 6) {
            s_activation_producer<kT>(p, s, rank, lane, abort_flag);
        }
    } else {
        dev::setmaxnreg_inc<192>();
        if (warp < 8 + kSEpiWarps) {
            s_epilogue_role<kT, kPartials>(p, s, rank, warp & 3, lane, tmem, abort_flag);
        } else {
            s_converter_role<kT>(p, s, rank, 1, (warp - 12) * 32 + lane, lane, abort_flag);
        }
    }

    dev::tc_fence_before();
    __syncthreads();
    dev::cluster_sync();   // the peer's MMAs, commits and arrivals on this CTA are done
    if (warp == 1) {
        dev::tc_fence_after();
        dev::tmem_dealloc_pair(tmem, kSTmemCols);
    }
}

template <int kT>
constexpr size_t small_smem_bytes() { return sizeof(SSmem<kT>) + 1024; }

int tokens_tile(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

template <int kT>
int small_max_pairs_t(const fmpq_layout& L) {
    static int cached[64] = {};
    const int dev = L.device;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int pairs = L.num_sms / 2 > 0 ? L.num_sms / 2 : 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = small_smem_bytes<kT>();
    int clusters = 0;
    if (ensure_smem_limit(reinterpret_cast<const void*>(w4ax_gemm_small_kernel<kT, false>),
                          static_cast<int>(small_smem_bytes<kT>())) == cudaSuccess &&
        cudaOccupancyMaxActiveClusters(&clusters, w4ax_gemm_small_kernel<kT, false>, &cfg) == cudaSuccess && clusters > 0 &&
        clusters < pairs)
        pairs = clusters;
    cudaGetLastError();   // a failed query leaves no sticky error behind
    if (dev >= 0 && dev < 64) cached[dev] = pairs;
    return pairs;
}

int small_max_pairs(const fmpq_layout& L, int T) {
    switch (T) {
        case 16: return small_max_pairs_t<16>(L);
        case 32: return small_max_pairs_t<32>(L);
        case 64: return small_max_pairs_t<64>(L);
        default: return small_max_pairs_t<128>(L);
    }
}

// Splits so that the units (tiles x splits) come close to one per resident pair.
int small_splits(const fmpq_layout& L, int64_t ntiles, int T) {
    const int pairs = small_max_pairs(L, T);
    if (ntiles * 2 > pairs) return 1;
    int s = static_cast<int>(pairs / ntiles);
    if (s > L.nb) s = L.nb;
    if (s > 16) s = 16;
    return s < 1 ? 1 : s;
}

template <int kT>
cudaError_t launch_small_t(const fmpq_layout& L, const SParams& p, int pairs, cudaStream_t stream) {
    const void* fn = p.P != nullptr ? reinterpret_cast<const void*>(w4ax_gemm_small_kernel<kT, true>)
                                    : reinterpret_cast<const void*>(w4ax_gemm_small_kernel<kT, false>);
    const cudaError_t e = ensure_smem_limit(fn, static_cast<int>(small_smem_bytes<kT>()));
    if (e != cudaSuccess) return e;
    if (p.P != nullptr)
        w4ax_gemm_small_kernel<kT, true><<<2 * pairs, kSThreads, small_smem_bytes<kT>(), stream>>>(p);
    else
        w4ax_gemm_small_kernel<kT, false><<<2 * pairs, kSThreads, small_smem_bytes<kT>(), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool gemm_small_path(int64_t M) { return M >= 1 && M <= 128; }

size_t gemm_small_counter_bytes(const fmpq_layout& L, int64_t M, int64_t N) {
    const int64_t ntiles = (N + kTileN - 1) / kTileN;
    if (small_splits(L, ntiles, tokens_tile(M)) == 1) return 0;
    return static_cast<size_t>(ntiles) * 2 * sizeof(int32_t) + 16;
}

size_t gemm_small_workspace_bytes(const fmpq_layout& L, int64_t M, int64_t N) {
    const int64_t ntiles = (N + kTileN - 1) / kTileN;
    const int T = tokens_tile(M);
    const int splits = small_splits(L, ntiles, T);
    if (splits == 1) return 0;
    return static_cast<size_t>(ntiles) * splits * 256 * T * sizeof(float) + gemm_small_counter_bytes(L, M, N);
}

cudaError_t launch_gemm_small(const fmpq_layout& L, const GemmArgs& a, cudaStream_t stream) {
    SParams p{};
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
    const int T = tokens_tile(a.M);
    p.ntiles = static_cast<int>((a.N + kTileN - 1) / kTileN);
    p.splits = small_splits(L, p.ntiles, T);
    if (a.P != nullptr) {
        // partial-sum export: every unit writes its blocks' sums directly (no workspace)
        p.P = a.P;
        p.pm0 = static_cast<int>(a.pm0);
        p.pmcount = static_cast<int>(a.pmcount);
        p.pn0 = static_cast<int>(a.pn0);
        p.pncount = static_cast<int>(a.pncount);
    } else if (p.splits > 1) {
        p.ws_partial = static_cast<float*>(a.workspace);
        p.ws_count = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a.workspace) +
                                                static_cast<size_t>(p.ntiles) * p.splits * 256 * T * sizeof(float));
    }
    const int64_t units = static_cast<int64_t>(p.ntiles) * p.splits;
    const int maxp = small_max_pairs(L, T);
    const int pairs = static_cast<int>(units < maxp ? units : maxp);
    switch (T) {
        case 16: return launch_small_t<16>(L, p, pairs, stream);
        case 32: return launch_small_t<32>(L, p, pairs, stream);
        case 64: return launch_small_t<64>(L, p, pairs, stream);
        default: return launch_small_t<128>(L, p, pairs, stream);
    }
}

}  // namespace fmpq
