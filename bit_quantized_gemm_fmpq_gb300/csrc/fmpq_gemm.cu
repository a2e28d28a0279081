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
//   * INT4 weights stay 4-bit in HBM: converter warps take the packed words from a
//     bulk-copy ring and turn each into 8 operand bytes with a mask and a rotate (the
//     sign-magnitude byte s0000mmm is the E4M3 value (-1)^s * m * 2^-9) -- the
//     restructured storage format that makes 4-bit -> 8-bit conversion a couple of
//     instructions (COMET news article, section 3).
//   * tcgen05.mma kind::f8f6f4 (M=128, N=256, K=32) with the accumulator in TMEM,
//     double-buffered so the MMA of the next block overlaps the epilogue of this one.
//   * Per block the epilogue warps read the tile (tcgen05.ld 16x256b: two rows and
//     column pairs per thread, so each weight scale read serves two rows) and accumulate
//     acc += D * (w_scale[n] * a_scale[m] * 2^18) in FP32 registers (packed f32x2 math).
//
// Warp roles (512 threads, one CTA per SM, persistent over pair tiles):
//   warp 0       weight producer: this CTA's half of each packed weight tile (bulk copies)
//   warp 1       even CTA: tcgen05 pair-MMA issuer; odd CTA: forwards operand readiness
//   warps 2-5    converters: packed weight codes -> 128B-swizzled E4M3 half-tile, and the
//                block's scales -> fp32 scale slot for the epilogue
//   warp 6       activation producer: this CTA's 128 rows of each block's plane(s)
//   warps 8-15   epilogue: per-block FP32 scale-and-sum, fp16 output (or split-K partials)
#include <cuda_fp16.h>

#include "fmpq_device.cuh"
#include "fmpq_internal.h"

namespace fmpq {
namespace {

constexpr int kThreads = 512;
constexpr int kPairM = 256;   // rows of a pair tile (128 per CTA)
constexpr int kASlots = 8;    // activation plane slots (an INT4 block takes one, INT8 two)
constexpr int kWStages = 7;   // packed weight half-tiles (bulk copies)
constexpr int kCvStages = 2;  // converted weight half-tiles
constexpr int kScStages = 4;  // per-block scales staged for the epilogue
constexpr int kBlk = 16;      // per-block readiness / release barriers (ring over blocks)
constexpr int kGroupM = 4;    // tile order: bands of 4 pair m-tiles, n-tiles inside a band
constexpr int kConvWarps = 4;
constexpr int kConvWarp0 = 2;   // converters are warps 2..5; warp 6 issues the activation copies
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;  // two 128 x 256 FP32 accumulators per CTA
constexpr uint32_t kIdesc = dev::idesc_e4m3_f32(256, 256);
// Weight scales of a block, staged for the epilogue: column n = 8g + 2c + j goes to
// [c][2g + j]. Each epilogue thread reads the 64 values of its column pairs contiguously;
// rows of 68 floats put the four c groups' 16-byte reads in distinct banks.
constexpr int kSwStride = 68;

struct ScaleSlot {
    float sw[4 * kSwStride];  // weight scales of the tile's 256 columns (permuted, see above)
    float sx[128];            // activation scales of this CTA's 128 rows, times 2^18
};

struct __align__(1024) Smem {
    uint8_t opA[kASlots][128 * 128];     // activation code planes (operand-ready, swizzled)
    uint8_t cvB[kCvStages][128 * 128];   // E4M3 weight operand: this CTA's 128 rows x 128 K
    uint8_t pkW[kWStages][128 * 64];     // packed weight codes of this CTA's 128 rows
    ScaleSlot sc[kScStages];             // per-block scales (fp32) for the epilogue
    // The layout's block tables, staged once: the MMA issuer and the activation producer
    // look them up every block.
    int32_t poff[kMaxBlocks];            // first code plane of each block
    uint8_t mask[kMaxBlocks];            // 1 = INT8 block (two planes)
    uint32_t maskw[kMaxBlocks / 32];     // the same, one bit per block
    // a_full[b % kBlk]: block b's activation planes have landed here (bulk-copy bytes only,
    //   so a drain after an abort can always wait for the copies in flight).
    // blk_full[b % kBlk]: block b's converted weight tile and scales are staged here
    //   (converter warps). In the even CTA it also gathers everything else the MMAs of block b
    //   wait for: the odd CTA's operands (one forwarded arrival) and the accumulator they
    //   overwrite (the epilogue warps of both CTAs, done with block b - 2).
    // blk_empty[b % kBlk]: block b's MMAs have finished (its activation slots and converted
    //   weight slot may be reused); committed by the even CTA to both CTAs.
    uint64_t a_full[kBlk], blk_full[kBlk], blk_empty[kBlk];
    uint64_t w_full[kWStages], w_empty[kWStages];
    uint64_t sc_full[kScStages], sc_empty[kScStages];
    uint64_t acc_full[2];
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
    // pair tiles (256 x 256): m-tiles [mt0, mt0 + mtiles) x n-tiles [nt0, nt0 + ntiles)
    int mt0, mtiles, nt0, ntiles;
    int splits;            // K splits per tile (1 = none)
    float* ws_partial;     // [tiles][splits][256][256] FP32 partial sums (splits > 1)
    int32_t* ws_count;     // [tiles][2] arrival counters per CTA half (zero between calls)
    // partial-sum export
    int32_t* P;
    int pm0, pmcount, pn0, pncount;
    // quantization variants (see GemmArgs)
    uint32_t wmask;        // code bits the converter keeps: 0x87878787 sign-magnitude, 0x0F0F0F0F unsigned
    int zero_kind;
    const uint16_t* ch_scales;
    const uint8_t* grp_scales;
    // the variants' zero-point term summed over all blocks on the tensor cores beforehand:
    // yz[m][n] (FP32, row stride N), the accumulators' starting value; nullptr for FMPQ
    const float* yz;
    // failure-detection test: polls before a device wait gives up, and the index of the packed
    // weight copy the first CTA withholds (-1: none)
    uint32_t poll_limit;
    int withhold;
};

// Codes 0-3 and 4-7 of a packed word as operand bytes. Sign-magnitude words keep |q| in bits
// 0-2 / 4-6 and the signs in bits 7 / 3 of the next byte (mask 0x87878787); unsigned words
// (QoQ) hold the codes in the low / high nibbles (mask 0x0F0F0F0F). Either way the byte is
// the E4M3 value (-1)^s * m * 2^-9 for m <= 15.
__device__ __forceinline__ uint32_t lo4(uint32_t w, uint32_t mask) { return w & mask; }
__device__ __forceinline__ uint32_t hi4(uint32_t w, uint32_t mask) { return __funnelshift_r(w, w, 4) & mask; }

// Work unit u -> (pair tile, split). Tiles run in bands of kGroupM m-tiles; inside a band
// the m-tile varies fastest, so the pairs running together share activation and weight
// blocks in L2.
struct Unit {
    int mt, nt, tile, split, b0, b1;
};
__device__ __forceinline__ Unit unit_of(const Params& p, int u) {
    Unit r;
    r.tile = u / p.splits;
    r.split = u % p.splits;
    const int band = r.tile / (kGroupM * p.ntiles);
    const int in_band = r.tile - band * kGroupM * p.ntiles;
    const int gm = min(kGroupM, p.mtiles - band * kGroupM);   // m-tiles in this band
    r.mt = p.mt0 + band * kGroupM + in_band % gm;
    r.nt = p.nt0 + in_band / gm;
    r.b0 = static_cast<int>((static_cast<int64_t>(r.split) * p.nb) / p.splits);
    r.b1 = static_cast<int>((static_cast<int64_t>(r.split + 1) * p.nb) / p.splits);
    return r;
}

__device__ __forceinline__ void fail(const Params& p, volatile int* abort_flag) {
    *abort_flag = 1;
    dev::report(p.status, dev::kStatusTimeout);
}

// ---------------------------------------------------------------- producers (warps 0 and 6)
// Warp 0 streams this CTA's 128 rows (8 KB) of each block's packed weight tile; warp 6
// streams this CTA's 128 activation rows of each block's plane(s). Separate threads, so the
// activation prefetch depth is set by its own ring, not by the weight conversion.
__device__ __forceinline__ void weight_producer(const Params& p, Smem& s, uint32_t rank, int lane,
                                                volatile int* abort_flag, uint32_t polls, int withhold) {
    const int num_units = p.mtiles * p.ntiles * p.splits;
    uint32_t wc = 0;
    bool ok = true;
    for (int u = blockIdx.x >> 1; ok && u < num_units; u += gridDim.x >> 1) {
        const Unit t = unit_of(p, u);
        for (int b = t.b0; b < t.b1; ++b, ++wc) {
            const int ws = wc % kWStages;
            // the whole warp waits (converged); lane 0 issues
            ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&s.w_empty[ws], ((wc / kWStages) & 1) ^ 1, abort_flag, polls));
            if (!ok) break;
            // (a failure-detection test withholds one copy of the first CTA: nothing is issued,
            // so the converters' wait on it runs out)
            if (lane == 0 && !(blockIdx.x == 0 && static_cast<int>(wc) == withhold)) {
                dev::mbar_arrive_expect_tx(&s.w_full[ws], 128 * 64);
                dev::bulk_g2s(s.pkW[ws], p.W + (static_cast<int64_t>(t.nt) * p.nb + b) * (256 * 64) + rank * (128 * 64),
                              128 * 64, &s.w_full[ws]);
            }
            __syncwarp();
        }
    }
    if (!ok && lane == 0) fail(p, abort_flag);
    if (lane == 0) {
        for (int ws = 0; ws < kWStages; ++ws) {   // drain copies in flight
            if (wc <= static_cast<uint32_t>(ws)) break;
            const uint32_t last = ws + ((wc - 1 - ws) / kWStages) * kWStages;
            dev::mbar_wait(&s.w_full[ws], (last / kWStages) & 1, nullptr, polls);
        }
    }
    __syncwarp();
}

__device__ __forceinline__ void activation_producer(const Params& p, Smem& s, uint32_t rank, int lane,
                                                    volatile int* abort_flag, uint32_t polls) {
    const int num_units = p.mtiles * p.ntiles * p.splits;
    uint32_t pc = 0, it = 0;        // planes and blocks issued
    int32_t slot_block[kASlots];    // block that last used each plane slot (-1: none)
#pragma unroll
    for (int i = 0; i < kASlots; ++i) slot_block[i] = -1;
    bool ok = true;
    const int64_t plane_bytes = static_cast<int64_t>(p.M) * kBlock;
    dev::pdl_wait();   // as the quantizer's programmatic dependent: its codes are complete after this
    for (int u = blockIdx.x >> 1; ok && u < num_units; u += gridDim.x >> 1) {
        const Unit t = unit_of(p, u);
        const int r0 = t.mt * kPairM + static_cast<int>(rank) * 128;
        const uint32_t abytes = static_cast<uint32_t>(max(0, min(128, p.M - r0))) * kBlock;
        for (int b = t.b0; ok && b < t.b1; ++b, ++it) {
            const int planes = s.mask[b] ? 2 : 1;
            // the slots of this block's planes must have been released by the MMAs of the
            // blocks that used them last (the whole warp waits, converged; lane 0 issues)
            for (int pl = 0; ok && pl < planes; ++pl) {
                const int sl = (pc + pl) % kASlots;
                int32_t last = -1;
#pragma unroll
                for (int i = 0; i < kASlots; ++i)
                    if (i == sl) last = slot_block[i];
                if (last >= 0)
                    ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&s.blk_empty[last % kBlk],
                                                                (static_cast<uint32_t>(last) / kBlk) & 1, abort_flag, polls));
            }
            if (!ok) break;
            uint64_t* bar = &s.a_full[it % kBlk];
            if (lane == 0) dev::mbar_arrive_expect_tx(bar, abytes * planes);   // rows past M: nothing to copy
            const uint8_t* a0 = p.A + static_cast<int64_t>(s.poff[b]) * plane_bytes + static_cast<int64_t>(r0) * kBlock;
            for (int pl = 0; pl < planes; ++pl, ++pc) {
                const int sl = pc % kASlots;
#pragma unroll
                for (int i = 0; i < kASlots; ++i)
                    if (i == sl) slot_block[i] = static_cast<int32_t>(it);
                if (lane == 0 && abytes > 0) dev::bulk_g2s(s.opA[sl], a0 + pl * plane_bytes, abytes, bar);
            }
            __syncwarp();
        }
    }
    if (!ok && lane == 0) fail(p, abort_flag);
    // drain copies in flight: a_full completes on the copies' bytes alone
    if (lane == 0) {
        for (uint32_t k = 0; k < kBlk && k < it; ++k) {
            const uint32_t b = it - 1 - k;
            dev::mbar_wait(&s.a_full[b % kBlk], (b / kBlk) & 1, nullptr, polls);
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------- MMA issuer / forwarder (warp 1)
// Even CTA: per block, waits for its planes (a_full) and blk_full (its converted weights, the
// odd CTA's forward and the free accumulator), issues the pair MMAs and commits blk_empty and
// acc_full to both CTAs. Odd CTA: forwards a_full + blk_full. This warp's time per block lies
// on the loop through the two accumulators (MMAs -> epilogue -> release -> next MMAs); the
// INT8 mask is read one 32-bit word per 32 blocks.
__device__ __forceinline__ void mma_role(const Params& p, Smem& s, uint32_t rank, int lane, uint32_t tmem,
                                         volatile int* abort_flag, uint32_t polls) {
    const int num_units = p.mtiles * p.ntiles * p.splits;
    uint32_t it = 0, pc = 0, mw = 0;
    bool ok = true;
    const uint32_t leader_blk_full = dev::mapa(&s.blk_full[0], 0);
    for (int u = blockIdx.x >> 1; ok && u < num_units; u += gridDim.x >> 1) {
        const Unit t = unit_of(p, u);
        for (int b = t.b0; ok && b < t.b1; ++b, ++it) {
            if (b == t.b0 || (b & 31) == 0) mw = s.maskw[b >> 5];
            const int planes = 1 + static_cast<int>((mw >> (b & 31)) & 1u);
            // the whole warp waits (converged); lane 0 issues
            ok = __all_sync(0xFFFFFFFFu, dev::mbar_wait(&s.a_full[it % kBlk], (it / kBlk) & 1, abort_flag, polls) &&
                                             dev::mbar_wait(&s.blk_full[it % kBlk], (it / kBlk) & 1, abort_flag, polls));
            if (!ok) break;
            if (rank != 0) {
                // odd CTA: this block's operands are in place here; tell the even CTA
                if (lane == 0) dev::mbar_arrive_remote(leader_blk_full + static_cast<uint32_t>(it % kBlk) * 8u);
                __syncwarp();
                pc += planes;
                continue;
            }
            const int ab = it & 1;
            if (lane == 0) {
                dev::tc_fence_after();
                const uint64_t bd = dev::sdesc_k_sw128(dev::smem_u32(s.cvB[it % kCvStages]));
                const uint32_t d = tmem + static_cast<uint32_t>(ab) * 256u;
                for (int pl = 0; pl < planes; ++pl) {
                    const uint64_t ad = dev::sdesc_k_sw128(dev::smem_u32(s.opA[(pc + pl) % kASlots]));
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dev::mma_e4m3_pair(d, ad + 2 * k, bd + 2 * k, kIdesc, (pl > 0 || k > 0) ? 1u : 0u);
                }
                dev::mma_commit_pair(&s.blk_empty[it % kBlk]);
                dev::mma_commit_pair(&s.acc_full[ab]);
            }
            __syncwarp();
            pc += planes;
        }
    }
    if (!ok && lane == 0) fail(p, abort_flag);
    if (rank == 0 && lane == 0) {
        // every MMA issued must finish before TMEM is released
        dev::mma_commit_pair(&s.mma_done);
        dev::mbar_wait(&s.mma_done, 0, nullptr, polls);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- converters (warps 2-5)
// The CTA's half of a weight tile (128 rows x 64 packed bytes) is 512 pieces of 16 bytes;
// piece i is row i/4, bytes 16*(i%4).. of the row, i.e. 32 codes = two 16-byte operand
// chunks. Thread ct (0..127) converts pieces ct + 128k, k = 0..3: 128 pieces = 32 rows, so
// the piece's column and the row's swizzle phase (row mod 8) are the same for every k and
// all addresses are the thread's base offsets plus constants. The converters also stage the
// block's scales -- entries ct, ct + 128, ct + 256 of [256 weight scales | this CTA's 128
// activation scales] -- for the epilogue, fetched one block ahead.
__device__ __forceinline__ void converter_role(const Params& p, Smem& s, uint32_t rank, int warp, int lane,
                                               volatile int* abort_flag, uint32_t polls) {
    const int num_units = p.mtiles * p.ntiles * p.splits;
    const int ct = (warp - kConvWarp0) * 32 + lane;
    const int r0 = ct >> 2, c4 = ct & 3;
    const uint32_t phase = static_cast<uint32_t>(r0 & 7);
    const uint32_t src0 = static_cast<uint32_t>(r0 * 64 + c4 * 16);
    const uint32_t dstA = static_cast<uint32_t>(r0 * 128) + (((2u * c4) ^ phase) << 4);
    const uint32_t dstB = static_cast<uint32_t>(r0 * 128) + (((2u * c4 + 1u) ^ phase) << 4);
    constexpr int kPieces = 512 / kConvThreads;               // 4 pieces per thread
    constexpr int kRowStep = kConvThreads / 4;                // 32 rows between a thread's pieces
    auto sw_pos = [](int i) { return ((i & 7) >> 1) * kSwStride + (i >> 3) * 2 + (i & 1); };
    const int swd0 = sw_pos(ct), swd1 = sw_pos(ct + 128);

    const uint32_t wm = p.wmask;
    int u = blockIdx.x >> 1;
    if (u >= num_units) return;
    Unit t = unit_of(p, u);
    int b = t.b0;
    // variants: as the converters reach a tile, its rows of the precomputed zero-point term go to
    // the L2 (one 1 KB row per thread), a few blocks before the epilogue starts from them
    auto prefetch_zero_term = [&](const Unit& tt) {
        const int row = tt.mt * kPairM + static_cast<int>(rank) * 128 + ct;
        if (p.yz != nullptr && tt.split == 0 && row < p.M) {
            const int cols = min(kTileN, p.N - tt.nt * kTileN);   // N % 16 == 0: a multiple of 64 bytes
            dev::bulk_prefetch_l2(p.yz + static_cast<int64_t>(row) * p.N + tt.nt * kTileN, static_cast<uint32_t>(cols) * 4u);
        }
    };
    prefetch_zero_term(t);
    dev::pdl_wait();   // the activation scales come from the quantizer (see activation_producer)
    // this thread's entries of the block's scales: weight columns ct and ct + 128, activation
    // row ct, fetched one block ahead as raw values and converted when they are staged, so that
    // the loads' latency hides behind a block
    uint32_t sc0 = 0, sc1 = 0, sc2 = 0;   // fp16 bits: weight scales (QoQ: s1) and activation scale
    uint32_t gc0 = 0, gc1 = 0;            // QoQ: the group scale s2 per column
    auto load_scales = [&](const Unit& tt, int bb) {
        const int n0 = tt.nt * kTileN, m0 = tt.mt * kPairM + static_cast<int>(rank) * 128;
        const int n_a = n0 + ct, n_b = n0 + ct + 128, m = m0 + ct;
        const int64_t wb = static_cast<int64_t>(bb) * p.N, xb = static_cast<int64_t>(bb) * p.M;
        if (p.zero_kind != kZeroQoq) {
            sc0 = n_a < p.N ? __ldg(p.w_scales + wb + n_a) : 0u;
            sc1 = n_b < p.N ? __ldg(p.w_scales + wb + n_b) : 0u;
            sc2 = m < p.M ? __ldg(p.a_scales + xb + m) : 0u;
        } else {
            sc0 = n_a < p.N ? __ldg(p.ch_scales + n_a) : 0u;
            sc1 = n_b < p.N ? __ldg(p.ch_scales + n_b) : 0u;
            sc2 = m < p.M ? __ldg(p.a_scales + m) : 0u;
            gc0 = n_a < p.N ? __ldg(p.grp_scales + wb + n_a) : 0u;
            gc1 = n_b < p.N ? __ldg(p.grp_scales + wb + n_b) : 0u;
        }
    };
    load_scales(t, b);
    bool ok = true;
    for (uint32_t it = 0;; ++it) {
        const int ws = it % kWStages;
        const int cs = it % kCvStages;
        const int ss = it % kScStages;
        // every lane waits (a converged warp polls faster than one lane with 31 parked);
        // the vote keeps the decision uniform
        ok = dev::mbar_wait(&s.w_full[ws], (it / kWStages) & 1, abort_flag, polls) &&
             dev::mbar_wait(&s.sc_empty[ss], ((it / kScStages) & 1) ^ 1, abort_flag, polls);
        if (ok && it >= static_cast<uint32_t>(kCvStages)) {   // converted slot: MMAs of block it - kCvStages done
            const uint32_t prev = it - kCvStages;
            ok = dev::mbar_wait(&s.blk_empty[prev % kBlk], (prev / kBlk) & 1, abort_flag, polls);
        }
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) break;
        const uint8_t* src = s.pkW[ws] + src0;
        uint8_t* dst = s.cvB[cs];
        uint4 w[kPieces];
#pragma unroll
        for (int k = 0; k < kPieces; ++k) w[k] = *reinterpret_cast<const uint4*>(src + k * kRowStep * 64);
#pragma unroll
        for (int k = 0; k < kPieces; ++k) {
            const uint4 v = w[k];
            *reinterpret_cast<uint4*>(dst + dstA + k * kRowStep * 128) =
                make_uint4(lo4(v.x, wm), hi4(v.x, wm), lo4(v.y, wm), hi4(v.y, wm));
            *reinterpret_cast<uint4*>(dst + dstB + k * kRowStep * 128) =
                make_uint4(lo4(v.z, wm), hi4(v.z, wm), lo4(v.w, wm), hi4(v.w, wm));
        }
        ScaleSlot& sl = s.sc[ss];
        auto h2f = [](uint32_t h) { return __half2float(__ushort_as_half(static_cast<unsigned short>(h))); };
        const float fx = h2f(sc2);
        sl.sx[ct] = fx * 262144.0f;   // 2^18 undoes the operand encoding
        if (p.zero_kind != kZeroQoq) {
            sl.sw[swd0] = h2f(sc0);
            sl.sw[swd1] = h2f(sc1);
        } else {
            // QoQ: weight scale s1 * s2 (exact in fp32)
            sl.sw[swd0] = h2f(sc0) * static_cast<float>(gc0);
            sl.sw[swd1] = h2f(sc1) * static_cast<float>(gc1);
        }
        dev::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            dev::mbar_arrive(&s.w_empty[ws]);
            dev::mbar_arrive(&s.blk_full[it % kBlk]);
            dev::mbar_arrive(&s.sc_full[ss]);
        }
        // next block
        if (++b == t.b1) {
            u += gridDim.x >> 1;
            if (u >= num_units) break;
            t = unit_of(p, u);
            b = t.b0;
            prefetch_zero_term(t);
        }
        load_scales(t, b);
    }
    if (!ok && lane == 0) fail(p, abort_flag);
}

// ---------------------------------------------------------------- epilogue (warps 8-15)
// Warp e (0..7) covers TMEM lanes 32*(warp%4) + 16*(e/4) + [0, 16) -- this CTA's tile rows --
// and all 256 columns, read with tcgen05.ld 16x256b: thread t holds rows t/4 and t/4 + 8 of
// that slab and columns 8g + 2(t%4) + {0, 1}, g = 0..31 (four registers per 8 columns:
// row0 col0, row0 col1, row1 col0, row1 col1).
// kYz: the quantization variants' zero-point term, summed over all blocks beforehand (yz,
// launch_zero_term), is the accumulators' starting value.
template <bool kPartials, bool kYz>
__device__ __forceinline__ void epilogue_role(const Params& p, Smem& s, uint32_t rank, int warp, int lane,
                                              uint32_t tmem, volatile int* abort_flag, uint32_t polls) {
    const int num_units = p.mtiles * p.ntiles * p.splits;
    const int ew = warp - 8;                         // 0..7
    const int q = warp & 3;                          // TMEM lane quarter of this warp
    const int slab = q * 32 + (ew >> 2) * 16;        // first local row of this warp
    const int tq = lane & 3, tr = lane >> 2;
    const int lr0 = slab + tr, lr1 = slab + tr + 8;  // this thread's local rows
    const int et = ew * 32 + lane;                   // 0..255
    const uint32_t lane_addr = static_cast<uint32_t>(slab) << 16;
    const uint32_t leader_blk_full = dev::mapa(&s.blk_full[0], 0);
    uint32_t v = 0;
    bool ok = true;
    for (int u = blockIdx.x >> 1; u < num_units; u += gridDim.x >> 1) {
        const Unit t = unit_of(p, u);
        const int m0 = t.mt * kPairM + static_cast<int>(rank) * 128, n0 = t.nt * kTileN;
        const int row0 = m0 + lr0, row1 = m0 + lr1;
        const bool ok0 = row0 < p.M, ok1 = row1 < p.M;
        float2 accA[32], accB[32];   // rows lr0 / lr1, column pair g
#pragma unroll
        for (int g = 0; g < 32; ++g) {
            accA[g] = make_float2(0.f, 0.f);
            accB[g] = make_float2(0.f, 0.f);
        }
        if constexpr (kYz && !kPartials) {
            // the accumulators start from the zero-point term summed over all blocks (one split of
            // a split-K tile carries it); the converters brought these rows to the L2
            if (t.split == 0) {
#pragma unroll
                for (int g = 0; g < 32; ++g) {
                    const int col = n0 + 8 * g + 2 * tq;
                    if (col < p.N) {
                        if (ok0) accA[g] = __ldg(reinterpret_cast<const float2*>(p.yz + static_cast<int64_t>(row0) * p.N + col));
                        if (ok1) accB[g] = __ldg(reinterpret_cast<const float2*>(p.yz + static_cast<int64_t>(row1) * p.N + col));
                    }
                }
            }
        }
        for (int b = t.b0; b < t.b1; ++b, ++v) {
            const int ab = v & 1;
            const int ss = v % kScStages;
            if (ok) {
                // every lane waits (each acquires the scales it reads); the vote keeps the
                // decision uniform
                ok = dev::mbar_wait(&s.sc_full[ss], (v / kScStages) & 1, abort_flag, polls) &&
                     dev::mbar_wait(&s.acc_full[ab], (v >> 1) & 1, abort_flag, polls);
                ok = __all_sync(0xFFFFFFFFu, ok);
            }
            const ScaleSlot& sl = s.sc[ss];
            // accumulator ab is free for block v + 2, whose MMAs the even CTA issues
            const uint32_t release = leader_blk_full + static_cast<uint32_t>((v + 2) % kBlk) * 8u;
            if (ok) {
                dev::tc_fence_after();
                const uint32_t taddr = tmem + lane_addr + ab * 256u;
                if constexpr (!kPartials) {
                    const float xa = sl.sx[lr0], xb = sl.sx[lr1];   // include 2^18 (operand encoding)
                    const float2 sxa = make_float2(xa, xa);
                    const float2 sxb = make_float2(xb, xb);
                    const float4* swv = reinterpret_cast<const float4*>(sl.sw + tq * kSwStride);
                    auto math = [&](const uint32_t* d, int g0, int n) {
#pragma unroll
                        for (int i = 0; i < n; i += 2) {
                            const float4 f = swv[(g0 + i) >> 1];
                            const float2 sp[2] = {make_float2(f.x, f.y), make_float2(f.z, f.w)};
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const int g = g0 + i + j, k = 4 * (i + j);
                                const float2 ca = dev::fmul2(sp[j], sxa);
                                const float2 cb = dev::fmul2(sp[j], sxb);
                                accA[g] = dev::ffma2(make_float2(__uint_as_float(d[k]), __uint_as_float(d[k + 1])), ca, accA[g]);
                                accB[g] = dev::ffma2(make_float2(__uint_as_float(d[k + 2]), __uint_as_float(d[k + 3])), cb, accB[g]);
                            }
                        }
                    };
                    // 4 chunks of 64 columns; the TMEM load of the next chunk is in flight during the
                    // math of the current one (a wait covers every load issued before it, so
                    // larger chunks, not more loads, are what cut the round trips)
                    uint32_t dA[32], dB[32];
                    dev::tmem_ld16x256b_x8(taddr, dA);
                    dev::tmem_ld_wait32(dA);
                    dev::tmem_ld16x256b_x8(taddr + 64, dB);
                    math(dA, 0, 8);
                    dev::tmem_ld_wait32(dB);
                    dev::tmem_ld16x256b_x8(taddr + 128, dA);
                    math(dB, 8, 8);
                    dev::tmem_ld_wait32(dA);
                    dev::tmem_ld16x256b_x8(taddr + 192, dB);
                    math(dA, 16, 8);
                    dev::tmem_ld_wait32(dB);
                    math(dB, 24, 8);
                } else {
                    // export exact partial sums of the requested window
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        uint32_t d[16];
                        dev::tmem_ld16x256b_x4(taddr + c * 32, d);
                        dev::tmem_ld_wait16(d);
                        for (int i = 0; i < 4; ++i) {
                            for (int e = 0; e < 4; ++e) {
                                const int row = (e < 2) ? row0 : row1;
                                const int n = n0 + 8 * (4 * c + i) + 2 * tq + (e & 1);
                                if (row >= p.M || row < p.pm0 || row >= p.pm0 + p.pmcount) continue;
                                if (n < p.pn0 || n >= p.pn0 + p.pncount || n >= p.N) continue;
                                p.P[(static_cast<int64_t>(row - p.pm0) * p.pncount + (n - p.pn0)) * p.nb + b] =
                                    __float2int_rn(__uint_as_float(d[4 * i + e]) * 262144.0f);
                            }
                        }
                    }
                }
                dev::tc_fence_before();
            }
            __syncwarp();
            if (lane == 0 && ok) {
                dev::mbar_arrive_remote(release);
                dev::mbar_arrive(&s.sc_empty[ss]);
            }
        }
        if constexpr (!kPartials) {
            auto store_rows = [&]() {
#pragma unroll
                for (int g = 0; g < 32; ++g) {
                    const int col = n0 + 8 * g + 2 * tq;
                    if (col < p.N) {
                        if (ok0) *reinterpret_cast<__half2*>(p.Y + static_cast<int64_t>(row0) * p.ldy + col) = __floats2half2_rn(accA[g].x, accA[g].y);
                        if (ok1) *reinterpret_cast<__half2*>(p.Y + static_cast<int64_t>(row1) * p.ldy + col) = __floats2half2_rn(accB[g].x, accB[g].y);
                    }
                }
            };
            if (p.splits == 1) {
                store_rows();
            } else {
                // split-K: publish this split's FP32 partial (this CTA's half of the tile); the
                // last split to arrive sums all of them in split order (deterministic).
                const int hrow = static_cast<int>(rank) * 128;
                float* base = p.ws_partial + (static_cast<int64_t>(t.tile) * p.splits + t.split) * kPairM * kTileN;
#pragma unroll
                for (int g = 0; g < 32; ++g) {
                    const int cc = 8 * g + 2 * tq;
                    __stcg(reinterpret_cast<float2*>(base + (hrow + lr0) * kTileN + cc), accA[g]);
                    __stcg(reinterpret_cast<float2*>(base + (hrow + lr1) * kTileN + cc), accB[g]);
                }
                __threadfence();
                dev::named_bar_sync(1, kEpiWarps * 32);
                if (et == 0) {
                    int32_t* cnt = p.ws_count + t.tile * 2 + rank;
                    const int prev = atomicAdd(cnt, 1);
                    const int last = (prev == p.splits - 1);
                    if (last) *cnt = 0;  // reusable for the next call
                    s.fixup_last = last;
                }
                dev::named_bar_sync(1, kEpiWarps * 32);
                if (s.fixup_last) {
                    // every split (this one included) is in the workspace: sum in split order
                    __threadfence();
#pragma unroll
                    for (int g = 0; g < 32; ++g) {
                        accA[g] = make_float2(0.f, 0.f);
                        accB[g] = make_float2(0.f, 0.f);
                    }
                    for (int sp = 0; sp < p.splits; ++sp) {
                        const float* o = p.ws_partial + (static_cast<int64_t>(t.tile) * p.splits + sp) * kPairM * kTileN;
#pragma unroll
                        for (int g = 0; g < 32; ++g) {
                            const int cc = 8 * g + 2 * tq;
                            const float2 fa = __ldcg(reinterpret_cast<const float2*>(o + (hrow + lr0) * kTileN + cc));
                            const float2 fb = __ldcg(reinterpret_cast<const float2*>(o + (hrow + lr1) * kTileN + cc));
                            accA[g].x += fa.x;
                            accA[g].y += fa.y;
                            accB[g].x += fb.x;
                            accB[g].y += fb.y;
                        }
                    }
                    store_rows();
                }
            }
        }
    }
    if (!ok && lane == 0) fail(p, abort_flag);
}

// kTest: the failure-detection test instantiation (runtime poll bound, a withheld weight copy);
// the others bound every wait by the compile-time dev::kMaxPolls.
template <bool kPartials, bool kYz, bool kTest = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) w4ax_gemm_kernel(const Params p) {
    extern __shared__ uint8_t smem_raw[];
    Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = dev::cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int i = 0; i < kBlk; ++i) {
            dev::mbar_init(&s.a_full[i], 1);   // the producer's expect-tx arrival
            // converter warps; in the even CTA also the odd CTA's forward and both CTAs'
            // epilogue warps (accumulator released)
            dev::mbar_init(&s.blk_full[i], kConvWarps + (rank == 0 ? 1 + 2 * kEpiWarps : 0));
            dev::mbar_init(&s.blk_empty[i], 1);
        }
        for (int i = 0; i < kWStages; ++i) {
            dev::mbar_init(&s.w_full[i], 1);
            dev::mbar_init(&s.w_empty[i], kConvWarps);
        }
        for (int i = 0; i < kScStages; ++i) {
            dev::mbar_init(&s.sc_full[i], kConvWarps);
            dev::mbar_init(&s.sc_empty[i], kEpiWarps);
        }
        for (int i = 0; i < 2; ++i) dev::mbar_init(&s.acc_full[i], 1);
        dev::mbar_init(&s.mma_done, 1);
        s.abort_flag = 0;
        if (rank == 0) {
            // blocks 0 and 1 find both accumulators free
            for (int i = 0; i < 2; ++i)
                for (int k = 0; k < 2 * kEpiWarps; ++k) dev::mbar_arrive(&s.blk_full[i]);
        }
        dev::fence_barrier_init();
    }
    for (int b = threadIdx.x; b < p.nb; b += kThreads) {
        s.mask[b] = p.mask[b];
        s.poff[b] = p.poff[b];
    }
    if (warp < kMaxBlocks / 32) {
        const int b = warp * 32 + lane;
        const uint32_t bits = __ballot_sync(0xFFFFFFFFu, b < p.nb && p.mask[b] != 0);
        if (lane == 0) s.maskw[warp] = bits;
    }
    if (warp == 1) dev::tmem_alloc_pair(&s.tmem_base, kTmemCols);
    dev::tc_fence_before();
    __syncthreads();
    dev::cluster_sync();   // both CTAs' barriers and TMEM exist before any cross-CTA traffic
    dev::tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int* abort_flag = &s.abort_flag;
    const uint32_t polls = kTest ? p.poll_limit : dev::kMaxPolls;
    const int withhold = kTest ? p.withhold : -1;

    if (warp < 8) {
        dev::setmaxnreg_dec<56>();
        if (warp == 0) {
            weight_producer(p, s, rank, lane, abort_flag, polls, withhold);
        } else if (warp == 1) {
            mma_role(p, s, rank, lane, tmem, abort_flag, polls);
        } else if (warp < kConvWarp0 + kConvWarps) {
            converter_role(p, s, rank, warp, lane, abort_flag, polls);
        } else if (warp == 6) {
            activation_producer(p, s, rank, lane, abort_flag, polls);
        }
    } else {
        dev::setmaxnreg_inc<200>();
        epilogue_role<kPartials, kYz>(p, s, rank, warp, lane, tmem, abort_flag, polls);
    }

    dev::tc_fence_before();
    __syncthreads();
    dev::cluster_sync();   // the peer's MMAs, commits and arrivals on this CTA are done
    if (warp == 1) {
        dev::tc_fence_after();
        dev::tmem_dealloc_pair(tmem, kTmemCols);
    }
}


constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory of the GEMM exceeds the 227 KB a CTA may use");

// Pairs (2-CTA clusters) that can be resident at once: the persistent grid never launches
// more, so no cluster waits for another to finish. Asked once per device.
int max_pairs(const fmpq_layout& L) {
    static int cached[64] = {};
    const int dev = L.device;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int pairs = L.num_sms / 2 > 0 ? L.num_sms / 2 : 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sizeof(Smem) + 1024;
    int clusters = 0;
    if (ensure_smem_limit(reinterpret_cast<const void*>(w4ax_gemm_kernel<false, false>),
                          static_cast<int>(sizeof(Smem) + 1024)) == cudaSuccess &&
        cudaOccupancyMaxActiveClusters(&clusters, w4ax_gemm_kernel<false, false>, &cfg) == cudaSuccess && clusters > 0 &&
        clusters < pairs)
        pairs = clusters;
    cudaGetLastError();   // a failed query leaves no sticky error behind
    if (dev >= 0 && dev < 64) cached[dev] = pairs;
    return pairs;
}

int choose_splits(const fmpq_layout& L, int64_t tiles) {
    const int pairs = max_pairs(L);
    if (tiles * 2 > pairs) return 1;
    int s = static_cast<int>(pairs / tiles);
    if (s > L.nb) s = L.nb;
    if (s > 16) s = 16;
    return s < 1 ? 1 : s;
}

int64_t pair_tiles(int64_t M, int64_t N) { return ((M + kPairM - 1) / kPairM) * ((N + kTileN - 1) / kTileN); }

}  // namespace

size_t gemm_counter_bytes(const fmpq_layout& L, int64_t M, int64_t N, bool variant) {
    if (!variant && gemm_small_path(M)) return gemm_small_counter_bytes(L, M, N);
    const int64_t tiles = pair_tiles(M, N);
    if (choose_splits(L, tiles) == 1) return 0;
    return static_cast<size_t>(tiles) * 2 * sizeof(int32_t) + 16;
}

size_t gemm_workspace_bytes(const fmpq_layout& L, int64_t M, int64_t N, bool variant) {
    if (!variant && gemm_small_path(M)) return gemm_small_workspace_bytes(L, M, N);
    const int64_t tiles = pair_tiles(M, N);
    const int splits = choose_splits(L, tiles);
    if (splits == 1) return 0;
    return static_cast<size_t>(tiles) * splits * kPairM * kTileN * sizeof(float) + gemm_counter_bytes(L, M, N, variant);
}

size_t variant_workspace_bytes(const fmpq_layout& L, int64_t M, int64_t N) {
    return ((gemm_workspace_bytes(L, M, N, true) + 1023) & ~size_t(1023)) + zero_term_bytes(L, M, N);
}

cudaError_t launch_gemm(const fmpq_layout& L, const GemmArgs& a, cudaStream_t stream) {
    const bool variant = a.zero_kind != kZeroNone || a.unsigned_w;
    if (!variant && gemm_small_path(a.M)) return launch_gemm_small(L, a, stream);
    for (auto fn : {w4ax_gemm_kernel<false, false>, w4ax_gemm_kernel<true, false>, w4ax_gemm_kernel<false, true>,
                    w4ax_gemm_kernel<false, false, true>}) {
        const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(fn), static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
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
    p.wmask = a.unsigned_w ? 0x0F0F0F0Fu : 0x87878787u;
    p.zero_kind = a.zero_kind;
    p.ch_scales = static_cast<const uint16_t*>(a.ch_scales);
    p.grp_scales = a.grp_scales;
    p.poll_limit = a.poll_limit != 0 ? a.poll_limit : dev::kMaxPolls;
    p.withhold = a.withhold;
    const bool partials = a.P != nullptr;
    if (partials) {
        p.mt0 = static_cast<int>(a.pm0 / kPairM);
        p.mtiles = static_cast<int>((a.pm0 + a.pmcount - 1) / kPairM) - p.mt0 + 1;
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
        p.mtiles = static_cast<int>((a.M + kPairM - 1) / kPairM);
        p.nt0 = 0;
        p.ntiles = static_cast<int>((a.N + kTileN - 1) / kTileN);
        p.splits = choose_splits(L, static_cast<int64_t>(p.mtiles) * p.ntiles);   // as gemm_workspace_bytes
        if (p.splits > 1) {
            const int64_t tiles = static_cast<int64_t>(p.mtiles) * p.ntiles;
            p.ws_partial = static_cast<float*>(a.workspace);
            p.ws_count = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a.workspace) +
                                                    static_cast<size_t>(tiles) * p.splits * kPairM * kTileN * sizeof(float));
        }
    }
    if (a.zero_kind != kZeroNone && !partials) {
        // the zero-point term for every output first, after the split-K part of the workspace
        uint8_t* zero_ws = static_cast<uint8_t*>(a.workspace) +
                           ((gemm_workspace_bytes(L, a.M, a.N, true) + 1023) & ~size_t(1023));
        bool maps_ok = true;
        const cudaError_t e = launch_zero_term(L, a, zero_ws, stream, &maps_ok);
        if (e != cudaSuccess) return e;
        if (!maps_ok) return cudaErrorInvalidValue;
        p.yz = reinterpret_cast<const float*>(zero_ws);
    }
    const int64_t units = static_cast<int64_t>(p.mtiles) * p.ntiles * p.splits;
    const int pairs = static_cast<int>(units < max_pairs(L) ? units : max_pairs(L));
    const int grid = 2 * pairs;   // clusters of two CTAs (one pair per two SMs)
    if (a.withhold >= 0)
        w4ax_gemm_kernel<false, false, true><<<grid, kThreads, kSmemBytes, stream>>>(p);
    else if (partials)
        w4ax_gemm_kernel<true, false><<<grid, kThreads, kSmemBytes, stream>>>(p);
    else if (p.yz != nullptr)
        w4ax_gemm_kernel<false, true><<<grid, kThreads, kSmemBytes, stream>>>(p);
    else if (a.pdl) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, w4ax_gemm_kernel<false, false>, p);
    } else
        w4ax_gemm_kernel<false, false><<<grid, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace fmpq
