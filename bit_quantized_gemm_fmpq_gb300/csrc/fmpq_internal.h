// Host-side internals shared by the C-ABI implementation and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

struct fmpq_layout {
    int32_t K = 0;
    int32_t K_in = 0;        // input row width the permutation selects from (K for a full permutation)
    int32_t nb = 0;          // K / 128
    int32_t n8 = 0;          // number of INT8 blocks
    int device = -1;
    int num_sms = 0;
    uint16_t* d_perm16 = nullptr;  // [K] gather permutation (K <= 65536)
    uint8_t* d_mask = nullptr;     // [nb] 1 = INT8 block
    int32_t* d_poff = nullptr;     // [nb] first code plane of each block (planes before it)
    int32_t* d_status = nullptr;   // device status word
    int32_t planes = 0;            // code planes: n4 + 2*n8
    uint32_t mask_bits[8] = {};    // the INT8 blocks as a bitmap (bit b % 32 of word b / 32)
    int64_t row_bytes = 0;         // packed-A bytes per token: 128 * planes
};

namespace fmpq {

constexpr int kBlock = 128;
constexpr int kMaxBlocks = 256;     // K <= 32768
constexpr int kTileN = 256;          // packed-weight row grouping and GEMM tile width

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device. Function
// attributes are per device: the first call for each (kernel, device) sets it, later calls
// return at once. Thread-safe.
cudaError_t ensure_smem_limit(const void* kernel, int bytes);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime (no link to
// libcuda); nullptr when the driver does not provide it.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled();

// Launchers (return cudaGetLastError() after the launch).
// gamma_perm != nullptr: the quantized values are the row's RMSNorm with that gamma (permuted
// channel order) and eps. mode: kQuantSym (FMPQ), kQuantAsym (QUIK asymmetric, aux = zero points
// fp16 [nb][M]), kQuantTok (QoQ per-token INT8, aux = block code sums int32 [nb][M]; scales [M]).
enum { kQuantSym = 0, kQuantAsym = 2, kQuantTok = 3 };
// QUIK input split fused into the quantizer: X_out[m][j] = X[m][cols[j]] (0 outside [0, K_in)),
// n a multiple of 8, cols and X_out 16-byte aligned.
struct QuantSplit {
    const int32_t* cols;
    int n;
    void* X_out;
};
cudaError_t launch_quantize(const fmpq_layout& L, const void* X, int64_t ldx, int64_t M, void* A, void* scales,
                            cudaStream_t stream, const void* gamma_perm = nullptr, float eps = 0.0f,
                            int mode = kQuantSym, void* aux = nullptr, const QuantSplit* split = nullptr);
// The quantizer fused with SwiGLU: G, U fp16 [M][ld] in the layout's permuted channel order.
cudaError_t launch_swiglu_quantize(const fmpq_layout& L, const void* G, int64_t ldg, const void* U, int64_t ldu,
                                   int64_t M, void* A, void* scales, cudaStream_t stream);
// QoQ progressive weights: unsigned 4-bit codes in the packed layout, s1 fp16 [N], s2 / z2 [nb][N].
cudaError_t launch_qoq_pack_weights(const fmpq_layout& L, const void* W, int64_t ldw, int64_t N, void* Wp,
                                    void* s1, uint8_t* s2, uint8_t* z2, cudaStream_t stream);
// QUIK zero-point term: wsum [nb][N] = w_scale * sum of the block's codes (packed sign-magnitude).
cudaError_t launch_weight_sums(const fmpq_layout& L, const void* Wp, const void* w_scales, int64_t N, float* wsum,
                               cudaStream_t stream);
cudaError_t launch_pack_weights(const fmpq_layout& L, const void* W, int64_t ldw, int64_t N, void* Wp,
                                void* scales, cudaStream_t stream);
cudaError_t launch_unpack_weights(const fmpq_layout& L, const void* Wp, int64_t N, int8_t* Wq, cudaStream_t stream,
                                  bool unsigned_codes = false);

enum { kZeroNone = 0, kZeroQuik = 1, kZeroQoq = 2 };

struct GemmArgs {
    const void* A;
    const void* a_scales;
    const void* W;
    const void* w_scales;
    int64_t M, N;
    void* Y;
    int64_t ldy;
    void* workspace;
    size_t workspace_bytes;
    // partial-sum export (debug): when P != nullptr the kernel writes P instead of Y
    int32_t* P;
    int64_t pm0, pmcount, pn0, pncount;
    // Quantization variants (the defaults are FMPQ: signed weight codes, per-block activation
    // scales, no zero-point term). Each block then adds x_zero[m] * w_zero[n] to the output:
    //   kZeroQuik: x_zero = a_zeros[b][m] (fp16), w_zero = w_sums[b][n] (fp32)

    //   kZeroQoq:  activation scale a_scales[m] for every block; weight scale
    //              ch_scales[n] * grp_scales[b][n]; x_zero = a_scales[m] * a_sums[b][m],
    //              w_zero = -ch_scales[n] * grp_scales[b][n] * grp_zeros[b][n]
    // Outside the partial-sum export the term is summed over the blocks on the tensor cores first
    // (launch_zero_term, in the workspace after the split-K part) and starts the accumulators.
    int zero_kind = kZeroNone;
    bool unsigned_w = false;          // weight codes are unsigned 4-bit (QoQ), not sign-magnitude
    const void* a_zeros = nullptr;
    const int32_t* a_sums = nullptr;
    const float* w_sums = nullptr;
    const void* ch_scales = nullptr;
    const uint8_t* grp_scales = nullptr;
    const uint8_t* grp_zeros = nullptr;
    // failure-detection test (2-SM kernel only): polls before a device wait gives up (0: the
    // default bound) and the packed weight copy the first CTA withholds (-1: none)
    uint32_t poll_limit = 0;
    int withhold = -1;
    // launched right after this library's quantizer as its programmatic dependent: the GEMM's
    // prologue and weight stream start while the quantizer runs; the roles that read its codes
    // and scales wait for its completion (griddepcontrol.wait)
    bool pdl = false;
};

// Workspace of a split-K launch: FP32 partial tiles followed by the arrival counters
// (gemm_counter_bytes of it, at the end). Both are 0 when the shape needs no split.
// `variant`: a quantization variant (they always run the 2-SM kernel, whatever M).
size_t gemm_workspace_bytes(const fmpq_layout& L, int64_t M, int64_t N, bool variant = false);
size_t gemm_counter_bytes(const fmpq_layout& L, int64_t M, int64_t N, bool variant = false);
// A quantization variant's workspace: the split-K part (rounded up to 1 KB), then the zero-point
// term (zero_term_bytes). Needed whatever the shape.
size_t variant_workspace_bytes(const fmpq_layout& L, int64_t M, int64_t N);
cudaError_t launch_gemm(const fmpq_layout& L, const GemmArgs& args, cudaStream_t stream);

// The variants' zero-point term on the tensor cores, for the GEMM to start its accumulators
// from: yz[m][n] = sum_b x_zero[b][m] * w_zero[b][n] (FP32) at the start of ws, its operands
// after it (zero_term_bytes in all). tcgen05 kind::f16 on operands split so that every product
// is exact (QUIK: the zero points and a scaled two-term split of w_sums; QoQ: the code sums in
// two parts and s2 * z2, with s1 and the token scale applied to each output).
size_t zero_term_bytes(const fmpq_layout& L, int64_t M, int64_t N);
cudaError_t launch_zero_term(const fmpq_layout& L, const GemmArgs& args, void* ws, cudaStream_t stream,
                             bool* maps_ok);

// Outlier split, FP16 path: gather X[:, cols] into X_out, Y += X_out * W_out^T (tcgen05 kind::f16
// tiles; device-side timeouts go to `status`). *maps_ok is false when a TMA tensor map cannot be
// encoded (nothing is launched then).
cudaError_t launch_outlier_gemm(const void* X, int64_t ldx, int64_t M, const int32_t* cols, int n_out,
                                const void* W_out, int64_t ldw_out, int64_t N, void* X_out, void* Y, int64_t ldy,
                                int num_sms, int32_t* status, cudaStream_t stream, bool* maps_ok);

// Calibration: per-channel absmax (zeroes `out`, then reduces) and the host layout planner.
cudaError_t launch_channel_absmax(const void* X, int64_t ldx, int64_t T, int K, uint32_t* out, int num_sms,
                                  cudaStream_t stream);
void plan_layout(int K, const uint32_t* absmax, int n8, int32_t* perm, uint8_t* mask);
// Largest relative quantization error ||x - xhat|| / ||x|| over T calibration tokens (fp16,
// host, [T][ldx]) under a layout; and the smallest n8 whose planned layout keeps it within eps
// (K/128 when none does), writing that layout and its error.
double layout_error(int K, const uint16_t* Xc, int64_t T, int64_t ldx, const int32_t* perm, const uint8_t* mask);
int plan_layout_budget(int K, const uint32_t* absmax, const uint16_t* Xc, int64_t T, int64_t ldx, double eps,
                       double* err, int32_t* perm, uint8_t* mask);

// Few tokens (M <= 128): the operand-swapped GEMM (output channels on the tensor core's M side,
// tokens on its N side). launch_gemm and the workspace queries dispatch to it.
bool gemm_small_path(int64_t M);
size_t gemm_small_workspace_bytes(const fmpq_layout& L, int64_t M, int64_t N);
size_t gemm_small_counter_bytes(const fmpq_layout& L, int64_t M, int64_t N);
cudaError_t launch_gemm_small(const fmpq_layout& L, const GemmArgs& args, cudaStream_t stream);

}  // namespace fmpq
