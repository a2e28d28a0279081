/*
 * fmpq.h -- C ABI of the GB300 (sm_103a) FMPQ W4Ax library.
 *
 * The method (COMET: Towards Practical W4A4KV4 LLMs Serving; FMPQ, "fine-grained
 * mixed-precision quantization"):
 *   - the K input channels of a linear layer are permuted so that outlier channels
 *     collect in a few blocks, and split into blocks of 128 channels
 *     (COMET news article, section 1 "outlier distribution");
 *   - activations are quantized per token and per block: INT8 for the outlier blocks,
 *     INT4 for the rest (same section, the "dynamic precision" sentence);
 *   - weights are INT4, per output channel and per block, prepared offline
 *     (QServe explainer, section "W4A8 GEMM core design": static weights are reordered
 *     offline at no runtime cost);
 *   - the W4Ax GEMM forms exact integer partial sums per block and applies the
 *     dequantization scales in an FP32 epilogue (COMET abstract: mixed W4A4/W4A8 matrix
 *     multiplication with a mixed-precision data layout; QUIK explainer, section "kernel
 *     fusion": dequantization fused into the GEMM epilogue).
 * Beside it: the layout derived from calibration data (fmpq_channel_absmax, fmpq_plan_layout),
 * the quantizer fused with RMSNorm (fmpq_rmsnorm_quantize) or SwiGLU (fmpq_swiglu_quantize), QUIK's FP16 outlier split
 * (fmpq_layout_create_select, fmpq_outlier_gemm_fp16), QUIK asymmetric activations
 * (fmpq_quantize_asym, w4ax_gemm_asym) and QoQ progressive group quantization with W4A8
 * GEMMs (qoq_pack_weights, qoq_quantize, qoq_gemm).
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless the parameter name ends in "_host".
 *   - The caller owns every device buffer and stream. The library owns only the layout
 *     handle (a host struct plus small device tables allocated once by
 *     fmpq_layout_create on the device current at that time).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream),
 *     never synchronize (except fmpq_layout_create/destroy and fmpq_device_status), and
 *     allocate no memory.
 *   - Argument errors are reported synchronously by the return value and launch nothing.
 *     A CUDA launch failure returns FMPQ_ERR_CUDA. A device-side wait that gives up (a
 *     bounded wait, never a hang) records FMPQ_ERR_TIMEOUT in the layout's device status
 *     word, read by fmpq_device_status. The library never aborts, traps or prints.
 *   - All data buffers must be 16-byte aligned (FMPQ_ERR_MISALIGNED otherwise).
 *   - Inputs must be finite (no NaN/Inf); results for non-finite inputs are unspecified.
 */
#ifndef FMPQ_H
#define FMPQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FMPQ_API __attribute__((visibility("default")))
#else
#define FMPQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fmpq_status {
    FMPQ_OK = 0,
    FMPQ_ERR_INVALID_ARG = 1,       /* null pointer, bad permutation, bad mask value, ... */
    FMPQ_ERR_UNSUPPORTED_SHAPE = 2, /* K % 128 != 0, N % 16 != 0, sizes out of range */
    FMPQ_ERR_MISALIGNED = 3,        /* pointer or leading dimension misaligned */
    FMPQ_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
    FMPQ_ERR_TIMEOUT = 5,           /* (device status) a bounded device wait gave up */
    FMPQ_ERR_DEVICE = 6,            /* no usable sm_103 device / layout used on another device */
    FMPQ_ERR_WORKSPACE = 7          /* workspace missing or too small */
} fmpq_status;

#define FMPQ_BLOCK 128              /* channels per quantization block */
#define FMPQ_MAX_K 32768            /* largest supported K */

/* Opaque, library-owned description of one layer's channel permutation and block mask. */
typedef struct fmpq_layout fmpq_layout;

/* Create a layout.
 *   K                  number of input channels; K % 128 == 0, 128 <= K <= FMPQ_MAX_K.
 *   perm_host[K]       gather permutation: permuted channel j is input channel perm[j]
 *                      (COMET news article, section 1: channel reordering gathers the
 *                      outliers into the same blocks). Must be a permutation of [0, K).
 *   outlier_block_mask_host[K/128]  1 = INT8 block (outlier block), 0 = INT4 block.
 *   out                receives the handle.
 * Uploads small device tables on the current device (synchronous). */
FMPQ_API fmpq_status fmpq_layout_create(int32_t K, const int32_t* perm_host,
                               const uint8_t* outlier_block_mask_host, fmpq_layout** out);
/* A layout that selects its K channels from wider input rows of K_in channels (K <= K_in <=
 * FMPQ_MAX_K, K_in % 8 == 0): select_host[K] holds distinct channel indices in [0, K_in). The
 * quantizer and the weight packing then take rows of at least K_in channels (ldx, ldw >= K_in).
 * This is the base part of an outlier split (QUIK explainer, "第二步: 前向传播"): the base
 * channels go through the INT4/INT8 GEMM, the outlier channels through fmpq_outlier_gemm_fp16.
 * fmpq_rmsnorm_quantize needs K_in == K. */
FMPQ_API fmpq_status fmpq_layout_create_select(int32_t K, int32_t K_in, const int32_t* select_host,
                                               const uint8_t* outlier_block_mask_host, fmpq_layout** out);
FMPQ_API void fmpq_layout_destroy(fmpq_layout* layout);
FMPQ_API int32_t fmpq_layout_k(const fmpq_layout* layout);
FMPQ_API int32_t fmpq_layout_num_blocks(const fmpq_layout* layout);
FMPQ_API int32_t fmpq_layout_num_int8_blocks(const fmpq_layout* layout);

/* Bytes of the packed activation buffer for M tokens: M * 128 * (n4 + 2 * n8).
 * Layout: operand-ready code planes (the method's "mixed-precision data layout", made
 * concrete for a tensor core whose narrowest exact integer path is 8-bit E4M3):
 *   - One byte per code: bit 7 = sign bit of the fp16 input, bits 0-6 = the E4M3 encoding
 *     of part * 2^-9, where part is |q| for an INT4 block. An INT8 block has two planes,
 *     part = |q| mod 16 (low plane) and part = |q| - |q| mod 16 (high plane); the parts of
 *     a code sum to |q|. (For part <= 15 the encoding is the integer part itself.)
 *   - Planes follow block order: block b's first plane is plane poff_b = n4 + 2*n8 counted
 *     over the blocks before b; plane p occupies bytes [p*M*128, (p+1)*M*128).
 *   - Row m of a plane is 128 bytes; the 16 channels 16c..16c+15 of the block are stored
 *     in order in the 16-byte chunk at position c XOR (m mod 8), so that a copy of 128
 *     rows starting at a multiple of 128 is a 128-byte-swizzled K-major operand tile. */
FMPQ_API size_t fmpq_packed_a_bytes(const fmpq_layout* layout, int64_t M);

/* Bytes of the packed weight buffer for N output channels: ceil(N/256)*256 * K/2.
 * The packed weight format is implementation-defined (tile-major, padded to 256 rows);
 * w4_unpack_weights decodes it. */
FMPQ_API size_t fmpq_packed_w_bytes(const fmpq_layout* layout, int64_t N);

/* Fused activation quantizer (one pass: gather-permute, per-(token, block) absmax,
 * fp16 scale, round-half-even quantization, INT4/INT8 packing).
 *   X         fp16 [M][ldx], ldx >= K, ldx % 8 == 0.
 *   M         1 <= M <= 2^31-1.
 *   A_packed  fmpq_packed_a_bytes(layout, M) bytes (layout above).
 *   a_scales  fp16 [K/128][M]: a_scales[b*M + m] = fp16_rne(fp32(absmax)/qmax),
 *             qmax = 127 (INT8 block) or 7 (INT4 block).
 * Codes: q = clamp(rne(fp32(x) / fp32(scale)), -qmax, qmax); a zero scale gives q = 0. */
FMPQ_API fmpq_status fmpq_quantize(const fmpq_layout* layout, const void* X, int64_t ldx, int64_t M,
                          void* A_packed, void* a_scales, void* stream);

/* The quantizer fused with the preceding RMSNorm: the activation quantization of the QKV
 * projection and the first FFN layer fused into the layer norm before them (QServe explainer,
 * "运行时设计"). Codes, scales and layout are those of fmpq_quantize applied to
 *   y[m][c] = fp16_rn( (fp32(x[m][c]) * r_m) * fp32(gamma[c]) ),
 *   r_m = 1 / sqrt(T_m / K + eps)   (IEEE fp32 division, square root and addition),
 * where T_m is the exact sum of x[m][c]^2 over the row, rounded once to fp32 (nearest, ties to
 * even). It does not depend on any summation order.
 *   gamma_perm  fp16 [K]: gamma in the permuted order, gamma_perm[j] = gamma[perm[j]]
 *               (prepared once, like the weights). 16-byte aligned.
 *   eps         positive and finite (FMPQ_ERR_INVALID_ARG otherwise).
 * Other arguments as fmpq_quantize. */
FMPQ_API fmpq_status fmpq_rmsnorm_quantize(const fmpq_layout* layout, const void* X, int64_t ldx, int64_t M,
                                           const void* gamma_perm, float eps, void* A_packed, void* a_scales,
                                           void* stream);

/* The quantizer fused with the SwiGLU activation before the second FFN layer (QServe explainer,
 * "运行时设计": activation quantization fused into the kernel that produces the activation). Codes,
 * scales and layout are those of fmpq_quantize applied to
 *   h[m][j] = fp16_rn( g[m][j] * u[m][j] / (1 + e^(-g[m][j])) )
 * rounded once from the real value (ties to even; exact unless that value lies within ~2^-50 of an
 * fp16 rounding boundary); a zero h keeps the IEEE sign of g * u.
 *   G_perm, U_perm  fp16 [M][ldg], [M][ldu]: the gate and up projections' outputs in the layout's
 *                   PERMUTED channel order (column j is channel perm[j]: the projections' output
 *                   channels are reordered offline by the layout's permutation, as the weights are);
 *                   ldg, ldu >= K, multiples of 8, 16-byte aligned.
 * Other arguments as fmpq_quantize. Results are unspecified where h overflows fp16. */
FMPQ_API fmpq_status fmpq_swiglu_quantize(const fmpq_layout* layout, const void* G_perm, int64_t ldg,
                                          const void* U_perm, int64_t ldu, int64_t M, void* A_packed, void* a_scales,
                                          void* stream);

/* Offline weight preparation: W fp16 [N][ldw] (ldw >= K, ldw % 8 == 0, N % 16 == 0)
 * -> W_packed (fmpq_packed_w_bytes) and w_scales fp16 [K/128][N], INT4 range [-7, 7]
 * per output channel and block, same scale and rounding rule as the activations, on the
 * permuted channel order. */
FMPQ_API fmpq_status w4_pack_weights(const fmpq_layout* layout, const void* W, int64_t ldw, int64_t N,
                            void* W_packed, void* w_scales, void* stream);

/* Debug/test: decode W_packed to codes Wq int8 [N][K] (permuted channel order). */
FMPQ_API fmpq_status w4_unpack_weights(const fmpq_layout* layout, const void* W_packed, int64_t N,
                              int8_t* Wq, void* stream);

/* Workspace bytes w4ax_gemm needs for this shape (0 when it needs none). With M > 64 and few
 * output tiles the GEMM splits K across CTA pairs; the workspace then holds the FP32 partial
 * tiles and one arrival counter per output tile. With M <= 64 (the few-token kernel) the
 * K-splits of a tile run as one thread-block cluster and meet in its shared memory: no
 * workspace. */
FMPQ_API size_t w4ax_gemm_workspace_bytes(const fmpq_layout* layout, int64_t M, int64_t N);

/* The W4Ax GEMM:
 *   Y[m][n] = fp16_rn( sum_b a_scales[b][m] * w_scales[b][n] * P[m][n][b] ),
 *   P[m][n][b] = sum over channels j of block b of qa[m][j] * qw[n][j]   (exact integers),
 * accumulated in FP32.
 *   Y          fp16 [M][ldy], ldy >= N, ldy % 8 == 0; N % 16 == 0.
 *   workspace  w4ax_gemm_workspace_bytes(layout, M, N) bytes (may be NULL when that is 0);
 *              zero-filled once before its first use; each call returns the arrival
 *              counters it uses to zero, so the buffer is reused without re-initialization.
 *              A call that records FMPQ_ERR_TIMEOUT may leave counters nonzero: zero-fill
 *              the workspace again before reusing it. Calls that share a workspace must not
 *              run concurrently.
 * The split-K reduction sums the K-splits in a fixed order, so results are deterministic. */
FMPQ_API fmpq_status w4ax_gemm(const fmpq_layout* layout, const void* A_packed, const void* a_scales,
                      const void* W_packed, const void* w_scales, int64_t M, int64_t N,
                      void* Y, int64_t ldy, void* workspace, size_t workspace_bytes, void* stream);

/* The same GEMM for callers that cannot allocate device memory (a pool that owns the whole
 * device, a serving path that must not allocate mid-flight, a host without access to the
 * allocator). It takes no workspace: when the shape needs one (w4ax_gemm_workspace_bytes > 0),
 * the library uses its own fixed device array of 20 MiB of partial tiles + 64 KiB of
 * counters, which every GPU that loads the library holds until exit. The paper has no
 * counterpart; this is an interface convenience.
 *   - Arguments and results are those of w4ax_gemm (no workspace arguments).
 *   - The first call on a device looks up the array's device address (host-side work only);
 *     make that first call before any stream capture.
 *   - When the shape needs the array, each call first clears the arrival counters it uses
 *     with a memset on `stream` (so a call after one that gave up with FMPQ_ERR_TIMEOUT still
 *     starts from zero), then launches the GEMM on `stream`.
 *   - Shapes whose workspace would exceed the array return FMPQ_ERR_WORKSPACE.
 *   - All calls share the array, which keeps the last call's contents: calls that overlap on
 *     the GPU (e.g. on two streams) race and must be serialized by the caller.
 *   - Allocates nothing. */
FMPQ_API fmpq_status w4ax_gemm_noalloc(const fmpq_layout* layout, const void* A_packed,
                                       const void* a_scales, const void* W_packed,
                                       const void* w_scales, int64_t M, int64_t N, void* Y,
                                       int64_t ldy, void* stream);

/* fmpq_quantize followed by w4ax_gemm on the same stream, as one call: the stand-alone
 * quantization node ahead of a GEMM whose input no fusable kernel produces, such as the
 * attention output projection (QServe explainer, "运行时设计"). The GEMM is launched as the
 * quantizer's programmatic dependent, so its prologue and weight stream run while the
 * quantizer does, and it reads the codes and activation scales only once the quantizer has
 * completed. Results, arguments (those of both calls; A_packed and a_scales are written,
 * then read) and errors as the two calls; every argument is checked before either kernel is
 * launched. */
FMPQ_API fmpq_status fmpq_quantize_gemm(const fmpq_layout* layout, const void* X, int64_t ldx, int64_t M,
                                        void* A_packed, void* a_scales, const void* W_packed,
                                        const void* w_scales, int64_t N, void* Y, int64_t ldy,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* Debug/test: the exact per-block integer partial sums P computed by the GEMM's own
 * tensor-core path, for the window [m0, m0+mcount) x [n0, n0+ncount):
 *   P int32 [mcount][ncount][K/128]. */
FMPQ_API fmpq_status w4ax_gemm_partials(const fmpq_layout* layout, const void* A_packed,
                               const void* W_packed, int64_t M, int64_t N, int64_t m0,
                               int64_t mcount, int64_t n0, int64_t ncount, int32_t* P,
                               void* stream);

/* Debug/test of failure detection: w4ax_gemm (the 2-SM kernel for M > 64, the few-token kernel
 * for M <= 64) in which the first CTA's weight producer never issues its withhold_copy-th packed
 * weight copy (counted from 0, < K/128; a few-token copy holds two blocks, and a copy the CTA
 * never reaches withholds nothing), and every device-side wait gives up after poll_limit polls
 * (>= 1024). The wait on the missing copy runs out, the kernel's roles leave their loops, wait
 * for the copies they did issue and release TMEM; the call records FMPQ_ERR_TIMEOUT in the
 * layout's device status word and Y is unspecified. Nothing faults or hangs: in the few-token
 * kernel's clusters the aborted CTA stops before any exchange with the other splits, whose
 * waits for it run out in turn. The next normal call is unaffected (a split-K workspace's
 * counters still return to zero). Other arguments as w4ax_gemm. */
FMPQ_API fmpq_status w4ax_gemm_fault_test(const fmpq_layout* layout, const void* A_packed, const void* a_scales,
                                          const void* W_packed, const void* w_scales, int64_t M, int64_t N, void* Y,
                                          int64_t ldy, void* workspace, size_t workspace_bytes,
                                          int32_t withhold_copy, uint32_t poll_limit, void* stream);

/* The FP16 path of an outlier split (QUIK explainer, "第二步: 前向传播": the outlier columns are
 * multiplied in FP16 by the unquantized outlier weights; the INT4 result, dequantized to FP16,
 * is added to this FP16 outlier result):
 *   X_out[m][j] = X[m][cols[j]]   (0 for an index outside [0, ldx))
 *   P[m][n]     = fp16_rn( sum_j X_out[m][j] * W_out[n][j] )   (FP32 accumulation: the FP16
 *                                                              outlier result)
 *   Y[m][n]     = fp16_rn( Y[m][n] + P[m][n] )   (the merge, an fp16 addition)
 *   layout     the base part's layout (fmpq_layout_create_select); only its device and its
 *              device status word are used (a device-side timeout is recorded there).
 *   X          fp16 [M][ldx] (device); cols int32 [n_out] (device); n_out % 8 == 0.
 *   W_out      fp16 [N][ldw_out], ldw_out >= n_out, the outlier columns of the weights (offline).
 *   X_out      fp16 [M][n_out] device workspace (caller-owned), overwritten.
 *   Y          fp16 [M][ldy], ldy >= N, N <= 8388480: read and updated in place (run the INT4
 *              path first).
 * The product runs on the tensor cores (tcgen05 kind::f16, FP32 accumulator in TMEM) in the
 * library's own kernel; nothing is allocated. FMPQ_ERR_CUDA if a launch fails. */
FMPQ_API fmpq_status fmpq_outlier_gemm_fp16(const fmpq_layout* layout, const void* X, int64_t ldx, int64_t M,
                                            const int32_t* cols, int32_t n_out, const void* W_out, int64_t ldw_out,
                                            int64_t N, void* X_out, void* Y, int64_t ldy, void* stream);

/* The input split fused into the quantizer (QUIK explainer, "核融合": one kernel reads the input,
 * takes the statistics, quantizes the base part and extracts the outlier part in one pass).
 * Writes what fmpq_quantize (asym = 0) or fmpq_quantize_asym (asym = 1) writes for the layout's
 * selected channels, and in the same pass over X
 *   X_out[m][j] = X[m][cols[j]]   (0 for an index outside [0, K_in)),
 * the operand of fmpq_outlier_product_fp16.
 *   cols    int32 [n_out] (device), 8 <= n_out <= FMPQ_MAX_K, n_out % 8 == 0, 16-byte aligned.
 *   X_out   fp16 [M][n_out] (device, caller-owned), 16-byte aligned.
 *   a_zeros asym = 1: fp16 [K/128][M] zero points (the layout must have no INT8 block); ignored
 *           for asym = 0.
 * Other arguments and errors as fmpq_quantize / fmpq_quantize_asym. */
FMPQ_API fmpq_status fmpq_quantize_split(const fmpq_layout* layout, const void* X, int64_t ldx, int64_t M,
                                         const int32_t* cols, int32_t n_out, int32_t asym, void* A_packed,
                                         void* a_scales, void* a_zeros, void* X_out, void* stream);

/* fmpq_outlier_gemm_fp16 without its gather: X_out fp16 [M][n_out] already holds the outlier
 * columns (fmpq_quantize_split). Y[m][n] = fp16_rn(Y[m][n] + fp16_rn(sum_j X_out[m][j] *
 * W_out[n][j])); arguments, limits and errors as fmpq_outlier_gemm_fp16. */
FMPQ_API fmpq_status fmpq_outlier_product_fp16(const fmpq_layout* layout, const void* X_out, int64_t M,
                                               int32_t n_out, const void* W_out, int64_t ldw_out, int64_t N,
                                               void* Y, int64_t ldy, void* stream);

/* ---- Offline layout derivation from calibration activations ----
 * The activation outliers sit in a small set of channels (about 10%: COMET news article,
 * section 1), and a permutation gathers them into the same 128-channel blocks, which take
 * INT8 codes. The outlier channels are found offline on calibration data and moved to the
 * end (QUIK explainer, "第一步: 识别与重排"). The statistic is each channel's absolute maximum.
 *
 * Per-channel absolute maximum over T calibration tokens (asynchronous on `stream`):
 *   X        fp16 [T][ldx] (device), 1 <= T, ldx >= K, ldx % 8 == 0, 16-byte aligned.
 *   K        K % 128 == 0, 128 <= K <= FMPQ_MAX_K.
 *   absmax   uint32 [K] (device, caller-owned): absmax[c] receives the fp16 bit pattern of
 *            max_t |X[t][c]| (sign bit clear; for finite inputs the bit patterns order like
 *            the magnitudes). The call zeroes it first, on the same stream. */
FMPQ_API fmpq_status fmpq_channel_absmax(const void* X, int64_t ldx, int64_t T, int32_t K, uint32_t* absmax,
                                         void* stream);

/* Layout from channel statistics (host only: no device work, callable without a GPU).
 *   absmax_host[K]   per-channel statistic, larger = more outlying (e.g. fmpq_channel_absmax).
 *   n8               INT8 blocks, 0 <= n8 <= K/128.
 *   perm_host[K]     out: the channels ranked by absmax (larger first, equal values by lower
 *                    index); the first 128*n8 of the ranking fill the last n8 blocks
 *                    (positions K-128*n8 .. K-1, in rank order), the other channels fill
 *                    positions 0 .. K-128*n8-1 in ascending channel order.
 *   mask_host[K/128] out: 1 for the last n8 blocks, 0 for the others.
 * The outputs feed fmpq_layout_create. */
FMPQ_API fmpq_status fmpq_plan_layout(int32_t K, const uint32_t* absmax_host, int32_t n8, int32_t* perm_host,
                                      uint8_t* mask_host);

/* Layout with the fewest INT8 blocks that keeps the quantization error of calibration tokens
 * within a budget (host only: no device work, callable without a GPU). The INT8 blocks are there
 * to keep the outliers' quantization error small (COMET news article, section 1); the error of a
 * layout on the calibration tokens is
 *   err = max over tokens t of ||x_t - xhat_t||_2 / ||x_t||_2   (0 for an all-zero token),
 * xhat_t the token's dequantized codes q * s under the layout (the rule of fmpq_quantize); both
 * squared norms are summed exactly and converted once to fp64, then one fp64 division and one
 * square root. For n8 = 0, 1, ..., K/128 the layout is fmpq_plan_layout(K, absmax_host, n8); the
 * first whose err <= eps is written, else the one for n8 = K/128 (every block INT8).
 *   absmax_host[K]       per-channel statistic (e.g. fmpq_channel_absmax of the same tokens).
 *   X_calib_host         fp16 [T][ldx] calibration tokens, input channel order, T >= 1, ldx >= K.
 *   eps                  the budget, finite and >= 0 (e.g. 0.05).
 *   n8_out, err_out      out: the INT8 blocks chosen and that layout's err (err > eps only when
 *                        even n8 = K/128 misses the budget).
 *   perm_host, mask_host out: as fmpq_plan_layout. */
FMPQ_API fmpq_status fmpq_plan_layout_budget(int32_t K, const uint32_t* absmax_host, const void* X_calib_host, int64_t T,
                                             int64_t ldx, double eps, int32_t* n8_out, double* err_out,
                                             int32_t* perm_host, uint8_t* mask_host);

/* INT8 blocks for an outlier fraction of the channels: ceil(round(fraction * K) / 128), with
 * round taking halves away from zero, at most K/128; -1 for an invalid K or a fraction
 * outside [0, 1]. */
FMPQ_API int32_t fmpq_outlier_blocks(int32_t K, double fraction);

/* ---- Quantization variants the pages describe beside FMPQ ----
 * Both run on the same layouts, packed formats and 2-SM GEMM kernel (for every M), with a
 * zero-point term. The term is summed over the blocks on the tensor cores first, into the
 * workspace, and starts the GEMM's accumulators. Their workspace (never 0; the same for both):
 * w4ax_gemm's split-K part plus the term (M*N*4 bytes and the term's operands). */
FMPQ_API size_t fmpq_variant_gemm_workspace_bytes(const fmpq_layout* layout, int64_t M, int64_t N);

/* QUIK asymmetric activations (QUIK explainer, "反量化背后的数学": activations take a scale and a
 * zero point, weights a scale only; the zero point's term z * sum(w) needs only the weights'
 * sum, computed offline). The layout must have no INT8 block (FMPQ_ERR_INVALID_ARG): QUIK keeps
 * its outliers in FP16 (fmpq_outlier_gemm_fp16). Per token m and block b:
 *   z = the block's smallest input (value order, -0 below +0)   -> a_zeros[b][m] (fp16 bits)
 *   s = fp16_rn( fp32( fp32(max) - fp32(z) ) / 15 )              -> a_scales[b][m]
 *   q = clamp( rne( fp32( fp32(x) - fp32(z) ) / fp32(s) ), 0, 15 ), q = 0 when s == 0
 * (IEEE fp32 subtraction and division, round half to even), so x ~ s * q + z. A_packed has the
 * fmpq_quantize format with the sign bits clear (byte = E4M3 of q * 2^-9).
 *   a_scales, a_zeros  fp16 [K/128][M], 16-byte aligned. Other arguments as fmpq_quantize. */
FMPQ_API fmpq_status fmpq_quantize_asym(const fmpq_layout* layout, const void* X, int64_t ldx, int64_t M,
                                        void* A_packed, void* a_scales, void* a_zeros, void* stream);

/* Offline weight sums of the zero-point term: w_sums[b][n] = w_scales[b][n] * (sum of the
 * block's codes of output channel n) in fp32 (exact), from w4_pack_weights' outputs.
 *   w_sums  fp32 [K/128][N] (device, caller-owned), 16-byte aligned. */
FMPQ_API fmpq_status w4_weight_sums(const fmpq_layout* layout, const void* W_packed, const void* w_scales,
                                    int64_t N, float* w_sums, void* stream);

/* The GEMM on asymmetric activations:
 *   Y[m][n] = fp16_rn( sum_b ( a_scales[b][m] * w_scales[b][n] * P[m][n][b]
 *                              + a_zeros[b][m] * w_sums[b][n] ) ),   FP32 accumulation,
 * P the exact integer sums of the unsigned activation codes times the weight codes. The zero-point
 * sum over b is formed first on the tensor cores (fp16 zero points times a scaled two-term fp16
 * split of w_sums, products exact) into the workspace, and added once per output. Shapes and alignment as
 * w4ax_gemm; workspace: fmpq_variant_gemm_workspace_bytes (never 0), else FMPQ_ERR_WORKSPACE. */
FMPQ_API fmpq_status w4ax_gemm_asym(const fmpq_layout* layout, const void* A_packed, const void* a_scales,
                                    const void* a_zeros, const void* W_packed, const void* w_scales,
                                    const float* w_sums, int64_t M, int64_t N, void* Y, int64_t ldy,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* QoQ progressive group quantization with W4A8 GEMMs (QServe explainer, "渐进式分组量化" and
 * "运行时设计"). The layout must have every block INT8 (FMPQ_ERR_INVALID_ARG) and K_in == K.
 *
 * Offline weights: per output channel n, then per group g (the layout's 128-channel blocks):
 *   s1[n] = fp16_rn( fp32(absmax of W[n][0..K)) / 119 )           (protective range [-119, 119])
 *   q8    = clamp( rne( fp32(w) / fp32(s1) ), -119, 119 )          (IEEE division; 0 if s1 == 0)
 *   [mn, mx] = the range of the group's q8 extended to include 0
 *   s2 = max(1, ceil((mx - mn) / 15)), z2 = clamp(rne(-mn / s2), 0, 15)   (integers)
 *   q4 = clamp( rne(q8 / s2) + z2, 0, 15 )                          (exact rationals, ties to even)
 * The dequantized (q4 - z2) * s2 stays in [-127, 127].
 *   W_packed    fmpq_packed_w_bytes(layout, N): unsigned 4-bit codes (permuted order).
 *   ch_scales   fp16 [N] (s1); grp_scales, grp_zeros uint8 [K/128][N] (s2, z2). 16-byte aligned. */
FMPQ_API fmpq_status qoq_pack_weights(const fmpq_layout* layout, const void* W, int64_t ldw, int64_t N,
                                      void* W_packed, void* ch_scales, uint8_t* grp_scales, uint8_t* grp_zeros,
                                      void* stream);

/* Debug/test: decode qoq_pack_weights' codes to q4 uint8 [N][K] (permuted order). */
FMPQ_API fmpq_status qoq_unpack_weights(const fmpq_layout* layout, const void* W_packed, int64_t N, uint8_t* q4,
                                        void* stream);

/* Per-token INT8 activations: s[m] = fp16_rn( fp32(absmax of row m) / 127 ),
 * q = clamp( rne(fp32(x) / fp32(s)), -127, 127 ), every block packed as an INT8 block of
 * fmpq_quantize's format (A_packed: fmpq_packed_a_bytes); a_sums[b][m] = the sum of the
 * block's codes (the term the group zero point multiplies).
 *   a_scales  fp16 [M]; a_sums int32 [K/128][M]. 16-byte aligned. */
FMPQ_API fmpq_status qoq_quantize(const fmpq_layout* layout, const void* X, int64_t ldx, int64_t M,
                                  void* A_packed, void* a_scales, int32_t* a_sums, void* stream);

/* The W4A8 GEMM, the group zero point subtracted after the multiplication (QServe explainer,
 * "W4A8逐组快速反量化"):
 *   Y[m][n] = fp16_rn( a_scales[m] * ch_scales[n] *
 *                      sum_b grp_scales[b][n] * ( P[m][n][b] - grp_zeros[b][n] * a_sums[b][m] ) ),
 * P the exact integer sums of the INT8 activation codes times the unsigned codes q4, FP32
 * accumulation. The zero-point part, -a_scales[m] * ch_scales[n] * sum_b grp_scales[b][n] *
 * grp_zeros[b][n] * a_sums[b][m], is summed first on the tensor cores (exact integer products)
 * into the workspace and starts the accumulators. Shapes and alignment as w4ax_gemm; workspace:
 * fmpq_variant_gemm_workspace_bytes (never 0), else FMPQ_ERR_WORKSPACE. */
FMPQ_API fmpq_status qoq_gemm(const fmpq_layout* layout, const void* A_packed, const void* a_scales,
                              const int32_t* a_sums, const void* W_packed, const void* ch_scales,
                              const uint8_t* grp_scales, const uint8_t* grp_zeros, int64_t M, int64_t N, void* Y,
                              int64_t ldy, void* workspace, size_t workspace_bytes, void* stream);

/* Debug/test: P of qoq_gemm (INT8 codes times q4), as w4ax_gemm_partials. */
FMPQ_API fmpq_status qoq_gemm_partials(const fmpq_layout* layout, const void* A_packed, const void* W_packed,
                                       int64_t M, int64_t N, int64_t m0, int64_t mcount, int64_t n0,
                                       int64_t ncount, int32_t* P, void* stream);

/* Read (and, if clear != 0, reset) the layout's device status word. Synchronizes the
 * device. *code = FMPQ_OK or the first error a kernel recorded (e.g. FMPQ_ERR_TIMEOUT). */
FMPQ_API fmpq_status fmpq_device_status(const fmpq_layout* layout, int32_t* code, int32_t clear);

/* Static description of a status code. */
FMPQ_API const char* fmpq_status_string(fmpq_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
FMPQ_API int32_t fmpq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FMPQ_H */
