// C ABI of the FMPQ W4Ax library (declared in include/fmpq.h): argument validation,
// layout handles, and kernel launches on the caller's stream.
#include <cuda_runtime.h>

#include <cstdint>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/fmpq.h"
#include "fmpq_internal.h"

static_assert(FMPQ_MAX_K / FMPQ_BLOCK <= fmpq::kMaxBlocks, "kernel block tables hold every block");

namespace fmpq {

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
    struct Entry {
        const void* kernel;
        int device;
        int bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& d : done)
        if (d.kernel == kernel && d.device == dev && d.bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    for (Entry& d : done)
        if (d.kernel == kernel && d.device == dev) {
            d.bytes = bytes;
            return cudaSuccess;
        }
    done.push_back(Entry{kernel, dev, bytes});
    return cudaSuccess;
}

}  // namespace fmpq

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fmpq_status check_device(const fmpq_layout* L) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FMPQ_ERR_CUDA;
    return dev == L->device ? FMPQ_OK : FMPQ_ERR_DEVICE;
}

fmpq_status launched(cudaError_t e) { return e == cudaSuccess ? FMPQ_OK : FMPQ_ERR_CUDA; }

// Layout over K gathered channels taken from input rows of K_in >= K channels.
fmpq_status create_layout(int32_t K, int32_t K_in, const int32_t* perm_host, const uint8_t* outlier_block_mask_host,
                          fmpq_layout** out) {
    if (out == nullptr || perm_host == nullptr || outlier_block_mask_host == nullptr) return FMPQ_ERR_INVALID_ARG;
    *out = nullptr;
    if (K < FMPQ_BLOCK || K > FMPQ_MAX_K || K % FMPQ_BLOCK != 0) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (K_in < K || K_in > FMPQ_MAX_K || K_in % 8 != 0) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    const int nb = K / FMPQ_BLOCK;
    std::vector<uint8_t> seen(static_cast<size_t>(K_in), 0);
    std::vector<uint16_t> perm16(static_cast<size_t>(K));
    for (int j = 0; j < K; ++j) {
        const int32_t c = perm_host[j];
        if (c < 0 || c >= K_in || seen[c]) return FMPQ_ERR_INVALID_ARG;
        seen[c] = 1;
        perm16[j] = static_cast<uint16_t>(c);
    }
    // plane offsets: an INT4 block has one code plane, an INT8 block two
    std::vector<int32_t> poff(static_cast<size_t>(nb));
    int n8 = 0;
    int32_t planes = 0;
    for (int b = 0; b < nb; ++b) {
        const uint8_t m = outlier_block_mask_host[b];
        if (m > 1) return FMPQ_ERR_INVALID_ARG;
        poff[b] = planes;
        planes += m ? 2 : 1;
        n8 += m;
    }
    int dev = -1, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FMPQ_ERR_DEVICE;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FMPQ_ERR_DEVICE;
    if (major != 10 || minor != 3) return FMPQ_ERR_DEVICE;  // built for sm_103a only

    fmpq_layout* L = new (std::nothrow) fmpq_layout();
    if (L == nullptr) return FMPQ_ERR_INVALID_ARG;
    L->K = K;
    L->K_in = K_in;
    L->nb = nb;
    L->n8 = n8;
    L->device = dev;
    L->num_sms = sms;
    L->planes = planes;
    L->row_bytes = static_cast<int64_t>(planes) * FMPQ_BLOCK;
    for (int b = 0; b < nb; ++b)
        if (outlier_block_mask_host[b]) L->mask_bits[b >> 5] |= 1u << (b & 31);
    bool ok = cudaMalloc(&L->d_perm16, sizeof(uint16_t) * K) == cudaSuccess &&
              cudaMalloc(&L->d_mask, static_cast<size_t>(nb)) == cudaSuccess &&
              cudaMalloc(&L->d_poff, sizeof(int32_t) * nb) == cudaSuccess &&
              cudaMalloc(&L->d_status, sizeof(int32_t)) == cudaSuccess;
    ok = ok && cudaMemcpy(L->d_perm16, perm16.data(), sizeof(uint16_t) * K, cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(L->d_mask, outlier_block_mask_host, static_cast<size_t>(nb), cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(L->d_poff, poff.data(), sizeof(int32_t) * nb, cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemset(L->d_status, 0, sizeof(int32_t)) == cudaSuccess;
    if (!ok) {
        fmpq_layout_destroy(L);
        return FMPQ_ERR_CUDA;
    }
    *out = L;
    return FMPQ_OK;
}

}  // namespace

extern "C" {

fmpq_status fmpq_layout_create(int32_t K, const int32_t* perm_host, const uint8_t* outlier_block_mask_host,
                               fmpq_layout** out) {
    return create_layout(K, K, perm_host, outlier_block_mask_host, out);
}

fmpq_status fmpq_layout_create_select(int32_t K, int32_t K_in, const int32_t* select_host,
                                      const uint8_t* outlier_block_mask_host, fmpq_layout** out) {
    return create_layout(K, K_in, select_host, outlier_block_mask_host, out);
}

void fmpq_layout_destroy(fmpq_layout* L) {
    if (L == nullptr) return;
    int prev = -1;
    const bool switched = cudaGetDevice(&prev) == cudaSuccess && prev != L->device && L->device >= 0 &&
                          cudaSetDevice(L->device) == cudaSuccess;
    cudaDeviceSynchronize();
    cudaFree(L->d_perm16);
    cudaFree(L->d_mask);
    cudaFree(L->d_poff);
    cudaFree(L->d_status);
    if (switched) cudaSetDevice(prev);
    delete L;
}

int32_t fmpq_layout_k(const fmpq_layout* L) { return L ? L->K : 0; }
int32_t fmpq_layout_num_blocks(const fmpq_layout* L) { return L ? L->nb : 0; }
int32_t fmpq_layout_num_int8_blocks(const fmpq_layout* L) { return L ? L->n8 : 0; }

size_t fmpq_packed_a_bytes(const fmpq_layout* L, int64_t M) {
    if (L == nullptr || M < 0) return 0;
    return static_cast<size_t>(M) * static_cast<size_t>(L->row_bytes);
}

size_t fmpq_packed_w_bytes(const fmpq_layout* L, int64_t N) {
    if (L == nullptr || N < 0) return 0;
    const int64_t npad = (N + fmpq::kTileN - 1) / fmpq::kTileN * fmpq::kTileN;
    return static_cast<size_t>(npad) * static_cast<size_t>(L->K / 2);
}

fmpq_status fmpq_quantize(const fmpq_layout* L, const void* X, int64_t ldx, int64_t M, void* A_packed,
                          void* a_scales, void* stream) {
    if (L == nullptr || X == nullptr || A_packed == nullptr || a_scales == nullptr) return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || ldx < L->K_in) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldx % 8 != 0 || !aligned16(X) || !aligned16(A_packed) || !aligned16(a_scales)) return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    return launched(fmpq::launch_quantize(*L, X, ldx, M, A_packed, a_scales, static_cast<cudaStream_t>(stream)));
}

fmpq_status fmpq_rmsnorm_quantize(const fmpq_layout* L, const void* X, int64_t ldx, int64_t M, const void* gamma_perm,
                                  float eps, void* A_packed, void* a_scales, void* stream) {
    if (L == nullptr || X == nullptr || gamma_perm == nullptr || A_packed == nullptr || a_scales == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (!(eps > 0.0f) || !(eps < 1e30f)) return FMPQ_ERR_INVALID_ARG;   // positive and finite
    if (M < 1 || M > INT32_MAX || ldx < L->K || L->K_in != L->K) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldx % 8 != 0 || !aligned16(X) || !aligned16(gamma_perm) || !aligned16(A_packed) || !aligned16(a_scales))
        return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    return launched(fmpq::launch_quantize(*L, X, ldx, M, A_packed, a_scales, static_cast<cudaStream_t>(stream),
                                          gamma_perm, eps));
}

fmpq_status fmpq_swiglu_quantize(const fmpq_layout* L, const void* G_perm, int64_t ldg, const void* U_perm,
                                 int64_t ldu, int64_t M, void* A_packed, void* a_scales, void* stream) {
    if (L == nullptr || G_perm == nullptr || U_perm == nullptr || A_packed == nullptr || a_scales == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || ldg < L->K || ldu < L->K) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldg % 8 != 0 || ldu % 8 != 0 || !aligned16(G_perm) || !aligned16(U_perm) || !aligned16(A_packed) ||
        !aligned16(a_scales))
        return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    return launched(fmpq::launch_swiglu_quantize(*L, G_perm, ldg, U_perm, ldu, M, A_packed, a_scales,
                                                 static_cast<cudaStream_t>(stream)));
}

fmpq_status w4_pack_weights(const fmpq_layout* L, const void* W, int64_t ldw, int64_t N, void* W_packed,
                            void* w_scales, void* stream) {
    if (L == nullptr || W == nullptr || W_packed == nullptr || w_scales == nullptr) return FMPQ_ERR_INVALID_ARG;
    if (N < 16 || N % 16 != 0 || N > INT32_MAX || ldw < L->K_in) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldw % 8 != 0 || !aligned16(W) || !aligned16(W_packed) || !aligned16(w_scales)) return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    return launched(fmpq::launch_pack_weights(*L, W, ldw, N, W_packed, w_scales, static_cast<cudaStream_t>(stream)));
}

fmpq_status w4_unpack_weights(const fmpq_layout* L, const void* W_packed, int64_t N, int8_t* Wq, void* stream) {
    if (L == nullptr || W_packed == nullptr || Wq == nullptr) return FMPQ_ERR_INVALID_ARG;
    if (N < 16 || N % 16 != 0 || N > INT32_MAX) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(W_packed) || !aligned16(Wq)) return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    return launched(fmpq::launch_unpack_weights(*L, W_packed, N, Wq, static_cast<cudaStream_t>(stream)));
}

size_t w4ax_gemm_workspace_bytes(const fmpq_layout* L, int64_t M, int64_t N) {
    if (L == nullptr || M < 1 || N < 1) return 0;
    return fmpq::gemm_workspace_bytes(*L, M, N);
}

fmpq_status w4ax_gemm(const fmpq_layout* L, const void* A_packed, const void* a_scales, const void* W_packed,
                      const void* w_scales, int64_t M, int64_t N, void* Y, int64_t ldy, void* workspace,
                      size_t workspace_bytes, void* stream) {
    if (L == nullptr || A_packed == nullptr || a_scales == nullptr || W_packed == nullptr || w_scales == nullptr ||
        Y == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || N < 16 || N % 16 != 0 || N > INT32_MAX || ldy < N)
        return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldy % 8 != 0 || !aligned16(A_packed) || !aligned16(a_scales) || !aligned16(W_packed) ||
        !aligned16(w_scales) || !aligned16(Y))
        return FMPQ_ERR_MISALIGNED;
    const size_t need = fmpq::gemm_workspace_bytes(*L, M, N);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return FMPQ_ERR_WORKSPACE;
    if (need > 0 && !aligned16(workspace)) return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    fmpq::GemmArgs a{};
    a.A = A_packed;
    a.a_scales = a_scales;
    a.W = W_packed;
    a.w_scales = w_scales;
    a.M = M;
    a.N = N;
    a.Y = Y;
    a.ldy = ldy;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return launched(fmpq::launch_gemm(*L, a, static_cast<cudaStream_t>(stream)));
}

fmpq_status fmpq_quantize_gemm(const fmpq_layout* L, const void* X, int64_t ldx, int64_t M, void* A_packed,
                               void* a_scales, const void* W_packed, const void* w_scales, int64_t N, void* Y,
                               int64_t ldy, void* workspace, size_t workspace_bytes, void* stream) {
    // every argument of both steps is checked before anything is launched
    if (L == nullptr || X == nullptr || A_packed == nullptr || a_scales == nullptr || W_packed == nullptr ||
        w_scales == nullptr || Y == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || ldx < L->K_in || N < 16 || N % 16 != 0 || N > INT32_MAX || ldy < N)
        return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldx % 8 != 0 || ldy % 8 != 0 || !aligned16(X) || !aligned16(A_packed) || !aligned16(a_scales) ||
        !aligned16(W_packed) || !aligned16(w_scales) || !aligned16(Y))
        return FMPQ_ERR_MISALIGNED;
    const size_t need = fmpq::gemm_workspace_bytes(*L, M, N);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return FMPQ_ERR_WORKSPACE;
    if (need > 0 && !aligned16(workspace)) return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fmpq_status st = launched(fmpq::launch_quantize(*L, X, ldx, M, A_packed, a_scales, s))) return st;
    fmpq::GemmArgs a{};
    a.A = A_packed;
    a.a_scales = a_scales;
    a.W = W_packed;
    a.w_scales = w_scales;
    a.M = M;
    a.N = N;
    a.Y = Y;
    a.ldy = ldy;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.pdl = true;   // the quantizer just launched on this stream is the GEMM's only prerequisite
    return launched(fmpq::launch_gemm(*L, a, s));
}

fmpq_status w4ax_gemm_partials(const fmpq_layout* L, const void* A_packed, const void* W_packed, int64_t M,
                               int64_t N, int64_t m0, int64_t mcount, int64_t n0, int64_t ncount, int32_t* P,
                               void* stream) {
    if (L == nullptr || A_packed == nullptr || W_packed == nullptr || P == nullptr) return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || N < 16 || N % 16 != 0 || N > INT32_MAX) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (m0 < 0 || mcount < 1 || m0 + mcount > M || n0 < 0 || ncount < 1 || n0 + ncount > N)
        return FMPQ_ERR_INVALID_ARG;
    if (!aligned16(A_packed) || !aligned16(W_packed)) return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    fmpq::GemmArgs a{};
    a.A = A_packed;
    a.W = W_packed;
    a.M = M;
    a.N = N;
    a.P = P;
    a.pm0 = m0;
    a.pmcount = mcount;
    a.pn0 = n0;
    a.pncount = ncount;
    // scales are not used by the partial-sum export; point them at valid memory
    a.a_scales = A_packed;
    a.w_scales = W_packed;
    return launched(fmpq::launch_gemm(*L, a, static_cast<cudaStream_t>(stream)));
}

fmpq_status w4ax_gemm_fault_test(const fmpq_layout* L, const void* A_packed, const void* a_scales, const void* W_packed,
                                 const void* w_scales, int64_t M, int64_t N, void* Y, int64_t ldy, void* workspace,
                                 size_t workspace_bytes, int32_t withhold_copy, uint32_t poll_limit, void* stream) {
    if (L == nullptr || A_packed == nullptr || a_scales == nullptr || W_packed == nullptr || w_scales == nullptr ||
        Y == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || N < 16 || N % 16 != 0 || N > INT32_MAX || ldy < N)
        return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (withhold_copy < 0 || withhold_copy >= L->nb || poll_limit < 1024) return FMPQ_ERR_INVALID_ARG;
    if (ldy % 8 != 0 || !aligned16(A_packed) || !aligned16(a_scales) || !aligned16(W_packed) ||
        !aligned16(w_scales) || !aligned16(Y))
        return FMPQ_ERR_MISALIGNED;
    const size_t need = fmpq::gemm_workspace_bytes(*L, M, N);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return FMPQ_ERR_WORKSPACE;
    if (fmpq_status st = check_device(L)) return st;
    fmpq::GemmArgs a{};
    a.A = A_packed;
    a.a_scales = a_scales;
    a.W = W_packed;
    a.w_scales = w_scales;
    a.M = M;
    a.N = N;
    a.Y = Y;
    a.ldy = ldy;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.withhold = withhold_copy;
    a.poll_limit = poll_limit;
    return launched(fmpq::launch_gemm(*L, a, static_cast<cudaStream_t>(stream)));
}

// ---- quantization variants: QUIK asymmetric activations, QoQ progressive group quantization

size_t fmpq_variant_gemm_workspace_bytes(const fmpq_layout* L, int64_t M, int64_t N) {
    if (L == nullptr || M < 1 || N < 1) return 0;
    return fmpq::variant_workspace_bytes(*L, M, N);
}

fmpq_status fmpq_quantize_asym(const fmpq_layout* L, const void* X, int64_t ldx, int64_t M, void* A_packed,
                               void* a_scales, void* a_zeros, void* stream) {
    if (L == nullptr || X == nullptr || A_packed == nullptr || a_scales == nullptr || a_zeros == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (L->n8 != 0) return FMPQ_ERR_INVALID_ARG;   // every block 4-bit
    if (M < 1 || M > INT32_MAX || ldx < L->K_in) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldx % 8 != 0 || !aligned16(X) || !aligned16(A_packed) || !aligned16(a_scales) || !aligned16(a_zeros))
        return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    return launched(fmpq::launch_quantize(*L, X, ldx, M, A_packed, a_scales, static_cast<cudaStream_t>(stream),
                                          nullptr, 0.0f, fmpq::kQuantAsym, a_zeros));
}

fmpq_status w4_weight_sums(const fmpq_layout* L, const void* W_packed, const void* w_scales, int64_t N, float* w_sums,
                           void* stream) {
    if (L == nullptr || W_packed == nullptr || w_scales == nullptr || w_sums == nullptr) return FMPQ_ERR_INVALID_ARG;
    if (N < 16 || N % 16 != 0 || N > INT32_MAX) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(W_packed) || !aligned16(w_scales) || !aligned16(w_sums)) return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    return launched(fmpq::launch_weight_sums(*L, W_packed, w_scales, N, w_sums, static_cast<cudaStream_t>(stream)));
}

fmpq_status w4ax_gemm_asym(const fmpq_layout* L, const void* A_packed, const void* a_scales, const void* a_zeros,
                           const void* W_packed, const void* w_scales, const float* w_sums, int64_t M, int64_t N,
                           void* Y, int64_t ldy, void* workspace, size_t workspace_bytes, void* stream) {
    if (L == nullptr || A_packed == nullptr || a_scales == nullptr || a_zeros == nullptr || W_packed == nullptr ||
        w_scales == nullptr || w_sums == nullptr || Y == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (L->n8 != 0) return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || N < 16 || N % 16 != 0 || N > INT32_MAX || ldy < N)
        return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldy % 8 != 0 || !aligned16(A_packed) || !aligned16(a_scales) || !aligned16(a_zeros) || !aligned16(W_packed) ||
        !aligned16(w_scales) || !aligned16(w_sums) || !aligned16(Y))
        return FMPQ_ERR_MISALIGNED;
    const size_t need = fmpq::variant_workspace_bytes(*L, M, N);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return FMPQ_ERR_WORKSPACE;
    if (need > 0 && !aligned16(workspace)) return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    fmpq::GemmArgs a{};
    a.A = A_packed;
    a.a_scales = a_scales;
    a.W = W_packed;
    a.w_scales = w_scales;
    a.M = M;
    a.N = N;
    a.Y = Y;
    a.ldy = ldy;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.zero_kind = fmpq::kZeroQuik;
    a.a_zeros = a_zeros;
    a.w_sums = w_sums;
    return launched(fmpq::launch_gemm(*L, a, static_cast<cudaStream_t>(stream)));
}

fmpq_status qoq_pack_weights(const fmpq_layout* L, const void* W, int64_t ldw, int64_t N, void* W_packed,
                             void* ch_scales, uint8_t* grp_scales, uint8_t* grp_zeros, void* stream) {
    if (L == nullptr || W == nullptr || W_packed == nullptr || ch_scales == nullptr || grp_scales == nullptr ||
        grp_zeros == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (N < 16 || N % 16 != 0 || N > INT32_MAX || ldw < L->K || L->K_in != L->K) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldw % 8 != 0 || !aligned16(W) || !aligned16(W_packed) || !aligned16(ch_scales) || !aligned16(grp_scales) ||
        !aligned16(grp_zeros))
        return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    return launched(fmpq::launch_qoq_pack_weights(*L, W, ldw, N, W_packed, ch_scales, grp_scales, grp_zeros,
                                                  static_cast<cudaStream_t>(stream)));
}

fmpq_status qoq_unpack_weights(const fmpq_layout* L, const void* W_packed, int64_t N, uint8_t* q4, void* stream) {
    if (L == nullptr || W_packed == nullptr || q4 == nullptr) return FMPQ_ERR_INVALID_ARG;
    if (N < 16 || N % 16 != 0 || N > INT32_MAX) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(W_packed) || !aligned16(q4)) return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    return launched(fmpq::launch_unpack_weights(*L, W_packed, N, reinterpret_cast<int8_t*>(q4),
                                                static_cast<cudaStream_t>(stream), true));
}

fmpq_status qoq_quantize(const fmpq_layout* L, const void* X, int64_t ldx, int64_t M, void* A_packed, void* a_scales,
                         int32_t* a_sums, void* stream) {
    if (L == nullptr || X == nullptr || A_packed == nullptr || a_scales == nullptr || a_sums == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (L->n8 != L->nb) return FMPQ_ERR_INVALID_ARG;   // every block INT8
    if (M < 1 || M > INT32_MAX || ldx < L->K || L->K_in != L->K) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldx % 8 != 0 || !aligned16(X) || !aligned16(A_packed) || !aligned16(a_scales) || !aligned16(a_sums))
        return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    return launched(fmpq::launch_quantize(*L, X, ldx, M, A_packed, a_scales, static_cast<cudaStream_t>(stream),
                                          nullptr, 0.0f, fmpq::kQuantTok, a_sums));
}

fmpq_status qoq_gemm(const fmpq_layout* L, const void* A_packed, const void* a_scales, const int32_t* a_sums,
                     const void* W_packed, const void* ch_scales, const uint8_t* grp_scales, const uint8_t* grp_zeros,
                     int64_t M, int64_t N, void* Y, int64_t ldy, void* workspace, size_t workspace_bytes,
                     void* stream) {
    if (L == nullptr || A_packed == nullptr || a_scales == nullptr || a_sums == nullptr || W_packed == nullptr ||
        ch_scales == nullptr || grp_scales == nullptr || grp_zeros == nullptr || Y == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (L->n8 != L->nb) return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || N < 16 || N % 16 != 0 || N > INT32_MAX || ldy < N)
        return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldy % 8 != 0 || !aligned16(A_packed) || !aligned16(a_scales) || !aligned16(a_sums) || !aligned16(W_packed) ||
        !aligned16(ch_scales) || !aligned16(grp_scales) || !aligned16(grp_zeros) || !aligned16(Y))
        return FMPQ_ERR_MISALIGNED;
    const size_t need = fmpq::variant_workspace_bytes(*L, M, N);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return FMPQ_ERR_WORKSPACE;
    if (need > 0 && !aligned16(workspace)) return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    fmpq::GemmArgs a{};
    a.A = A_packed;
    a.a_scales = a_scales;
    a.W = W_packed;
    a.w_scales = ch_scales;   // not read by the QoQ path; a valid pointer
    a.M = M;
    a.N = N;
    a.Y = Y;
    a.ldy = ldy;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.zero_kind = fmpq::kZeroQoq;
    a.unsigned_w = true;
    a.a_sums = a_sums;
    a.ch_scales = ch_scales;
    a.grp_scales = grp_scales;
    a.grp_zeros = grp_zeros;
    return launched(fmpq::launch_gemm(*L, a, static_cast<cudaStream_t>(stream)));
}

fmpq_status qoq_gemm_partials(const fmpq_layout* L, const void* A_packed, const void* W_packed, int64_t M, int64_t N,
                              int64_t m0, int64_t mcount, int64_t n0, int64_t ncount, int32_t* P, void* stream) {
    if (L == nullptr || A_packed == nullptr || W_packed == nullptr || P == nullptr) return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || N < 16 || N % 16 != 0 || N > INT32_MAX) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (m0 < 0 || mcount < 1 || m0 + mcount > M || n0 < 0 || ncount < 1 || n0 + ncount > N)
        return FMPQ_ERR_INVALID_ARG;
    if (!aligned16(A_packed) || !aligned16(W_packed)) return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    fmpq::GemmArgs a{};
    a.A = A_packed;
    a.W = W_packed;
    a.M = M;
    a.N = N;
    a.P = P;
    a.pm0 = m0;
    a.pmcount = mcount;
    a.pn0 = n0;
    a.pncount = ncount;
    a.unsigned_w = true;
    a.a_scales = A_packed;   // scales are not read by the partial-sum export
    a.w_scales = W_packed;
    return launched(fmpq::launch_gemm(*L, a, static_cast<cudaStream_t>(stream)));
}

fmpq_status fmpq_channel_absmax(const void* X, int64_t ldx, int64_t T, int32_t K, uint32_t* absmax, void* stream) {
    if (X == nullptr || absmax == nullptr) return FMPQ_ERR_INVALID_ARG;
    if (K < FMPQ_BLOCK || K > FMPQ_MAX_K || K % FMPQ_BLOCK != 0 || T < 1 || ldx < K) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldx % 8 != 0 || !aligned16(X) || !aligned16(absmax)) return FMPQ_ERR_MISALIGNED;
    int dev = -1, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FMPQ_ERR_DEVICE;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FMPQ_ERR_DEVICE;
    if (major != 10 || minor != 3) return FMPQ_ERR_DEVICE;
    return launched(fmpq::launch_channel_absmax(X, ldx, T, K, absmax, sms, static_cast<cudaStream_t>(stream)));
}

fmpq_status fmpq_outlier_gemm_fp16(const fmpq_layout* L, const void* X, int64_t ldx, int64_t M, const int32_t* cols,
                                   int32_t n_out, const void* W_out, int64_t ldw_out, int64_t N, void* X_out, void* Y,
                                   int64_t ldy, void* stream) {
    if (L == nullptr || X == nullptr || cols == nullptr || W_out == nullptr || X_out == nullptr || Y == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || n_out < 8 || n_out % 8 != 0 || n_out > FMPQ_MAX_K || N < 1 ||
        N > 65535ll * 128 || ldx < 1 || ldw_out < n_out || ldy < N || ldw_out > INT32_MAX || ldy > INT32_MAX)
        return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldx % 8 != 0 || ldw_out % 8 != 0 || ldy % 8 != 0 || !aligned16(X) || !aligned16(cols) || !aligned16(W_out) ||
        !aligned16(X_out) || !aligned16(Y))
        return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    bool maps_ok = true;
    const cudaError_t e = fmpq::launch_outlier_gemm(X, ldx, M, cols, n_out, W_out, ldw_out, N, X_out, Y, ldy,
                                                    L->num_sms, L->d_status, static_cast<cudaStream_t>(stream),
                                                    &maps_ok);
    return (e == cudaSuccess && maps_ok) ? FMPQ_OK : FMPQ_ERR_CUDA;
}

fmpq_status fmpq_quantize_split(const fmpq_layout* L, const void* X, int64_t ldx, int64_t M, const int32_t* cols,
                                int32_t n_out, int32_t asym, void* A_packed, void* a_scales, void* a_zeros,
                                void* X_out, void* stream) {
    if (L == nullptr || X == nullptr || cols == nullptr || A_packed == nullptr || a_scales == nullptr ||
        X_out == nullptr || (asym != 0 && a_zeros == nullptr) || (asym != 0 && asym != 1))
        return FMPQ_ERR_INVALID_ARG;
    if (asym != 0 && L->n8 != 0) return FMPQ_ERR_INVALID_ARG;   // asymmetric: every block 4-bit
    if (M < 1 || M > INT32_MAX || ldx < L->K_in || n_out < 8 || n_out % 8 != 0 || n_out > FMPQ_MAX_K)
        return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldx % 8 != 0 || !aligned16(X) || !aligned16(A_packed) || !aligned16(a_scales) || !aligned16(cols) ||
        !aligned16(X_out) || (asym != 0 && !aligned16(a_zeros)))
        return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    const fmpq::QuantSplit split{cols, n_out, X_out};
    return launched(fmpq::launch_quantize(*L, X, ldx, M, A_packed, a_scales, static_cast<cudaStream_t>(stream),
                                          nullptr, 0.0f, asym ? fmpq::kQuantAsym : fmpq::kQuantSym,
                                          asym ? a_zeros : nullptr, &split));
}

fmpq_status fmpq_outlier_product_fp16(const fmpq_layout* L, const void* X_out, int64_t M, int32_t n_out,
                                      const void* W_out, int64_t ldw_out, int64_t N, void* Y, int64_t ldy,
                                      void* stream) {
    if (L == nullptr || X_out == nullptr || W_out == nullptr || Y == nullptr) return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || n_out < 8 || n_out % 8 != 0 || n_out > FMPQ_MAX_K || N < 1 ||
        N > 65535ll * 128 || ldw_out < n_out || ldy < N || ldw_out > INT32_MAX || ldy > INT32_MAX)
        return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldw_out % 8 != 0 || ldy % 8 != 0 || !aligned16(W_out) || !aligned16(X_out) || !aligned16(Y))
        return FMPQ_ERR_MISALIGNED;
    if (fmpq_status st = check_device(L)) return st;
    bool maps_ok = true;
    const cudaError_t e = fmpq::launch_outlier_gemm(nullptr, 0, M, nullptr, n_out, W_out, ldw_out, N,
                                                    const_cast<void*>(X_out), Y, ldy, L->num_sms, L->d_status,
                                                    static_cast<cudaStream_t>(stream), &maps_ok);
    return (e == cudaSuccess && maps_ok) ? FMPQ_OK : FMPQ_ERR_CUDA;
}

fmpq_status fmpq_plan_layout(int32_t K, const uint32_t* absmax_host, int32_t n8, int32_t* perm_host,
                             uint8_t* mask_host) {
    if (absmax_host == nullptr || perm_host == nullptr || mask_host == nullptr) return FMPQ_ERR_INVALID_ARG;
    if (K < FMPQ_BLOCK || K > FMPQ_MAX_K || K % FMPQ_BLOCK != 0) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (n8 < 0 || n8 > K / FMPQ_BLOCK) return FMPQ_ERR_INVALID_ARG;
    try {
        fmpq::plan_layout(K, absmax_host, n8, perm_host, mask_host);
    } catch (const std::bad_alloc&) {
        return FMPQ_ERR_INVALID_ARG;
    }
    return FMPQ_OK;
}

fmpq_status fmpq_plan_layout_budget(int32_t K, const uint32_t* absmax_host, const void* X_calib_host, int64_t T,
                                    int64_t ldx, double eps, int32_t* n8_out, double* err_out, int32_t* perm_host,
                                    uint8_t* mask_host) {
    if (absmax_host == nullptr || X_calib_host == nullptr || n8_out == nullptr || err_out == nullptr ||
        perm_host == nullptr || mask_host == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (K < FMPQ_BLOCK || K > FMPQ_MAX_K || K % FMPQ_BLOCK != 0 || T < 1 || ldx < K) return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (!(eps >= 0.0) || !std::isfinite(eps)) return FMPQ_ERR_INVALID_ARG;
    try {
        *n8_out = fmpq::plan_layout_budget(K, absmax_host, static_cast<const uint16_t*>(X_calib_host), T, ldx, eps,
                                           err_out, perm_host, mask_host);
    } catch (const std::bad_alloc&) {
        return FMPQ_ERR_INVALID_ARG;
    }
    return FMPQ_OK;
}

int32_t fmpq_outlier_blocks(int32_t K, double fraction) {
    if (K < FMPQ_BLOCK || K > FMPQ_MAX_K || K % FMPQ_BLOCK != 0 || !(fraction >= 0.0 && fraction <= 1.0)) return -1;
    const long long n_out = std::llround(fraction * K);
    const long long n8 = (n_out + FMPQ_BLOCK - 1) / FMPQ_BLOCK;
    return static_cast<int32_t>(n8 < K / FMPQ_BLOCK ? n8 : K / FMPQ_BLOCK);
}

fmpq_status fmpq_device_status(const fmpq_layout* L, int32_t* code, int32_t clear) {
    if (L == nullptr || code == nullptr) return FMPQ_ERR_INVALID_ARG;
    if (fmpq_status st = check_device(L)) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return FMPQ_ERR_CUDA;
    if (cudaMemcpy(code, L->d_status, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return FMPQ_ERR_CUDA;
    if (clear && cudaMemset(L->d_status, 0, sizeof(int32_t)) != cudaSuccess) return FMPQ_ERR_CUDA;
    return FMPQ_OK;
}

const char* fmpq_status_string(fmpq_status s) {
    switch (s) {
        case FMPQ_OK: return "ok";
        case FMPQ_ERR_INVALID_ARG: return "invalid argument";
        case FMPQ_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case FMPQ_ERR_MISALIGNED: return "misaligned pointer or leading dimension";
        case FMPQ_ERR_CUDA: return "CUDA error";
        case FMPQ_ERR_TIMEOUT: return "device wait timed out";
        case FMPQ_ERR_DEVICE: return "unsupported or wrong device";
        case FMPQ_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

int32_t fmpq_version(void) { return 100; }

}  // extern "C"
