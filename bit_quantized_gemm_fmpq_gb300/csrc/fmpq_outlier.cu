// The FP16 outlier path of an outlier split (QUIK explainer, "第二步: 前向传播"): the input's
// outlier columns are multiplied in FP16 by the unquantized outlier weights and the result is
// added to the output of the INT4 path (the base columns, fmpq_layout_create_select +
// w4ax_gemm).
//
//   outlier_gather_kernel  X[:, cols] -> a dense fp16 [M][n_out] operand (one element per thread)
//   the product            a plain FP16 GEMM from cuBLAS (FP32 accumulation, beta = 1 adds it to Y),
//                          loaded at run time on the first call, so that the library neither links
//                          nor needs cuBLAS for anything else; one handle per device with a fixed
//                          device workspace (no allocation per call).
#include <cublas_v2.h>
#include <cuda_runtime.h>
#include <dlfcn.h>

#include <cstdint>
#include <mutex>

#include "../../include/fmpq.h"
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

constexpr size_t kCublasWorkspace = size_t(4) << 20;
__device__ __align__(256) unsigned char g_cublas_ws[kCublasWorkspace];

// The exported C entry point cublasGemmEx (the C++ header also overloads the name).
using GemmExFn = cublasStatus_t (*)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int, const void*,
                                    const void*, cudaDataType, int, const void*, cudaDataType, int, const void*, void*,
                                    cudaDataType, int, cublasComputeType_t, cublasGemmAlgo_t);

struct CublasApi {
    decltype(&cublasCreate_v2) create = nullptr;
    decltype(&cublasSetStream_v2) set_stream = nullptr;
    decltype(&cublasSetWorkspace_v2) set_workspace = nullptr;
    GemmExFn gemm_ex = nullptr;
};

std::mutex g_mu;
CublasApi g_api;
bool g_api_tried = false;
cublasHandle_t g_handle[64] = {};

bool load_api() {
    if (g_api_tried) return g_api.gemm_ex != nullptr;
    g_api_tried = true;
    void* h = dlopen("libcublas.so.13", RTLD_NOW | RTLD_LOCAL);
    if (h == nullptr) h = dlopen("libcublas.so", RTLD_NOW | RTLD_LOCAL);
    if (h == nullptr) return false;
    g_api.create = reinterpret_cast<decltype(&cublasCreate_v2)>(dlsym(h, "cublasCreate_v2"));
    g_api.set_stream = reinterpret_cast<decltype(&cublasSetStream_v2)>(dlsym(h, "cublasSetStream_v2"));
    g_api.set_workspace = reinterpret_cast<decltype(&cublasSetWorkspace_v2)>(dlsym(h, "cublasSetWorkspace_v2"));
    g_api.gemm_ex = reinterpret_cast<GemmExFn>(dlsym(h, "cublasGemmEx"));
    if (!g_api.create || !g_api.set_stream || !g_api.set_workspace || !g_api.gemm_ex) {
        g_api.gemm_ex = nullptr;
        return false;
    }
    return true;
}

// The device's handle, created (once) with the fixed workspace.
cublasHandle_t handle_for(int dev) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (dev < 0 || dev >= 64 || !load_api()) return nullptr;
    if (g_handle[dev] != nullptr) return g_handle[dev];
    cublasHandle_t h = nullptr;
    if (g_api.create(&h) != CUBLAS_STATUS_SUCCESS) return nullptr;
    void* ws = nullptr;
    if (cudaGetSymbolAddress(&ws, g_cublas_ws) != cudaSuccess ||
        g_api.set_workspace(h, ws, kCublasWorkspace) != CUBLAS_STATUS_SUCCESS) {
        cudaGetLastError();
        return nullptr;
    }
    g_handle[dev] = h;
    return h;
}

}  // namespace

cudaError_t launch_outlier_gemm(const void* X, int64_t ldx, int64_t M, const int32_t* cols, int n_out,
                                const void* W_out, int64_t ldw_out, int64_t N, void* X_out, void* Y, int64_t ldy,
                                cudaStream_t stream, bool* cublas_ok) {
    *cublas_ok = true;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cublasHandle_t h = handle_for(dev);
    if (h == nullptr) {
        *cublas_ok = false;
        return cudaSuccess;
    }
    const unsigned gy = static_cast<unsigned>(M < 65535 ? M : 65535);
    outlier_gather_kernel<<<dim3(static_cast<unsigned>((n_out + 255) / 256), gy), 256, 0, stream>>>(
        static_cast<const uint16_t*>(X), ldx, M, cols, n_out, static_cast<uint16_t*>(X_out));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // Column-major view: Y^T (N x M, ld ldy) += W_out^T-as-stored (n_out x N, ld ldw_out)^T * X_out^T (n_out x M)
    const float one = 1.0f;
    std::lock_guard<std::mutex> lock(g_mu);   // the handle is shared by the device's callers
    if (g_api.set_stream(h, stream) != CUBLAS_STATUS_SUCCESS ||
        g_api.gemm_ex(h, CUBLAS_OP_T, CUBLAS_OP_N, static_cast<int>(N), static_cast<int>(M), n_out, &one, W_out,
                      CUDA_R_16F, static_cast<int>(ldw_out), X_out, CUDA_R_16F, n_out, &one, Y, CUDA_R_16F,
                      static_cast<int>(ldy), CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS) {
        *cublas_ok = false;
    }
    return cudaGetLastError();
}

}  // namespace fmpq
