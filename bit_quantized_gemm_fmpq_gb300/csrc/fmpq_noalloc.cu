// w4ax_gemm_noalloc: the W4Ax GEMM for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all. Examples: code running inside a memory pool
// that owns every byte of the device, code paths that must not allocate in the middle of
// serving traffic, and hosts whose allocator is not reachable from this library. For
// shapes with few output tiles the GEMM splits K across CTAs and needs a workspace
// (w4ax_gemm_workspace_bytes). Here that workspace lives in a fixed array inside the
// library instead of a caller buffer.
//
// The array is a file-scope device variable of kScratchBytes + kCounterBytes bytes; every
// GPU that loads the library keeps it until the process exits. Host code only holds a
// stand-in for it, not a device address, so the address is looked up once per device
// with cudaGetSymbolAddress (with that device current) and cached.
//
// The split-K kernel needs its per-tile arrival counters at zero when it starts. A call that
// completes leaves them at zero, but one that gave up on a device-side wait (FMPQ_ERR_TIMEOUT)
// may not, so every call clears the counters it will use with a cudaMemsetAsync on the
// caller's stream (no allocation) before the launch.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fmpq.h"
#include "fmpq_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(20) << 20;  // split-K partial tiles (FP32)
constexpr size_t kCounterBytes = size_t(64) << 10;  // per-tile arrival counters (int32)
constexpr int kMaxDevices = 64;

// Partial tiles occupy [kScratchBytes - used, kScratchBytes); the counters always start at
// kScratchBytes, so they never overlap partials written by a call with another shape.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes + kCounterBytes];

std::mutex g_mutex;
unsigned char* g_base[kMaxDevices] = {};

// Device address of the scratch array on `dev` (which must be current). The first call on
// a device looks it up (host-side work only: no device work, no allocation).
fmpq_status scratch_base(int dev, unsigned char** out) {
    if (dev < 0 || dev >= kMaxDevices) return FMPQ_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_base[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return FMPQ_ERR_CUDA;
        }
        g_base[dev] = static_cast<unsigned char*>(ptr);
    }
    *out = g_base[dev];
    return FMPQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

fmpq_status w4ax_gemm_noalloc(const fmpq_layout* L, const void* A_packed, const void* a_scales,
                              const void* W_packed, const void* w_scales, int64_t M, int64_t N, void* Y,
                              int64_t ldy, void* stream) {
    if (L == nullptr || A_packed == nullptr || a_scales == nullptr || W_packed == nullptr || w_scales == nullptr ||
        Y == nullptr)
        return FMPQ_ERR_INVALID_ARG;
    if (M < 1 || M > INT32_MAX || N < 16 || N % 16 != 0 || N > INT32_MAX || ldy < N)
        return FMPQ_ERR_UNSUPPORTED_SHAPE;
    if (ldy % 8 != 0 || !aligned16(A_packed) || !aligned16(a_scales) || !aligned16(W_packed) ||
        !aligned16(w_scales) || !aligned16(Y))
        return FMPQ_ERR_MISALIGNED;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FMPQ_ERR_CUDA;
    if (dev != L->device) return FMPQ_ERR_DEVICE;

    fmpq::GemmArgs a{};
    a.A = A_packed;
    a.a_scales = a_scales;
    a.W = W_packed;
    a.w_scales = w_scales;
    a.M = M;
    a.N = N;
    a.Y = Y;
    a.ldy = ldy;
    const size_t need = fmpq::gemm_workspace_bytes(*L, M, N);
    if (need > 0) {
        const size_t counters = fmpq::gemm_counter_bytes(*L, M, N);
        if (need < counters) return FMPQ_ERR_WORKSPACE;
        const size_t partials = need - counters;
        if (partials > kScratchBytes || counters > kCounterBytes) return FMPQ_ERR_WORKSPACE;  // shape too large
        unsigned char* base = nullptr;
        if (fmpq_status st = scratch_base(dev, &base)) return st;
        // the launcher places the counters right after the partials: end the partials at
        // kScratchBytes so the counters land at the fixed counter region
        a.workspace = base + (kScratchBytes - partials);
        a.workspace_bytes = need;
        // counters start at zero even after an earlier call that gave up on a device wait
        if (cudaMemsetAsync(base + kScratchBytes, 0, counters, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return FMPQ_ERR_CUDA;
    }
    return fmpq::launch_gemm(*L, a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FMPQ_OK : FMPQ_ERR_CUDA;
}

}  // extern "C"
