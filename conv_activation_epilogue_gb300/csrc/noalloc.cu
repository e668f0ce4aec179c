// noalloc.cu -- the two-kernel GEMM path for callers that cannot allocate
// device memory when they call us.
//
// mmact_gemm_split needs an fp32 workspace of M*N elements between its two
// kernels, and expects the caller to provide it.  Some callers have no way to
// do that at call time: a plugin that is handed only its input and output
// buffers by a host framework, a framework whose caching allocator already
// owns the whole device budget, or a latency-critical loop where cudaMalloc /
// cudaFree may block or synchronise the device and stall unrelated streams.
// mmact_gemm_split_noalloc serves them from a fixed scratch array that lives
// in this library's own device image: it calls no cudaMalloc, cudaFree or any
// other allocating routine.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library reserves MMACT_NOALLOC_MAX_ELEMENTS * 4 bytes (16 MiB) until the
// process exits.  Host code cannot use the symbol itself as a device
// address (on the host it names a shadow variable), so the first call on each
// device asks the runtime for the array's device address with
// cudaGetSymbolAddress, with that device current, and caches it.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "mmact.h"

#define MMACT_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

static __device__ __align__(256) float g_noalloc_scratch[MMACT_NOALLOC_MAX_ELEMENTS];

constexpr int MAX_DEVICES = 64;
float *g_scratch_ptr[MAX_DEVICES] = {};
std::mutex g_scratch_mutex;

// Device address of this device's scratch array (looked up once per device).
mmact_status scratch_address(float **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return MMACT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MMACT_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_scratch_ptr[dev];
    return MMACT_OK;
}

}  // namespace

MMACT_EXPORT mmact_status mmact_gemm_split_noalloc(const void *A, const void *B, const float *bias,
                                                   void *C, int64_t M, int64_t N, int64_t K,
                                                   mmact_dtype ab_dtype, mmact_dtype c_dtype,
                                                   mmact_act act, float alpha, void *stream)
{
    const int64_t max_dim = (int64_t(1) << 31) - 1;
    if (M < 0 || N < 0 || M > max_dim || N > max_dim) return MMACT_ERR_INVALID_ARG;
    if (M * N > (int64_t)MMACT_NOALLOC_MAX_ELEMENTS) return MMACT_ERR_UNSUPPORTED;
    float *ws = nullptr;
    const mmact_status s = scratch_address(&ws);
    if (s != MMACT_OK) return s;
    // The first kernel overwrites all M*N workspace elements before the
    // second reads them, so nothing left by an earlier call is ever read.
    return mmact_gemm_split(A, B, bias, C, M, N, K, ab_dtype, c_dtype, act, alpha, ws, stream);
}
