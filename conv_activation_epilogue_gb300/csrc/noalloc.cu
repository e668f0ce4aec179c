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
// cudaGetSymbolAddress, with that device current, and caches it.  The cache
// entry is tied to the CUDA context it was looked up in (by the context's
// process-unique id): after cudaDeviceReset the next call finds a new context
// and looks the address up again instead of reusing a stale one.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "mmact.h"

#define MMACT_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

static __device__ __align__(256) float g_noalloc_scratch[MMACT_NOALLOC_MAX_ELEMENTS];

constexpr int MAX_DEVICES = 64;
struct ScratchEntry {
    unsigned long long ctx_id = 0;   // id of the context the address belongs to (0: none yet)
    float *ptr = nullptr;
};
ScratchEntry g_scratch[MAX_DEVICES];
std::mutex g_scratch_mutex;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

template <typename Fn>
bool driver_entry(const char *name, Fn *out)
{
    if (*out != nullptr) return true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    *out = reinterpret_cast<Fn>(fn);
    return true;
}

// Device address of the current device's scratch array in the current
// context: looked up once per device and context, under a lock.
mmact_status scratch_address(float **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return MMACT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!driver_entry("cuCtxGetCurrent", &g_ctx_get_current) || !driver_entry("cuCtxGetId", &g_ctx_get_id))
        return MMACT_ERR_CUDA;
    // id of the current context, 0 when the runtime has not made one current yet
    auto current_id = [](unsigned long long *id) {
        CUcontext ctx = nullptr;
        *id = 0;
        if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return false;
        return ctx == nullptr || g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
    };
    unsigned long long id = 0;
    if (!current_id(&id)) return MMACT_ERR_CUDA;
    ScratchEntry &e = g_scratch[dev];
    if (id == 0 || e.ptr == nullptr || e.ctx_id != id) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MMACT_ERR_CUDA;
        if (!current_id(&id) || id == 0) return MMACT_ERR_CUDA;   // the lookup made the context current
        e.ptr = static_cast<float *>(p);
        e.ctx_id = id;
    }
    *out = e.ptr;
    return MMACT_OK;
}

}  // namespace

MMACT_EXPORT mmact_status mmact_gemm_split_noalloc(const void *A, const void *B, const float *bias,
                                                   void *C, int64_t M, int64_t N, int64_t K,
                                                   mmact_dtype ab_dtype, mmact_dtype c_dtype,
                                                   mmact_act act, float alpha, void *stream)
{
    // the same argument checks as mmact_gemm_split, before anything else
    mmact_status s = mmact::gemm_check(A, B, bias, C, M, N, K, ab_dtype, c_dtype, act);
    if (s != MMACT_OK) return s;
    if (M * N > (int64_t)MMACT_NOALLOC_MAX_ELEMENTS) return MMACT_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return MMACT_OK;
    float *ws = nullptr;
    s = scratch_address(&ws);
    if (s != MMACT_OK) return s;
    // The first kernel overwrites all M*N workspace elements before the
    // second reads them, so nothing left by an earlier call is ever read.
    return mmact_gemm_split(A, B, bias, C, M, N, K, ab_dtype, c_dtype, act, alpha, ws, stream);
}
