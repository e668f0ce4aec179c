// elementwise.cu -- the HBM-bound kernels: the second kernel of the two-kernel
// ablation (fp32 workspace -> activation -> output dtype), the degenerate
// empty-contraction case (output = act(bias), plus the residual when one is
// given), and the bounded-wait self-test.
//
// The ablation follows the "multimodal-ops Fused ConvTanh" article, section
// on how the two kernels split the work: its second kernel reads the fp32
// workspace back from HBM, runs the activation entirely in fp32, casts last
// and writes the output contiguously.  Here the workspace is already in the
// output's element order (row-major [M,N] for GEMM, NCHW for conv), so the
// pass is a straight streaming map: 32 bytes read and 16 (or 32) bytes
// written per thread and iteration, grid-stride over the tensor.
#include "common.cuh"
#include "kernels.h"

namespace mmact {

template <int OUT, int ACT>
__global__ void __launch_bounds__(256) act_kernel(const float *__restrict__ ws, void *__restrict__ out,
                                                  int64_t count, float alpha)
{
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the workspace is the previous kernel's output
    const int64_t n8 = count >> 3;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const float4 *src = reinterpret_cast<const float4 *>(ws);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const float4 a = __ldcs(src + 2 * i);
        const float4 b = __ldcs(src + 2 * i + 1);
        float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = act_f32<ACT>(v[e], alpha);
        if constexpr (OUT == OUT_F32) {
            float4 *dst = reinterpret_cast<float4 *>(out) + 2 * i;
            __stcs(dst, make_float4(v[0], v[1], v[2], v[3]));
            __stcs(dst + 1, make_float4(v[4], v[5], v[6], v[7]));
        } else {
            uint4 w;
            w.x = pack2<OUT>(v[0], v[1]);
            w.y = pack2<OUT>(v[2], v[3]);
            w.z = pack2<OUT>(v[4], v[5]);
            w.w = pack2<OUT>(v[6], v[7]);
            __stcs(reinterpret_cast<uint4 *>(out) + i, w);
        }
    }
    // ragged tail (count % 8 elements), one thread each
    if (blockIdx.x == 0 && threadIdx.x < (count & 7)) {
        const int64_t k = (n8 << 3) + threadIdx.x;
        const float v = act_f32<ACT>(ws[k], alpha);
        if constexpr (OUT == OUT_F32) reinterpret_cast<float *>(out)[k] = v;
        else if constexpr (OUT == OUT_BF16) reinterpret_cast<__nv_bfloat16 *>(out)[k] = __float2bfloat16_rn(v);
        else reinterpret_cast<__half *>(out)[k] = __float2half_rn(v);
    }
}

template <int OUT>
__device__ __forceinline__ float load_out(const void *p, int64_t k)
{
    if constexpr (OUT == OUT_F32) return static_cast<const float *>(p)[k];
    else if constexpr (OUT == OUT_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[k]);
    else return __half2float(static_cast<const __half *>(p)[k]);
}

template <int OUT, int ACT>
__global__ void __launch_bounds__(256) bias_act_kernel(const float *__restrict__ bias,
                                                       void *out, int64_t rows,
                                                       int64_t cols, int per_row, int64_t bias_len,
                                                       float alpha, const void *res)
{
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    const int64_t total = rows * cols;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total; k += stride) {
        const int64_t r = k / cols, c = k - r * cols;
        float b = bias == nullptr ? 0.0f : bias[per_row ? (r % bias_len) : c];
        if (res != nullptr) b += load_out<OUT>(res, k);   // may alias out: read before the write
        const float v = act_f32<ACT>(b, alpha);
        if constexpr (OUT == OUT_F32) reinterpret_cast<float *>(out)[k] = v;
        else if constexpr (OUT == OUT_BF16) reinterpret_cast<__nv_bfloat16 *>(out)[k] = __float2bfloat16_rn(v);
        else reinterpret_cast<__half *>(out)[k] = __float2half_rn(v);
    }
}

// Waits on an mbarrier that nothing arrives at; the bounded wait must give up
// and record the timeout in the status word.
__global__ void wait_selftest_kernel(unsigned int *status, unsigned long long timeout_ns)
{
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    const uint32_t b = ptx::smem_addr(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    ptx::cta_sync();
    if (threadIdx.x == 0) {
        if (!ptx::mbar_wait_bounded(b, 0, timeout_ns, &abort_flag)) atomicOr(status, ST_TIMEOUT);
    }
}

template <int OUT>
static cudaError_t launch_act_o(const float *ws, void *out, int64_t count, int act, float alpha,
                                int grid, cudaStream_t s)
{
    switch (act) {
    case ACT_RELU: return launch_k(act_kernel<OUT, ACT_RELU>, grid, 256, 0, s, ws, out, count, alpha);
    case ACT_LEAKY: return launch_k(act_kernel<OUT, ACT_LEAKY>, grid, 256, 0, s, ws, out, count, alpha);
    case ACT_TANH: return launch_k(act_kernel<OUT, ACT_TANH>, grid, 256, 0, s, ws, out, count, alpha);
    case ACT_SIGMOID: return launch_k(act_kernel<OUT, ACT_SIGMOID>, grid, 256, 0, s, ws, out, count, alpha);
    case ACT_GELU: return launch_k(act_kernel<OUT, ACT_GELU>, grid, 256, 0, s, ws, out, count, alpha);
    default: return launch_k(act_kernel<OUT, ACT_NONE>, grid, 256, 0, s, ws, out, count, alpha);
    }
}

cudaError_t launch_act(const float *ws, void *out, int64_t count, int out_kind, int act, float alpha,
                       int grid, cudaStream_t stream)
{
    if (count <= 0) return cudaSuccess;
    if (out_kind == OUT_BF16) return launch_act_o<OUT_BF16>(ws, out, count, act, alpha, grid, stream);
    if (out_kind == OUT_F16) return launch_act_o<OUT_F16>(ws, out, count, act, alpha, grid, stream);
    return launch_act_o<OUT_F32>(ws, out, count, act, alpha, grid, stream);
}

template <int OUT>
static cudaError_t launch_bias_act_o(const float *bias, void *out, int64_t rows, int64_t cols,
                                     int per_row, int64_t bias_len, int act, float alpha,
                                     cudaStream_t s, const void *res)
{
    const int64_t total = rows * cols;
    const int grid = (int)std::min<int64_t>((total + 255) / 256, 4096);
#define MMACT_BA(A_) \
    return launch_k(bias_act_kernel<OUT, A_>, grid, 256, 0, s, bias, out, rows, cols, per_row, bias_len, \
                    alpha, res)
    switch (act) {
    case ACT_RELU: MMACT_BA(ACT_RELU);
    case ACT_LEAKY: MMACT_BA(ACT_LEAKY);
    case ACT_TANH: MMACT_BA(ACT_TANH);
    case ACT_SIGMOID: MMACT_BA(ACT_SIGMOID);
    case ACT_GELU: MMACT_BA(ACT_GELU);
    default: MMACT_BA(ACT_NONE);
    }
#undef MMACT_BA
    return cudaGetLastError();
}

cudaError_t launch_bias_act(const float *bias, void *out, int64_t rows, int64_t cols, int per_row,
                            int64_t bias_len, int out_kind, int act, float alpha, cudaStream_t stream,
                            const void *res)
{
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    if (out_kind == OUT_BF16)
        return launch_bias_act_o<OUT_BF16>(bias, out, rows, cols, per_row, bias_len, act, alpha, stream, res);
    if (out_kind == OUT_F16)
        return launch_bias_act_o<OUT_F16>(bias, out, rows, cols, per_row, bias_len, act, alpha, stream, res);
    return launch_bias_act_o<OUT_F32>(bias, out, rows, cols, per_row, bias_len, act, alpha, stream, res);
}

cudaError_t launch_wait_selftest(unsigned int *status, unsigned long long timeout_ns,
                                 cudaStream_t stream)
{
    return launch_k(wait_selftest_kernel, 1, 32, 0, stream, status, timeout_ns);
}

}  // namespace mmact
