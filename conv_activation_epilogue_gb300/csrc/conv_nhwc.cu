// conv_nhwc.cu -- channels-last (NHWC) conv2d + bias + activation as an
// implicit GEMM fed entirely by TMA:
//
//   y[n][oh][ow][co] = act(bias[co] + sum_{r,q,ci} w[co][r][q][ci] *
//                          x[n][oh*sh - pt + r*dh][ow*sw - pl + q*dw][ci])
//
// M = output pixels, N = output channels, K = (r, q, ci) with channels
// fastest.  This is the layout-converting member of the fusion families the
// "ops-nn fused_matmul_relu" article lists (NHWC / NCHW conversion) applied to
// the "multimodal-ops Fused ConvTanh" operator.  An M tile is TH output rows x
// TW output columns of one image (TW * TH = 128 pixels).  With channels
// innermost, the A tile of tap (r, q) and channel block cb is one 4-D TMA box
// of x {C, W, H, N}: box {64, TW*sw, TH*sh, 1} with element strides
// {1, sw, sh, 1}, at (64 cb, ow0*sw - pl + q*dw, oh0*sh - pt + r*dh, n).  It
// lands as 128 pixel rows of 128 bytes with the 128-byte swizzle -- exactly
// the K-major operand layout -- and the TMA's out-of-range zero fill is the
// convolution's zero padding.  The filter, stored [Co][kh][kw][C], is the
// K-major B operand through a 3-D map {C, kh*kw, Co}.  The epilogue is the
// GEMM's (per-column bias, activation, swizzled staging) with a 4-D TMA store
// into y {Co, Wo, Ho, N}; pixels past Wo or Ho are clipped by the store.
//
// Warps: 0 TMA producer (x and filter tiles), 1 TMEM + MMA, 2..9 epilogue
// (two warps per TMEM lane quarter, splitting each tile's output units, which
// halves the exposed epilogue of the last tile on small problems).
#include "common.cuh"
#include "kernels.h"

namespace mmact {

template <int BN>
struct NhwcCfg {
    static constexpr int A_BYTES = 128 * 64 * 2;                 // 16 KB
    static constexpr int B_BYTES = BN * 64 * 2;                  // BN rows x 128 B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_BYTES = 8 * 4096;                  // one 4 KB buffer per epilogue warp
    static constexpr int STAGES = (232448 - EPI_BYTES - 256) / STAGE_BYTES > 8
                                      ? 8
                                      : (232448 - EPI_BYTES - 256) / STAGE_BYTES;
    static constexpr int TMEM_COLS = (int)TileN<BN>::TMEM_COLS;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int THREADS = 320;                      // 8 epilogue warps
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// tile -> (pixel block (n, row block, column block), output-channel block);
// grouped M-first raster as for the GEMM (group_m pixel blocks share a sweep
// over the channel blocks).
__device__ __forceinline__ void nhwc_tile(int t, const NhwcArgs &p, int &n, int &toh, int &tow, int &nb)
{
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int m_first = g * p.group_m;
    const int gm = min(p.tiles_m - m_first, p.group_m);
    const int r = t - g * per_group;
    const int mb = m_first + r % gm;
    nb = r / gm;
    tow = mb % p.tiles_ow;
    const int rr = mb / p.tiles_ow;
    toh = rr % p.tiles_oh;
    n = rr / p.tiles_oh;
}

template <int BN, int OUT, bool TF32>
__global__ void __launch_bounds__(NhwcCfg<BN>::THREADS, 1)
    conv_nhwc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmY, const NhwcArgs p)
{
    using Cfg = NhwcCfg<BN>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int COLS = OUT == OUT_F32 ? 32 : 64;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t base = ptx::smem_addr(smem);
    // let the next kernel in the stream start its set-up; fetch the tensor
    // maps while this one sets up
    ptx::griddep_launch_dependents();
    if (threadIdx.x == 0) {
        ptx::prefetch_tensormap(&tmX);
        ptx::prefetch_tensormap(&tmW);
    }
    if (base & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.status, ST_SMEM_ALIGN);
        return;
    }
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    Pipe pp;
    pp.full0 = base + Cfg::OFF_BAR;
    pp.empty0 = pp.full0 + 8 * STAGES;
    pp.tfull0 = pp.empty0 + 8 * STAGES;
    pp.tempty0 = pp.tfull0 + 16;
    pp.drain = pp.tempty0 + 16;
    pp.abort = misc + 1;
    pp.status = p.status;
    pp.wait_ns = p.wait_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(pp.full0 + 8 * s, 1);
            ptx::mbar_init(pp.empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(pp.tfull0 + 8 * a, 1);
            ptx::mbar_init(pp.tempty0 + 8 * a, 8);
        }
        ptx::mbar_init(pp.drain, 1);
        misc[1] = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(base + Cfg::OFF_MISC, Cfg::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    ptx::cta_sync();
    ptx::tc_fence_after();
    pp.tmem = misc[0];
    ptx::griddep_wait();   // inputs and outputs may belong to the previous kernel

    const uint32_t sA = base + Cfg::OFF_A, sB = base + Cfg::OFF_B;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- producer --
            ptx::prefetch_tensormap(&tmX);
            ptx::prefetch_tensormap(&tmW);
            uint32_t stage = 0, phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
                int n, toh, tow, nb;
                nhwc_tile(t, p, n, toh, tow, nb);
                const int iy0 = toh * p.TH * p.sh - p.pt;
                const int ix0 = tow * p.TW * p.sw - p.pl;
                int r = 0, q = 0, cb = 0;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!pipe_wait(pp, pp.empty0 + 8 * stage, phase ^ 1u)) { ok = false; break; }
                    const uint32_t fb = pp.full0 + 8 * stage;
                    ptx::mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
                    ptx::tma_load_4d(sA + stage * Cfg::A_BYTES, &tmX, fb, cb * p.kc, ix0 + q * p.dw,
                                     iy0 + r * p.dh, n);
                    ptx::tma_load_3d(sB + stage * Cfg::B_BYTES, &tmW, fb, cb * p.kc, r * p.kw + q, nb * BN);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if (++cb == p.ncb) {
                        cb = 0;
                        if (++q == p.kw) { q = 0; ++r; }
                    }
                }
            }
            if (!ok) pipe_fail(pp);
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s))
                    ptx::mbar_wait_bounded(pp.full0 + 8 * s, (last_par >> s) & 1u, DRAIN_NS, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0)
            mma_role<BN, STAGES, true, false, TF32>(pp, sA, sB, p.num_tiles, p.num_kb,
                                                    TF32 ? ptx::idesc_tf32(128, BN)
                                                         : ptx::idesc_f16(p.ab_bf16 != 0, false, false, 128, BN));
    } else {
        // -------------------------------------------------------- epilogue --
        // TMEM lane quarter qd holds tile pixels 32qd..32qd+31, which lie in
        // one output row (TW is 32 or 64): row toh*TH + 32qd/TW, columns
        // tow*TW + (32qd mod TW) + 0..31.
        const int qd = warp & 3;
        const int half = (warp - 2) >> 2;                // which of the quarter's two warps
        const uint32_t my_buf = base + Cfg::OFF_EPI + (uint32_t)(warp - 2) * 4096u;
        uint32_t acc = 0, acc_phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
            int n, toh, tow, nb;
            nhwc_tile(t, p, n, toh, tow, nb);
            const int n0 = nb * BN;
            const int oh = toh * p.TH + (qd * 32) / p.TW;
            const int ow = tow * p.TW + (qd * 32) % p.TW;
            if (!warp_epi_wait(pp, pp.tfull0 + 8 * acc, acc_phase)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t tbase = pp.tmem + ((uint32_t)(qd * 32) << 16) + acc * TileN<BN>::ACC_STRIDE;
#pragma unroll 1
            for (int u = half; u < BN / COLS; u += 2) {
                const uint32_t buf = my_buf;             // one 4 KB staging buffer per warp
                if (lane == 0) ptx::bulk_wait_read<0>();
                __syncwarp();
                const int col0 = n0 + u * COLS;
                const void *rrow = nullptr;      // this lane's pixel: channels col0.. of the residual
                if (p.res != nullptr && oh < p.Ho && ow + lane < p.Wo) {
                    constexpr int ESZ = OUT == OUT_F32 ? 4 : 2;
                    rrow = static_cast<const char *>(p.res) +
                           ((((int64_t)n * p.Ho + oh) * p.Wo + ow + lane) * p.Co + col0) * ESZ;
                }
                epi_unit_dispatch<OUT, false>(p.act, tbase + u * COLS,
                                              p.bias != nullptr ? p.bias + col0 : nullptr, p.Co - col0,
                                              0.0f, p.alpha, buf, lane, rrow, p.res != nullptr);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && oh < p.Ho && ow < p.Wo && col0 < p.Co) {
                    ptx::tma_store_4d(&tmY, buf, col0, ow, oh, n);
                    ptx::bulk_commit();
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(pp.tempty0 + 8 * acc);
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (!ok) pipe_fail(pp);
        if (lane == 0) ptx::bulk_wait<0>();
        __syncwarp();
    }

    ptx::tc_fence_before();
    ptx::cta_sync();
    __syncwarp();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(pp.tmem, Cfg::TMEM_COLS);
    }
}

template <int BN, int OUT>
static cudaError_t launch_nhwc_t(const NhwcLaunch &L, cudaStream_t stream)
{
    if (L.args.tf32)
        return launch_k(conv_nhwc_kernel<BN, OUT, true>, L.grid, NhwcCfg<BN>::THREADS,
                        NhwcCfg<BN>::SMEM_BYTES, stream, L.tmX, L.tmW, L.tmY, L.args);
    return launch_k(conv_nhwc_kernel<BN, OUT, false>, L.grid, NhwcCfg<BN>::THREADS, NhwcCfg<BN>::SMEM_BYTES,
                    stream, L.tmX, L.tmW, L.tmY, L.args);
}

template <int BN, int OUT>
static cudaError_t setup_nhwc_t()
{
    cudaError_t e = cudaFuncSetAttribute(conv_nhwc_kernel<BN, OUT, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, NhwcCfg<BN>::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(conv_nhwc_kernel<BN, OUT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 NhwcCfg<BN>::SMEM_BYTES);
    return e;
}

cudaError_t setup_nhwc_kernels()
{
    cudaError_t e = cudaSuccess;
#define MMACT_NHWC_SETUP(BN_, OUT_) \
    if (e == cudaSuccess) e = setup_nhwc_t<BN_, OUT_>();
    MMACT_NHWC_SETUP(256, OUT_BF16)
    MMACT_NHWC_SETUP(256, OUT_F16)
    MMACT_NHWC_SETUP(256, OUT_F32)
    MMACT_NHWC_SETUP(128, OUT_BF16)
    MMACT_NHWC_SETUP(128, OUT_F16)
    MMACT_NHWC_SETUP(128, OUT_F32)
    MMACT_NHWC_SETUP(64, OUT_BF16)
    MMACT_NHWC_SETUP(64, OUT_F16)
    MMACT_NHWC_SETUP(64, OUT_F32)
#undef MMACT_NHWC_SETUP
    return e;
}

cudaError_t launch_conv_nhwc(const NhwcLaunch &L, cudaStream_t stream)
{
#define MMACT_NHWC_CASE(BN_, OUT_) \
    if (L.tile_n == BN_ && L.out == OUT_) return launch_nhwc_t<BN_, OUT_>(L, stream);
    MMACT_NHWC_CASE(256, OUT_BF16)
    MMACT_NHWC_CASE(256, OUT_F16)
    MMACT_NHWC_CASE(256, OUT_F32)
    MMACT_NHWC_CASE(128, OUT_BF16)
    MMACT_NHWC_CASE(128, OUT_F16)
    MMACT_NHWC_CASE(128, OUT_F32)
    MMACT_NHWC_CASE(64, OUT_BF16)
    MMACT_NHWC_CASE(64, OUT_F16)
    MMACT_NHWC_CASE(64, OUT_F32)
#undef MMACT_NHWC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace mmact
