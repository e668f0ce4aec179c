// gemm.cu -- persistent, warp-specialised tcgen05 GEMM with the fused
// bias + activation epilogue:  C = act(A x B + bias).
//
// "MatmulLeakyRelu fusion walkthrough" (pyasc examples/05_matmul_leakyrelu)
// computes the same operator in one kernel on an Ascend core: the Cube unit
// produces base_m x base_n blocks of A x B + Bias that stay on chip, the
// Vector unit applies LeakyReLU in place, and a strided block copy writes
// each block to global memory (sections on the fused kernel and on the
// tiling / multi-core split, whose block order is M-first).  Here the same
// dataflow is mapped onto one GB300 SM:
//
//   warp 0      TMA producer: A [128 x 64] and B [64 x BN] tiles into a
//               STAGES-deep shared-memory ring (mbarrier full/empty pairs)
//   warp 1      allocates TMEM, issues tcgen05.mma (fp32 accumulators in TMEM,
//               two accumulator buffers so the epilogue of one tile overlaps
//               the main loop of the next), commits stages and tiles
//   warps 2..5  epilogue: tcgen05.ld -> + bias -> act (fp32) -> convert ->
//               swizzled shared buffer -> TMA store; the fp32 intermediate
//               never leaves the SM
//
// One CTA per SM walks the output tiles in a grouped M-first order (group_m
// M tiles sweep all N tiles before the next group starts) for L2 reuse.
// Every wait is bounded; on a timeout the kernel stops, drains its in-flight
// copies and MMAs, frees TMEM and records the error in the status word.
#include "common.cuh"
#include "kernels.h"

namespace mmact {

template <int BN>
struct GemmCfg {
    static constexpr int BM = 128, BK = 64;
    static constexpr int A_BYTES = BM * BK * 2;                  // 16 KB
    static constexpr int B_BYTES = (int)TileN<BN>::B_BYTES;      // ceil(BN/64) chunks of 8 KB
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_BYTES = 4 * 2 * 4096;               // 4 warps x 2 x (32 x 128 B)
    // as many stages as fit next to the epilogue staging buffers
    static constexpr int STAGES = (232448 - EPI_BYTES - 256) / STAGE_BYTES > 8
                                      ? 8
                                      : (232448 - EPI_BYTES - 256) / STAGE_BYTES;
    static constexpr int TMEM_COLS = (int)TileN<BN>::TMEM_COLS;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;      // [0] tmem base, [1] abort
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

__device__ __forceinline__ void gemm_tile(int t, const GemmArgs &p, int &mb, int &nb)
{
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int m_first = g * p.group_m;
    const int gm = min(p.tiles_m - m_first, p.group_m);
    const int r = t - g * per_group;
    mb = m_first + r % gm;
    nb = r / gm;
}

// tmCt: the map for the 32-column tail unit of a 224-wide tile with a 16-bit
// output (unswizzled 64-byte rows); unused otherwise.
// Start of output row `row`'s residual segment at column col0, or null (no
// residual, or a row past M).
template <int OUT>
__device__ __forceinline__ const void *residual_row(const GemmArgs &p, int row, int col0)
{
    if (p.res == nullptr || row >= p.M) return nullptr;
    constexpr int ESZ = OUT == OUT_F32 ? 4 : 2;
    return static_cast<const char *>(p.res) + ((int64_t)row * p.N + col0) * ESZ;
}

template <int BN, int OUT>
__global__ void __launch_bounds__(192, 1)
    gemm_act_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmCt,
                    const GemmArgs p)
{
    using Cfg = GemmCfg<BN>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int COLS = OUT == OUT_F32 ? 32 : 64;   // output columns per 128-byte row segment
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t base = ptx::smem_addr(smem);
    // let the next kernel in the stream start its set-up; fetch the tensor
    // maps while this one sets up
    ptx::griddep_launch_dependents();
    if (threadIdx.x == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    if (base & 1023u) {   // the swizzle patterns assume a 1024-byte aligned ring
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
            ptx::mbar_init(pp.tempty0 + 8 * a, 4);
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
            ptx::prefetch_tensormap(&tmA);
            ptx::prefetch_tensormap(&tmB);
            uint32_t stage = 0, phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
                int mb, nb;
                gemm_tile(t, p, mb, nb);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!pipe_wait(pp, pp.empty0 + 8 * stage, phase ^ 1u)) { ok = false; break; }
                    const uint32_t fb = pp.full0 + 8 * stage;
                    ptx::mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
                    ptx::tma_load_2d(sA + stage * Cfg::A_BYTES, &tmA, fb, kb * 64, mb * 128);
#pragma unroll
                    for (int c = 0; c < TileN<BN>::NCHUNK; ++c)
                        ptx::tma_load_2d(sB + stage * Cfg::B_BYTES + c * 8192, &tmB, fb,
                                         nb * BN + c * 64, kb * 64);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) pipe_fail(pp);
            // Every copy issued must land before the CTA may exit.
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s))
                    ptx::mbar_wait_bounded(pp.full0 + 8 * s, (last_par >> s) & 1u, DRAIN_NS, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0)
            mma_role<BN, STAGES>(pp, sA, sB, p.num_tiles, p.num_kb,
                                 ptx::idesc_f16(p.ab_bf16 != 0, false, true, 128, BN));
    } else {
        // -------------------------------------------------------- epilogue --
        const int q = warp & 3;                  // TMEM lane quarter this warp may read
        const uint32_t my_buf = base + Cfg::OFF_EPI + (uint32_t)q * 8192u;
        uint32_t acc = 0, acc_phase = 0;
        uint32_t units = 0;      // running count: picks the staging buffer
        bool ok = true;
        for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
            int mb, nb;
            gemm_tile(t, p, mb, nb);
            const int n0 = nb * BN;
            if (!warp_epi_wait(pp, pp.tfull0 + 8 * acc, acc_phase)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t tbase = pp.tmem + ((uint32_t)(q * 32) << 16) + acc * TileN<BN>::ACC_STRIDE;
            const int row0 = mb * 128 + q * 32;
            if (p.res != nullptr) {
                // this lane's residual row segment of the first unit (one 128-byte line)
                const void *r0 = residual_row<OUT>(p, row0 + lane, n0);
                if (r0 != nullptr) ptx::prefetch_l1(r0);
            }
#pragma unroll 1
            for (int u = 0; u < BN / COLS; ++u) {
                if (p.res != nullptr && u + 1 < BN / COLS + (BN % COLS != 0 ? 1 : 0)) {
                    // the next unit's segment, fetched while this unit runs
                    const void *rn = residual_row<OUT>(p, row0 + lane, n0 + (u + 1) * COLS);
                    if (rn != nullptr && n0 + (u + 1) * COLS < p.N) ptx::prefetch_l1(rn);
                }
                const uint32_t buf = my_buf + (units++ & 1u) * 4096u;
                if (lane == 0) ptx::bulk_wait_read<1>();   // the store that last used `buf` has read it
                __syncwarp();
                const int col0 = n0 + u * COLS;
                epi_unit_dispatch<OUT, false>(p.act, tbase + u * COLS,
                                              p.bias != nullptr ? p.bias + col0 : nullptr,
                                              p.N - col0, 0.0f, p.alpha, buf, lane,
                                              residual_row<OUT>(p, row0 + lane, col0), p.res != nullptr);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && row0 < p.M && col0 < p.N) {
                    ptx::tma_store_2d(&tmC, buf, col0, row0);
                    ptx::bulk_commit();
                }
            }
            if constexpr (BN % COLS != 0) {
                // tail: the last 32 columns of a 224-wide tile (16-bit output)
                static_assert(BN % COLS == 32 && OUT != OUT_F32, "tail unit is 32 16-bit columns");
                const uint32_t buf = my_buf + (units++ & 1u) * 4096u;
                if (lane == 0) ptx::bulk_wait_read<1>();
                __syncwarp();
                const int col0 = n0 + (BN / COLS) * COLS;
                epi_unit_dispatch<OUT, false, 32>(p.act, tbase + (BN / COLS) * COLS,
                                                  p.bias != nullptr ? p.bias + col0 : nullptr,
                                                  p.N - col0, 0.0f, p.alpha, buf, lane,
                                                  residual_row<OUT>(p, row0 + lane, col0), p.res != nullptr);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && row0 < p.M && col0 < p.N) {
                    ptx::tma_store_2d(&tmCt, buf, col0, row0);
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

    // Every role must be done before TMEM is released.  In the producer and
    // MMA warps only lane 0 ran the role loop, so the warps arrive here
    // diverged: the thread-counting barrier waits for every thread, where the
    // warp-counting bar.sync behind __syncthreads() could complete early.
    ptx::tc_fence_before();
    ptx::cta_sync();
    __syncwarp();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(pp.tmem, Cfg::TMEM_COLS);
    }
}

template <int BN, int OUT>
static cudaError_t launch_gemm_t(const GemmLaunch &L, cudaStream_t stream)
{
    return launch_k(gemm_act_kernel<BN, OUT>, L.grid, 192, GemmCfg<BN>::SMEM_BYTES, stream, L.tmA, L.tmB,
                    L.tmC, L.tmCt, L.args);
}

template <int BN, int OUT>
static cudaError_t setup_gemm_t()
{
    return cudaFuncSetAttribute(gemm_act_kernel<BN, OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GemmCfg<BN>::SMEM_BYTES);
}

cudaError_t setup_gemm_kernels()
{
    cudaError_t e = cudaSuccess;
#define MMACT_GEMM_SETUP(BN_, OUT_) \
    if (e == cudaSuccess) e = setup_gemm_t<BN_, OUT_>();
    MMACT_GEMM_SETUP(224, OUT_BF16)
    MMACT_GEMM_SETUP(224, OUT_F16)
    MMACT_GEMM_SETUP(224, OUT_F32)
    MMACT_GEMM_SETUP(192, OUT_BF16)
    MMACT_GEMM_SETUP(192, OUT_F16)
    MMACT_GEMM_SETUP(192, OUT_F32)
    MMACT_GEMM_SETUP(256, OUT_BF16)
    MMACT_GEMM_SETUP(256, OUT_F16)
    MMACT_GEMM_SETUP(256, OUT_F32)
    MMACT_GEMM_SETUP(128, OUT_BF16)
    MMACT_GEMM_SETUP(128, OUT_F16)
    MMACT_GEMM_SETUP(128, OUT_F32)
    MMACT_GEMM_SETUP(64, OUT_BF16)
    MMACT_GEMM_SETUP(64, OUT_F16)
    MMACT_GEMM_SETUP(64, OUT_F32)
#undef MMACT_GEMM_SETUP
    return e;
}

cudaError_t launch_gemm(const GemmLaunch &L, cudaStream_t stream)
{
#define MMACT_GEMM_CASE(BN_, OUT_) \
    if (L.tile_n == BN_ && L.out == OUT_) return launch_gemm_t<BN_, OUT_>(L, stream);
    MMACT_GEMM_CASE(224, OUT_BF16)
    MMACT_GEMM_CASE(224, OUT_F16)
    MMACT_GEMM_CASE(224, OUT_F32)
    MMACT_GEMM_CASE(192, OUT_BF16)
    MMACT_GEMM_CASE(192, OUT_F16)
    MMACT_GEMM_CASE(192, OUT_F32)
    MMACT_GEMM_CASE(256, OUT_BF16)
    MMACT_GEMM_CASE(256, OUT_F16)
    MMACT_GEMM_CASE(256, OUT_F32)
    MMACT_GEMM_CASE(128, OUT_BF16)
    MMACT_GEMM_CASE(128, OUT_F16)
    MMACT_GEMM_CASE(128, OUT_F32)
    MMACT_GEMM_CASE(64, OUT_BF16)
    MMACT_GEMM_CASE(64, OUT_F16)
    MMACT_GEMM_CASE(64, OUT_F32)
#undef MMACT_GEMM_CASE
    return cudaErrorInvalidValue;
}

}  // namespace mmact
