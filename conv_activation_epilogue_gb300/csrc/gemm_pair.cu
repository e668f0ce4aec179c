// gemm_pair.cu -- the fused GEMM C = act(A x B + bias [+ R]) with one
// tcgen05.mma per CTA pair (cta_group::2): 256 x 256 output tiles on two SMs.
//
// The persistent kernel of gemm.cu gives every SM a 128 x 256 tile and so
// fills its shared memory with 48 KB per K block of 64 (A 16 KB + B 32 KB).
// Here the two CTAs of a cluster pair share a 256 x 256 tile: CTA r holds A
// rows [128r, 128r + 128) and B columns [128r, 128r + 128) of it, and one
// M = 256 MMA issued by the even CTA reads both halves of B from both CTAs'
// shared memory while each SM accumulates its own 128 rows x 256 columns in
// its own TMEM.  Each SM then fills 32 KB per K block for the same MMA work,
// two thirds of the bytes, which buys two more ring stages.  The block order,
// epilogue and fused bias / activation / residual are those of gemm.cu
// ("MatmulLeakyRelu fusion walkthrough", pyasc examples/05_matmul_leakyrelu:
// the fused kernel and the tiling sections).
//
//   warp 0      (both CTAs) TMA producer: its A and B halves into its own
//               ring; the copies complete on the even CTA's full barrier,
//               which counts the bytes of both
//   warp 1      (both CTAs) the pair's TMEM allocation; in the even CTA the
//               MMA issuer, whose commits arrive on the stage and tile
//               barriers of both CTAs (multicast)
//   warps 2..5  (both CTAs) epilogue of the CTA's 128 rows; a finished
//               accumulator buffer is released on the even CTA's barrier
//               (4 warps x 2 CTAs)
//
// Every wait is bounded.  Both CTAs pass a final cluster barrier before TMEM
// is released, so no commit or arrival can target a CTA that has exited.
#include "common.cuh"
#include "kernels.h"

namespace mmact {

struct PairCfg {
    static constexpr int BM = 128, BN = 256, BK = 64;             // per CTA: 128 rows x 256 columns
    static constexpr int A_BYTES = BM * BK * 2;                   // 16 KB: this CTA's A rows
    static constexpr int B_BYTES = 2 * 8192;                      // 8 KB x 2: this CTA's 128 B columns
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_BYTES = 4 * 2 * 4096;
    static constexpr int STAGES = (232448 - EPI_BYTES - 256) / STAGE_BYTES > 8
                                      ? 8
                                      : (232448 - EPI_BYTES - 256) / STAGE_BYTES;
    static constexpr uint32_t ACC_STRIDE = 256, TMEM_COLS = 512;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 5 + 8;           // + residual loads: 4 warps x 2 buffers
    static constexpr int OFF_RBAR = OFF_BAR + (2 * STAGES + 5) * 8;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;       // [0] tmem base, [1] abort
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Pair tile t -> (M block of 256 rows, N block of 256 columns), grouped
// M-first as in the persistent kernel (tiles_m / tiles_n count pair tiles).
__device__ __forceinline__ void pair_tile(int t, const GemmArgs &p, int &mb, int &nb)
{
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int m_first = g * p.group_m;
    const int gm = min(p.tiles_m - m_first, p.group_m);
    const int r = t - g * per_group;
    mb = m_first + r % gm;
    nb = r / gm;
}

template <int OUT>
__global__ void __launch_bounds__(192, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmR,
                     const GemmArgs p)
{
    using Cfg = PairCfg;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int COLS = OUT == OUT_F32 ? 32 : 64;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = ptx::smem_addr(smem);
    const uint32_t rank = ptx::cluster_ctarank();    // 0: issues the MMAs; 1: its peer
    const bool leader = rank == 0;
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);

    ptx::griddep_launch_dependents();
    if (threadIdx.x == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    // The dynamic shared memory starts at the same offset in every CTA of a
    // launch, so both CTAs of a pair agree on `aligned`.
    const bool aligned = (base & 1023u) == 0;
    if (!aligned && threadIdx.x == 0) atomicOr(p.status, ST_SMEM_ALIGN);

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

    if (aligned) {
        if (threadIdx.x == 0) {
            for (int s = 0; s < STAGES; ++s) {
                ptx::mbar_init(pp.full0 + 8 * s, 1);      // the even CTA's producer arrives
                ptx::mbar_init(pp.empty0 + 8 * s, 1);     // one multicast commit per use
            }
            for (int a = 0; a < 2; ++a) {
                ptx::mbar_init(pp.tfull0 + 8 * a, 1);
                ptx::mbar_init(pp.tempty0 + 8 * a, 8);    // 4 epilogue warps x 2 CTAs
            }
            ptx::mbar_init(pp.drain, 1);
            for (int b = 0; b < 8; ++b) ptx::mbar_init(base + Cfg::OFF_RBAR + 8 * b, 1);
            misc[1] = 0;
            ptx::fence_mbar_init();
        }
        if (warp == 1) {
            ptx::tmem_alloc_pair(base + Cfg::OFF_MISC, Cfg::TMEM_COLS);
            ptx::tmem_relinquish_pair();
        }
    }
    ptx::tc_fence_before();
    ptx::cta_sync();
    ptx::tc_fence_after();
    // barrier initialisation of both CTAs visible before either signals the other
    ptx::cluster_sync();
    pp.tmem = misc[0];
    // The pair's MMAs address both CTAs' accumulators through the even CTA's
    // TMEM base, so the two allocations must have returned the same columns;
    // a pair that disagrees records an error and does no work.
    const bool usable = aligned && ptx::ld_cluster_u32(ptx::mapa(base + Cfg::OFF_MISC, rank ^ 1u)) == pp.tmem;
    if (aligned && !usable && threadIdx.x == 0) atomicOr(p.status, ST_PAIR_TMEM);
    ptx::griddep_wait();

    const uint32_t sA = base + Cfg::OFF_A, sB = base + Cfg::OFF_B;

    // Both CTAs read both bases, so `usable` is the same in the pair.
    ptx::cluster_sync();

    if (usable && warp == 0) {
        if (lane == 0) {
            // -------------------------------------------------------- producer --
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            // A strips are reused by every wave of a raster group (8 M blocks of 256 rows);
            // a B strip only by the tiles of one wave.  With l2_policy the A loads carry
            // the evict-last policy so that the group's A rows stay in L2 across its waves.
            const uint64_t pol_a = ptx::createpolicy_evict_last();
            for (int t = pair; t < p.num_tiles && ok; t += npairs) {
                int mb, nb;
                pair_tile(t, p, mb, nb);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!pipe_wait(pp, pp.empty0 + 8 * stage, phase ^ 1u)) { ok = false; break; }
                    const uint32_t fb = pp.full0 + 8 * stage;
                    if (leader) ptx::mbar_arrive_expect_tx(fb, 2u * Cfg::STAGE_BYTES);
                    const uint32_t fb_leader = ptx::mapa(fb, 0);
                    if (p.l2_policy != 0)
                        ptx::tma_load_2d_pair_hint(sA + stage * Cfg::A_BYTES, &tmA, fb_leader, kb * 64,
                                                   mb * 256 + (int)rank * 128, pol_a);
                    else
                        ptx::tma_load_2d_pair(sA + stage * Cfg::A_BYTES, &tmA, fb_leader, kb * 64,
                                              mb * 256 + (int)rank * 128);
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        ptx::tma_load_2d_pair(sB + stage * Cfg::B_BYTES + c * 8192, &tmB, fb_leader,
                                              nb * 256 + (int)rank * 128 + c * 64, kb * 64);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) pipe_fail(pp);
            // The copies of both CTAs complete on the even CTA's full barriers;
            // its MMA issuer consumes (so waits for) every stage issued, and
            // the final cluster barrier keeps both CTAs resident until then.
        }
    } else if (usable && warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------------ MMA issuer --
            const uint32_t idesc = ptx::idesc_f16(p.ab_bf16 != 0, false, true, 256, 256);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int t = pair; t < p.num_tiles && ok; t += npairs) {
                if (!pipe_wait(pp, pp.tempty0 + 8 * acc, acc_phase ^ 1u)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d = pp.tmem + acc * Cfg::ACC_STRIDE;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!pipe_wait(pp, pp.full0 + 8 * stage, phase)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t a0 = sA + stage * Cfg::A_BYTES, b0 = sB + stage * Cfg::B_BYTES;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t ad = ptx::smem_desc(a0 + 32u * k, 16u, 1024u, ptx::SWIZZLE_128B);
                        const uint64_t bd = ptx::smem_desc(b0 + 2048u * k, 8192u, 1024u, ptx::SWIZZLE_128B);
                        ptx::mma_f16_pair(d, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    ptx::mma_commit_pair_mc(pp.empty0 + 8 * stage, 3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit_pair_mc(pp.tfull0 + 8 * acc, 3);
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) pipe_fail(pp);
            // every MMA issued must finish before TMEM is released
            ptx::mma_commit_pair_mc(pp.drain, 1);
            ptx::mbar_wait_bounded(pp.drain, 0, DRAIN_NS, nullptr);
        }
    } else if (usable && warp >= 2) {
        // ------------------------------------------------------------ epilogue --
        const int q = warp & 3;
        const uint32_t my_buf = base + Cfg::OFF_EPI + (uint32_t)q * 8192u;
        const uint32_t tempty_leader = ptx::mapa(pp.tempty0, 0);
        const uint64_t pol_c = ptx::createpolicy_evict_first();   // C is never read back here
        // Residual: each unit's R tile [32 rows][128 B] is loaded by TMA (the output's
        // tensor map layout, on R) into the staging buffer the unit's output will use,
        // one unit ahead: the load for unit i+1 is issued, into the other buffer, once
        // every earlier store has read its buffer, and unit i waits only for its own.
        // Each lane reads its R row segment before overwriting it with its output, and
        // every element of R is loaded before the store of the same element of C (R
        // may be C itself).
        const bool has_res = p.res != nullptr;
        const uint32_t rbar0 = base + Cfg::OFF_RBAR + (uint32_t)q * 16u;
        uint32_t rphase = 0, rpending = 0;
        constexpr int NU = 256 / COLS;                      // units per tile for this warp
        auto load_r = [&](int t_, int u_, uint32_t b) {     // lane 0 only
            int mb_, nb_;
            pair_tile(t_, p, mb_, nb_);
            const uint32_t bar = rbar0 + 8u * b;
            ptx::mbar_arrive_expect_tx(bar, 4096u);
            ptx::tma_load_2d(my_buf + b * 4096u, &tmR, bar, nb_ * 256 + u_ * COLS, mb_ * 256 + (int)rank * 128 + q * 32);
            rpending |= 1u << b;
        };
        if (has_res && pair < p.num_tiles && lane == 0) {
            ptx::prefetch_tensormap(&tmR);
            load_r(pair, 0, 0u);                            // units == 0: buffer 0
        }
        uint32_t acc = 0, acc_phase = 0, units = 0;
        bool ok = true;
        for (int t = pair; t < p.num_tiles; t += npairs) {
            int mb, nb;
            pair_tile(t, p, mb, nb);
            const int n0 = nb * 256;
            if (!warp_epi_wait(pp, pp.tfull0 + 8 * acc, acc_phase)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t tbase = pp.tmem + ((uint32_t)(q * 32) << 16) + acc * Cfg::ACC_STRIDE;
            const int row0 = mb * 256 + (int)rank * 128 + q * 32;
#pragma unroll 1
            for (int u = 0; u < NU; ++u) {
                const uint32_t cur = units++ & 1u;
                const uint32_t buf = my_buf + cur * 4096u;
                const int col0 = n0 + u * COLS;
                if (has_res) {
                    if (lane == 0) {
                        // the next unit's R into the other buffer, once every store has read it
                        const int tn = u + 1 < NU ? t : t + npairs;
                        if (tn < p.num_tiles) {
                            ptx::bulk_wait_read<0>();
                            load_r(tn, u + 1 < NU ? u + 1 : 0, cur ^ 1u);
                        }
                    }
                    __syncwarp();
                    if (!warp_epi_wait(pp, rbar0 + 8u * cur, (rphase >> cur) & 1u)) { ok = false; break; }
                    rphase ^= 1u << cur;
                    rpending &= ~(1u << cur);
                    epi_unit_dispatch_rsmem<OUT>(p.act, tbase + u * COLS, p.bias != nullptr ? p.bias + col0 : nullptr,
                                                 p.N - col0, p.alpha, buf, lane);
                } else {
                    if (lane == 0) ptx::bulk_wait_read<1>();
                    __syncwarp();
                    epi_unit_dispatch<OUT, false>(p.act, tbase + u * COLS,
                                                  p.bias != nullptr ? p.bias + col0 : nullptr, p.N - col0,
                                                  0.0f, p.alpha, buf, lane);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && row0 < p.M && col0 < p.N) {
                    if (p.l2_policy != 0) ptx::tma_store_2d_hint(&tmC, buf, col0, row0, pol_c);
                    else ptx::tma_store_2d(&tmC, buf, col0, row0);
                    ptx::bulk_commit();
                }
            }
            if (!ok) break;                                 // a residual wait gave up
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) ptx::mbar_arrive(pp.tempty0 + 8 * acc);
                else ptx::mbar_arrive_cluster(tempty_leader + 8 * acc);
            }
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (!ok) pipe_fail(pp);
        if (lane == 0) {
            // a residual load still in flight (after a failed wait) lands before exit
            for (uint32_t b = 0; b < 2; ++b)
                if (rpending & (1u << b))
                    ptx::mbar_wait_bounded(rbar0 + 8u * b, (rphase >> b) & 1u, DRAIN_NS, nullptr);
            ptx::bulk_wait<0>();
        }
        __syncwarp();
    }

    // Both CTAs done with every role: no commit, copy or arrival is still
    // addressed to either of them.  Thread-counting barriers, so the lanes of
    // the producer and MMA warps may arrive at different times.
    ptx::tc_fence_before();
    ptx::cluster_sync();
    ptx::cta_sync();
    __syncwarp();
    if (aligned && warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(pp.tmem, Cfg::TMEM_COLS);
    }
}

template <int OUT>
static cudaError_t launch_pair_t(const GemmLaunch &L, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)L.grid);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = PairCfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<OUT>, L.tmA, L.tmB, L.tmC, L.tmR, L.args);
}

cudaError_t setup_pair_kernels()
{
    cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<OUT_BF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_pair_kernel<OUT_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PairCfg::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_pair_kernel<OUT_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PairCfg::SMEM_BYTES);
    return e;
}

int pair_max_clusters()
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 128);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = PairCfg::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<OUT_BF16>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_gemm_pair(const GemmLaunch &L, cudaStream_t stream)
{
    if (L.out == OUT_BF16) return launch_pair_t<OUT_BF16>(L, stream);
    if (L.out == OUT_F16) return launch_pair_t<OUT_F16>(L, stream);
    if (L.out == OUT_F32) return launch_pair_t<OUT_F32>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mmact
