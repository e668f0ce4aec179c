// gemm_splitk.cu -- the fused GEMM C = act(A x B + bias) for shapes with few
// output tiles (small M), split along K over a thread-block cluster.
//
// "MatmulLeakyRelu fusion walkthrough" (pyasc examples/05_matmul_leakyrelu)
// splits the work over cores by output blocks only (section on the tiling /
// multi-core split): every core owns whole base_m x base_n blocks and runs
// the full K loop.  With M = 128 and N = 8192 that leaves a GB300 with 32
// blocks of 256 columns for 152 SMs, or narrow tiles whose A block is
// re-read from L2 once per 64 columns.  Here each 128 x 256 output tile is
// instead owned by a cluster of S CTAs; CTA r accumulates the K blocks
// [r*num_kb/S, (r+1)*num_kb/S) into its own TMEM, and the S fp32 partial
// tiles are summed through distributed shared memory before the epilogue:
//
//   warp 0      TMA producer: A [128 x 64] and B [64 x 256] stages of this
//               CTA's K range (mbarrier full/empty ring)
//   warp 1      TMEM allocation and the tcgen05.mma issuer (one accumulator)
//   warps 2..5  (a) write the partial sums of the S-1 column slices that the
//                   other CTAs finish into send slots of this CTA's (now idle)
//                   operand ring;
//               cluster barrier (every ring in the cluster is idle);
//               one thread pushes each send slot into its owner's receive
//               slot with a bulk shared::cta -> shared::cluster copy that
//               completes on the owner's receive mbarrier;
//               (b) wait for the S-1 incoming slices, add them to this CTA's
//                   own slice (256/S columns) of its TMEM accumulator, then
//                   the residual (if any), bias, activation, conversion and
//                   TMA store as in the persistent kernel;
//               cluster barrier (no CTA leaves while a copy is in flight).
//
// The exchange moves 32 KB blocks through the copy engine: reading the
// peers' slices with per-lane ld.shared::cluster instead was measured at
// about 3 bytes per clock per SM, half of the kernel's time.
//
// The sum over K is therefore formed in fp32 in a fixed order (own partial
// first, then the peers by rank), as the persistent kernel forms it in fp32
// in K order; the fp32 intermediate still never leaves the SM cluster.
//
// Every thread of every CTA passes both cluster barriers exactly once, on
// every path (a timed-out wait, a misaligned shared-memory base): the
// pipeline waits are bounded, so a cluster can never wait on a thread that
// does not come.
#include "common.cuh"
#include "kernels.h"

namespace mmact {

template <int S>
struct SplitCfg {
    static constexpr int BN = 256, BM = 128, BK = 64;
    static constexpr int SLICE = BN / S;                          // columns finished per CTA
    static constexpr int A_BYTES = BM * BK * 2;                   // 16 KB
    static constexpr int B_BYTES = (int)TileN<BN>::B_BYTES;       // 4 chunks of 8 KB
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_BYTES = 4 * 4096;                    // 4 warps x (32 x 128 B)
    static constexpr int STAGES = (232448 - EPI_BYTES - 256) / STAGE_BYTES;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 4;              // ring, tile full, drain, receive
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;       // [0] tmem base, [1] abort
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    // a partial slice: [128 rows][SLICE fp32], row pitch SLICE * 4 bytes,
    // 16-byte chunk c of row m stored at chunk c ^ (m & 7).  S-1 send slots
    // (one per peer) then S-1 receive slots (one per peer) in the ring.
    static constexpr int PART_BYTES = BM * SLICE * 4;
    static constexpr int OFF_SEND = 0;
    static constexpr int OFF_RECV = (S - 1) * PART_BYTES;
    static_assert(S == 2 || S == 4, "cluster of 2 or 4 CTAs");
    static_assert(SLICE % 64 == 0, "slices are written 64 columns at a time");
    static_assert(STAGES >= 2, "operand ring");
    static_assert(2 * (S - 1) * PART_BYTES <= STAGES * STAGE_BYTES, "partials fit in the operand ring");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Slot of peer `j` among the S-1 peers of CTA `self` (ranks in order, self
// left out).
__device__ __forceinline__ int peer_slot(int j, int self) { return j < self ? j : j - 1; }

// Byte offset of the 16-byte chunk holding columns [4c, 4c+4) of row m in a
// partial slice.  Eight consecutive rows (one phase of a 16-byte-per-lane
// access) land on eight different bank groups.
template <int SLICE>
__device__ __forceinline__ uint32_t part_off(int m, int c)
{
    return (uint32_t)m * (uint32_t)(SLICE * 4) + ((uint32_t)(c ^ (m & 7)) << 4);
}

// 32 summed accumulator columns of one row -> + bias -> act -> output dtype,
// written into the lane's 128-byte row of a swizzled TMA staging buffer
// starting at 16-byte chunk `c0` (0, or 4 for the second half of a 16-bit
// row).  `bias` points at the first column's bias (null: none); columns at
// or past `nvalid` get no bias.
template <int OUT, int ACT>
__device__ __forceinline__ void finish32(float (&v)[32], const float *bias, int nvalid, float alpha,
                                         uint32_t row, uint32_t sw, int c0)
{
    if (bias != nullptr) {
        if (nvalid >= 32 && (reinterpret_cast<uintptr_t>(bias) & 15u) == 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 b4 = __ldg(reinterpret_cast<const float4 *>(bias + j));
                v[j] += b4.x;
                v[j + 1] += b4.y;
                v[j + 2] += b4.z;
                v[j + 3] += b4.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < nvalid) v[j] += __ldg(bias + j);
        }
    }
    if constexpr (OUT == OUT_F32) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
            ptx::st_shared_v4(row + (((uint32_t)(c0 + c) ^ sw) << 4),
                              __float_as_uint(act_f32<ACT>(v[4 * c], alpha)),
                              __float_as_uint(act_f32<ACT>(v[4 * c + 1], alpha)),
                              __float_as_uint(act_f32<ACT>(v[4 * c + 2], alpha)),
                              __float_as_uint(act_f32<ACT>(v[4 * c + 3], alpha)));
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                w[e] = pack2<OUT>(act_f32<ACT>(v[8 * c + 2 * e], alpha), act_f32<ACT>(v[8 * c + 2 * e + 1], alpha));
            ptx::st_shared_v4(row + (((uint32_t)(c0 + c) ^ sw) << 4), w[0], w[1], w[2], w[3]);
        }
    }
}

template <int OUT>
__device__ __forceinline__ void finish32_act(int act, float (&v)[32], const float *bias, int nvalid,
                                             float alpha, uint32_t row, uint32_t sw, int c0)
{
    switch (act) {
    case ACT_RELU: finish32<OUT, ACT_RELU>(v, bias, nvalid, alpha, row, sw, c0); break;
    case ACT_LEAKY: finish32<OUT, ACT_LEAKY>(v, bias, nvalid, alpha, row, sw, c0); break;
    case ACT_TANH: finish32<OUT, ACT_TANH>(v, bias, nvalid, alpha, row, sw, c0); break;
    case ACT_SIGMOID: finish32<OUT, ACT_SIGMOID>(v, bias, nvalid, alpha, row, sw, c0); break;
    case ACT_GELU: finish32<OUT, ACT_GELU>(v, bias, nvalid, alpha, row, sw, c0); break;
    default: finish32<OUT, ACT_NONE>(v, bias, nvalid, alpha, row, sw, c0); break;
    }
}

template <int S, int OUT>
__global__ void __launch_bounds__(192, 1)
    gemm_splitk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const GemmArgs p)
{
    using Cfg = SplitCfg<S>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int SLICE = Cfg::SLICE;
    constexpr int COLS = OUT == OUT_F32 ? 32 : 64;   // output columns per 128-byte staging row
    constexpr int ESZ = OUT == OUT_F32 ? 4 : 2;      // output (and residual) element bytes
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = ptx::smem_addr(smem);
    const uint32_t rank = ptx::cluster_ctarank();

    ptx::griddep_launch_dependents();
    if (threadIdx.x == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    // The swizzle patterns assume a 1024-byte aligned ring.  A CTA without
    // one does no work but still passes both cluster barriers below.
    const bool aligned = (base & 1023u) == 0;
    if (!aligned && threadIdx.x == 0) atomicOr(p.status, ST_SMEM_ALIGN);

    // this cluster's tile (M tiles fastest: tiles that share a B column
    // block run together) and this CTA's K range
    const int t = (int)(blockIdx.x / S);
    const int mb = t % p.tiles_m, nb = t / p.tiles_m;
    const int kb0 = (int)(((int64_t)rank * p.num_kb) / S);
    const int kb1 = (int)(((int64_t)(rank + 1) * p.num_kb) / S);

    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    Pipe pp;
    pp.full0 = base + Cfg::OFF_BAR;
    pp.empty0 = pp.full0 + 8 * STAGES;
    pp.tfull0 = pp.empty0 + 8 * STAGES;
    pp.tempty0 = 0;
    pp.drain = pp.tfull0 + 8;
    const uint32_t recv_bar = pp.drain + 8;
    pp.abort = misc + 1;
    pp.status = p.status;
    pp.wait_ns = p.wait_ns;

    if (aligned) {
        if (threadIdx.x == 0) {
            for (int s = 0; s < STAGES; ++s) {
                ptx::mbar_init(pp.full0 + 8 * s, 1);
                ptx::mbar_init(pp.empty0 + 8 * s, 1);
            }
            ptx::mbar_init(pp.tfull0, 1);
            ptx::mbar_init(pp.drain, 1);
            ptx::mbar_init(recv_bar, 1);
            misc[1] = 0;
            ptx::fence_mbar_init();
            // the S-1 incoming slices complete the receive barrier's first phase
            ptx::mbar_arrive_expect_tx(recv_bar, (uint32_t)((S - 1) * Cfg::PART_BYTES));
        }
        if (warp == 1) {
            ptx::tmem_alloc(base + Cfg::OFF_MISC, (uint32_t)Cfg::BN);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    ptx::cta_sync();
    ptx::tc_fence_after();
    pp.tmem = misc[0];
    ptx::griddep_wait();   // inputs and outputs may belong to the previous kernel

    const uint32_t sA = base + Cfg::OFF_A, sB = base + Cfg::OFF_B;
    const int q = warp & 3;                          // TMEM lane quarter of an epilogue warp
    const int m = q * 32 + lane;                     // this epilogue lane's row of the tile
    const uint32_t tbase = pp.tmem + ((uint32_t)(q * 32) << 16);
    bool ok = true;

    if (aligned) {
        if (warp == 0) {
            if (lane == 0) {
                // -------------------------------------------------- producer --
                uint32_t stage = 0, phase = 0, issued = 0, last_par = 0;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!pipe_wait(pp, pp.empty0 + 8 * stage, phase ^ 1u)) { ok = false; break; }
                    const uint32_t fb = pp.full0 + 8 * stage;
                    ptx::mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
                    ptx::tma_load_2d(sA + stage * Cfg::A_BYTES, &tmA, fb, kb * 64, mb * 128);
#pragma unroll
                    for (int c = 0; c < TileN<Cfg::BN>::NCHUNK; ++c)
                        ptx::tma_load_2d(sB + stage * Cfg::B_BYTES + c * 8192, &tmB, fb,
                                         nb * Cfg::BN + c * 64, kb * 64);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) pipe_fail(pp);
                // every copy issued must land before the ring is reused or the CTA exits
                for (int s = 0; s < STAGES; ++s)
                    if (issued & (1u << s))
                        ptx::mbar_wait_bounded(pp.full0 + 8 * s, (last_par >> s) & 1u, DRAIN_NS, nullptr);
            }
        } else if (warp == 1) {
            if (lane == 0) {
                // ------------------------------------------------ MMA issuer --
                const uint32_t idesc = ptx::idesc_f16(p.ab_bf16 != 0, false, true, 128, Cfg::BN);
                uint32_t stage = 0, phase = 0;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!pipe_wait(pp, pp.full0 + 8 * stage, phase)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t a0 = sA + stage * Cfg::A_BYTES, b0 = sB + stage * Cfg::B_BYTES;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t ad = ptx::smem_desc(a0 + 32u * k, 16u, 1024u, ptx::SWIZZLE_128B);
                        const uint64_t bd = ptx::smem_desc(b0 + 2048u * k, 8192u, 1024u, ptx::SWIZZLE_128B);
                        ptx::mma_f16(pp.tmem, ad, bd, idesc, (kb > kb0 || k != 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(pp.empty0 + 8 * stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) pipe_fail(pp);
                // the tile's MMAs (possibly none) are done when this fires
                ptx::mma_commit(pp.tfull0);
                ptx::mma_commit(pp.drain);
                ptx::mbar_wait_bounded(pp.drain, 0, DRAIN_NS, nullptr);
            }
        } else {
            // ------------------------------ epilogue (a): partials for peers --
            ok = warp_epi_wait(pp, pp.tfull0, 0);
            ptx::tc_fence_after();
            if (ok) {
                const bool empty = kb1 == kb0;           // no K block: the partial is zero
#pragma unroll 1
                for (int j = 0; j < S; ++j) {
                    if (j == (int)rank) continue;
                    const uint32_t part =
                        base + (uint32_t)(Cfg::OFF_SEND + peer_slot(j, (int)rank) * Cfg::PART_BYTES);
#pragma unroll 1
                    for (int h = 0; h < SLICE / 32; h += 2) {
                        // two TMEM loads in flight per wait
                        uint32_t r0[32], r1[32];
                        ptx::tmem_ld32(tbase + (uint32_t)(j * SLICE + 32 * h), r0);
                        ptx::tmem_ld32(tbase + (uint32_t)(j * SLICE + 32 * h + 32), r1);
                        ptx::tmem_ld_wait(r0);
                        ptx::tmem_ld_wait(r1);
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const uint32_t a = part + part_off<SLICE>(m, 8 * h + c);
                            const uint32_t *r = c < 8 ? r0 + 4 * c : r1 + 4 * (c - 8);
                            if (empty)
                                ptx::st_shared_v4(a, 0u, 0u, 0u, 0u);
                            else
                                ptx::st_shared_v4(a, r[0], r[1], r[2], r[3]);
                        }
                    }
                }
            } else {
                pipe_fail(pp);
            }
            ptx::fence_proxy_async_smem();               // the copy engine reads the send slots
        }
    }

    // Send slots written (or abandoned), every ring of the cluster idle.  The
    // barrier counts threads, so the lanes of the producer and MMA warps may
    // arrive at different times.  (The dynamic shared memory starts at the
    // same offset in every CTA of a launch, so `aligned` is the same for the
    // whole cluster: either every CTA sends and receives, or none does.)
    ptx::cluster_sync();

    if (aligned && threadIdx.x == 64) {
        // push slice j to CTA j, into its receive slot for this rank
#pragma unroll 1
        for (int j = 0; j < S; ++j) {
            if (j == (int)rank) continue;
            const uint32_t src = base + (uint32_t)(Cfg::OFF_SEND + peer_slot(j, (int)rank) * Cfg::PART_BYTES);
            const uint32_t dst = ptx::mapa(
                base + (uint32_t)(Cfg::OFF_RECV + peer_slot((int)rank, j) * Cfg::PART_BYTES), (uint32_t)j);
            ptx::bulk_copy_to_cluster(dst, src, (uint32_t)Cfg::PART_BYTES, ptx::mapa(recv_bar, (uint32_t)j));
        }
    }

    if (aligned && warp >= 2) {
        // -------------------------- epilogue (b): finish this CTA's slice --
        // the slice's bias lines and this lane's residual row segment,
        // fetched while the peers' slices arrive
        const int slice0 = nb * Cfg::BN + (int)rank * SLICE;
        if (p.bias != nullptr && warp == 2 && lane < SLICE / 32 && slice0 + 32 * lane < p.N)
            ptx::prefetch_l1(p.bias + slice0 + 32 * lane);
        const char *res_row = nullptr;                   // residual at (row m, column slice0)
        if (p.res != nullptr && mb * 128 + m < p.M) {
            res_row = static_cast<const char *>(p.res) + ((int64_t)(mb * 128 + m) * p.N + slice0) * ESZ;
#pragma unroll
            for (int b = 0; b < SLICE * ESZ; b += 128)
                if (slice0 + b / ESZ < p.N) ptx::prefetch_l1(res_row + b);
        }
        // The peers' slices of this CTA's columns.  Every aligned CTA sends,
        // failed or not, and this wait does not give up on an abort: no copy
        // may still be writing into this CTA's shared memory when it exits.
        const uint32_t landed = ptx::mbar_wait_bounded(recv_bar, 0, DRAIN_NS, nullptr, 1000) ? 1u : 0u;
        const bool got = __shfl_sync(0xffffffffu, landed, 0) != 0u;
        if (!got) pipe_fail(pp);
        ok = __all_sync(0xffffffffu, ok && got && *pp.abort == 0u);
        const bool empty = kb1 == kb0;
        const uint32_t buf = base + Cfg::OFF_EPI + (uint32_t)q * 4096u;
        const uint32_t row = buf + (uint32_t)lane * 128u;
        const uint32_t sw = (uint32_t)(lane & 7);
        const uint32_t recv = base + (uint32_t)Cfg::OFF_RECV;
        const int row0 = mb * 128 + q * 32;          // first row of this warp's store
        ptx::tc_fence_after();
#pragma unroll 1
        for (int u = 0; u < SLICE / COLS && ok; ++u) {
            const int scol = u * COLS;                   // first column within the slice
            const int col0 = nb * Cfg::BN + (int)rank * SLICE + scol;   // in C
            if (u > 0) {                                 // the previous unit's store has read buf
                if (lane == 0) ptx::bulk_wait_read<0>();
                __syncwarp();
            }
#pragma unroll 1
            for (int h = 0; h < COLS / 32; ++h) {
                uint32_t r[32];
                ptx::tmem_ld32(tbase + (uint32_t)((int)rank * SLICE + scol + 32 * h), r);
                ptx::tmem_ld_wait(r);
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = empty ? 0.0f : __uint_as_float(r[j]);
                // peers in rank order (slot i holds the i-th peer)
#pragma unroll 1
                for (int i = 0; i < S - 1; ++i) {
                    const uint32_t slot = recv + (uint32_t)(i * Cfg::PART_BYTES);
                    uint4 w[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        w[c] = ptx::ld_shared_v4(slot + part_off<SLICE>(m, (scol + 32 * h) / 4 + c));
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        v[4 * c] += __uint_as_float(w[c].x);
                        v[4 * c + 1] += __uint_as_float(w[c].y);
                        v[4 * c + 2] += __uint_as_float(w[c].z);
                        v[4 * c + 3] += __uint_as_float(w[c].w);
                    }
                }
                const int c32 = col0 + 32 * h;
                if (p.res != nullptr)                    // warp-uniform; null rows add nothing
                    add_residual<OUT, 32>(res_row != nullptr ? res_row + (scol + 32 * h) * ESZ : nullptr,
                                          p.N - c32, v);
                finish32_act<OUT>(p.act, v, p.bias != nullptr ? p.bias + c32 : nullptr, p.N - c32,
                                  p.alpha, row, sw, 4 * h);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && row0 < p.M && col0 < p.N) {
                ptx::tma_store_2d(&tmC, buf, col0, row0);
                ptx::bulk_commit();
            }
        }
        if (!ok) pipe_fail(pp);
        if (lane == 0) ptx::bulk_wait<0>();
        __syncwarp();
    }

    // every CTA has received its slices (or given up): no copy is in flight
    // when a CTA releases its shared memory
    ptx::cluster_sync();

    ptx::tc_fence_before();
    ptx::cta_sync();
    __syncwarp();
    if (aligned && warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(pp.tmem, (uint32_t)Cfg::BN);
    }
}

template <int S, int OUT>
static cudaError_t launch_splitk_t(const GemmLaunch &L, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)L.grid);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = SplitCfg<S>::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_splitk_kernel<S, OUT>, L.tmA, L.tmB, L.tmC, L.args);
}

template <int S, int OUT>
static cudaError_t setup_splitk_t()
{
    return cudaFuncSetAttribute(gemm_splitk_kernel<S, OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SplitCfg<S>::SMEM_BYTES);
}

cudaError_t setup_splitk_kernels()
{
    cudaError_t e = cudaSuccess;
#define MMACT_SPLITK_SETUP(S_, OUT_) \
    if (e == cudaSuccess) e = setup_splitk_t<S_, OUT_>();
    MMACT_SPLITK_SETUP(2, OUT_BF16)
    MMACT_SPLITK_SETUP(2, OUT_F16)
    MMACT_SPLITK_SETUP(2, OUT_F32)
    MMACT_SPLITK_SETUP(4, OUT_BF16)
    MMACT_SPLITK_SETUP(4, OUT_F16)
    MMACT_SPLITK_SETUP(4, OUT_F32)
#undef MMACT_SPLITK_SETUP
    return e;
}

// Clusters of S split-K CTAs that can be resident on the device at once
// (0 when the query fails).
template <int S>
static int splitk_max_clusters_t()
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(S * 64));
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = SplitCfg<S>::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_splitk_kernel<S, OUT_BF16>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

int splitk_max_clusters(int S)
{
    return S == 2 ? splitk_max_clusters_t<2>() : S == 4 ? splitk_max_clusters_t<4>() : 0;
}

cudaError_t launch_gemm_splitk(const GemmLaunch &L, cudaStream_t stream)
{
#define MMACT_SPLITK_CASE(S_, OUT_) \
    if (L.split_k == S_ && L.out == OUT_) return launch_splitk_t<S_, OUT_>(L, stream);
    MMACT_SPLITK_CASE(2, OUT_BF16)
    MMACT_SPLITK_CASE(2, OUT_F16)
    MMACT_SPLITK_CASE(2, OUT_F32)
    MMACT_SPLITK_CASE(4, OUT_BF16)
    MMACT_SPLITK_CASE(4, OUT_F16)
    MMACT_SPLITK_CASE(4, OUT_F32)
#undef MMACT_SPLITK_CASE
    return cudaErrorInvalidValue;
}

}  // namespace mmact
