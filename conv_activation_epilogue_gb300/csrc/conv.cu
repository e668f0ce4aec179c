// conv.cu -- persistent, warp-specialised implicit-GEMM conv2d (NCHW) with the
// fused bias + activation epilogue:  y = act(conv2d(x, w) + bias).
//
// "multimodal-ops Fused ConvTanh" article, section on how the two kernels
// split the work: the convolution is an implicit GEMM whose A operand is the
// filter [Co x K] (K = Ci*kh*kw in the filter's own (ci, r, q) order) and whose
// B operand is the input features [K x Ho*Wo], so each image's result
// [Co, Ho*Wo] is already NCHW.  Per image n the GEMM view is
//
//   y[n][co][p] = act(bias[co] + sum_k w[co][k] * X_n[k][p]),
//   X_n[(ci,r,q)][(oh,ow)] = x[n][ci][oh*sh - pt + r*dh][ow*sw - pl + q*dw]
//                            (0 outside the image),
//
// with X_n never materialised: producer warps gather each [64 K x 128 pixel]
// B tile straight from x into shared memory, in the MN-major 128-byte
// swizzled layout tcgen05.mma reads (the im2col addresses for stride, pad and
// dilation are generated on the fly).  The filter tile [128 co x 64 K] comes
// by TMA when its row pitch allows (K * 2 bytes a multiple of 16), else it is
// gathered too.  The MMA issuer and the epilogue are the GEMM kernel's; the
// epilogue adds bias per output channel (per accumulator row) and stores each
// 32-channel x 64-pixel block with a 3-D TMA store into y viewed as
// [N][Co][Ho*Wo] (or with plain stores when y's row pitch is not 16-byte
// aligned).  The article's stride-2 odd/even column split is not needed:
// address generation handles any stride.
//
// fp32 inputs (F32): x and w are fp32 and are used to fp32 accuracy by
// splitting each value v into bf16 hi = rn(v) and lo = rn(v - hi), so that
// hi + lo carries 16 significant bits and x*w = xh*wh + xl*wh + xh*wl up to the
// dropped xl*wl term (below 2^-16 of |x*w|) and the roundings of hi and lo
// (about 2^-17 of |v| each).  The gather warps split both operands (the filter
// is always gathered in this mode) into hi and lo tiles, and the MMA issuer
// accumulates the three products per K step in the same fp32 TMEM
// accumulator.  The same kernel runs an fp32 GEMM C[M,N] = A[M,K] B[K,N] as
// the 1x1 conv w = A ([M, K, 1, 1]), x = B ([1, K, 1, N]), with the bias along
// the output columns (bias_col), and channels-last fp32 convs (nhwc): x
// [N,H,W,C] and the filter [Co,kh,kw,C] gathered with K = (r, q, ci), y
// [N,Ho,Wo,Co] written with plain stores (the 32 lanes of a warp hold 32
// consecutive output channels of one pixel).
//
// Warps: 0 filter TMA, 1 TMEM + MMA, 2..5 epilogue, 6..9 B-tile gather.
#include "common.cuh"
#include "kernels.h"

namespace mmact {

template <bool F32>
struct ConvCfgT {
    static constexpr int BM = 128, BN = 128, BK = 64;
    static constexpr int A_BYTES = BM * BK * 2 * (F32 ? 2 : 1);   // hi tile, then lo tile (F32)
    static constexpr int B_BYTES = BK * BN * 2 * (F32 ? 2 : 1);
    static constexpr int STAGES = F32 ? 3 : 6;
    static constexpr int EPI_BYTES = 4 * 2 * 4096;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int THREADS = 320;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};
using ConvCfg = ConvCfgT<false>;

// tile -> (image, pixel block, channel block); channel blocks vary fastest so
// CTAs running side by side share the same input pixels in L2.
__device__ __forceinline__ void conv_tile(int t, const ConvArgs &p, int &n, int &pb, int &cb)
{
    cb = t % p.tiles_co;
    const int r = t / p.tiles_co;
    pb = r % p.tiles_p;
    n = r / p.tiles_p;
}

// Byte offset of element (k, j) inside an MN-major 128B-swizzled [64 x 128] tile.
__device__ __forceinline__ uint32_t b_tile_offset(int k, int j)
{
    return (uint32_t)((j >> 6) * 8192 + k * 128 + ((((j >> 3) & 7) ^ (k & 7)) << 4) + ((j & 7) << 1));
}

// Byte offset of element (m, k) inside a K-major 128B-swizzled [128 x 64] tile.
__device__ __forceinline__ uint32_t a_tile_offset(int m, int k)
{
    return (uint32_t)(m * 128 + ((((k >> 3) & 7) ^ (m & 7)) << 4) + ((k & 7) << 1));
}

// v = hi + lo with hi, lo bf16 (round to nearest even both times).
__device__ __forceinline__ void split_bf16(float v, uint16_t &hi, uint16_t &lo)
{
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    const __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
    hi = *reinterpret_cast<const uint16_t *>(&h);
    lo = *reinterpret_cast<const uint16_t *>(&l);
}

template <int OUT, bool F32>
__global__ void __launch_bounds__(ConvCfgT<F32>::THREADS, 1)
    conv_act_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmY,
                    const ConvArgs p)
{
    using Cfg = ConvCfgT<F32>;
    constexpr int STAGES = Cfg::STAGES, BN = Cfg::BN;
    constexpr int COLS = OUT == OUT_F32 ? 32 : 64;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t base = ptx::smem_addr(smem);
    // let the next kernel in the stream start its set-up; fetch the tensor
    // maps while this one sets up
    ptx::griddep_launch_dependents();
    if (threadIdx.x == 0) {
        if (p.a_tma) ptx::prefetch_tensormap(&tmW);
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
        // full: the 4 gather warps, plus the filter TMA producer when it is used
        const uint32_t full_count = (p.a_tma && !F32) ? 5u : 4u;
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(pp.full0 + 8 * s, full_count);
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
        if (lane == 0 && p.a_tma && !F32) {
            // ---------------------------------------------- filter producer --
            ptx::prefetch_tensormap(&tmW);
            uint32_t stage = 0, phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
                int n, pb, cb;
                conv_tile(t, p, n, pb, cb);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!pipe_wait(pp, pp.empty0 + 8 * stage, phase ^ 1u)) { ok = false; break; }
                    const uint32_t fb = pp.full0 + 8 * stage;
                    ptx::mbar_arrive_expect_tx(fb, Cfg::A_BYTES);
                    ptx::tma_load_2d(sA + stage * Cfg::A_BYTES, &tmW, fb, kb * 64, cb * 128);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) pipe_fail(pp);
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s))
                    ptx::mbar_wait_bounded(pp.full0 + 8 * s, (last_par >> s) & 1u, DRAIN_NS, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            if constexpr (F32) {
                // split precision: per K step of 16, hi*hi + lo*hi + hi*lo (bf16 operands)
                const uint32_t idesc = ptx::idesc_f16(true, false, true, 128, BN);
                constexpr uint32_t AH = 128 * 64 * 2, BH = 64 * 128 * 2;   // offset of the lo tiles
                uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
                bool ok = true;
                for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
                    if (!pipe_wait(pp, pp.tempty0 + 8 * acc, acc_phase ^ 1u)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t d = pp.tmem + acc * BN;
                    for (int kb = 0; kb < p.num_kb; ++kb) {
                        if (!pipe_wait(pp, pp.full0 + 8 * stage, phase)) { ok = false; break; }
                        ptx::fence_proxy_async_smem();
                        ptx::tc_fence_after();
                        const uint32_t a0 = sA + stage * Cfg::A_BYTES, b0 = sB + stage * Cfg::B_BYTES;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t ah = ptx::smem_desc(a0 + 32u * k, 16u, 1024u, ptx::SWIZZLE_128B);
                            const uint64_t al = ptx::smem_desc(a0 + AH + 32u * k, 16u, 1024u, ptx::SWIZZLE_128B);
                            const uint64_t bh = ptx::smem_desc(b0 + 2048u * k, 8192u, 1024u, ptx::SWIZZLE_128B);
                            const uint64_t bl = ptx::smem_desc(b0 + BH + 2048u * k, 8192u, 1024u, ptx::SWIZZLE_128B);
                            ptx::mma_f16(d, ah, bh, idesc, (kb | k) != 0 ? 1u : 0u);
                            ptx::mma_f16(d, al, bh, idesc, 1u);
                            ptx::mma_f16(d, ah, bl, idesc, 1u);
                        }
                        ptx::mma_commit(pp.empty0 + 8 * stage);
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                    if (!ok) break;
                    ptx::mma_commit(pp.tfull0 + 8 * acc);
                    acc ^= 1u;
                    if (acc == 0) acc_phase ^= 1u;
                }
                if (!ok) pipe_fail(pp);
                ptx::mma_commit(pp.drain);
                ptx::mbar_wait_bounded(pp.drain, 0, DRAIN_NS, nullptr);
            } else {
                mma_role<BN, STAGES, false, true>(pp, sA, sB, p.num_tiles, p.num_kb,
                                                  ptx::idesc_f16(p.ab_bf16 != 0, false, true, 128, BN));
            }
        }
    } else if (warp >= 6) {
        // ---------------------------------------------------- B-tile gather --
        // Thread j owns pixel column j of every B tile.  For each stage it
        // first issues all 64 of its loads into registers -- independent, so
        // they are in flight together, and issued before waiting for the ring
        // slot so their latency overlaps the wait -- then writes them into
        // the swizzled tile.
        const int j = threadIdx.x - 192;              // this thread's pixel column, 0..127
        const int HW = p.H * p.W;                     // C*H*W < 2^31 is checked on the host
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
            int n, pb, cb;
            conv_tile(t, p, n, pb, cb);
            const int pix = pb * BN + j;
            const bool pvalid = pix < p.P;
            const int oh = pvalid ? pix / p.Wo : 0;
            const int ow = pvalid ? pix - oh * p.Wo : 0;
            const int ih0 = oh * p.sh - p.pt, iw0 = ow * p.sw - p.pl;
            const uint16_t *xn = p.x + (int64_t)n * p.C * HW;
            const int co_rows = p.Co - cb * 128;      // filter rows valid in this tile (gathered A)
            // (ci, r, q) of the next K index, advanced one step per element
            int r = 0, q = 0, k = 0, cbase = 0;       // cbase = ci * H * W
            for (int kb = 0; kb < p.num_kb; ++kb) {
                if constexpr (F32) {
                    // fp32 values, split into hi and lo tiles (x, then the filter rows m = j)
                    const float *xf = reinterpret_cast<const float *>(p.x) + (int64_t)n * p.C * HW;
                    float xv[64];
                    if (p.nhwc) {
                        // K = (r, q, ci), channels fastest; cbase holds ci here
#pragma unroll
                        for (int kl = 0; kl < 64; ++kl) {
                            const int ih = ih0 + r * p.dh, iw = iw0 + q * p.dw;
                            const bool in = pvalid && k < p.K && (unsigned)ih < (unsigned)p.H &&
                                            (unsigned)iw < (unsigned)p.W;
                            xv[kl] = in ? __ldg(xf + ((int64_t)ih * p.W + iw) * p.C + cbase) : 0.0f;
                            ++k;
                            if (++cbase == p.C) {
                                cbase = 0;
                                if (++q == p.kw) { q = 0; ++r; }
                            }
                        }
                    } else {
#pragma unroll
                        for (int kl = 0; kl < 64; ++kl) {
                            const int ih = ih0 + r * p.dh, iw = iw0 + q * p.dw;
                            const bool in = pvalid && k < p.K && (unsigned)ih < (unsigned)p.H &&
                                            (unsigned)iw < (unsigned)p.W;
                            xv[kl] = in ? __ldg(xf + cbase + ih * p.W + iw) : 0.0f;
                            ++k;
                            if (++q == p.kw) {
                                q = 0;
                                if (++r == p.kh) { r = 0; cbase += HW; }
                            }
                        }
                    }
                    if (!warp_pipe_wait(pp, pp.empty0 + 8 * stage, phase ^ 1u)) { ok = false; break; }
                    const uint32_t bt = sB + stage * Cfg::B_BYTES;
#pragma unroll
                    for (int kl = 0; kl < 64; ++kl) {
                        uint16_t hi, lo;
                        split_bf16(xv[kl], hi, lo);
                        ptx::st_shared_u16(bt + b_tile_offset(kl, j), hi);
                        ptx::st_shared_u16(bt + 64 * 128 * 2 + b_tile_offset(kl, j), lo);
                    }
                    const uint32_t at = sA + stage * Cfg::A_BYTES;
                    const float *wr = reinterpret_cast<const float *>(p.w) + (int64_t)(cb * 128 + j) * p.K;
#pragma unroll 8
                    for (int kl = 0; kl < 64; ++kl) {
                        const int kk = kb * 64 + kl;
                        const float v = (j < co_rows && kk < p.K) ? __ldg(wr + kk) : 0.0f;
                        uint16_t hi, lo;
                        split_bf16(v, hi, lo);
                        ptx::st_shared_u16(at + a_tile_offset(j, kl), hi);
                        ptx::st_shared_u16(at + 128 * 64 * 2 + a_tile_offset(j, kl), lo);
                    }
                    __syncwarp();   // the MMA thread fences the stores into the async proxy
                    if (lane == 0) ptx::mbar_arrive(pp.full0 + 8 * stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    continue;
                }
                uint16_t vals[64];
#pragma unroll
                for (int kl = 0; kl < 64; ++kl) {
                    const int ih = ih0 + r * p.dh, iw = iw0 + q * p.dw;
                    const bool in = pvalid && k < p.K && (unsigned)ih < (unsigned)p.H &&
                                    (unsigned)iw < (unsigned)p.W;
                    vals[kl] = in ? __ldg(xn + cbase + ih * p.W + iw) : (uint16_t)0;
                    ++k;
                    if (++q == p.kw) {
                        q = 0;
                        if (++r == p.kh) { r = 0; cbase += HW; }
                    }
                }
                if (!warp_pipe_wait(pp, pp.empty0 + 8 * stage, phase ^ 1u)) { ok = false; break; }
                const uint32_t bt = sB + stage * Cfg::B_BYTES;
#pragma unroll
                for (int kl = 0; kl < 64; ++kl) ptx::st_shared_u16(bt + b_tile_offset(kl, j), vals[kl]);
                if (!p.a_tma) {
                    // filter tile rows m = j: w[cb*128 + m][kb*64 .. +64)
                    const uint32_t at = sA + stage * Cfg::A_BYTES;
                    const uint16_t *wr = p.w + (int64_t)(cb * 128 + j) * p.K;
                    for (int kl = 0; kl < 64; ++kl) {
                        const int kk = kb * 64 + kl;
                        const uint16_t v = (j < co_rows && kk < p.K) ? __ldg(wr + kk) : (uint16_t)0;
                        ptx::st_shared_u16(at + a_tile_offset(j, kl), v);
                    }
                }
                __syncwarp();   // the MMA thread fences the stores into the async proxy
                if (lane == 0) ptx::mbar_arrive(pp.full0 + 8 * stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok) pipe_fail(pp);
    } else {
        // -------------------------------------------------------- epilogue --
        const int qd = warp & 3;
        const uint32_t my_buf = base + Cfg::OFF_EPI + (uint32_t)qd * 8192u;
        uint32_t acc = 0, acc_phase = 0;
        uint32_t units = 0;      // running count: picks the staging buffer
        bool ok = true;
        for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
            int n, pb, cb;
            conv_tile(t, p, n, pb, cb);
            const int co_row0 = cb * 128 + qd * 32;
            const int co = co_row0 + lane;
            const float brow = (p.bias != nullptr && !p.bias_col && co < p.Co) ? __ldg(p.bias + co) : 0.0f;
            if (!warp_epi_wait(pp, pp.tfull0 + 8 * acc, acc_phase)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t tbase = pp.tmem + ((uint32_t)(qd * 32) << 16) + acc * BN;
#pragma unroll 1
            for (int u = 0; u < BN / COLS; ++u) {
                const uint32_t buf = my_buf + (units++ & 1u) * 4096u;
                const int pix0 = pb * BN + u * COLS;
                if (lane == 0) ptx::bulk_wait_read<1>();
                __syncwarp();
                const void *rrow = nullptr;      // this lane's channel, pixels pix0.. (contiguous in y)
                if (p.res != nullptr && co < p.Co && pix0 < p.P) {
                    rrow = static_cast<const char *>(p.res) +
                           (((int64_t)n * p.Co + co) * p.P + pix0) * (OUT == OUT_F32 ? 4 : 2);
                    ptx::prefetch_l1(rrow);
                }
                if (p.bias_col)          // a GEMM run as a 1x1 conv: bias along the output columns
                    epi_unit_dispatch<OUT, false>(p.act, tbase + u * COLS, p.bias != nullptr ? p.bias + pix0 : nullptr,
                                                  p.P - pix0, 0.0f, p.alpha, buf, lane, rrow, p.res != nullptr);
                else
                    epi_unit_dispatch<OUT, true>(p.act, tbase + u * COLS, nullptr, p.P - pix0, brow, p.alpha, buf,
                                                 lane, rrow, p.res != nullptr);
                if (p.y_tma) {
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && co_row0 < p.Co && pix0 < p.P) {
                        ptx::tma_store_3d(&tmY, buf, pix0, co_row0, n);
                        ptx::bulk_commit();
                    }
                } else if (!p.nhwc) {
                    // plain stores, coalesced: for each of the unit's 32 channel rows the
                    // lanes store consecutive pixels, read back from the swizzled staging rows
                    __syncwarp();
                    const int nvalid = min(COLS, p.P - pix0);
                    const int ebytes = p.out_elem_bytes;
                    const uint8_t *stage_rows = smem + (buf - base);
                    for (int r = 0; r < 32 && co_row0 + r < p.Co; ++r) {
                        uint8_t *dst = reinterpret_cast<uint8_t *>(p.y) +
                                       (((int64_t)n * p.Co + co_row0 + r) * p.P + pix0) * ebytes;
                        for (int e = lane; e < nvalid; e += 32) {
                            const int byte = e * ebytes;
                            const uint8_t *src = stage_rows + r * 128 + (((byte >> 4) ^ (r & 7)) << 4) + (byte & 15);
                            if (ebytes == 4)
                                *reinterpret_cast<uint32_t *>(dst + byte) = *reinterpret_cast<const uint32_t *>(src);
                            else
                                *reinterpret_cast<uint16_t *>(dst + byte) = *reinterpret_cast<const uint16_t *>(src);
                        }
                    }
                    __syncwarp();
                } else if (co < p.Co) {
                    // channels-last: each lane stores its channel for the segment's pixels (the
                    // 32 lanes' channels are contiguous in y; pixel e is Co elements after e - 1)
                    const uint8_t *row = smem + (buf - base) + lane * 128;
                    const int64_t pstride = p.nhwc ? (int64_t)p.Co * p.out_elem_bytes : p.out_elem_bytes;
                    uint8_t *dst = reinterpret_cast<uint8_t *>(p.y) +
                                   (p.nhwc ? (((int64_t)n * p.P + pix0) * p.Co + co)
                                           : (((int64_t)n * p.Co + co) * p.P + pix0)) * p.out_elem_bytes;
                    const int nvalid = min(COLS, p.P - pix0);
                    for (int e = 0; e < nvalid; ++e) {
                        const int byte = e * p.out_elem_bytes;
                        const int chunk = (byte >> 4) ^ (lane & 7);
                        const uint8_t *src = row + chunk * 16 + (byte & 15);
                        uint8_t *d = dst + (int64_t)e * pstride;
                        if (p.out_elem_bytes == 4)
                            *reinterpret_cast<uint32_t *>(d) = *reinterpret_cast<const uint32_t *>(src);
                        else
                            *reinterpret_cast<uint16_t *>(d) = *reinterpret_cast<const uint16_t *>(src);
                    }
                    __syncwarp();
                } else {
                    __syncwarp();
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

template <int OUT, bool F32>
static cudaError_t launch_conv_t(const ConvLaunch &L, cudaStream_t stream)
{
    using Cfg = ConvCfgT<F32>;
    return launch_k(conv_act_kernel<OUT, F32>, L.grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream, L.tmW, L.tmY,
                    L.args);
}

template <int OUT, bool F32>
static cudaError_t setup_conv_t()
{
    return cudaFuncSetAttribute(conv_act_kernel<OUT, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                ConvCfgT<F32>::SMEM_BYTES);
}

cudaError_t setup_conv_kernels()
{
    cudaError_t e = setup_conv_t<OUT_BF16, false>();
    if (e == cudaSuccess) e = setup_conv_t<OUT_F16, false>();
    if (e == cudaSuccess) e = setup_conv_t<OUT_F32, false>();
    if (e == cudaSuccess) e = setup_conv_t<OUT_BF16, true>();
    if (e == cudaSuccess) e = setup_conv_t<OUT_F16, true>();
    if (e == cudaSuccess) e = setup_conv_t<OUT_F32, true>();
    return e;
}

cudaError_t launch_conv(const ConvLaunch &L, cudaStream_t stream)
{
    if (L.args.vec) return launch_conv_vec(L, stream);
    if (L.args.f32) {
        if (L.out == OUT_BF16) return launch_conv_t<OUT_BF16, true>(L, stream);
        if (L.out == OUT_F16) return launch_conv_t<OUT_F16, true>(L, stream);
        if (L.out == OUT_F32) return launch_conv_t<OUT_F32, true>(L, stream);
        return cudaErrorInvalidValue;
    }
    if (L.out == OUT_BF16) return launch_conv_t<OUT_BF16, false>(L, stream);
    if (L.out == OUT_F16) return launch_conv_t<OUT_F16, false>(L, stream);
    if (L.out == OUT_F32) return launch_conv_t<OUT_F32, false>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mmact
