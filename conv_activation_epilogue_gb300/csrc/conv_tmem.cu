// conv_tmem.cu -- NCHW implicit-GEMM conv2d + bias + activation with the
// im2col operand assembled in tensor memory.
//
//   y[n][co][p] = act(bias[co] + sum_k w[co][k] * x_col[n][k][p]),
//   k = (ci, r, q) in the filter's own order, p = oh * Wo + ow.
//
// The GEMM view is the "multimodal-ops Fused ConvTanh" article's (section on
// how the two kernels split the work: the filter [Co x Ci*kh*kw] against the
// input features [Ci*kh*kw x pixels]), with the roles of the MMA operands
// swapped so that the im2col operand can live in tensor memory: the MMA
// computes D[pixel][co] = A[pixel][k] * B[k][co] with
//   A = 128 consecutive output pixels of one image x 64 K per K block, written
//       into TMEM by producer warps (tcgen05.st; lane m = pixel m, two 16-bit
//       K values per 32-bit column, the lower K in the low half), and
//   B = the filter tile [BN output channels][64 K] as stored ([Co][Ci*kh*kw]
//       is K-major), loaded by TMA with the 128-byte swizzle.
// The tensor core then reads only the filter from shared memory; the im2col
// tile is never written to shared memory at all.  Each producer lane builds
// the A row of one pixel: per K block the TMA warp stages the raw input
// window the block needs (the channels its 64 K values span, the input rows
// the tile's output rows read for every filter row, an 8-aligned column span
// covering every filter column; zero fill outside the image is the padding),
// and the lane picks its 64 values from it with 16-bit shared loads at
// offsets from a per-CTA table (a K value's offset depends only on its
// position in the K block and the block's phase).  The windows are small (a
// few KB to 32 KB), so as many window slots as the shared-memory budget allows
// (up to 8) keep their TMA latency off the producers' path.  The result
// D[pixel][co] is transposed through shared memory into [co][pixel] blocks of
// 32 x 32 (for each output channel the 32 lanes of a warp hold 32 consecutive
// pixels) and written to NCHW y by TMA stores.
//
// Three rings, each advancing in K-block order: filter tiles in shared memory
// (3-4 stages), im2col tiles in TMEM (8 stages of 32 columns), input windows
// in shared memory (up to 8 slots).  Each has its own full/empty barriers so
// that no ring waits for another's slowest consumer.
//
// Warps: 0 TMA for filter tiles, 14 TMA for input windows, 1 TMEM allocation + MMA issue,
// 2..5 epilogue (one per TMEM lane quarter), 6..13 im2col producers in two
// groups of four (one warp per lane quarter) that build alternate K blocks,
// so that two blocks are assembled at once; once the CTA's
// last accumulator is complete the producer warps take two of every three of
// its epilogue units, staged in the filter ring that no MMA reads any more.
#include "common.cuh"
#include "kernels.h"

namespace mmact {

template <int BN>
struct TmemConvCfg {
    static constexpr int STAGES = BN == 256 ? 3 : 4;      // filter tiles in shared memory
    static constexpr int B_BYTES = BN * 128;              // [BN rows][64 K] 16-bit, 128-byte rows
    static constexpr int EPI_BUF = 4096;                  // [32 channels][32 pixels] (fp32; 2 KB for 16-bit)
    static constexpr int EPI_BYTES = 4 * 2 * EPI_BUF;     // two buffers per epilogue warp
    static constexpr int TABLE = CONV_TMEM_TABLE_MAX;     // K-offset table entries
    static constexpr int MAX_WSTAGES = CONV_TMEM_MAX_WSTAGES;
    static constexpr int ACC_BUFS = BN == 256 ? 1 : 2;    // accumulator buffers of BN columns
    static constexpr uint32_t A_COL0 = ACC_BUFS * BN;     // TMEM column of im2col stage 0
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int ASTAGES = (TMEM_COLS - A_COL0) / 32 > 8 ? 8 : (TMEM_COLS - A_COL0) / 32;   // im2col tiles in TMEM
    static constexpr int OFF_B = 0;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_TAB = OFF_EPI + EPI_BYTES;
    static constexpr int OFF_BAR = OFF_TAB + TABLE * 4;
    static constexpr int NUM_BARS = 2 * STAGES + 2 * ASTAGES + 2 * MAX_WSTAGES + 2 * ACC_BUFS + 2;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_WIN = (OFF_MISC + 16 + 1023) / 1024 * 1024;   // window ring: the rest
    static constexpr int SMEM_BYTES = 232448;
    static constexpr int WIN_REGION = SMEM_BYTES - OFF_WIN;
    static constexpr int HELPER_BUFS = STAGES * B_BYTES >= 8 * 2 * EPI_BUF ? 2 : 1;
    static constexpr int PRODUCER_WARPS = 8;
    static constexpr int WINDOW_WARP = 6 + PRODUCER_WARPS;
    static constexpr int THREADS = (7 + PRODUCER_WARPS) * 32;
    static_assert(A_COL0 + ASTAGES * 32 <= TMEM_COLS, "tensor memory budget");
    static_assert(STAGES * B_BYTES >= 8 * EPI_BUF, "helper staging fits in the filter ring");
    static_assert(WIN_REGION >= 2 * CONV_TMEM_WIN_MAX_BYTES, "two windows of the largest size");
    static_assert(B_BYTES % 1024 == 0, "slot alignment");
};

// tile -> (image, 128-pixel block, output-channel block); the channel block
// varies fastest so that CTAs reading the same input window run together.
__device__ __forceinline__ void tconv_tile(int t, const TmemConvArgs &p, int &n, int &pb, int &cb)
{
    cb = t % p.tiles_co;
    const int r = t / p.tiles_co;
    pb = r % p.tiles_p;
    n = r / p.tiles_p;
}

template <int OUT>
__device__ __forceinline__ void store_out(void *y, int64_t idx, float v)
{
    if constexpr (OUT == OUT_F32) static_cast<float *>(y)[idx] = v;
    else if constexpr (OUT == OUT_BF16) static_cast<__nv_bfloat16 *>(y)[idx] = __float2bfloat16_rn(v);
    else static_cast<__half *>(y)[idx] = __float2half_rn(v);
}

template <int OUT>
__device__ __forceinline__ float load_res(const void *r, int64_t idx)
{
    if constexpr (OUT == OUT_F32) return static_cast<const float *>(r)[idx];
    else if constexpr (OUT == OUT_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(r)[idx]);
    else return __half2float(static_cast<const __half *>(r)[idx]);
}

// One epilogue unit: this warp's 32 pixels (lanes) x 32 output channels
// co0..co0+31 of the accumulator at taddr, act(acc + bias (+ residual)).
// With Y_TMA the values are transposed into `buf` as [32 channels][32
// pixels] and the lane 0 stores the block with one TMA store (the store
// clips pixels past P and channels past Co); otherwise every lane stores its
// own values (for each channel the warp's 32 consecutive pixels).
template <int OUT, int ACT, bool RES, bool Y_TMA>
__device__ __forceinline__ void tconv_epi_unit(const TmemConvArgs &p, const CUtensorMap *tmY, uint32_t taddr,
                                               int n, int co0, int px0, int lane, uint32_t buf)
{
    const int px = px0 + lane;
    const bool px_ok = px < p.P;
    uint32_t acc[32];
    ptx::tmem_ld32(taddr, acc);
    float b[32];
    if (p.bias != nullptr && co0 + 32 <= p.Co && (reinterpret_cast<uintptr_t>(p.bias + co0) & 15u) == 0) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p.bias + co0 + j));
            b[j] = v.x;
            b[j + 1] = v.y;
            b[j + 2] = v.z;
            b[j + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) b[j] = (p.bias != nullptr && co0 + j < p.Co) ? __ldg(p.bias + co0 + j) : 0.0f;
    }
    const int64_t base = ((int64_t)n * p.Co + co0) * p.P + px;   // y index of (co0, px)
    if constexpr (RES) {
        // channel j of this pixel is P elements after channel j - 1
        constexpr int ESZ = OUT == OUT_F32 ? 4 : 2;
        const char *rp = static_cast<const char *>(p.res) + base * ESZ;
        const int64_t rstep = (int64_t)p.P * ESZ;
        const int nco = min(32, p.Co - co0);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (px_ok && j < nco) b[j] += load_res<OUT>(rp, 0);
            rp += rstep;
        }
    }
    ptx::tmem_ld_wait(acc);
    float (&v)[32] = b;                            // the activations replace the biases in place
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = act_f32<ACT>(__uint_as_float(acc[j]) + b[j], p.alpha);
    if constexpr (Y_TMA) {
        if constexpr (OUT == OUT_F32) {
            // row j = channel co0 + j: 32 pixels x 4 bytes
#pragma unroll
            for (int j = 0; j < 32; ++j) ptx::st_shared_u32(buf + (uint32_t)j * 128u + 4u * (uint32_t)lane, __float_as_uint(v[j]));
        } else {
            // lane pair (2i, 2i+1): the even lane writes channel j, the odd lane
            // channel j+1, each the pixel pair (2i, 2i+1) as one 32-bit word
            const bool odd = (lane & 1) != 0;
            const uint32_t col = 4u * (uint32_t)(lane >> 1);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float send = odd ? v[j] : v[j + 1];
                const float got = __shfl_xor_sync(0xffffffffu, send, 1);
                const uint32_t w = odd ? pack2<OUT>(got, v[j + 1]) : pack2<OUT>(v[j], got);
                ptx::st_shared_u32(buf + (uint32_t)(j + (odd ? 1 : 0)) * 64u + col, w);
            }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            ptx::tma_store_3d(tmY, buf, px0, co0, n);
            ptx::bulk_commit();
        }
        return;
    }
    constexpr int ESZ = OUT == OUT_F32 ? 4 : 2;
    char *yp = static_cast<char *>(p.y) + base * ESZ;
    const int64_t ystep = (int64_t)p.P * ESZ;
    const int nco = min(32, p.Co - co0);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        if (px_ok && j < nco) store_out<OUT>(yp, 0, v[j]);
        yp += ystep;
    }
}

template <int OUT, bool RES, bool Y_TMA>
__device__ __forceinline__ void tconv_epi_unit_act(const TmemConvArgs &p, const CUtensorMap *tmY, uint32_t taddr,
                                                   int n, int co0, int px0, int lane, uint32_t buf)
{
    switch (p.act) {
    case ACT_RELU: tconv_epi_unit<OUT, ACT_RELU, RES, Y_TMA>(p, tmY, taddr, n, co0, px0, lane, buf); break;
    case ACT_LEAKY: tconv_epi_unit<OUT, ACT_LEAKY, RES, Y_TMA>(p, tmY, taddr, n, co0, px0, lane, buf); break;
    case ACT_TANH: tconv_epi_unit<OUT, ACT_TANH, RES, Y_TMA>(p, tmY, taddr, n, co0, px0, lane, buf); break;
    case ACT_SIGMOID: tconv_epi_unit<OUT, ACT_SIGMOID, RES, Y_TMA>(p, tmY, taddr, n, co0, px0, lane, buf); break;
    case ACT_GELU: tconv_epi_unit<OUT, ACT_GELU, RES, Y_TMA>(p, tmY, taddr, n, co0, px0, lane, buf); break;
    default: tconv_epi_unit<OUT, ACT_NONE, RES, Y_TMA>(p, tmY, taddr, n, co0, px0, lane, buf); break;
    }
}

// The units u0, u0 + ustep, ... of tile t's accumulator at tbase (this warp's
// lane quarter qd), staged alternately in nbufs buffers of EPI_BUF bytes from
// buf0.  Returns with this warp's TMA stores committed (not waited for).
template <int BN, int OUT>
__device__ __forceinline__ void tconv_epi_units(const TmemConvArgs &p, const CUtensorMap *tmY, uint32_t tbase,
                                                int t, int qd, int u0, int ustep, uint32_t buf0, int nbufs,
                                                uint32_t &units, int lane)
{
    int n, pb, cb;
    tconv_tile(t, p, n, pb, cb);
    const int px0 = pb * 128 + qd * 32;
    // this tile's bias lines (BN floats) into L1 before the first unit needs them
    if (p.bias != nullptr && lane < BN / 32 && cb * BN + lane * 32 < p.Co) ptx::prefetch_l1(p.bias + cb * BN + lane * 32);
#pragma unroll 1
    for (int u = u0; u < BN / 32; u += ustep) {
        const int co0 = cb * BN + u * 32;
        if (co0 >= p.Co) break;                    // warp-uniform
        const uint32_t buf = buf0 + (nbufs == 2 ? (units & 1u) : 0u) * (uint32_t)TmemConvCfg<BN>::EPI_BUF;
        ++units;
        if (p.y_tma) {
            if (lane == 0) {
                if (nbufs == 2) ptx::bulk_wait_read<1>();
                else ptx::bulk_wait_read<0>();
            }
            __syncwarp();
            if (p.res != nullptr)
                tconv_epi_unit_act<OUT, true, true>(p, tmY, tbase + u * 32, n, co0, px0, lane, buf);
            else
                tconv_epi_unit_act<OUT, false, true>(p, tmY, tbase + u * 32, n, co0, px0, lane, buf);
        } else {
            if (p.res != nullptr)
                tconv_epi_unit_act<OUT, true, false>(p, tmY, tbase + u * 32, n, co0, px0, lane, buf);
            else
                tconv_epi_unit_act<OUT, false, false>(p, tmY, tbase + u * 32, n, co0, px0, lane, buf);
        }
    }
}

template <int BN, int OUT>
__global__ void __launch_bounds__(TmemConvCfg<BN>::THREADS)
    conv_tmem_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmY, const TmemConvArgs p)
{
    using Cfg = TmemConvCfg<BN>;
    constexpr int STAGES = Cfg::STAGES, MAXW = Cfg::MAX_WSTAGES, ACC_BUFS = Cfg::ACC_BUFS;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t base = ptx::smem_addr(smem);
    ptx::griddep_launch_dependents();
    if (threadIdx.x == 0) {
        ptx::prefetch_tensormap(&tmW);
        ptx::prefetch_tensormap(&tmX);
        if (p.y_tma) ptx::prefetch_tensormap(&tmY);
    }
    if (base & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.status, ST_SMEM_ALIGN);
        return;
    }
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    int *tab = reinterpret_cast<int *>(smem + Cfg::OFF_TAB);
    const int WST = p.wstages;                          // window slots (2..MAXW)
    Pipe pp;
    constexpr int ASTAGES = Cfg::ASTAGES;
    pp.full0 = base + Cfg::OFF_BAR;                      // filter ring
    pp.empty0 = pp.full0 + 8 * STAGES;
    const uint32_t afull0 = pp.empty0 + 8 * STAGES;      // im2col ring (TMEM)
    const uint32_t aempty0 = afull0 + 8 * ASTAGES;
    const uint32_t wfull0 = aempty0 + 8 * ASTAGES;       // input-window ring
    const uint32_t wempty0 = wfull0 + 8 * MAXW;
    pp.tfull0 = wempty0 + 8 * MAXW;
    pp.tempty0 = pp.tfull0 + 8 * ACC_BUFS;
    pp.drain = pp.tempty0 + 8 * ACC_BUFS;
    const uint32_t tlast = pp.drain + 8;                // the CTA's last accumulator is complete
    pp.abort = misc + 1;
    pp.status = p.status;
    pp.wait_ns = p.wait_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(pp.full0 + 8 * s, 1);        // filter TMA
            ptx::mbar_init(pp.empty0 + 8 * s, 1);       // MMA commit
        }
        for (int s = 0; s < ASTAGES; ++s) {
            ptx::mbar_init(afull0 + 8 * s, 4);          // the producer group of the block
            ptx::mbar_init(aempty0 + 8 * s, 1);         // MMA commit
        }
        for (int s = 0; s < MAXW; ++s) {
            ptx::mbar_init(wfull0 + 8 * s, 1);
            ptx::mbar_init(wempty0 + 8 * s, 4);          // the producer group that read it
        }
        for (int a = 0; a < ACC_BUFS; ++a) {
            ptx::mbar_init(pp.tfull0 + 8 * a, 1);
            ptx::mbar_init(pp.tempty0 + 8 * a, 4);
        }
        ptx::mbar_init(pp.drain, 1);
        ptx::mbar_init(tlast, 1);
        misc[1] = 0;
        ptx::fence_mbar_init();
    }
    // K-offset table: entry j is the window offset (elements) of K value j of
    // a block, for the block phases 0..tab_period-1 (the pattern repeats).
    {
        const int taps = p.kh * p.kw;
        const int plane = p.HB * p.WB;
        for (int j = threadIdx.x; j < p.tab_period * 64; j += blockDim.x) {
            const int ci = j / taps;
            const int tap = j - ci * taps;
            const int r = tap / p.kw;
            const int q = tap - r * p.kw;
            const int c_lo = ((j >> 6) << 6) / taps;
            tab[j] = (ci - c_lo) * plane + r * p.rstep * p.WB + q * p.dw;
        }
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

    const uint32_t sB = base + Cfg::OFF_B, sWin = base + Cfg::OFF_WIN;
    const uint32_t slot = (uint32_t)p.win_slot;
    const int taps = p.kh * p.kw;
    // the CTA's last tile (its epilogue is shared with the producer warps)
    const int my_tiles = blockIdx.x < (unsigned)p.num_tiles
                             ? (p.num_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int t_last = (int)blockIdx.x + (my_tiles - 1) * (int)gridDim.x;

    if (warp == 0) {
        if (lane == 0) {
            // --------------------------------------------------- filter tiles --
            uint32_t stage = 0, phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
                int n, pb, cb;
                tconv_tile(t, p, n, pb, cb);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!pipe_wait(pp, pp.empty0 + 8 * stage, phase ^ 1u)) { ok = false; break; }
                    const uint32_t fb = pp.full0 + 8 * stage;
                    ptx::mbar_arrive_expect_tx(fb, Cfg::B_BYTES);
                    ptx::tma_load_2d(sB + stage * Cfg::B_BYTES, &tmW, fb, kb * 64, cb * BN);
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
    } else if (warp == Cfg::WINDOW_WARP) {
        if (lane == 0) {
            // -------------------------------------------------- input windows --
            uint32_t ws = 0, wph = 0, wissued = 0, wlast = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
                int n, pb, cb;
                tconv_tile(t, p, n, pb, cb);
                const int y0 = ((pb * 128) / p.Wo) * p.sh - p.pt;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!pipe_wait(pp, wempty0 + 8 * ws, wph ^ 1u)) { ok = false; break; }
                    const uint32_t wb = wfull0 + 8 * ws;
                    ptx::mbar_arrive_expect_tx(wb, (uint32_t)p.raw_bytes);
                    ptx::tma_load_4d(sWin + ws * slot, &tmX, wb, p.x0, y0, (kb * 64) / taps, n);
                    wissued |= 1u << ws;
                    wlast = (wlast & ~(1u << ws)) | (wph << ws);
                    if (++ws == (uint32_t)WST) { ws = 0; wph ^= 1u; }
                }
            }
            if (!ok) pipe_fail(pp);
            for (int s = 0; s < WST; ++s)
                if (wissued & (1u << s))
                    ptx::mbar_wait_bounded(wfull0 + 8 * s, (wlast >> s) & 1u, DRAIN_NS, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA --
            const uint32_t idesc = ptx::idesc_f16(p.ab_bf16 != 0, false, false, 128, BN);
            uint32_t stage = 0, phase = 0, as = 0, aph = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
                if (!pipe_wait(pp, pp.tempty0 + 8 * acc, acc_phase ^ 1u)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d = pp.tmem + acc * BN;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    // the filter tile (normally landed long before) first, so that its wait
                    // overlaps the previous block's MMAs; then the im2col tile
                    if (!pipe_wait(pp, pp.full0 + 8 * stage, phase) || !pipe_wait_spin(pp, afull0 + 8 * as, aph)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a0 = pp.tmem + Cfg::A_COL0 + as * 32u;
                    const uint32_t b0 = sB + stage * Cfg::B_BYTES;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        ptx::mma_f16_tmem_a(d, a0 + 8u * k, ptx::smem_desc(b0 + 32u * k, 16u, 1024u, ptx::SWIZZLE_128B),
                                            idesc, (kb | k) != 0 ? 1u : 0u);
                    ptx::mma_commit(pp.empty0 + 8 * stage);
                    ptx::mma_commit(aempty0 + 8 * as);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if (++as == (uint32_t)ASTAGES) { as = 0; aph ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit(pp.tfull0 + 8 * acc);
                if (t + (int)gridDim.x >= p.num_tiles) ptx::mma_commit(tlast);
                if (++acc == (uint32_t)ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
            }
            if (!ok) pipe_fail(pp);
            ptx::mma_commit(pp.drain);
            ptx::mbar_wait_bounded(pp.drain, 0, DRAIN_NS, nullptr);
        }
    } else if (warp >= 6) {
        // ------------------------------------------------ im2col into TMEM --
        // Group g (warps 6..9 or 10..13) builds the K blocks whose running
        // index G (over all of the CTA's tiles) has G % 2 == g; its warp for
        // lane quarter qd writes all 64 K values of pixels 32qd..32qd+31: TMEM
        // lanes 32qd.., columns A_COL0 + 32 * (G % ASTAGES) .. + 31 (two per column).
        const int qd = warp & 3, g = (warp - 6) >> 2, h = g;
        const uint32_t tlane = (uint32_t)(qd * 32) << 16;
        bool ok = true;
        int G = 0;                                   // running K-block index of the CTA
        for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
            int n, pb, cb;
            tconv_tile(t, p, n, pb, cb);
            const int p0 = pb * 128;
            const int px = min(p0 + qd * 32 + lane, p.P - 1);   // past P: any in-tile pixel (result discarded)
            const int oh = px / p.Wo, ow = px - (px / p.Wo) * p.Wo;
            const int lane_off = (oh - p0 / p.Wo) * p.rowmul * p.WB + ow * p.sw + p.xoff;
            for (int kb = (G & 1) == g ? 0 : 1; kb < p.num_kb; kb += 2) {
                const int Gk = G + kb;
                const uint32_t stage = (uint32_t)(Gk % ASTAGES), phase = (uint32_t)((Gk / ASTAGES) & 1);
                const uint32_t ws = (uint32_t)(Gk % WST), wph = (uint32_t)((Gk / WST) & 1);
                const uint32_t tb = base + Cfg::OFF_TAB + 4u * (uint32_t)((kb % p.tab_period) * 64);
                if (!warp_pipe_wait_spin(pp, aempty0 + 8 * stage, phase ^ 1u) ||
                    !warp_pipe_wait_spin(pp, wfull0 + 8 * ws, wph)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t wbase = sWin + ws * slot + 2u * (uint32_t)lane_off;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    uint4 o[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) o[j] = ptx::ld_shared_v4(tb + 128u * half + 16u * j);
                    uint32_t e[32];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        e[4 * j] = ptx::ld_shared_u16(wbase + 2u * o[j].x);
                        e[4 * j + 1] = ptx::ld_shared_u16(wbase + 2u * o[j].y);
                        e[4 * j + 2] = ptx::ld_shared_u16(wbase + 2u * o[j].z);
                        e[4 * j + 3] = ptx::ld_shared_u16(wbase + 2u * o[j].w);
                    }
                    uint32_t r[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) r[j] = __byte_perm(e[2 * j], e[2 * j + 1], 0x5410);
                    ptx::tmem_st16(pp.tmem + tlane + Cfg::A_COL0 + stage * 32u + 16u * (uint32_t)half, r);
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(afull0 + 8 * stage);
                    ptx::mbar_arrive(wempty0 + 8 * ws);
                }
            }
            G += p.num_kb;
        }
        if (ok && my_tiles > 0) {
            // ------------------------------- help with the last tile's epilogue --
            // Units u = 1 + h (mod 3) of quarter qd, staged in the filter ring:
            // the last accumulator is complete only after every MMA has read it.
            // Its commit is also signalled on tlast (phase 0): these warps can run
            // far ahead of the MMAs, and a parity wait on the accumulator barrier
            // could then match an earlier tile's phase.
            const uint32_t hacc = (uint32_t)((my_tiles - 1) % ACC_BUFS);
            if (warp_epi_wait(pp, tlast, 0)) {
                ptx::tc_fence_after();
                const uint32_t tbase = pp.tmem + tlane + hacc * BN;
                const uint32_t hbuf = sB + (uint32_t)(warp - 6) * (uint32_t)(Cfg::HELPER_BUFS * Cfg::EPI_BUF);
                uint32_t units = 0;
                tconv_epi_units<BN, OUT>(p, &tmY, tbase, t_last, qd, 1 + h, 3, hbuf, Cfg::HELPER_BUFS, units, lane);
                ptx::tc_fence_before();
                if (lane == 0) ptx::bulk_wait<0>();
                __syncwarp();
            } else {
                ok = false;
            }
        }
        if (!ok) pipe_fail(pp);
    } else {
        // -------------------------------------------------------- epilogue --
        const int qd = warp & 3;
        const uint32_t my_buf = base + Cfg::OFF_EPI + (uint32_t)qd * 2u * Cfg::EPI_BUF;
        uint32_t acc = 0, acc_phase = 0, units = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
            if (!warp_epi_wait(pp, pp.tfull0 + 8 * acc, acc_phase)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t tbase = pp.tmem + ((uint32_t)(qd * 32) << 16) + acc * BN;
            // the last tile's units are shared with the producer warps (this warp: u = 0, 3, 6, ...)
            tconv_epi_units<BN, OUT>(p, &tmY, tbase, t, qd, 0, t == t_last ? 3 : 1, my_buf, 2, units, lane);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(pp.tempty0 + 8 * acc);
            if (++acc == (uint32_t)ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
        }
        if (!ok) pipe_fail(pp);
        if (lane == 0) ptx::bulk_wait<0>();
        __syncwarp();
    }

    // Every role must be done before TMEM is released (thread-counting barrier:
    // the single-lane roles arrive diverged).
    ptx::tc_fence_before();
    ptx::cta_sync();
    __syncwarp();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(pp.tmem, Cfg::TMEM_COLS);
    }
}

template <int BN, int OUT>
static cudaError_t launch_tconv_t(const TmemConvLaunch &L, cudaStream_t stream)
{
    using Cfg = TmemConvCfg<BN>;
    return launch_k(conv_tmem_kernel<BN, OUT>, L.grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream, L.tmW, L.tmX,
                    L.tmY, L.args);
}

template <int BN, int OUT>
static cudaError_t setup_tconv_t()
{
    return cudaFuncSetAttribute(conv_tmem_kernel<BN, OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TmemConvCfg<BN>::SMEM_BYTES);
}

int conv_tmem_window_region(int tile_n)
{
    return tile_n == 256 ? TmemConvCfg<256>::WIN_REGION
                         : (tile_n == 128 ? TmemConvCfg<128>::WIN_REGION : TmemConvCfg<64>::WIN_REGION);
}

cudaError_t setup_conv_tmem_kernels()
{
    cudaError_t e = cudaSuccess;
#define MMACT_TCONV_SETUP(BN_, OUT_) \
    if (e == cudaSuccess) e = setup_tconv_t<BN_, OUT_>();
    MMACT_TCONV_SETUP(256, OUT_BF16)
    MMACT_TCONV_SETUP(256, OUT_F16)
    MMACT_TCONV_SETUP(256, OUT_F32)
    MMACT_TCONV_SETUP(128, OUT_BF16)
    MMACT_TCONV_SETUP(128, OUT_F16)
    MMACT_TCONV_SETUP(128, OUT_F32)
    MMACT_TCONV_SETUP(64, OUT_BF16)
    MMACT_TCONV_SETUP(64, OUT_F16)
    MMACT_TCONV_SETUP(64, OUT_F32)
#undef MMACT_TCONV_SETUP
    return e;
}

cudaError_t launch_conv_tmem(const TmemConvLaunch &L, cudaStream_t stream)
{
#define MMACT_TCONV_CASE(BN_, OUT_) \
    if (L.tile_n == BN_ && L.out == OUT_) return launch_tconv_t<BN_, OUT_>(L, stream);
    MMACT_TCONV_CASE(256, OUT_BF16)
    MMACT_TCONV_CASE(256, OUT_F16)
    MMACT_TCONV_CASE(256, OUT_F32)
    MMACT_TCONV_CASE(128, OUT_BF16)
    MMACT_TCONV_CASE(128, OUT_F16)
    MMACT_TCONV_CASE(128, OUT_F32)
    MMACT_TCONV_CASE(64, OUT_BF16)
    MMACT_TCONV_CASE(64, OUT_F16)
    MMACT_TCONV_CASE(64, OUT_F32)
#undef MMACT_TCONV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace mmact
