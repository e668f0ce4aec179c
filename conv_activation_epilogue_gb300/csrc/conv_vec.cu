// conv_vec.cu -- implicit-GEMM conv2d + bias + activation, vectorised
// producer for the common NCHW geometries (input width a multiple of 8,
// horizontal stride 1 or 2, filter rows whose pitch allows TMA).
//
// Same GEMM view as conv.cu ("multimodal-ops Fused ConvTanh" article, section
// on how the two kernels split the work: A = filter [Co x Ci*kh*kw], B = input
// features [Ci*kh*kw x pixels], result [Co, pixels] = NCHW), with a 128 x 256
// output tile: 128 output channels x 256 output pixels, the pixels being TH
// output rows x TW output columns (4 x 64, or 8 x 32 when the output is exactly
// 32 wide, in which case the tile is 256 consecutive pixels of one image).
//
// B-tile producer.  Each gather warp owns 16 consecutive K rows (ci, r, q) of
// every 64-row stage; for each row every lane builds one 16-byte vector of 8
// consecutive output pixels.  Those pixels read input row
// ih = oh*sh - pt + r*dh at columns iws + S*e (e = 0..7), iws = ow*S - pl + q*dw.
// Because W is a multiple of 8, the input row splits into aligned 8-element
// chunks that never straddle two rows; the lane loads the 2 (S = 1) or 3
// (S = 2) aligned chunks covering the window -- chunks outside the row or rows
// outside the image read as zero, which is exactly the zero padding -- and
// picks its 8 elements with byte permutes.  The shift iws mod 8 is the same
// for every lane of the warp, so the selection is a warp-uniform switch.  The
// vector is stored with one 16-byte shared store into the 128-byte swizzled
// MN-major tile that tcgen05.mma reads.
//
// Window variant (WIN).  Read straight from global memory, every input
// element is fetched once per filter tap that touches it (9 times for a 3x3
// filter), and those redundant 16-byte loads are what limits the producer.
// With WIN the TMA warp also loads, per 64-row K block, the raw input window
// the block needs -- the <= CB channels its rows (ci, r, q) span, every input
// row the tile's output rows read for any r, and an 8-aligned column span
// covering every q -- as one 4-D box of x {W, H, C, N} into shared memory
// (zero fill outside the image is the padding; a row traversal stride of sh
// skips the rows no tap reads when dh is a multiple of sh).  The gather
// warps then build the B tile from that window with 16-byte shared loads and
// the same byte picks, so global memory sees each input element about once
// per tile and channel block.
#include "common.cuh"
#include "kernels.h"

namespace mmact {

template <bool WIN>
struct ConvVecCfg {
    static constexpr int BM = 128, BN = 256, BK = 64;
    static constexpr int A_BYTES = BM * BK * 2;          // 16 KB
    static constexpr int B_BYTES = BK * BN * 2;          // 32 KB (4 chunks of 64 pixels)
    static constexpr int STAGES = WIN ? 3 : 4;
    static constexpr int RSTAGES = WIN ? 2 : 0;          // input-window ring
    static constexpr int RAW_MAX = CONV_WIN_MAX_BYTES;   // bytes of one window slot
    static constexpr int EPI_BYTES = 4 * 2 * 4096;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_RAW = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_EPI = OFF_RAW + RSTAGES * RAW_MAX;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 6 + 2 * RSTAGES;   // + the last tile's accumulator
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int GATHER_WARPS = 8;
    static constexpr int THREADS = (6 + GATHER_WARPS) * 32;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// tile -> (image, output-row block, output-column block, channel block); the
// channel block varies fastest so neighbouring CTAs share input pixels in L2.
__device__ __forceinline__ void vconv_tile(int t, const ConvArgs &p, int &n, int &toh, int &tow,
                                           int &cb)
{
    cb = t % p.tiles_co;
    int r = t / p.tiles_co;
    tow = r % p.tiles_ow;
    r /= p.tiles_ow;
    toh = r % p.tiles_oh;
    n = r / p.tiles_oh;
}

__device__ __forceinline__ uint4 ldg16(const uint16_t *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// Eight output elements e = 0..7 taken from the concatenated chunk words w
// (4*NCH words, two 16-bit elements each) at element positions sh + S*e.
// Branch-free: shift the word array left by sh/2 words with two levels of
// selects, then build each output word with one byte permute whose selector
// depends on whether sh is odd.
template <int S>
__device__ __forceinline__ void pick8(int sh, const uint32_t *w, uint32_t (&o)[4])
{
    constexpr int NW = S == 1 ? 8 : 12;
    const bool s1 = (sh & 2) != 0, s2 = (sh & 4) != 0, odd = (sh & 1) != 0;
    uint32_t u[NW - 1], v[NW - 3];
#pragma unroll
    for (int i = 0; i < NW - 1; ++i) u[i] = s1 ? w[i + 1] : w[i];
#pragma unroll
    for (int i = 0; i < NW - 3; ++i) v[i] = s2 ? u[i + 2] : u[i];
    if constexpr (S == 1) {
        const uint32_t sel = odd ? 0x5432u : 0x3210u;
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = __byte_perm(v[j], v[j + 1], sel);
    } else {
        const uint32_t sel = odd ? 0x7632u : 0x5410u;
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = __byte_perm(v[2 * j], v[2 * j + 1], sel);
    }
}

template <int OUT, int S, bool WIN>
__global__ void __launch_bounds__(ConvVecCfg<WIN>::THREADS, 1)
    conv_vec_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmY,
                    const __grid_constant__ CUtensorMap tmY4, const __grid_constant__ CUtensorMap tmX,
                    const ConvArgs p)
{
    using Cfg = ConvVecCfg<WIN>;
    constexpr int STAGES = Cfg::STAGES, BN = Cfg::BN;
    constexpr int COLS = OUT == OUT_F32 ? 32 : 64;
    constexpr int NCH = S == 1 ? 2 : 3;                 // aligned chunks per output vector
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t base = ptx::smem_addr(smem);
    // let the next kernel in the stream start its set-up; fetch the tensor
    // maps while this one sets up
    ptx::griddep_launch_dependents();
    if (threadIdx.x == 0) {
        ptx::prefetch_tensormap(&tmW);
        if constexpr (WIN) ptx::prefetch_tensormap(&tmX);
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
    const uint32_t rfull0 = pp.drain + 8;                // input-window ring (WIN)
    const uint32_t rempty0 = rfull0 + 8 * Cfg::RSTAGES;
    const uint32_t tlast = rempty0 + 8 * Cfg::RSTAGES;   // the CTA's last accumulator is complete

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(pp.full0 + 8 * s, Cfg::GATHER_WARPS + 1);   // gather warps + filter TMA
            ptx::mbar_init(pp.empty0 + 8 * s, 1);
        }
        for (int s = 0; s < Cfg::RSTAGES; ++s) {
            ptx::mbar_init(rfull0 + 8 * s, 1);                         // window TMA
            ptx::mbar_init(rempty0 + 8 * s, Cfg::GATHER_WARPS);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(pp.tfull0 + 8 * a, 1);
            ptx::mbar_init(pp.tempty0 + 8 * a, 4);
        }
        ptx::mbar_init(pp.drain, 1);
        ptx::mbar_init(tlast, 1);
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

    // One epilogue unit: 32 output channels (this warp's TMEM lane quarter,
    // starting at co_row0) x COLS pixels of the tile, from accumulator column
    // tbase + u * COLS, staged in `buf` and stored by TMA.
    auto store_unit = [&](int n, int toh, int tow, int co_row0, float brow, uint32_t tbase, int u,
                          uint32_t buf) {
        // this lane's channel: the unit's pixels are contiguous in y (one output
        // row when TW = 64, consecutive pixels of the image when TW = 32)
        const void *rrow = nullptr;
        int rvalid = 0;
        if (p.res != nullptr && co_row0 + lane < p.Co) {
            constexpr int ESZ = OUT == OUT_F32 ? 4 : 2;
            const int col = u * COLS;
            int64_t off = -1;
            if (p.TW == 32) {
                const int pix0 = toh * p.TH * p.Wo + col;
                if (pix0 < p.P) {
                    off = ((int64_t)n * p.Co + co_row0 + lane) * p.P + pix0;
                    rvalid = p.P - pix0;
                }
            } else {
                const int oh = toh * p.TH + col / 64, ow = tow * 64 + (col & 63);
                if (oh < p.Ho && ow < p.Wo) {
                    off = (((int64_t)n * p.Co + co_row0 + lane) * p.Ho + oh) * p.Wo + ow;
                    rvalid = p.Wo - ow;
                }
            }
            if (off >= 0) {
                rrow = static_cast<const char *>(p.res) + off * ESZ;
                ptx::prefetch_l1(rrow);                   // read chunk by chunk in the epilogue unit
                ptx::prefetch_l1(static_cast<const char *>(rrow) + 64);
            }
        }
        epi_unit_dispatch<OUT, true>(p.act, tbase + u * COLS, nullptr, rvalid, brow, p.alpha, buf, lane,
                                     rrow, p.res != nullptr);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && co_row0 < p.Co) {
            const int col = u * COLS;                    // first B-tile column of this unit
            if (p.TW == 32) {
                // the tile is 256 consecutive pixels of image n
                const int pix0 = toh * p.TH * p.Wo + col;
                if (pix0 < p.P) {
                    ptx::tma_store_3d(&tmY, buf, pix0, co_row0, n);
                    ptx::bulk_commit();
                }
            } else {
                const int oh = toh * p.TH + col / 64;
                const int ow = tow * 64 + (col & 63);
                if (oh < p.Ho && ow < p.Wo) {
                    ptx::tma_store_4d(&tmY4, buf, ow, oh, co_row0, n);
                    ptx::bulk_commit();
                }
            }
        }
    };

    // The CTA's last tile: its accumulator buffer and phase, and the number of
    // warps sharing its epilogue (each CTA of a small conv owns one tile, so
    // that epilogue is not hidden behind any main loop: the gather warps, idle
    // by then, take two of every three units).
    const int my_tiles = blockIdx.x < (unsigned)p.num_tiles
                             ? (p.num_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int t_last = (int)blockIdx.x + (my_tiles - 1) * (int)gridDim.x;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------- filter producer --
            ptx::prefetch_tensormap(&tmW);
            if constexpr (WIN) ptx::prefetch_tensormap(&tmX);
            const int taps = p.kh * p.kw;
            uint32_t stage = 0, phase = 0, issued = 0, last_par = 0;
            uint32_t rst = 0, rph = 0, rissued = 0, rlast = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
                int n, toh, tow, cb;
                vconv_tile(t, p, n, toh, tow, cb);
                const int y0 = toh * p.TH * p.sh - p.pt;                  // window origin (WIN)
                const int x0 = (tow * p.TW * S - p.pl) & ~7;              // 8-aligned: TMA x rule
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!pipe_wait(pp, pp.empty0 + 8 * stage, phase ^ 1u)) { ok = false; break; }
                    const uint32_t fb = pp.full0 + 8 * stage;
                    ptx::mbar_arrive_expect_tx(fb, Cfg::A_BYTES);
                    ptx::tma_load_2d(sA + stage * Cfg::A_BYTES, &tmW, fb, kb * 64, cb * 128);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if constexpr (WIN) {
                        if (!pipe_wait(pp, rempty0 + 8 * rst, rph ^ 1u)) { ok = false; break; }
                        const uint32_t rb = rfull0 + 8 * rst;
                        ptx::mbar_arrive_expect_tx(rb, (uint32_t)p.raw_bytes);
                        ptx::tma_load_4d(base + Cfg::OFF_RAW + rst * Cfg::RAW_MAX, &tmX, rb, x0, y0,
                                         (kb * 64) / taps, n);
                        rissued |= 1u << rst;
                        rlast = (rlast & ~(1u << rst)) | (rph << rst);
                        if (++rst == (uint32_t)Cfg::RSTAGES) { rst = 0; rph ^= 1u; }
                    }
                }
            }
            if (!ok) pipe_fail(pp);
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s))
                    ptx::mbar_wait_bounded(pp.full0 + 8 * s, (last_par >> s) & 1u, DRAIN_NS, nullptr);
            for (int s = 0; s < Cfg::RSTAGES; ++s)
                if (rissued & (1u << s))
                    ptx::mbar_wait_bounded(rfull0 + 8 * s, (rlast >> s) & 1u, DRAIN_NS, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0)
            mma_role<BN, STAGES, false, true>(pp, sA, sB, p.num_tiles, p.num_kb,
                                              ptx::idesc_f16(p.ab_bf16 != 0, false, true, 128, BN), tlast);
    } else if (warp >= 6 && WIN) {
        // ------------------------------------ B-tile build from the window --
        // Same lane -> (tile row, 8-pixel vector) mapping and B-tile
        // addressing as the global-load gather below.  Window element
        // (cc, hr, wc) is x[n][c_lo + cc][y0 + hr*esh][x0 + wc]; row k =
        // (ci, r, q) of output pixel (t_row, 8 t_vec + e) reads window row
        // (ci - c_lo, t_row*rowmul + r*rstep) at column u + 8 S t_vec + S e
        // with u = (tile column origin - x0) + q*dw.
        constexpr int ROWS = 64 / Cfg::GATHER_WARPS;
        constexpr int GRP = S == 1 ? 8 : 4;
        static_assert(ROWS % GRP == 0, "row split");
        const int gw = warp - 6;
        const int taps = p.kh * p.kw;
        const int vpr = p.TW >> 3;
        const int t_row = lane / vpr, t_vec = lane - (lane / vpr) * vpr;
        const int pcol = t_row * p.TW + t_vec * 8;
        const uint32_t lane_off = (uint32_t)((pcol >> 6) * 8192);
        const uint32_t pc8 = (uint32_t)((pcol >> 3) & 7);
        const int lane_raw = t_row * p.rowmul * p.WB + t_vec * 8 * S;
        uint32_t stage = 0, phase = 0, rst = 0, rph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
            int n, toh, tow, cb;
            vconv_tile(t, p, n, toh, tow, cb);
            const int xs = tow * p.TW * S - p.pl;
            const int off0 = xs - (xs & ~7);
            for (int kb = 0; kb < p.num_kb; ++kb) {
                // lanes 0..ROWS-1 decode this warp's rows before the waits
                int my_row = 0, my_u = 0, my_ok = 0;
                if (lane < ROWS) {
                    const int k = kb * 64 + gw * ROWS + lane;
                    if (k < p.K) {
                        const int ci = k / taps;
                        const int tap = k - ci * taps;
                        const int r = tap / p.kw;
                        my_row = ((ci - (kb * 64) / taps) * p.HB + r * p.rstep) * p.WB;
                        my_u = off0 + (tap - r * p.kw) * p.dw;
                        my_ok = 1;
                    }
                }
                if (!warp_pipe_wait(pp, rfull0 + 8 * rst, rph) ||
                    !warp_pipe_wait(pp, pp.empty0 + 8 * stage, phase ^ 1u)) {
                    ok = false;
                    break;
                }
                const uint32_t rbuf = base + Cfg::OFF_RAW + rst * Cfg::RAW_MAX + 2u * (uint32_t)lane_raw;
                const uint32_t bt = sB + stage * Cfg::B_BYTES + lane_off;
#pragma unroll
                for (int g = 0; g < ROWS; g += GRP) {
                    uint4 ch[GRP][NCH];
                    int shift[GRP], rok[GRP];
#pragma unroll
                    for (int i = 0; i < GRP; ++i) {
                        const int row = __shfl_sync(0xffffffffu, my_row, g + i);
                        const int u = __shfl_sync(0xffffffffu, my_u, g + i);
                        rok[i] = __shfl_sync(0xffffffffu, my_ok, g + i);
                        shift[i] = u & 7;
                        const uint32_t a = rbuf + 2u * (uint32_t)(row + (u & ~7));
#pragma unroll
                        for (int c = 0; c < NCH; ++c) ch[i][c] = ptx::ld_shared_v4(a + 16u * c);
                    }
#pragma unroll
                    for (int i = 0; i < GRP; ++i) {
                        uint32_t w[4 * NCH];
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            w[4 * c + 0] = ch[i][c].x;
                            w[4 * c + 1] = ch[i][c].y;
                            w[4 * c + 2] = ch[i][c].z;
                            w[4 * c + 3] = ch[i][c].w;
                        }
                        uint32_t o[4];
                        pick8<S>(shift[i], w, o);
                        if (!rok[i]) o[0] = o[1] = o[2] = o[3] = 0u;   // rows past K
                        const int kl = gw * ROWS + g + i;
                        ptx::st_shared_v4(bt + (uint32_t)kl * 128u + ((pc8 ^ (uint32_t)(kl & 7)) << 4), o[0],
                                          o[1], o[2], o[3]);
                    }
                }
                __syncwarp();   // the MMA thread fences the stores into the async proxy
                if (lane == 0) {
                    ptx::mbar_arrive(rempty0 + 8 * rst);
                    ptx::mbar_arrive(pp.full0 + 8 * stage);
                }
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                if (++rst == (uint32_t)Cfg::RSTAGES) { rst = 0; rph ^= 1u; }
            }
        }
        if (ok && my_tiles > 0) {
            // ------------------------------- help with the last tile's epilogue --
            // Gather warp g (lane quarter g & 3) takes units u = 1 + (g >> 2)
            // (mod 3) of the CTA's last tile, staged in the operand ring, which
            // no MMA reads any more once that tile's accumulator is complete
            // (signalled on tlast, which only the last tile's commit reaches).
            const int hq = warp & 3, hslot = 1 + ((warp - 6) >> 2);
            const uint32_t hacc = (uint32_t)((my_tiles - 1) & 1);
            int n, toh, tow, cb;
            vconv_tile(t_last, p, n, toh, tow, cb);
            const int co_row0 = cb * 128 + hq * 32;
            const int co = co_row0 + lane;
            const float brow = (p.bias != nullptr && co < p.Co) ? __ldg(p.bias + co) : 0.0f;
            if (warp_epi_wait(pp, tlast, 0)) {
                ptx::tc_fence_after();
                const uint32_t tbase = pp.tmem + ((uint32_t)(hq * 32) << 16) + hacc * BN;
                const uint32_t hbuf = sB + (uint32_t)(warp - 6) * 8192u;
                uint32_t hunits = 0;
#pragma unroll 1
                for (int u = hslot; u < BN / COLS; u += 3) {
                    const uint32_t buf = hbuf + (hunits++ & 1u) * 4096u;
                    if (lane == 0) ptx::bulk_wait_read<1>();
                    __syncwarp();
                    store_unit(n, toh, tow, co_row0, brow, tbase, u, buf);
                }
                ptx::tc_fence_before();
                if (lane == 0) ptx::bulk_wait<0>();
                __syncwarp();
            } else {
                ok = false;
            }
        }
        if (!ok) pipe_fail(pp);
    } else if (warp >= 6) {
        // ---------------------------------------------------- B-tile gather --
        // Rows are handled in groups of 4: the loads of a whole group are
        // issued before any of its byte-picks, and the first group's loads go
        // out before the wait for the ring slot, so load latency overlaps.
        constexpr int ROWS = 64 / Cfg::GATHER_WARPS;     // K rows per warp and stage
        constexpr int GRP = S == 1 ? 8 : 4;                // rows whose loads are issued together
        static_assert(ROWS <= 32 && ROWS % GRP == 0, "row split");
        const int gw = warp - 6;                         // owns K rows [gw*ROWS, +ROWS) of a stage
        const int HW = p.H * p.W;
        const int taps = p.kh * p.kw;
        const int vpr = p.TW >> 3;                       // vectors per tile row: 8 or 4
        const int t_row = lane / vpr, t_vec = lane - (lane / vpr) * vpr;
        const int pcol = t_row * p.TW + t_vec * 8;       // B-tile column of this lane's first pixel
        const uint32_t lane_off = (uint32_t)((pcol >> 6) * 8192);
        const uint32_t pc8 = (uint32_t)((pcol >> 3) & 7);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
            int n, toh, tow, cb;
            vconv_tile(t, p, n, toh, tow, cb);
            const int oh = toh * p.TH + t_row;
            const int ihb = oh * p.sh - p.pt;            // input row of tap r = 0
            const int iwb = (tow * p.TW + t_vec * 8) * S - p.pl;
            const int ihbW = ihb * p.W;
            const uint16_t *xn = p.x + (int64_t)n * p.C * HW;
            for (int kb = 0; kb < p.num_kb; ++kb) {
                // Lanes 0..ROWS-1 decode this warp's K rows k = (ci, r, q) in
                // parallel; each row's offsets are then broadcast by shuffles,
                // so the row loop below has no divisions and no branches.  A
                // row past K gets an r*dh that puts every lane out of range.
                int my_rowoff = 0, my_rdh = 1 << 28, my_qdw = 0;
                if (lane < ROWS) {
                    const int k = kb * 64 + gw * ROWS + lane;
                    if (k < p.K) {
                        const int ci = k / taps;
                        const int tap = k - ci * taps;
                        const int r = tap / p.kw;
                        my_rdh = r * p.dh;
                        my_qdw = (tap - r * p.kw) * p.dw;
                        my_rowoff = ci * HW + my_rdh * p.W;
                    }
                }
                const uint32_t bt = sB + stage * Cfg::B_BYTES + lane_off;
#pragma unroll 1
                for (int g = 0; g < ROWS; g += GRP) {
                    uint4 ch[GRP][NCH];
                    int shift[GRP];
#pragma unroll
                    for (int i = 0; i < GRP; ++i) {
                        const int rowoff = __shfl_sync(0xffffffffu, my_rowoff, g + i);
                        const int rdh = __shfl_sync(0xffffffffu, my_rdh, g + i);
                        const int qdw = __shfl_sync(0xffffffffu, my_qdw, g + i);
                        const bool rowok = (unsigned)(ihb + rdh) < (unsigned)p.H;
                        const int iws = iwb + qdw;
                        const int c0 = iws >> 3;                 // floor(iws / 8)
                        const int e0 = rowoff + ihbW + c0 * 8;   // element offset of chunk c0
                        shift[i] = iws & 7;
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            ch[i][c] = make_uint4(0u, 0u, 0u, 0u);
                            if (rowok && (unsigned)(c0 + c) < (unsigned)p.W8) ch[i][c] = ldg16(xn + e0 + c * 8);
                        }
                    }
                    if (g == 0) {
                        if (!warp_pipe_wait(pp, pp.empty0 + 8 * stage, phase ^ 1u)) { ok = false; break; }
                    }
#pragma unroll
                    for (int i = 0; i < GRP; ++i) {
                        uint32_t w[4 * NCH];
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            w[4 * c + 0] = ch[i][c].x;
                            w[4 * c + 1] = ch[i][c].y;
                            w[4 * c + 2] = ch[i][c].z;
                            w[4 * c + 3] = ch[i][c].w;
                        }
                        uint32_t o[4];
                        pick8<S>(shift[i], w, o);
                        const int kl = gw * ROWS + g + i;
                        ptx::st_shared_v4(bt + (uint32_t)kl * 128u + ((pc8 ^ (uint32_t)(kl & 7)) << 4), o[0],
                                          o[1], o[2], o[3]);
                    }
                }
                if (!ok) break;
                __syncwarp();   // the MMA thread fences the stores into the async proxy
                if (lane == 0) ptx::mbar_arrive(pp.full0 + 8 * stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (ok && my_tiles > 0) {
            // ------------------------------- help with the last tile's epilogue --
            // Gather warp g (lane quarter g & 3) takes units u = 1 + (g >> 2)
            // (mod 3) of the CTA's last tile, staged in the operand ring, which
            // no MMA reads any more once that tile's accumulator is complete
            // (signalled on tlast, which only the last tile's commit reaches).
            const int hq = warp & 3, hslot = 1 + ((warp - 6) >> 2);
            const uint32_t hacc = (uint32_t)((my_tiles - 1) & 1);
            int n, toh, tow, cb;
            vconv_tile(t_last, p, n, toh, tow, cb);
            const int co_row0 = cb * 128 + hq * 32;
            const int co = co_row0 + lane;
            const float brow = (p.bias != nullptr && co < p.Co) ? __ldg(p.bias + co) : 0.0f;
            if (warp_epi_wait(pp, tlast, 0)) {
                ptx::tc_fence_after();
                const uint32_t tbase = pp.tmem + ((uint32_t)(hq * 32) << 16) + hacc * BN;
                const uint32_t hbuf = sB + (uint32_t)(warp - 6) * 8192u;
                uint32_t hunits = 0;
#pragma unroll 1
                for (int u = hslot; u < BN / COLS; u += 3) {
                    const uint32_t buf = hbuf + (hunits++ & 1u) * 4096u;
                    if (lane == 0) ptx::bulk_wait_read<1>();
                    __syncwarp();
                    store_unit(n, toh, tow, co_row0, brow, tbase, u, buf);
                }
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
        const uint32_t my_buf = base + Cfg::OFF_EPI + (uint32_t)qd * 8192u;
        uint32_t acc = 0, acc_phase = 0, units = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
            int n, toh, tow, cb;
            vconv_tile(t, p, n, toh, tow, cb);
            const int co_row0 = cb * 128 + qd * 32;
            const int co = co_row0 + lane;
            const float brow = (p.bias != nullptr && co < p.Co) ? __ldg(p.bias + co) : 0.0f;
            if (!warp_epi_wait(pp, pp.tfull0 + 8 * acc, acc_phase)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t tbase = pp.tmem + ((uint32_t)(qd * 32) << 16) + acc * BN;
            const int ustep = t == t_last ? 3 : 1;      // last tile: units 0, 3, 6 (helpers: the rest)
#pragma unroll 1
            for (int u = 0; u < BN / COLS; u += ustep) {
                const uint32_t buf = my_buf + (units++ & 1u) * 4096u;
                if (lane == 0) ptx::bulk_wait_read<1>();
                __syncwarp();
                store_unit(n, toh, tow, co_row0, brow, tbase, u, buf);
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

template <int OUT, int S, bool WIN>
static cudaError_t launch_vec_t(const ConvLaunch &L, cudaStream_t stream)
{
    using Cfg = ConvVecCfg<WIN>;
    return launch_k(conv_vec_kernel<OUT, S, WIN>, L.grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream, L.tmW,
                    L.tmY, L.tmY4, L.tmX, L.args);
}

template <int OUT, int S, bool WIN>
static cudaError_t setup_vec_t()
{
    return cudaFuncSetAttribute(conv_vec_kernel<OUT, S, WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                ConvVecCfg<WIN>::SMEM_BYTES);
}

template <bool WIN>
static cudaError_t setup_vec_w()
{
    cudaError_t e = setup_vec_t<OUT_BF16, 1, WIN>();
    if (e == cudaSuccess) e = setup_vec_t<OUT_F16, 1, WIN>();
    if (e == cudaSuccess) e = setup_vec_t<OUT_F32, 1, WIN>();
    if (e == cudaSuccess) e = setup_vec_t<OUT_BF16, 2, WIN>();
    if (e == cudaSuccess) e = setup_vec_t<OUT_F16, 2, WIN>();
    if (e == cudaSuccess) e = setup_vec_t<OUT_F32, 2, WIN>();
    return e;
}

cudaError_t setup_conv_vec_kernels()
{
    cudaError_t e = setup_vec_w<false>();
    if (e == cudaSuccess) e = setup_vec_w<true>();
    return e;
}

template <bool WIN>
static cudaError_t launch_vec_w(const ConvLaunch &L, cudaStream_t stream)
{
    const int s = L.args.sw;
    if (s == 1) {
        if (L.out == OUT_BF16) return launch_vec_t<OUT_BF16, 1, WIN>(L, stream);
        if (L.out == OUT_F16) return launch_vec_t<OUT_F16, 1, WIN>(L, stream);
        if (L.out == OUT_F32) return launch_vec_t<OUT_F32, 1, WIN>(L, stream);
    } else if (s == 2) {
        if (L.out == OUT_BF16) return launch_vec_t<OUT_BF16, 2, WIN>(L, stream);
        if (L.out == OUT_F16) return launch_vec_t<OUT_F16, 2, WIN>(L, stream);
        if (L.out == OUT_F32) return launch_vec_t<OUT_F32, 2, WIN>(L, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_conv_vec(const ConvLaunch &L, cudaStream_t stream)
{
    return L.args.win ? launch_vec_w<true>(L, stream) : launch_vec_w<false>(L, stream);
}

}  // namespace mmact
