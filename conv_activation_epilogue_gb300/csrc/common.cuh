// common.cuh -- device code shared by the fused GEMM and implicit-GEMM conv
// kernels: the activation functions, output packing, the tcgen05 MMA issuer
// role and the TMEM -> registers -> swizzled shared memory epilogue unit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace mmact {

enum : int { ACT_NONE = 0, ACT_RELU = 1, ACT_LEAKY = 2, ACT_TANH = 3, ACT_SIGMOID = 4, ACT_GELU = 5 };
enum : int { OUT_F32 = 0, OUT_F16 = 1, OUT_BF16 = 2 };

// Bits of the per-device status word.
enum : unsigned { ST_TIMEOUT = 1u, ST_SMEM_ALIGN = 2u, ST_PAIR_TMEM = 4u };

constexpr uint64_t DRAIN_NS = 1000000000ull;   // bound on end-of-kernel drains

// tanh in fp32 with the hardware's tanh.approx.f32 (one MUFU operation; the
// ratio-of-exponentials form (e^z - e^-z)/(e^z + e^-z) would take two, an
// exponential and a reciprocal).  Its relative error, about 2^-11, is well
// inside the output tolerance; it saturates to +-1 without overflow.
__device__ __forceinline__ float tanh_f32(float z)
{
    return ptx::tanh_approx(z);
}

// 1 / (1 + e^-z) = (1 + tanh(z/2)) / 2: one MUFU operation, absolute error
// about 2^-12, saturating to 0 and 1.
__device__ __forceinline__ float sigmoid_f32(float z)
{
    return fmaf(0.5f, ptx::tanh_approx(0.5f * z), 0.5f);
}

// erf(x) by Abramowitz and Stegun, Handbook of Mathematical Functions, formula
// 7.1.26: for x >= 0, erf(x) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5))))
// e^{-x^2} with t = 1 / (1 + p x), absolute error below 1.5e-7 (5.4e-7 in this
// fp32 evaluation); erf is odd.  Branch-free: one hardware exponential, one
// hardware reciprocal (fast division, a few ulp: far below the formula's own
// error) and five FMAs, so a warp can keep many in flight -- the epilogue of
// a small tile evaluates dozens per thread.
__device__ __forceinline__ float erf_as7126(float x)
{
    const float ax = fabsf(x);
    const float t = __fdividef(1.0f, fmaf(0.3275911f, ax, 1.0f));
    float poly = fmaf(1.061405429f, t, -1.453152027f);
    poly = fmaf(poly, t, 1.421413741f);
    poly = fmaf(poly, t, -0.284496736f);
    poly = fmaf(poly, t, 0.254829592f);
    const float e = 1.0f - poly * t * __expf(-ax * ax);
    return copysignf(e, x);
}

// z * Phi(z) = z/2 * (1 + erf(z / sqrt(2))).
__device__ __forceinline__ float gelu_f32(float z)
{
    return 0.5f * z * (1.0f + erf_as7126(z * 0.7071067811865476f));
}

template <int ACT>
__device__ __forceinline__ float act_f32(float z, float alpha)
{
    if constexpr (ACT == ACT_RELU) return z > 0.0f ? z : 0.0f;
    else if constexpr (ACT == ACT_LEAKY) return z > 0.0f ? z : alpha * z;
    else if constexpr (ACT == ACT_TANH) return tanh_f32(z);
    else if constexpr (ACT == ACT_SIGMOID) return sigmoid_f32(z);
    else if constexpr (ACT == ACT_GELU) return gelu_f32(z);
    else return z;
}

template <int OUT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    if constexpr (OUT == OUT_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

// Launches `kernel` with programmatic stream serialization: the next kernel
// in the stream may begin its set-up (barrier init, TMEM allocation,
// tensor-map prefetch) while this one finishes, and every kernel of this
// library waits in ptx::griddep_wait() before it touches global data.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Shared-memory addresses of the pipeline's barriers and flags.
struct Pipe {
    uint32_t full0, empty0;      // operand ring: barrier s at +8*s
    uint32_t tfull0, tempty0;    // accumulator ring (2 buffers)
    uint32_t drain;
    uint32_t tmem;               // TMEM base address of the accumulators
    volatile uint32_t *abort;    // set when any role gives up
    unsigned int *status;        // device status word
    uint64_t wait_ns;
};

__device__ __forceinline__ void pipe_fail(const Pipe &pp)
{
    *pp.abort = 1u;
    atomicOr(pp.status, ST_TIMEOUT);
}

// Pipeline waits pass a suspend-time hint: a waiting thread is parked until
// the phase completes (or the hint runs out) instead of re-polling the
// barrier, which otherwise competes with the gather warps' shared-memory
// traffic (measured: the windowed conv producer ran up to 7x slower per
// stage while the MMA and TMA threads polled without a hint).
constexpr uint32_t PIPE_SUSPEND_NS = 100000;

__device__ __forceinline__ bool pipe_wait(const Pipe &pp, uint32_t bar, uint32_t parity)
{
    return ptx::mbar_wait_bounded(bar, parity, pp.wait_ns, pp.abort, PIPE_SUSPEND_NS);
}

// Spinning variant for waits on the critical path whose phase is completed
// by thread arrivals (no suspend hint: the waiting thread re-polls).
__device__ __forceinline__ bool pipe_wait_spin(const Pipe &pp, uint32_t bar, uint32_t parity)
{
    return ptx::mbar_wait_bounded(bar, parity, pp.wait_ns, pp.abort, 0);
}

__device__ __forceinline__ bool warp_pipe_wait_spin(const Pipe &pp, uint32_t bar, uint32_t parity)
{
    const uint32_t r = pipe_wait_spin(pp, bar, parity) ? 1u : 0u;
    return __shfl_sync(0xffffffffu, r, 0) != 0u;
}

// The epilogue's wait for a finished accumulator: long, and not on the
// critical path, so the waiting warps are parked between polls.
__device__ __forceinline__ bool epi_wait(const Pipe &pp, uint32_t bar, uint32_t parity)
{
    return ptx::mbar_wait_bounded(bar, parity, pp.wait_ns, pp.abort, 1000);
}

// Waits made on behalf of a whole warp: every lane polls, and the warp takes
// lane 0's verdict so that it leaves convergent.  (Polling from lane 0 alone
// while the other 31 lanes sat at a warp-synchronous shuffle was measured to
// slow the other warps of the SM several-fold: a conv producer stage took
// ~7.4k cycles instead of ~1.0k while epilogue warps waited that way.)
__device__ __forceinline__ bool warp_pipe_wait(const Pipe &pp, uint32_t bar, uint32_t parity)
{
    const uint32_t r = pipe_wait(pp, bar, parity) ? 1u : 0u;
    return __shfl_sync(0xffffffffu, r, 0) != 0u;
}

__device__ __forceinline__ bool warp_epi_wait(const Pipe &pp, uint32_t bar, uint32_t parity)
{
    const uint32_t r = epi_wait(pp, bar, parity) ? 1u : 0u;
    return __shfl_sync(0xffffffffu, r, 0) != 0u;
}

// The MMA issuer (one thread).  For every tile of this CTA it waits for a free
// accumulator buffer, then for each K block waits for the operand stage,
// issues BK/16 tcgen05.mma instructions and commits the stage back to the
// producer; the finished accumulator is committed to the epilogue.
//   A stage: [128 rows x 64 K] K-major, 128-byte swizzle (rows 128 B apart,
//            8-row groups 1024 B apart); the K step of 16 moves 32 bytes.
//   B stage: [64 K x BN] MN-major, 128-byte swizzle, BN/64 column chunks of
//            64 K rows x 128 B each (chunk stride 8192 B); the K step of 16
//            moves 16 rows = 2048 bytes.
// Tile geometry shared by the producer, MMA issuer and epilogue: BN columns
// per tile, stored as ceil(BN/64) chunks of 64 columns; the two TMEM
// accumulator buffers start 256 columns apart when BN > 128 (BN apart below).
template <int BN>
struct TileN {
    static constexpr int NCHUNK = (BN + 63) / 64;
    static constexpr uint32_t B_BYTES = 64u * 64u * 2u * NCHUNK;
    static constexpr uint32_t ACC_STRIDE = BN > 128 ? 256u : (uint32_t)BN;
    static constexpr uint32_t TMEM_COLS = 2u * ACC_STRIDE;
};

//
// B_KMAJOR: the B stage is instead [BN rows x 64 K] K-major with the same
// 128-byte swizzle as A (rows are output columns; used when B is given as
// [N, K] with K contiguous, e.g. a channels-last filter).
//
// THREAD_FILLED: some operand stage bytes were written by ordinary shared
// stores of producer threads (the conv gathers) rather than by TMA.  Those
// threads only store and arrive on the full barrier (release); this thread,
// after acquiring the barrier, issues the one generic-to-async proxy fence
// that makes the stores visible to the tensor core's operand reads.
// TF32: the operands are fp32 (kind::tf32, 8 K per instruction = 32 bytes,
// the same K step as the 16-bit kinds; both operands must be K-major).
// last_bar (optional, 0 = none): an mbarrier of count 1 that also receives the
// commit of the CTA's last tile, so that warps which only help with that
// tile's epilogue can wait for it by phase 0 (a parity wait on the
// accumulator barrier alone could match an earlier tile's phase when those
// warps run far ahead of the MMAs).
template <int BN, int STAGES, bool B_KMAJOR = false, bool THREAD_FILLED = false, bool TF32 = false>
__device__ void mma_role(const Pipe &pp, uint32_t sA, uint32_t sB, int num_tiles, int num_kb,
                         uint32_t idesc, uint32_t last_bar = 0)
{
    constexpr uint32_t A_BYTES = 128 * 64 * 2;
    constexpr uint32_t B_BYTES = B_KMAJOR ? (uint32_t)BN * 128u : TileN<BN>::B_BYTES;
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        if (!pipe_wait(pp, pp.tempty0 + 8 * acc, acc_phase ^ 1u)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t d = pp.tmem + acc * TileN<BN>::ACC_STRIDE;
        for (int kb = 0; kb < num_kb; ++kb) {
            if (!pipe_wait(pp, pp.full0 + 8 * stage, phase)) { ok = false; break; }
            if constexpr (THREAD_FILLED) ptx::fence_proxy_async_smem();
            ptx::tc_fence_after();
            const uint32_t a0 = sA + stage * A_BYTES, b0 = sB + stage * B_BYTES;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint64_t ad = ptx::smem_desc(a0 + 32u * k, 16u, 1024u, ptx::SWIZZLE_128B);
                const uint64_t bd = B_KMAJOR ? ptx::smem_desc(b0 + 32u * k, 16u, 1024u, ptx::SWIZZLE_128B)
                                             : ptx::smem_desc(b0 + 2048u * k, 8192u, 1024u, ptx::SWIZZLE_128B);
                if constexpr (TF32) ptx::mma_tf32(d, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                else ptx::mma_f16(d, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            }
            ptx::mma_commit(pp.empty0 + 8 * stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit(pp.tfull0 + 8 * acc);
        if (last_bar != 0 && t + (int)gridDim.x >= num_tiles) ptx::mma_commit(last_bar);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) pipe_fail(pp);
    // Every MMA this thread issued must finish before TMEM is released.
    ptx::mma_commit(pp.drain);
    ptx::mbar_wait_bounded(pp.drain, 0, DRAIN_NS, nullptr);
}

// Two 16-bit output values (one 32-bit word, low half first) as floats.
template <int OUT>
__device__ __forceinline__ float2 unpack2(uint32_t w)
{
    if constexpr (OUT == OUT_BF16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        __half2 h = *reinterpret_cast<__half2 *>(&w);
        return __half22float2(h);
    }
}

// PER residual values of this lane's row segment starting at column c0 (the
// segment holds elements of the output dtype; columns at or past nvalid read
// as 0).  One 16-byte load when the chunk is whole and aligned.  Plain,
// coherent loads (not the read-only path): the residual may be the output
// tensor itself, each element read here before this unit's store writes it.
template <int OUT, int PER>
__device__ __forceinline__ void residual_chunk(const void *res, int nvalid, int c0, float (&v)[PER])
{
    constexpr int ESZ = OUT == OUT_F32 ? 4 : 2;
    static_assert(PER * ESZ == 16, "one chunk is 16 bytes");
    if (res == nullptr) {                              // this lane's row is out of range
#pragma unroll
        for (int j = 0; j < PER; ++j) v[j] = 0.0f;
        return;
    }
    const char *p = static_cast<const char *>(res) + c0 * ESZ;
    if (c0 + PER <= nvalid && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if constexpr (OUT == OUT_F32) {
                v[e] = __uint_as_float(w[e]);
            } else {
                const float2 f = unpack2<OUT>(w[e]);
                v[2 * e] = f.x;
                v[2 * e + 1] = f.y;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            float x = 0.0f;
            if (c0 + j < nvalid) {
                if constexpr (OUT == OUT_F32) x = reinterpret_cast<const float *>(p)[j];
                else if constexpr (OUT == OUT_BF16) x = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[j]);
                else x = __half2float(reinterpret_cast<const __half *>(p)[j]);
            }
            v[j] = x;
        }
    }
}

// a + r when the residual is read in the packing loop, a otherwise (no add:
// a + 0.0f is not an identity in IEEE arithmetic, -0 + 0 = +0).
template <bool ADD>
__device__ __forceinline__ float plus_if(float a, float r)
{
    if constexpr (ADD) return a + r;
    else return a;
}

// Adds this lane's residual row segment -- COLS elements of the output dtype
// from `res` -- to v[0..min(nvalid, COLS)): one branch, then all of its
// 16-byte loads issued together (coherent loads: the residual may be the
// output tensor itself, each element read before this unit's store).
template <int OUT, int COLS>
__device__ __forceinline__ void add_residual(const void *res, int nvalid, float (&v)[COLS])
{
    constexpr int PER = OUT == OUT_F32 ? 4 : 8;      // elements per 16 bytes
    if (res == nullptr) return;                        // this lane's row is out of range
    if (nvalid >= COLS && (reinterpret_cast<uintptr_t>(res) & 15u) == 0) {
        const uint4 *q = reinterpret_cast<const uint4 *>(res);
        uint4 u[COLS / PER];
#pragma unroll
        for (int c = 0; c < COLS / PER; ++c) u[c] = q[c];
#pragma unroll
        for (int c = 0; c < COLS / PER; ++c) {
            const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if constexpr (OUT == OUT_F32) {
                    v[4 * c + e] += __uint_as_float(w[e]);
                } else {
                    const float2 f = unpack2<OUT>(w[e]);
                    v[8 * c + 2 * e] += f.x;
                    v[8 * c + 2 * e + 1] += f.y;
                }
            }
        }
    } else {
#pragma unroll
        for (int c = 0; c < COLS; c += PER) {
            float rv[PER];
            residual_chunk<OUT, PER>(res, nvalid, c, rv);
#pragma unroll
            for (int j = 0; j < PER; ++j) v[c + j] += rv[j];
        }
    }
}

// Adds this lane's residual row segment staged in shared memory by a TMA load
// through the output's tensor map (128-byte rows, 16-byte chunk c of row r at
// chunk c ^ (r & 7)): the 8 chunks of `row`, swizzled by `sw`.
template <int OUT, int COLS>
__device__ __forceinline__ void add_residual_smem(uint32_t row, uint32_t sw, float (&v)[COLS])
{
    constexpr int PER = OUT == OUT_F32 ? 4 : 8;
    static_assert(COLS == 8 * PER, "one 128-byte row segment");
    uint4 u[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) u[c] = ptx::ld_shared_v4(row + (((uint32_t)c ^ sw) << 4));
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if constexpr (OUT == OUT_F32) {
                v[4 * c + e] += __uint_as_float(w[e]);
            } else {
                const float2 f = unpack2<OUT>(w[e]);
                v[8 * c + 2 * e] += f.x;
                v[8 * c + 2 * e + 1] += f.y;
            }
        }
    }
}

// One epilogue unit: 32 rows (this warp's TMEM lane quarter) x one 128-byte
// output row segment (32 fp32 or 64 16-bit columns).  Loads the fp32
// accumulators from TMEM, adds the fp32 bias (per column from global memory
// `bias_col[0..nvalid)`, zero beyond it or when null; or the per-row `brow`),
// adds the lane's residual row segment when `res` is not null (with RSMEM: the
// segment already staged in `buf` at this lane's row, which the output then
// overwrites in place), applies the
// activation in fp32, converts, and writes the row into a
// 32 x 128 B shared buffer in the 128-byte swizzled order a TMA store expects
// (16-byte chunk c of row r lands at chunk c ^ (r & 7)).
//
// NCOL = 32 with a 16-bit output is the narrow tail unit of a 224-wide tile:
// 64-byte rows, written densely without swizzle (its TMA store uses an
// unswizzled map).
template <int OUT, int ACT, bool BIAS_ROW, int NCOL, bool RES, bool RSMEM = false>
__device__ __forceinline__ void epi_unit(uint32_t taddr, const float *bias_col, int nvalid,
                                         float brow, float alpha, uint32_t buf, int lane,
                                         const void *res)
{
    static_assert(!RSMEM || (RES && !BIAS_ROW && NCOL * (OUT == OUT_F32 ? 4 : 2) == 128),
                  "a staged residual is a whole 128-byte row segment with a per-column bias");
    constexpr int COLS = NCOL;
    constexpr bool WIDE = COLS == 64;                  // two TMEM loads per unit
    uint32_t r0[32];
    uint32_t r1[32];
    ptx::tmem_ld32(taddr, r0);
    if constexpr (WIDE) ptx::tmem_ld32(taddr + 32, r1);
    float bc[COLS];
    if (!BIAS_ROW && bias_col != nullptr && nvalid >= COLS &&
        (reinterpret_cast<uintptr_t>(bias_col) & 15u) == 0) {
        // the whole segment is in range and 16-byte aligned: vector loads
#pragma unroll
        for (int j = 0; j < COLS; j += 4) {
            const float4 b4 = __ldg(reinterpret_cast<const float4 *>(bias_col + j));
            bc[j] = b4.x;
            bc[j + 1] = b4.y;
            bc[j + 2] = b4.z;
            bc[j + 3] = b4.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < COLS; ++j)
            bc[j] = BIAS_ROW ? brow : ((bias_col != nullptr && j < nvalid) ? __ldg(bias_col + j) : 0.0f);
    }
    // Residual.  With a per-column bias (GEMM, channels-last conv) bc[] is a
    // per-lane array already: the whole row segment is added into it, its
    // loads issued together before the TMEM wait.  With a per-row bias (NCHW
    // conv) bc[] folds to one register, so the residual is read chunk by
    // chunk in the packing loops instead (from L1: the caller prefetches).
    if constexpr (RSMEM) {
        add_residual_smem<OUT, COLS>(buf + (uint32_t)lane * 128u, (uint32_t)(lane & 7), bc);
    } else if constexpr (RES && !BIAS_ROW) {
        add_residual<OUT, COLS>(res, nvalid, bc);
        __syncwarp();                                  // converge before the warp-collective wait
    }
    constexpr bool CHUNKED = RES && BIAS_ROW;
    ptx::tmem_ld_wait(r0);
    if constexpr (WIDE) ptx::tmem_ld_wait(r1);
    if constexpr (OUT != OUT_F32 && !WIDE) {
        // 32 columns of a 16-bit output: 4 chunks of 16 bytes, row pitch 64 bytes
        const uint32_t row = buf + (uint32_t)lane * 64u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float rv[8] = {};
            if constexpr (CHUNKED) residual_chunk<OUT, 8>(res, nvalid, 8 * c, rv);
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = 8 * c + 2 * e;
                w[e] = pack2<OUT>(act_f32<ACT>(plus_if<CHUNKED>(__uint_as_float(r0[col]) + bc[col], rv[2 * e]), alpha),
                                  act_f32<ACT>(plus_if<CHUNKED>(__uint_as_float(r0[col + 1]) + bc[col + 1], rv[2 * e + 1]),
                                               alpha));
            }
            ptx::st_shared_v4(row + (uint32_t)c * 16u, w[0], w[1], w[2], w[3]);
        }
        return;
    }
    const uint32_t row = buf + (uint32_t)lane * 128u;
    const uint32_t sw = (uint32_t)(lane & 7);
    if constexpr (OUT == OUT_F32) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float rv[4] = {};
            if constexpr (CHUNKED) residual_chunk<OUT, 4>(res, nvalid, 4 * c, rv);
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = 4 * c + e;
                v[e] = act_f32<ACT>(plus_if<CHUNKED>(__uint_as_float(r0[col]) + bc[col], rv[e]), alpha);
            }
            ptx::st_shared_v4(row + (((uint32_t)c ^ sw) << 4), __float_as_uint(v[0]),
                              __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
        }
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float rv[8] = {};
            if constexpr (CHUNKED) residual_chunk<OUT, 8>(res, nvalid, 8 * c, rv);
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = 8 * c + 2 * e;
                const uint32_t ua = col < 32 ? r0[col] : r1[col - 32];
                const uint32_t ub = col + 1 < 32 ? r0[col + 1] : r1[col + 1 - 32];
                w[e] = pack2<OUT>(act_f32<ACT>(plus_if<CHUNKED>(__uint_as_float(ua) + bc[col], rv[2 * e]), alpha),
                                  act_f32<ACT>(plus_if<CHUNKED>(__uint_as_float(ub) + bc[col + 1], rv[2 * e + 1]), alpha));
            }
            ptx::st_shared_v4(row + (((uint32_t)c ^ sw) << 4), w[0], w[1], w[2], w[3]);
        }
    }
}

template <int OUT, bool BIAS_ROW, int NCOL, bool RES, bool RSMEM = false>
__device__ __forceinline__ void epi_unit_act(int act, uint32_t taddr, const float *bias_col, int nvalid,
                                             float brow, float alpha, uint32_t buf, int lane,
                                             const void *res)
{
    switch (act) {
    case ACT_RELU:
        epi_unit<OUT, ACT_RELU, BIAS_ROW, NCOL, RES, RSMEM>(taddr, bias_col, nvalid, brow, alpha, buf, lane, res);
        break;
    case ACT_LEAKY:
        epi_unit<OUT, ACT_LEAKY, BIAS_ROW, NCOL, RES, RSMEM>(taddr, bias_col, nvalid, brow, alpha, buf, lane, res);
        break;
    case ACT_TANH:
        epi_unit<OUT, ACT_TANH, BIAS_ROW, NCOL, RES, RSMEM>(taddr, bias_col, nvalid, brow, alpha, buf, lane, res);
        break;
    case ACT_SIGMOID:
        epi_unit<OUT, ACT_SIGMOID, BIAS_ROW, NCOL, RES, RSMEM>(taddr, bias_col, nvalid, brow, alpha, buf, lane, res);
        break;
    case ACT_GELU:
        epi_unit<OUT, ACT_GELU, BIAS_ROW, NCOL, RES, RSMEM>(taddr, bias_col, nvalid, brow, alpha, buf, lane, res);
        break;
    default:
        epi_unit<OUT, ACT_NONE, BIAS_ROW, NCOL, RES, RSMEM>(taddr, bias_col, nvalid, brow, alpha, buf, lane, res);
        break;
    }
}

// One epilogue unit with the activation and the presence of a residual
// resolved once: the residual-free code carries no residual work.  `has_res`
// must be the same for every lane of the warp (the unit's tcgen05.ld is
// warp-collective); a lane whose row is out of range passes res == nullptr
// and adds nothing.
template <int OUT, bool BIAS_ROW, int NCOL = (OUT == OUT_F32 ? 32 : 64)>
__device__ __forceinline__ void epi_unit_dispatch(int act, uint32_t taddr, const float *bias_col,
                                                  int nvalid, float brow, float alpha, uint32_t buf,
                                                  int lane, const void *res = nullptr, bool has_res = false)
{
    if (has_res)
        epi_unit_act<OUT, BIAS_ROW, NCOL, true>(act, taddr, bias_col, nvalid, brow, alpha, buf, lane, res);
    else
        epi_unit_act<OUT, BIAS_ROW, NCOL, false>(act, taddr, bias_col, nvalid, brow, alpha, buf, lane, res);
}

// The same unit with the residual already staged in `buf` (warp-uniform
// choice between the two by the caller).
template <int OUT, int NCOL = (OUT == OUT_F32 ? 32 : 64)>
__device__ __forceinline__ void epi_unit_dispatch_rsmem(int act, uint32_t taddr, const float *bias_col,
                                                        int nvalid, float alpha, uint32_t buf, int lane)
{
    epi_unit_act<OUT, false, NCOL, true, true>(act, taddr, bias_col, nvalid, 0.0f, alpha, buf, lane, nullptr);
}

}  // namespace mmact
