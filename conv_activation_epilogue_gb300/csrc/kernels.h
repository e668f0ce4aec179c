// kernels.h -- host-side view of the kernels: argument blocks and launchers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "mmact.h"

namespace mmact {

struct GemmArgs {
    int M, N, K;
    int tiles_m, tiles_n, num_tiles, num_kb;
    int group_m;         // M tiles that share one sweep over N (L2 reuse)
    int ab_bf16;         // 1: bf16 operands, 0: fp16
    int act;             // ACT_*
    float alpha;
    const float *bias;   // [N] or null
    const void *res;     // residual [M, N] in the output dtype, or null
    unsigned int *status;
    unsigned long long wait_ns;
    int l2_policy;       // CTA-pair kernel: 0 no hints; 1 B and C evict-first (A strips stay in L2)
};

struct GemmLaunch {
    CUtensorMap tmA, tmB, tmC, tmCt;   // tmCt: 32-column tail store map (224-wide tiles)
    CUtensorMap tmR;                   // residual, laid out as tmC (CTA-pair kernel; when res != null)
    GemmArgs args;
    int tile_n;          // 64, 128, 192, 224 or 256
    int out;             // OUT_*
    int grid;
    int split_k;         // 0: persistent kernel; 2 or 4: split-K cluster kernel (tile_n 256)
    int pair;            // 1: CTA-pair kernel (256 x 256 tiles over two SMs)
};

struct ConvArgs {
    int Nb, C, H, W, Co, kh, kw;
    int sh, sw, pt, pl, dh, dw;
    int Ho, Wo, P;       // P = Ho * Wo
    int K;               // C * kh * kw
    int tiles_co, tiles_p, num_tiles, num_kb;
    int ab_bf16;
    int act;
    float alpha;
    int vec;             // 1: vectorised producer (conv_vec.cu), 0: per-element gather
    int TW, TH;          // vectorised path: output tile of TH rows x TW columns (TW * TH = 256)
    int tiles_oh, tiles_ow, W8;
    int win;             // vectorised path: 1 = input window staged in smem by TMA (below)
    int WB, HB, CB;      //   window box: WB columns x HB rows x CB channels
    int rstep, rowmul;   //   window rows per filter row r, per output row of the tile
    int raw_bytes;       //   bytes of one window
    int a_tma;           // 1: filter tiles by TMA, 0: gathered by the producer warps
    int y_tma;           // 1: output tiles by TMA store, 0: direct global stores
    int f32;             // 1: fp32 x and w, each split into bf16 hi + lo (three MMAs per K step)
    int bias_col;        // 1: bias per output pixel column (a GEMM run as a 1x1 conv), 0: per channel
    int nhwc;            // 1 (with f32): channels-last x [N,H,W,C], filter [Co,kh,kw,C], y [N,Ho,Wo,Co]
    int out_elem_bytes;
    const uint16_t *x;
    const uint16_t *w;
    const float *bias;
    const void *res;     // residual shaped like y (output dtype), or null
    void *y;
    unsigned int *status;
    unsigned long long wait_ns;
};

// Largest input window (bytes) the vectorised conv kernel stages per K block.
constexpr int CONV_WIN_MAX_BYTES = 24576;

struct ConvLaunch {
    CUtensorMap tmW, tmY, tmY4, tmX;
    ConvArgs args;
    int out;
    int grid;
};

// One-time per-device set-up (dynamic shared-memory opt-in of every instance);
// must run with the device current, before the first launch on it.
cudaError_t setup_gemm_kernels();
cudaError_t setup_conv_kernels();
cudaError_t setup_conv_vec_kernels();
cudaError_t launch_conv_vec(const ConvLaunch &L, cudaStream_t stream);
// Channels-last conv2d as implicit GEMM: M = output pixels (n, oh, ow),
// N = output channels, K = (r, q, ci).
struct NhwcArgs {
    int Nb, C, H, W, Co, kh, kw;
    int sh, sw, pt, pl, dh, dw;
    int Ho, Wo;
    int M;               // Nb * Ho * Wo output pixels
    int ncb;             // channel blocks of kc per tap
    int kc;              // channels per K block: 64 (16-bit inputs) or 32 (fp32 inputs): 128 bytes
    int tf32;            // 1: fp32 inputs, tcgen05 kind::tf32
    int TW, TH;          // output pixels per tile: TH rows x TW columns (TW * TH = 128)
    int tiles_oh, tiles_ow;
    int tiles_m, tiles_n, num_tiles, num_kb;   // tiles_m = Nb * tiles_oh * tiles_ow; num_kb = kh * kw * ncb
    int group_m;
    int ab_bf16;
    int act;
    float alpha;
    const void *x;
    const float *bias;   // [Co] or null
    const void *res;     // residual shaped like y (output dtype), or null
    unsigned int *status;
    unsigned long long wait_ns;
};

struct NhwcLaunch {
    CUtensorMap tmX, tmW, tmY;   // x as {C, W, H, N}; filter as {C, kh*kw, Co}; y as {Co, Wo, Ho, N}
    NhwcArgs args;
    int tile_n;
    int out;
    int grid;
};

// NCHW conv with the im2col operand in tensor memory (conv_tmem.cu).
// Largest raw input window (bytes) staged per K block, and the size of the
// K-offset table (entries: lcm(64, kh*kw) must fit).
constexpr int CONV_TMEM_WIN_MAX_BYTES = 40960;
constexpr int CONV_TMEM_TABLE_MAX = 3136;
constexpr int CONV_TMEM_MAX_WSTAGES = 8;

struct TmemConvArgs {
    int Nb, C, H, W, Co, kh, kw;
    int sh, sw, pt, pl, dh, dw;
    int Ho, Wo, P, K;
    int tiles_co, tiles_p, num_tiles, num_kb;   // tiles: 128 consecutive pixels of one image x BN channels
    int ab_bf16;
    int act;
    float alpha;
    int WB, HB, CB;      // raw window per K block: WB columns x HB rows x CB channels
    int esh;             // TMA row traversal stride of the window (sh when every used row is a multiple of sh apart)
    int rowmul, rstep;   // window rows per output row of the tile, per filter row r
    int x0, xoff;        // window column origin (8-aligned) and -pl - x0
    int raw_bytes;
    int win_slot;        // bytes per window slot (raw_bytes rounded up to 1 KB)
    int wstages;         // window slots in the ring (2..CONV_TMEM_MAX_WSTAGES)
    int y_tma;           // 1: output blocks by TMA store (P * out bytes a multiple of 16)
    int tab_period;      // K-offset table covers tab_period blocks of 64 (the pattern's period)
    const float *bias;
    const void *res;     // residual shaped like y (output dtype), or null
    void *y;
    unsigned int *status;
    unsigned long long wait_ns;
};

struct TmemConvLaunch {
    CUtensorMap tmW, tmX, tmY;   // filter as {K, Co}; x as {W, H, C, N}; y as {P, Co, N}
    TmemConvArgs args;
    int tile_n;             // BN: 64, 128 or 256 output channels per tile
    int out;
    int grid;
};

cudaError_t setup_conv_tmem_kernels();
cudaError_t launch_conv_tmem(const TmemConvLaunch &L, cudaStream_t stream);
// Bytes of shared memory the kernel with tile_n output channels leaves for its window ring.
int conv_tmem_window_region(int tile_n);

cudaError_t setup_nhwc_kernels();
cudaError_t launch_conv_nhwc(const NhwcLaunch &L, cudaStream_t stream);
cudaError_t launch_gemm(const GemmLaunch &L, cudaStream_t stream);
// Split-K over a cluster of L.split_k CTAs, one 128 x 256 tile per cluster
// (grid = tiles x split_k).
cudaError_t setup_splitk_kernels();
cudaError_t launch_gemm_splitk(const GemmLaunch &L, cudaStream_t stream);
// Split-K clusters of S CTAs that fit on the device at once (0: unknown).
int splitk_max_clusters(int S);
// CTA-pair GEMM: one M = 256 tcgen05.mma per pair of SMs (cta_group::2);
// args.tiles_m / tiles_n / num_tiles count 256 x 256 pair tiles, grid = 2 x pairs.
cudaError_t setup_pair_kernels();
cudaError_t launch_gemm_pair(const GemmLaunch &L, cudaStream_t stream);
int pair_max_clusters();

cudaError_t launch_conv(const ConvLaunch &L, cudaStream_t stream);
// out[i] = act(ws[i]) for i < count (ws fp32, out of dtype `out`).
cudaError_t launch_act(const float *ws, void *out, int64_t count, int out_kind, int act,
                       float alpha, int grid, cudaStream_t stream);
// out[r][c] = act(bias[c]) (bias may be null) for an [rows x cols] output;
// with per_row != 0 the bias runs along rows: out[r][c] = act(bias[r % bias_len]).
// out = act(bias (+ res)) for the empty contraction; res, if not null, has
// out's dtype and element order.
cudaError_t launch_bias_act(const float *bias, void *out, int64_t rows, int64_t cols, int per_row,
                            int64_t bias_len, int out_kind, int act, float alpha,
                            cudaStream_t stream, const void *res = nullptr);
cudaError_t launch_wait_selftest(unsigned int *status, unsigned long long timeout_ns,
                                 cudaStream_t stream);

// Host argument checks of the mmact_gemm family (api.cu): MMACT_OK (0), or the
// status the entry points return for these arguments.
mmact_status gemm_check(const void *A, const void *B, const float *bias, const void *C, int64_t M,
                        int64_t N, int64_t K, mmact_dtype ab, mmact_dtype cd, mmact_act act);

}  // namespace mmact
