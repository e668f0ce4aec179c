// api.cu -- the C ABI declared in include/mmact.h: argument validation, the
// launch planner (tile shape, persistent grid, tensor-map encoding) and the
// per-device status word.
//
// Argument checks mirror the MatmulLeakyRelu walkthrough's entry-point
// validation (an invalid value is rejected with the supported set named,
// before anything runs): every check here happens before any launch, and a
// failed check enqueues nothing.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "mmact.h"

#define MMACT_EXPORT extern "C" __attribute__((visibility("default")))

namespace mmact {
namespace {

__device__ unsigned int g_status;   // per-device kernel status word (ST_* bits)

constexpr uint64_t DEFAULT_WAIT_NS = 2000000000ull;
std::atomic<uint64_t> g_wait_ns{DEFAULT_WAIT_NS};
std::atomic<int> g_tile_n{0};
std::atomic<int> g_split_k{0};   // 0: chosen per shape; 1: never; 2 or 4: whenever legal
std::atomic<int> g_pair{0};      // CTA-pair GEMM kernel: 0 chosen per shape; 1 never; 2 always
std::atomic<int> g_conv_tmem{0}; // NCHW conv, im2col operand in TMEM: 0 when supported; 1 never
std::atomic<int> g_l2_policy{1}; // CTA-pair GEMM: 1 A evict-last, C evict-first (default); 0 no cache hints

constexpr int MAX_DEVICES = 64;
struct DeviceInfo {
    bool ready = false;
    int sm_count = 0;
    int splitk_clusters[2] = {0, 0};  // resident split-K clusters of 2 and of 4 CTAs
    int pair_clusters = 0;            // resident CTA pairs of the pair kernel
    unsigned int *status = nullptr;   // device address of g_status
};
DeviceInfo g_dev[MAX_DEVICES];
std::mutex g_dev_mutex;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

mmact_status device_info(DeviceInfo **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return MMACT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MMACT_ERR_CUDA;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_status) != cudaSuccess)
            return MMACT_ERR_CUDA;
        if (setup_gemm_kernels() != cudaSuccess || setup_conv_kernels() != cudaSuccess ||
            setup_conv_vec_kernels() != cudaSuccess || setup_nhwc_kernels() != cudaSuccess ||
            setup_splitk_kernels() != cudaSuccess || setup_pair_kernels() != cudaSuccess ||
            setup_conv_tmem_kernels() != cudaSuccess)
            return MMACT_ERR_CUDA;
        d.pair_clusters = pair_max_clusters();
        d.splitk_clusters[0] = splitk_max_clusters(2);
        d.splitk_clusters[1] = splitk_max_clusters(4);
        if (g_encode == nullptr) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return MMACT_ERR_CUDA;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        d.ready = true;
    }
    *out = &d;
    return MMACT_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int out_kind(mmact_dtype d)
{
    return d == MMACT_BF16 ? OUT_BF16 : (d == MMACT_F16 ? OUT_F16 : OUT_F32);
}
int elem_bytes(mmact_dtype d) { return (d == MMACT_F32 || d == MMACT_TF32) ? 4 : 2; }
CUtensorMapDataType tmap_type(mmact_dtype d)
{
    return d == MMACT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                           : (d == MMACT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32);   // F32, TF32
}

// Tiled map over a row-major tensor given innermost-first dims (elements) and
// the byte strides of dims 1..rank-1, with a 128-byte swizzle (or none).
// `estrides` (optional) are TMA traversal strides per dimension: a box of
// box[i] elements along dimension i then delivers ceil(box[i] / estrides[i]).
//
// A tensor map is a pure function of these arguments (it holds the address,
// not the memory), so encoded maps are kept in a small per-thread cache keyed
// by every argument: a repeated call with the same tensors, shapes and dtypes
// copies 128 bytes instead of encoding again, and a stale entry cannot exist.
// A set-associative cache: the few maps of one call could share a slot of a
// direct-mapped one and evict each other on every call.
struct TmapKey {
    int32_t dt, rank, swizzle, pad;
    const void *ptr;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
};
struct TmapEntry {
    CUtensorMap map;
    TmapKey key;
    bool valid;
};
// 64 sets of 4 entries, per host thread: one call encodes at most 4 maps, so the
// maps of a call never evict one another, whatever their hashes.
constexpr int TMAP_SETS = 64, TMAP_WAYS = 4;
thread_local TmapEntry t_tmap_cache[TMAP_SETS][TMAP_WAYS];
thread_local uint8_t t_tmap_next[TMAP_SETS];   // way to replace next in each set (round robin)
std::atomic<uint64_t> g_tmap_hits{0}, g_tmap_encodes{0};

uint64_t tmap_hash(const TmapKey &k)
{
    // FNV-1a over the key's bytes (the key is zero-filled, so padding is defined)
    const unsigned char *b = reinterpret_cast<const unsigned char *>(&k);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof(k); ++i) h = (h ^ b[i]) * 1099511628211ull;
    return h;
}

bool encode(CUtensorMap *m, mmact_dtype dt, int rank, const void *ptr, const uint64_t *dims,
            const uint64_t *strides_bytes, const uint32_t *box, bool swizzle = true,
            const uint32_t *estrides = nullptr)
{
    TmapKey k;
    std::memset(&k, 0, sizeof(k));
    k.dt = (int32_t)tmap_type(dt);
    k.rank = rank;
    k.swizzle = swizzle ? 1 : 0;
    k.ptr = ptr;
    for (int i = 0; i < rank; ++i) {
        k.gd[i] = dims[i];
        k.bx[i] = box[i];
        k.es[i] = estrides ? estrides[i] : 1;
    }
    for (int i = 0; i + 1 < rank; ++i) k.gs[i] = strides_bytes[i];
    const int set = (int)(tmap_hash(k) % TMAP_SETS);
    for (int w = 0; w < TMAP_WAYS; ++w) {
        const TmapEntry &e = t_tmap_cache[set][w];
        if (e.valid && std::memcmp(&e.key, &k, sizeof(k)) == 0) {
            *m = e.map;
            g_tmap_hits.fetch_add(1, std::memory_order_relaxed);
            return true;
        }
    }
    CUresult r = g_encode(m, (CUtensorMapDataType)k.dt, (cuuint32_t)rank, const_cast<void *>(ptr), k.gd, k.gs,
                          k.bx, k.es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    g_tmap_encodes.fetch_add(1, std::memory_order_relaxed);
    TmapEntry &e = t_tmap_cache[set][t_tmap_next[set]];
    t_tmap_next[set] = (uint8_t)((t_tmap_next[set] + 1) % TMAP_WAYS);
    e.key = k;
    e.map = *m;
    e.valid = true;
    return true;
}

bool valid_act(mmact_act a) { return a >= MMACT_ACT_NONE && a <= MMACT_ACT_GELU; }
bool valid_in(mmact_dtype d) { return d == MMACT_F16 || d == MMACT_BF16; }
bool valid_out(mmact_dtype d) { return d == MMACT_F16 || d == MMACT_BF16 || d == MMACT_F32; }

constexpr int64_t MAX_DIM = (int64_t(1) << 31) - 1;

// Output tile width for a GEMM: the candidate with the least estimated time
// = (waves of persistent tiles over the SMs) x (tile width) / (throughput of
// that width relative to 256).  The relative throughputs were measured on
// GB300 at 8192^3 (one CTA per SM, 128-row tiles): 1757, 1443, 1397, 1133 and
// 576 TFLOP/s for widths 256, 224, 192, 128 and 64.  Ties go to the wider tile.
int choose_tile_n(int64_t tiles_m, int64_t N, int sms)
{
    static const int widths[] = {256, 224, 192, 128, 64};
    static const double rel_rate[] = {1.0, 0.82, 0.80, 0.61, 0.32};
    int best = 256;
    double best_cost = 1e300;
    for (int i = 0; i < 5; ++i) {
        const int64_t tiles = tiles_m * ((N + widths[i] - 1) / widths[i]);
        const int64_t waves = (tiles + sms - 1) / sms;
        const double cost = (double)waves * widths[i] / rel_rate[i];
        if (cost < best_cost * 0.999) {
            best_cost = cost;
            best = widths[i];
        }
    }
    return best;
}

// Split-K factor for a GEMM (0: use the persistent kernel).  The split-K
// kernel runs one 128 x 256 tile per cluster of S CTAs, each over 1/S of the
// K blocks, then sums the S partial tiles across the cluster (a fixed cost of
// a few microseconds: slice exchange through distributed shared memory and
// the cluster barriers).  It is taken when all its clusters are resident at
// once (one wave) and each CTA still has enough K blocks to amortise that
// cost: at least 16 with S = 4, at least 64 with S = 2 (S = 2 halves the
// per-CTA work only twice for the same exchange cost).  Measured on GB300 against the persistent kernel's own choice of
// tile (bf16, us): 128x8192x8192 39.4 -> 30.7 (S=4); 1024x1024x8192 38.8 ->
// 21.3 (4); 256x4096x8192 38.8 -> 22.2 (4); 128x4096x4096 21.0 -> 15.2 (4);
// 384x2048x4096 21.1 -> 16.0 (4); 256x8192x8192 40.7 -> 36.2 (2); and
// 128x16384x4096 27.4 vs 29.3 with S=2, where the rule keeps the persistent
// kernel (32 K blocks per CTA).
int choose_split_k(const DeviceInfo &dev, int64_t tiles_m, int64_t N, int64_t num_kb)
{
    const int mode = g_split_k.load();
    if (mode == 1) return 0;
    const int64_t tiles = tiles_m * ((N + 255) / 256);
    if (mode == 2 || mode == 4) return num_kb >= mode ? mode : 0;
    if (g_tile_n.load() != 0) return 0;   // a fixed tile width asks for the persistent kernel
    if (tiles <= dev.splitk_clusters[1] && num_kb >= 4 * 16) return 4;
    if (tiles <= dev.splitk_clusters[0] && num_kb >= 2 * 64) return 2;
    return 0;
}

// Whether a GEMM that takes neither split-K nor a forced tile width runs on
// the CTA-pair kernel: 256 x 256 tiles on pairs of SMs, one M = 256
// tcgen05.mma per pair (each SM fills 32 KB of shared memory per K block
// instead of 48 KB for the same MMA work).  Taken when the persistent kernel
// would use 256-wide tiles and the pair grid needs no more waves than the
// persistent one: each wave of either does 128 x 256 outputs per SM, and a
// pair wave was measured faster (bf16 on GB300: 8192^3 639 -> 577 us,
// 8192x8192x4096 326 -> 282, 4096^3 94.6 -> 81.8, 16384x4096x1024
// 89.8 -> 82.8).  With a residual too, since the pair kernel stages the
// residual tiles by TMA one epilogue unit ahead (16384x4096x1024 with
// residual: 98.4 us on the pair, 103.9 us persistent).
bool choose_pair(const DeviceInfo &dev, int64_t M, int64_t N, int64_t num_kb, bool has_res)
{
    (void)num_kb;
    (void)has_res;
    const int mode = g_pair.load();
    if (mode == 1 || dev.pair_clusters <= 0) return false;
    if (mode == 2) return true;
    if (g_tile_n.load() != 0) return false;
    const int64_t tiles_m = (M + 127) / 128;
    if (choose_tile_n(tiles_m, N, dev.sm_count) != 256) return false;
    const int64_t tiles_n = (N + 255) / 256;
    const int64_t waves = (tiles_m * tiles_n + dev.sm_count - 1) / dev.sm_count;
    const int64_t pair_waves = (((M + 255) / 256) * tiles_n + dev.pair_clusters - 1) / dev.pair_clusters;
    return pair_waves <= waves;
}

mmact_status conv_f32_gemm_enqueue(const void *A, const void *B, const float *bias, void *C, int64_t M,
                                   int64_t N, int64_t K, mmact_dtype cd, mmact_act act, float alpha,
                                   cudaStream_t stream, const void *res, const DeviceInfo *dev);

// Shared by mmact_gemm, mmact_gemm_residual and the first kernel of
// mmact_gemm_split.  `res`: residual [M, N] in the output dtype, or null.
mmact_status gemm_enqueue(const void *A, const void *B, const float *bias, void *C, int64_t M,
                          int64_t N, int64_t K, mmact_dtype ab, mmact_dtype cd, mmact_act act,
                          float alpha, cudaStream_t stream, const void *res = nullptr)
{
    DeviceInfo *dev = nullptr;
    mmact_status st = device_info(&dev);
    if (st != MMACT_OK) return st;
    if (K == 0) {
        cudaError_t e = launch_bias_act(bias, C, M, N, 0, N, out_kind(cd), (int)act, alpha, stream, res);
        return e == cudaSuccess ? MMACT_OK : MMACT_ERR_CUDA;
    }
    if (ab == MMACT_F32) return conv_f32_gemm_enqueue(A, B, bias, C, M, N, K, cd, act, alpha, stream, res, dev);
    GemmLaunch L;
    std::memset(&L, 0, sizeof(L));
    const int tiles_m = (int)((M + 127) / 128);
    const int split = choose_split_k(*dev, tiles_m, N, (K + 63) / 64);
    const bool pair = split == 0 && choose_pair(*dev, M, N, (K + 63) / 64, res != nullptr);
    int bn = split != 0 || pair ? 256 : g_tile_n.load();
    if (bn == 0) bn = choose_tile_n(tiles_m, N, dev->sm_count);
    const int tiles_n = (int)((N + bn - 1) / bn);
    GemmArgs &a = L.args;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.tiles_m = tiles_m;
    a.tiles_n = tiles_n;
    a.num_tiles = tiles_m * tiles_n;
    a.num_kb = (int)((K + 63) / 64);
    // M blocks per raster group: 16 of 128 rows; on CTA pairs 8 of 256 rows (a wave
    // of 76 pair tiles then spans ~8 x 9.5 blocks, near the least A + B read per
    // wave, and with the evict-last hint the group's A rows stay in L2 across its
    // waves; measured on GB300 at 6144^3: 406 MB of DRAM traffic per launch, 1.9x
    // the algorithmic bytes, and 4096^3 88 -> 82 us)
    a.group_m = pair ? 8 : 16;
    a.ab_bf16 = ab == MMACT_BF16 ? 1 : 0;
    a.act = (int)act;
    a.alpha = alpha;
    a.bias = bias;
    a.res = res;
    a.status = dev->status;
    a.wait_ns = g_wait_ns.load();
    a.l2_policy = g_l2_policy.load();
    L.tile_n = bn;
    L.out = out_kind(cd);
    L.grid = (int)std::min<int64_t>(a.num_tiles, dev->sm_count);
    L.split_k = split;
    if (pair) {
        // 256 x 256 tiles, one per CTA pair
        a.tiles_m = (int)((M + 255) / 256);
        a.num_tiles = a.tiles_m * tiles_n;
        L.pair = 1;
        L.grid = 2 * (int)std::min<int64_t>(a.num_tiles, dev->pair_clusters);
    }
    if (split != 0) {
        if ((int64_t)a.num_tiles * split > MAX_DIM) return MMACT_ERR_UNSUPPORTED;
        L.grid = a.num_tiles * split;   // one cluster per tile
    }

    const uint64_t dA[2] = {(uint64_t)K, (uint64_t)M}, sA[1] = {(uint64_t)K * 2};
    const uint32_t bA[2] = {64, 128};
    const uint64_t dB[2] = {(uint64_t)N, (uint64_t)K}, sB[1] = {(uint64_t)N * 2};
    const uint32_t bB[2] = {64, 64};
    const int ce = elem_bytes(cd);
    const uint64_t dC[2] = {(uint64_t)N, (uint64_t)M}, sC[1] = {(uint64_t)N * ce};
    const uint32_t bC[2] = {(uint32_t)(128 / ce), 32};
    if (!encode(&L.tmA, ab, 2, A, dA, sA, bA) || !encode(&L.tmB, ab, 2, B, dB, sB, bB) ||
        !encode(&L.tmC, cd, 2, C, dC, sC, bC))
        return MMACT_ERR_CUDA;
    if (bn == 224 && ce == 2) {
        const uint32_t bT[2] = {32, 32};
        if (!encode(&L.tmCt, cd, 2, C, dC, sC, bT, false)) return MMACT_ERR_CUDA;
    }
    if (pair && res != nullptr && !encode(&L.tmR, cd, 2, res, dC, sC, bC)) return MMACT_ERR_CUDA;
    const cudaError_t e = split != 0 ? launch_gemm_splitk(L, stream)
                          : pair       ? launch_gemm_pair(L, stream)
                                       : launch_gemm(L, stream);
    return e == cudaSuccess ? MMACT_OK : MMACT_ERR_CUDA;
}

struct ConvGeom {
    int64_t Ho, Wo;
};

mmact_status conv_geom(int64_t H, int64_t W, int64_t kh, int64_t kw, const int32_t *st,
                       const int32_t *pd, const int32_t *dl, ConvGeom *g)
{
    if (st == nullptr || pd == nullptr || dl == nullptr) return MMACT_ERR_INVALID_ARG;
    if (H < 0 || W < 0 || kh <= 0 || kw <= 0) return MMACT_ERR_INVALID_ARG;
    if (st[0] <= 0 || st[1] <= 0 || dl[0] <= 0 || dl[1] <= 0) return MMACT_ERR_INVALID_ARG;
    if (pd[0] < 0 || pd[1] < 0 || pd[2] < 0 || pd[3] < 0) return MMACT_ERR_INVALID_ARG;
    const int64_t sh = H + pd[0] + pd[1] - (int64_t)dl[0] * (kh - 1) - 1;
    const int64_t sw = W + pd[2] + pd[3] - (int64_t)dl[1] * (kw - 1) - 1;
    if (sh < 0 || sw < 0) return MMACT_ERR_INVALID_ARG;
    g->Ho = sh / st[0] + 1;
    g->Wo = sw / st[1] + 1;
    return MMACT_OK;
}

mmact_status conv_check(const void *x, const void *w, const float *bias, const void *y, int64_t N,
                        int64_t C, int64_t H, int64_t W, int64_t Co, int64_t kh, int64_t kw,
                        const int32_t *st, const int32_t *pd, const int32_t *dl, mmact_dtype in,
                        mmact_dtype out, mmact_act act, ConvGeom *g, bool tf32_in = false)
{
    if (N < 0 || C < 0 || Co < 0) return MMACT_ERR_INVALID_ARG;
    const bool in_ok = valid_in(in) || in == MMACT_F32 || (tf32_in && in == MMACT_TF32);
    if (!in_ok || !valid_out(out) || !valid_act(act)) return MMACT_ERR_INVALID_ARG;
    mmact_status s = conv_geom(H, W, kh, kw, st, pd, dl, g);
    if (s != MMACT_OK) return s;
    // a pointer may be null only when its tensor is empty
    if ((x == nullptr && N * C * H * W != 0) || (w == nullptr && Co * C != 0) ||
        (y == nullptr && N * Co != 0))
        return MMACT_ERR_INVALID_ARG;
    if (bias != nullptr && !aligned4(bias)) return MMACT_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return MMACT_ERR_UNSUPPORTED;
    // every index the kernel forms fits in 32 bits per image / 64 bits overall
    if (C * H * W > MAX_DIM || Co * g->Ho * g->Wo > MAX_DIM || C * kh * kw > MAX_DIM ||
        N > MAX_DIM || H > MAX_DIM || W > MAX_DIM)
        return MMACT_ERR_UNSUPPORTED;
    return MMACT_OK;
}

// Host-side plan of a conv launch: the GEMM view, the producer (general
// gather, vectorised global-load gather, or vectorised window), the tile
// shape and the window box.  No device work.
void conv_plan(int64_t N, int64_t C, int64_t H, int64_t W, int64_t Co, int64_t kh, int64_t kw,
               const int32_t *st, const int32_t *pd, const int32_t *dl, const ConvGeom &g,
               mmact_dtype in, mmact_dtype out, ConvArgs &a)
{
    const int64_t P = g.Ho * g.Wo;
    std::memset(&a, 0, sizeof(a));
    a.Nb = (int)N;
    a.C = (int)C;
    a.H = (int)H;
    a.W = (int)W;
    a.Co = (int)Co;
    a.kh = (int)kh;
    a.kw = (int)kw;
    a.sh = st[0];
    a.sw = st[1];
    a.pt = pd[0];
    a.pl = pd[2];
    a.dh = dl[0];
    a.dw = dl[1];
    a.Ho = (int)g.Ho;
    a.Wo = (int)g.Wo;
    a.P = (int)P;
    a.K = (int)(C * kh * kw);
    a.tiles_co = (int)((Co + 127) / 128);
    a.tiles_p = (int)((P + 127) / 128);
    a.num_tiles = (int)(N * a.tiles_co * a.tiles_p);
    a.num_kb = (a.K + 63) / 64;
    a.ab_bf16 = in == MMACT_BF16 ? 1 : 0;
    a.out_elem_bytes = elem_bytes(out);
    a.f32 = in == MMACT_F32 ? 1 : 0;
    a.a_tma = (a.K % 8 == 0 && !a.f32) ? 1 : 0;
    a.y_tma = ((P * a.out_elem_bytes) % 16 == 0) ? 1 : 0;
    if (a.f32) return;   // fp32 inputs: the general gather producer, split precision
    // Vectorised producer: whole 16-byte input chunks per row (W % 8 == 0),
    // horizontal stride 1 or 2, filter by TMA, and an output TMA store:
    // 8 x 32 tiles when the output is exactly 32 wide (256 consecutive
    // pixels), else 4 x 64 tiles stored through a 4-D map (rows of y must be
    // 16-byte multiples).
    a.W8 = (int)(W / 8);
    if (a.a_tma && W % 8 == 0 && (a.sw == 1 || a.sw == 2)) {
        if (g.Wo == 32 && a.y_tma) {
            a.vec = 1;
            a.TW = 32;
            a.TH = 8;
        } else if ((g.Wo * a.out_elem_bytes) % 16 == 0) {
            a.vec = 1;
            a.TW = 64;
            a.TH = 4;
        }
    }
    if (!a.vec) return;
    a.tiles_oh = (int)((g.Ho + a.TH - 1) / a.TH);
    a.tiles_ow = (int)((g.Wo + a.TW - 1) / a.TW);
    a.num_tiles = (int)(N * a.tiles_oh * a.tiles_ow * a.tiles_co);
    // Input window per 64-row K block (conv_vec.cu, WIN): the channels 64
    // consecutive rows (ci, r, q) can span; the rows of every tap r (a row
    // stride of sh when dh is a multiple of sh); an 8-aligned column span wide
    // enough for every lane's chunk loads at every q.
    const int64_t taps = kh * kw;
    const int S = a.sw, nch = S == 1 ? 2 : 3, vpr = a.TW / 8;
    const int64_t CB = std::min<int64_t>(C, (62 + taps) / taps + 1);
    const bool hstride = a.sh > 1 && a.sh <= 8 && (kh == 1 || a.dh % a.sh == 0);
    const int64_t esh = hstride ? a.sh : 1;
    const int64_t HB = hstride ? a.TH + (kh - 1) * (a.dh / a.sh)
                               : (int64_t)(a.TH - 1) * a.sh + (kh - 1) * a.dh + 1;
    const int64_t c0max = ((int64_t)(vpr - 1) * 8 * S + 7 + (kw - 1) * a.dw) >> 3;
    const int64_t WB = 8 * (c0max + nch);
    const int64_t raw = WB * HB * CB * 2;
    if (raw <= CONV_WIN_MAX_BYTES && WB <= 256 && HB * esh <= 256 && CB <= 256) {
        a.win = 1;
        a.WB = (int)WB;
        a.HB = (int)HB;
        a.CB = (int)CB;
        a.rstep = hstride ? a.dh / a.sh : a.dh;
        a.rowmul = hstride ? 1 : a.sh;
        a.raw_bytes = (int)raw;
    }
}

// An fp32 GEMM C[M,N] = act(A[M,K] B[K,N] + bias) run by the general conv
// kernel in split precision as the 1x1 conv w = A ([M, K, 1, 1]), x = B ([1, K,
// 1, N]): output channels are the rows of C, output pixels its columns, and
// the bias runs along the columns.
mmact_status conv_f32_gemm_enqueue(const void *A, const void *B, const float *bias, void *C, int64_t M,
                                   int64_t N, int64_t K, mmact_dtype cd, mmact_act act, float alpha,
                                   cudaStream_t stream, const void *res, const DeviceInfo *dev)
{
    if (M > MAX_DIM || N * M > ((int64_t)1 << 62)) return MMACT_ERR_UNSUPPORTED;
    ConvLaunch L;
    std::memset(&L, 0, sizeof(L));
    ConvArgs &a = L.args;
    a.Nb = 1;
    a.C = (int)K;
    a.H = 1;
    a.W = (int)N;
    a.Co = (int)M;
    a.kh = a.kw = 1;
    a.sh = a.sw = 1;
    a.dh = a.dw = 1;
    a.Ho = 1;
    a.Wo = (int)N;
    a.P = (int)N;
    a.K = (int)K;
    a.tiles_co = (int)((M + 127) / 128);
    a.tiles_p = (int)((N + 127) / 128);
    if ((int64_t)a.tiles_co * a.tiles_p > MAX_DIM) return MMACT_ERR_UNSUPPORTED;
    a.num_tiles = a.tiles_co * a.tiles_p;
    a.num_kb = (int)((K + 63) / 64);
    a.f32 = 1;
    a.bias_col = 1;
    a.out_elem_bytes = elem_bytes(cd);
    a.y_tma = ((N * a.out_elem_bytes) % 16 == 0) ? 1 : 0;
    a.act = (int)act;
    a.alpha = alpha;
    a.x = static_cast<const uint16_t *>(B);
    a.w = static_cast<const uint16_t *>(A);
    a.bias = bias;
    a.res = res;
    a.y = C;
    a.status = dev->status;
    a.wait_ns = g_wait_ns.load();
    L.out = out_kind(cd);
    L.grid = (int)std::min<int64_t>(a.num_tiles, dev->sm_count);
    if (a.y_tma) {
        const int e = a.out_elem_bytes;
        const uint64_t d[3] = {(uint64_t)N, (uint64_t)M, 1};
        const uint64_t sb[2] = {(uint64_t)N * e, (uint64_t)M * N * e};
        const uint32_t bx[3] = {(uint32_t)(128 / e), 32, 1};
        if (!encode(&L.tmY, cd, 3, C, d, sb, bx)) return MMACT_ERR_CUDA;
    }
    return launch_conv(L, stream) == cudaSuccess ? MMACT_OK : MMACT_ERR_CUDA;
}

int64_t gcd64(int64_t a, int64_t b)
{
    while (b != 0) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// Plan of the NCHW conv kernel whose im2col operand lives in tensor memory
// (conv_tmem.cu): tiles of 128 consecutive output pixels of one image x BN
// output channels; per 64-value K block one raw input window box.  Returns
// false when the geometry needs another kernel: 16-bit inputs, filter rows
// and input rows with 16-byte pitches (K % 8, W % 8), a window that fits its
// slot and the TMA box limits, and a K-offset table that fits.
bool tconv_plan(int64_t N, int64_t C, int64_t H, int64_t W, int64_t Co, int64_t kh, int64_t kw,
                const int32_t *st, const int32_t *pd, const int32_t *dl, const ConvGeom &g,
                mmact_dtype in, TmemConvArgs &a, int &bn)
{
    std::memset(&a, 0, sizeof(a));
    if (!valid_in(in)) return false;
    const int64_t taps = kh * kw, K = C * taps, P = g.Ho * g.Wo;
    if (K % 8 != 0 || W % 8 != 0 || P <= 0) return false;
    const int64_t period = taps / gcd64(64, taps);          // blocks until the K pattern repeats
    if (period * 64 > CONV_TMEM_TABLE_MAX) return false;
    // output rows a 128-pixel tile can span (tiles start at multiples of 128)
    const int64_t tiles_p = (P + 127) / 128;
    int64_t nrows = 1;
    const int64_t starts = std::min<int64_t>(g.Wo / gcd64(128, g.Wo), tiles_p);
    for (int64_t i = 0; i < starts; ++i) {
        const int64_t s = (128 * i) % g.Wo;
        nrows = std::max<int64_t>(nrows, (s + 127) / g.Wo + 1);
    }
    nrows = std::min<int64_t>(nrows, g.Ho);
    const int64_t sh = st[0], sw = st[1], dh = dl[0], dw = dl[1];
    const bool lattice = sh > 1 && (kh == 1 || dh % sh == 0);
    const int64_t HB = lattice ? nrows + (kh - 1) * (dh / sh) : (nrows - 1) * sh + (kh - 1) * dh + 1;
    const int64_t esh = lattice ? sh : 1;
    const int64_t x0 = -(((int64_t)pd[2] + 7) / 8) * 8;
    const int64_t xoff = -(int64_t)pd[2] - x0;
    const int64_t WB = ((xoff + (g.Wo - 1) * sw + (kw - 1) * dw + 1) + 7) / 8 * 8;
    const int64_t CB = (64 % taps == 0) ? 64 / taps : 63 / taps + 2;
    const int64_t raw = WB * HB * CB * 2;
    if (raw > CONV_TMEM_WIN_MAX_BYTES || WB > 256 || HB * esh > 256 || CB > 256) return false;
    bn = Co <= 64 ? 64 : (Co <= 128 ? 128 : 256);
    // window ring: as many 1 KB-rounded slots as the kernel's shared memory leaves, up to 8
    const int64_t slot = (raw + 1023) / 1024 * 1024;
    const int64_t wstages = std::min<int64_t>(CONV_TMEM_MAX_WSTAGES, conv_tmem_window_region(bn) / slot);
    if (wstages < 2) return false;
    a.Nb = (int)N;
    a.C = (int)C;
    a.H = (int)H;
    a.W = (int)W;
    a.Co = (int)Co;
    a.kh = (int)kh;
    a.kw = (int)kw;
    a.sh = (int)sh;
    a.sw = (int)sw;
    a.pt = pd[0];
    a.pl = pd[2];
    a.dh = (int)dh;
    a.dw = (int)dw;
    a.Ho = (int)g.Ho;
    a.Wo = (int)g.Wo;
    a.P = (int)P;
    a.K = (int)K;
    a.tiles_co = (int)((Co + bn - 1) / bn);
    a.tiles_p = (int)tiles_p;
    if (N * a.tiles_co * tiles_p > MAX_DIM) return false;
    a.num_tiles = (int)(N * a.tiles_co * tiles_p);
    a.num_kb = (int)((K + 63) / 64);
    a.ab_bf16 = in == MMACT_BF16 ? 1 : 0;
    a.WB = (int)WB;
    a.HB = (int)HB;
    a.CB = (int)CB;
    a.esh = (int)esh;
    a.rowmul = lattice ? 1 : (int)sh;
    a.rstep = lattice ? (int)(dh / sh) : (int)dh;
    a.x0 = (int)x0;
    a.xoff = (int)xoff;
    a.raw_bytes = (int)raw;
    a.win_slot = (int)slot;
    a.wstages = (int)wstages;
    a.tab_period = (int)period;
    return true;
}

bool use_tconv() { return g_conv_tmem.load() == 0; }

mmact_status tconv_enqueue(const void *x, const void *w, const float *bias, void *y, int64_t N, int64_t C,
                           int64_t H, int64_t W, int64_t Co, int64_t kh, int64_t kw,
                           const TmemConvArgs &plan, int bn, const DeviceInfo *dev, mmact_dtype in,
                           mmact_dtype out, mmact_act act, float alpha, cudaStream_t stream, const void *res)
{
    TmemConvLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.args = plan;
    TmemConvArgs &a = L.args;
    a.act = (int)act;
    a.alpha = alpha;
    a.bias = bias;
    a.res = res;
    a.y = y;
    a.status = dev->status;
    a.wait_ns = g_wait_ns.load();
    L.tile_n = bn;
    L.out = out_kind(out);
    L.grid = (int)std::min<int64_t>(a.num_tiles, dev->sm_count);
    const int e = elem_bytes(out);
    a.y_tma = ((int64_t)a.P * e) % 16 == 0 ? 1 : 0;
    const uint64_t dW[2] = {(uint64_t)a.K, (uint64_t)Co}, sW[1] = {(uint64_t)a.K * 2};
    const uint32_t bW[2] = {64, (uint32_t)bn};
    const uint64_t dX[4] = {(uint64_t)W, (uint64_t)H, (uint64_t)C, (uint64_t)N};
    const uint64_t sX[3] = {(uint64_t)W * 2, (uint64_t)H * W * 2, (uint64_t)C * H * W * 2};
    const uint32_t bX[4] = {(uint32_t)a.WB, (uint32_t)(a.HB * a.esh), (uint32_t)a.CB, 1};
    const uint32_t eX[4] = {1, (uint32_t)a.esh, 1, 1};
    if (!encode(&L.tmW, in, 2, w, dW, sW, bW) || !encode(&L.tmX, in, 4, x, dX, sX, bX, false, eX))
        return MMACT_ERR_CUDA;
    if (a.y_tma) {
        // y as {P, Co, N}: 32 pixels x 32 channels per store, unswizzled [channel][pixel] rows
        const uint64_t dY[3] = {(uint64_t)a.P, (uint64_t)Co, (uint64_t)N};
        const uint64_t sY[2] = {(uint64_t)a.P * e, (uint64_t)Co * a.P * e};
        const uint32_t bY[3] = {32, 32, 1};
        if (!encode(&L.tmY, out, 3, y, dY, sY, bY, false)) return MMACT_ERR_CUDA;
    }
    return launch_conv_tmem(L, stream) == cudaSuccess ? MMACT_OK : MMACT_ERR_CUDA;
}

mmact_status conv_enqueue(const void *x, const void *w, const float *bias, void *y, int64_t N,
                          int64_t C, int64_t H, int64_t W, int64_t Co, int64_t kh, int64_t kw,
                          const int32_t *st, const int32_t *pd, const int32_t *dl, const ConvGeom &g,
                          mmact_dtype in, mmact_dtype out, mmact_act act, float alpha,
                          cudaStream_t stream, const void *res = nullptr)
{
    DeviceInfo *dev = nullptr;
    mmact_status s = device_info(&dev);
    if (s != MMACT_OK) return s;
    const int64_t P = g.Ho * g.Wo;
    if (N == 0 || Co == 0 || P == 0) return MMACT_OK;
    if (C == 0) {
        cudaError_t e = launch_bias_act(bias, y, N * Co, P, 1, Co, out_kind(out), (int)act, alpha, stream,
                                        res);
        return e == cudaSuccess ? MMACT_OK : MMACT_ERR_CUDA;
    }
    if (use_tconv()) {
        TmemConvArgs tp;
        int bn = 0;
        if (tconv_plan(N, C, H, W, Co, kh, kw, st, pd, dl, g, in, tp, bn))
            return tconv_enqueue(x, w, bias, y, N, C, H, W, Co, kh, kw, tp, bn, dev, in, out, act, alpha,
                                 stream, res);
    }
    ConvLaunch L;
    std::memset(&L, 0, sizeof(L));
    ConvArgs &a = L.args;
    conv_plan(N, C, H, W, Co, kh, kw, st, pd, dl, g, in, out, a);
    a.act = (int)act;
    a.alpha = alpha;
    a.x = static_cast<const uint16_t *>(x);
    a.w = static_cast<const uint16_t *>(w);
    a.bias = bias;
    a.res = res;
    a.y = y;
    a.status = dev->status;
    a.wait_ns = g_wait_ns.load();
    L.out = out_kind(out);
    L.grid = (int)std::min<int64_t>(a.num_tiles, dev->sm_count);
    if (a.win) {
        const uint32_t esh = (uint32_t)(a.rowmul == 1 && a.sh > 1 ? a.sh : 1);
        const uint64_t d[4] = {(uint64_t)W, (uint64_t)H, (uint64_t)C, (uint64_t)N};
        const uint64_t sb[3] = {(uint64_t)W * 2, (uint64_t)H * W * 2, (uint64_t)C * H * W * 2};
        const uint32_t bx[4] = {(uint32_t)a.WB, (uint32_t)a.HB * esh, (uint32_t)a.CB, 1};
        const uint32_t es[4] = {1, esh, 1, 1};
        if (!encode(&L.tmX, in, 4, x, d, sb, bx, false, es)) return MMACT_ERR_CUDA;
    }
    if (a.vec && a.TW == 64) {
        const int e = a.out_elem_bytes;
        const uint64_t d[4] = {(uint64_t)g.Wo, (uint64_t)g.Ho, (uint64_t)Co, (uint64_t)N};
        const uint64_t sb[3] = {(uint64_t)g.Wo * e, (uint64_t)P * e, (uint64_t)Co * P * e};
        const uint32_t bx[4] = {(uint32_t)(128 / e), 1, 32, 1};
        if (!encode(&L.tmY4, out, 4, y, d, sb, bx)) return MMACT_ERR_CUDA;
    }
    if (a.a_tma) {
        const uint64_t d[2] = {(uint64_t)a.K, (uint64_t)Co}, sb[1] = {(uint64_t)a.K * 2};
        const uint32_t bx[2] = {64, 128};
        if (!encode(&L.tmW, in, 2, w, d, sb, bx)) return MMACT_ERR_CUDA;
    }
    if (a.y_tma) {
        const int e = a.out_elem_bytes;
        const uint64_t d[3] = {(uint64_t)P, (uint64_t)Co, (uint64_t)N};
        const uint64_t sb[2] = {(uint64_t)P * e, (uint64_t)Co * P * e};
        const uint32_t bx[3] = {(uint32_t)(128 / e), 32, 1};
        if (!encode(&L.tmY, out, 3, y, d, sb, bx)) return MMACT_ERR_CUDA;
    }
    return launch_conv(L, stream) == cudaSuccess ? MMACT_OK : MMACT_ERR_CUDA;
}

int act_grid(const DeviceInfo *dev) { return dev->sm_count * 8; }

mmact_status nhwc_enqueue(const void *x, const void *w, const float *bias, void *y, int64_t N,
                          int64_t C, int64_t H, int64_t W, int64_t Co, int64_t kh, int64_t kw,
                          const int32_t *st, const int32_t *pd, const int32_t *dl, const ConvGeom &g,
                          mmact_dtype in, mmact_dtype out, mmact_act act, float alpha,
                          cudaStream_t stream, const void *res = nullptr)
{
    DeviceInfo *dev = nullptr;
    mmact_status s = device_info(&dev);
    if (s != MMACT_OK) return s;
    const int64_t M = N * g.Ho * g.Wo;
    if (M == 0 || Co == 0) return MMACT_OK;
    if (C == 0) {
        cudaError_t e = launch_bias_act(bias, y, M, Co, 0, Co, out_kind(out), (int)act, alpha, stream, res);
        return e == cudaSuccess ? MMACT_OK : MMACT_ERR_CUDA;
    }
    if (in == MMACT_F32) {
        // fp32 inputs to fp32 accuracy: the general gather kernel in split precision, channels-last
        ConvLaunch CL;
        std::memset(&CL, 0, sizeof(CL));
        conv_plan(N, C, H, W, Co, kh, kw, st, pd, dl, g, in, out, CL.args);
        ConvArgs &c = CL.args;
        c.nhwc = 1;
        c.y_tma = 0;
        c.act = (int)act;
        c.alpha = alpha;
        c.x = static_cast<const uint16_t *>(x);
        c.w = static_cast<const uint16_t *>(w);
        c.bias = bias;
        c.y = y;
        c.status = dev->status;
        c.wait_ns = g_wait_ns.load();
        CL.out = out_kind(out);
        CL.grid = (int)std::min<int64_t>(c.num_tiles, dev->sm_count);
        return launch_conv(CL, stream) == cudaSuccess ? MMACT_OK : MMACT_ERR_CUDA;
    }
    NhwcLaunch L;
    std::memset(&L, 0, sizeof(L));
    NhwcArgs &a = L.args;
    a.Nb = (int)N;
    a.C = (int)C;
    a.H = (int)H;
    a.W = (int)W;
    a.Co = (int)Co;
    a.kh = (int)kh;
    a.kw = (int)kw;
    a.sh = st[0];
    a.sw = st[1];
    a.pt = pd[0];
    a.pl = pd[2];
    a.dh = dl[0];
    a.dw = dl[1];
    a.Ho = (int)g.Ho;
    a.Wo = (int)g.Wo;
    a.M = (int)M;
    a.tf32 = in == MMACT_TF32 ? 1 : 0;
    const int ie = elem_bytes(in);              // 2, or 4 for fp32 inputs
    a.kc = 128 / ie;                            // one 128-byte row of K per block
    a.ncb = (int)((C + a.kc - 1) / a.kc);
    // M tile: TH output rows x TW output columns of one image, 128 pixels
    a.TW = g.Wo <= 32 ? 32 : 64;
    if (a.TW * a.sw > 256) a.TW = 32;
    a.TH = 128 / a.TW;
    if (a.TW * a.sw > 256 || a.TH * a.sh > 256) return MMACT_ERR_UNSUPPORTED;
    a.tiles_oh = (int)((g.Ho + a.TH - 1) / a.TH);
    a.tiles_ow = (int)((g.Wo + a.TW - 1) / a.TW);
    a.tiles_m = (int)(N * a.tiles_oh * a.tiles_ow);
    // channels-last tiles come in widths 256, 128 and 64 (same cost model as the GEMM)
    int bn = 256;
    {
        static const int widths[] = {256, 128, 64};
        static const double rel_rate[] = {1.0, 0.61, 0.32};
        double best = 1e300;
        for (int i = 0; i < 3; ++i) {
            const int64_t tiles = (int64_t)a.tiles_m * ((Co + widths[i] - 1) / widths[i]);
            const double cost = (double)((tiles + dev->sm_count - 1) / dev->sm_count) * widths[i] / rel_rate[i];
            if (cost < best * 0.999) {
                best = cost;
                bn = widths[i];
            }
        }
    }
    a.tiles_n = (int)((Co + bn - 1) / bn);
    a.num_tiles = a.tiles_m * a.tiles_n;
    a.num_kb = (int)(kh * kw) * a.ncb;
    a.group_m = 16;
    a.ab_bf16 = in == MMACT_BF16 ? 1 : 0;
    a.act = (int)act;
    a.alpha = alpha;
    a.x = x;
    a.bias = bias;
    a.res = res;
    a.status = dev->status;
    a.wait_ns = g_wait_ns.load();
    L.tile_n = bn;
    L.out = out_kind(out);
    L.grid = (int)std::min<int64_t>(a.num_tiles, dev->sm_count);
    const uint64_t dX[4] = {(uint64_t)C, (uint64_t)W, (uint64_t)H, (uint64_t)N};
    const uint64_t sX[3] = {(uint64_t)C * ie, (uint64_t)W * C * ie, (uint64_t)H * W * C * ie};
    const uint32_t bX[4] = {(uint32_t)a.kc, (uint32_t)(a.TW * a.sw), (uint32_t)(a.TH * a.sh), 1};
    const uint32_t eX[4] = {1, (uint32_t)a.sw, (uint32_t)a.sh, 1};
    const uint64_t dW[3] = {(uint64_t)C, (uint64_t)(kh * kw), (uint64_t)Co};
    const uint64_t sW[2] = {(uint64_t)C * ie, (uint64_t)(kh * kw) * C * ie};
    const uint32_t bW[3] = {(uint32_t)a.kc, 1, (uint32_t)bn};
    const int e = elem_bytes(out);
    const uint64_t dY[4] = {(uint64_t)Co, (uint64_t)g.Wo, (uint64_t)g.Ho, (uint64_t)N};
    const uint64_t sY[3] = {(uint64_t)Co * e, (uint64_t)g.Wo * Co * e, (uint64_t)g.Ho * g.Wo * Co * e};
    const uint32_t bY[4] = {(uint32_t)(128 / e), 32, 1, 1};
    if (!encode(&L.tmX, in, 4, x, dX, sX, bX, true, eX) || !encode(&L.tmW, in, 3, w, dW, sW, bW) ||
        !encode(&L.tmY, out, 4, y, dY, sY, bY))
        return MMACT_ERR_CUDA;
    return launch_conv_nhwc(L, stream) == cudaSuccess ? MMACT_OK : MMACT_ERR_CUDA;
}

// Fused single kernel or two-kernel split: the fused_matmul_relu article's
// run-time decision (fuse, or fall back to the matmul and a separate
// activation through a device temporary), decided here from a measured
// fused-versus-split grid on GB300 (GEMMs with K from 64 to 1024 and M, N
// from 64 to 8192, small-channel convs; every activation) rather than from
// an on-chip buffer budget.  The fused kernel wins on every shape with ReLU,
// LeakyReLU and tanh (1.2x to 3x) and on every GEMM with GELU whose output has
// more than 512 Ki elements (1.04x to 1.36x); between 64 Ki and 512 Ki
// elements the two are mixed (0.96x to 1.13x) and the fused kernel is kept.
// The split path wins (a) with GELU on a small output (M*N <= 64 Ki: one or two tiles, where
// the fused epilogue's few warps are latency-bound on the activation and the
// split's activation pass spreads over the whole GPU; 64x64x64: 4.8 against
// 5.7 us) and on small-channel convs with GELU (C*kh*kw <= 288, Co >= 64:
// up to 10 %); and (b) for an NCHW conv whose fused kernel would store its
// 16-bit output element by element (neither the tensor-memory nor the
// vectorised producer applies and the output row pitch rules out TMA
// stores), where the split's fp32 intermediate is stored by TMA (1x1
// stride 2 on 28 x 28: 8.4 against 16.8 us).
constexpr int64_t SPLIT_GELU_MAX_OUTPUT = 65536;
constexpr int64_t SPLIT_GELU_MAX_CONV_K = 288;

bool gemm_prefers_split(int64_t M, int64_t N, int64_t K, mmact_dtype ab, mmact_act act)
{
    if (M == 0 || N == 0 || K == 0 || ab == MMACT_F32) return false;
    return act == MMACT_ACT_GELU && M * N <= SPLIT_GELU_MAX_OUTPUT;
}

bool conv_prefers_split(int64_t N, int64_t C, int64_t H, int64_t W, int64_t Co, int64_t kh, int64_t kw,
                        const int32_t *st, const int32_t *pd, const int32_t *dl, const ConvGeom &g,
                        mmact_dtype in, mmact_dtype out, mmact_act act)
{
    if (N == 0 || Co == 0 || C == 0 || in == MMACT_F32) return false;
    if (act == MMACT_ACT_GELU && C * kh * kw <= SPLIT_GELU_MAX_CONV_K && Co >= 64) return true;
    TmemConvArgs tp;
    int bn = 0;
    if (use_tconv() && tconv_plan(N, C, H, W, Co, kh, kw, st, pd, dl, g, in, tp, bn)) return false;
    ConvArgs a;
    conv_plan(N, C, H, W, Co, kh, kw, st, pd, dl, g, in, out, a);
    return !a.vec && !a.y_tma;
}

// R is read element by element before the same element of the output is
// written, so R == out is allowed; any other overlap is not.
mmact_status residual_check(const void *R, const void *out, int64_t bytes)
{
    if (R == nullptr && bytes != 0) return MMACT_ERR_INVALID_ARG;
    if (!aligned16(R)) return MMACT_ERR_UNSUPPORTED;
    const char *r = static_cast<const char *>(R), *c = static_cast<const char *>(out);
    if (r != c && bytes != 0 && r < c + bytes && c < r + bytes) return MMACT_ERR_INVALID_ARG;
    return MMACT_OK;
}

}  // namespace

// Host validation shared by every mmact_gemm-family entry point (also used by
// the no-allocation entry point in noalloc.cu, before its own size limit).
mmact_status gemm_check(const void *A, const void *B, const float *bias, const void *C, int64_t M,
                        int64_t N, int64_t K, mmact_dtype ab, mmact_dtype cd, mmact_act act)
{
    if (M < 0 || N < 0 || K < 0 || M > MAX_DIM || N > MAX_DIM || K > MAX_DIM)
        return MMACT_ERR_INVALID_ARG;
    // a pointer may be null only when its tensor is empty
    if ((A == nullptr && M * K != 0) || (B == nullptr && K * N != 0) || (C == nullptr && M * N != 0))
        return MMACT_ERR_INVALID_ARG;
    const bool in_ok = valid_in(ab) || ab == MMACT_F32 || ab == MMACT_TF32;
    if (!in_ok || !valid_out(cd) || !valid_act(act)) return MMACT_ERR_INVALID_ARG;
    if (bias != nullptr && !aligned4(bias)) return MMACT_ERR_INVALID_ARG;
    if (ab == MMACT_TF32) return MMACT_ERR_UNSUPPORTED;   // one-pass tf32: channels-last conv only
    if (ab == MMACT_F32) {
        // fp32 operands are gathered element by element: 4-byte alignment, any K and N
        if (!aligned4(A) || !aligned4(B) || !aligned16(C)) return MMACT_ERR_UNSUPPORTED;
        return MMACT_OK;
    }
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return MMACT_ERR_UNSUPPORTED;
    if (K % 8 != 0 || N % 8 != 0) return MMACT_ERR_UNSUPPORTED;
    return MMACT_OK;
}

}  // namespace mmact

using namespace mmact;

MMACT_EXPORT mmact_status mmact_gemm(const void *A, const void *B, const float *bias, void *C,
                                     int64_t M, int64_t N, int64_t K, mmact_dtype ab_dtype,
                                     mmact_dtype c_dtype, mmact_act act, float alpha, void *stream)
{
    mmact_status s = gemm_check(A, B, bias, C, M, N, K, ab_dtype, c_dtype, act);
    if (s != MMACT_OK) return s;
    if (M == 0 || N == 0) return MMACT_OK;
    return gemm_enqueue(A, B, bias, C, M, N, K, ab_dtype, c_dtype, act, alpha,
                        static_cast<cudaStream_t>(stream));
}

MMACT_EXPORT mmact_status mmact_gemm_residual(const void *A, const void *B, const float *bias,
                                              const void *R, void *C, int64_t M, int64_t N, int64_t K,
                                              mmact_dtype ab_dtype, mmact_dtype c_dtype, mmact_act act,
                                              float alpha, void *stream)
{
    mmact_status s = gemm_check(A, B, bias, C, M, N, K, ab_dtype, c_dtype, act);
    if (s != MMACT_OK) return s;
    if (R == nullptr && M * N != 0) return MMACT_ERR_INVALID_ARG;
    if (!aligned16(R)) return MMACT_ERR_UNSUPPORTED;
    // R is read element by element before the same element of C is written,
    // so R == C is allowed; any other overlap is not.
    const int64_t bytes = M * N * elem_bytes(c_dtype);
    const char *r = static_cast<const char *>(R), *c = static_cast<const char *>(C);
    if (r != c && bytes != 0 && r < c + bytes && c < r + bytes) return MMACT_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return MMACT_OK;
    return gemm_enqueue(A, B, bias, C, M, N, K, ab_dtype, c_dtype, act, alpha,
                        static_cast<cudaStream_t>(stream), R);
}

MMACT_EXPORT mmact_status mmact_gemm_split(const void *A, const void *B, const float *bias, void *C,
                                           int64_t M, int64_t N, int64_t K, mmact_dtype ab_dtype,
                                           mmact_dtype c_dtype, mmact_act act, float alpha,
                                           float *workspace, void *stream)
{
    mmact_status s = gemm_check(A, B, bias, C, M, N, K, ab_dtype, c_dtype, act);
    if (s != MMACT_OK) return s;
    if (workspace == nullptr) return MMACT_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return MMACT_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return MMACT_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = gemm_enqueue(A, B, bias, workspace, M, N, K, ab_dtype, MMACT_F32, MMACT_ACT_NONE, 0.0f, st);
    if (s != MMACT_OK) return s;
    DeviceInfo *dev = nullptr;
    if ((s = device_info(&dev)) != MMACT_OK) return s;
    return launch_act(workspace, C, M * N, out_kind(c_dtype), (int)act, alpha, act_grid(dev), st) ==
                   cudaSuccess
               ? MMACT_OK
               : MMACT_ERR_CUDA;
}

MMACT_EXPORT mmact_status mmact_gemm_auto_choice(int64_t M, int64_t N, int64_t K, mmact_dtype ab_dtype,
                                                 mmact_dtype c_dtype, mmact_act act, int *split)
{
    if (split == nullptr || M < 0 || N < 0 || K < 0) return MMACT_ERR_INVALID_ARG;
    const bool in_ok = valid_in(ab_dtype) || ab_dtype == MMACT_F32;
    if (!in_ok || !valid_out(c_dtype) || !valid_act(act)) return MMACT_ERR_INVALID_ARG;
    *split = gemm_prefers_split(M, N, K, ab_dtype, act) ? 1 : 0;
    return MMACT_OK;
}

MMACT_EXPORT mmact_status mmact_gemm_auto(const void *A, const void *B, const float *bias, void *C,
                                          int64_t M, int64_t N, int64_t K, mmact_dtype ab_dtype,
                                          mmact_dtype c_dtype, mmact_act act, float alpha,
                                          float *workspace, void *stream)
{
    mmact_status s = gemm_check(A, B, bias, C, M, N, K, ab_dtype, c_dtype, act);
    if (s != MMACT_OK) return s;
    if (workspace != nullptr && !aligned16(workspace)) return MMACT_ERR_UNSUPPORTED;
    if (workspace != nullptr && gemm_prefers_split(M, N, K, ab_dtype, act))
        return mmact_gemm_split(A, B, bias, C, M, N, K, ab_dtype, c_dtype, act, alpha, workspace, stream);
    return mmact_gemm(A, B, bias, C, M, N, K, ab_dtype, c_dtype, act, alpha, stream);
}

MMACT_EXPORT mmact_status mmact_conv2d(const void *x, const void *w, const float *bias, void *y,
                                       int64_t N, int64_t C, int64_t H, int64_t W, int64_t Co,
                                       int64_t kh, int64_t kw, const int32_t strides[2],
                                       const int32_t pads[4], const int32_t dilations[2],
                                       mmact_dtype in_dtype, mmact_dtype out_dtype, mmact_act act,
                                       float alpha, void *stream)
{
    ConvGeom g;
    mmact_status s = conv_check(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations,
                                in_dtype, out_dtype, act, &g);
    if (s != MMACT_OK) return s;
    return conv_enqueue(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations, g, in_dtype,
                        out_dtype, act, alpha, static_cast<cudaStream_t>(stream));
}

MMACT_EXPORT mmact_status mmact_conv2d_residual(const void *x, const void *w, const float *bias,
                                                const void *R, void *y, int64_t N, int64_t C, int64_t H,
                                                int64_t W, int64_t Co, int64_t kh, int64_t kw,
                                                const int32_t strides[2], const int32_t pads[4],
                                                const int32_t dilations[2], mmact_dtype in_dtype,
                                                mmact_dtype out_dtype, mmact_act act, float alpha,
                                                void *stream)
{
    ConvGeom g;
    mmact_status s = conv_check(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations,
                                in_dtype, out_dtype, act, &g);
    if (s != MMACT_OK) return s;
    s = residual_check(R, y, N * Co * g.Ho * g.Wo * elem_bytes(out_dtype));
    if (s != MMACT_OK) return s;
    return conv_enqueue(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations, g, in_dtype,
                        out_dtype, act, alpha, static_cast<cudaStream_t>(stream), R);
}

MMACT_EXPORT mmact_status mmact_conv2d_nhwc_residual(const void *x, const void *w, const float *bias,
                                                     const void *R, void *y, int64_t N, int64_t C,
                                                     int64_t H, int64_t W, int64_t Co, int64_t kh,
                                                     int64_t kw, const int32_t strides[2],
                                                     const int32_t pads[4], const int32_t dilations[2],
                                                     mmact_dtype in_dtype, mmact_dtype out_dtype,
                                                     mmact_act act, float alpha, void *stream)
{
    ConvGeom g;
    mmact_status s = conv_check(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations,
                                in_dtype, out_dtype, act, &g, true);
    if (s != MMACT_OK) return s;
    if ((C * elem_bytes(in_dtype)) % 16 != 0 || Co % 8 != 0) return MMACT_ERR_UNSUPPORTED;
    if (N * g.Ho * g.Wo > MAX_DIM) return MMACT_ERR_UNSUPPORTED;
    if (in_dtype == MMACT_F32) return MMACT_ERR_UNSUPPORTED;   // split precision: no channels-last residual
    s = residual_check(R, y, N * Co * g.Ho * g.Wo * elem_bytes(out_dtype));
    if (s != MMACT_OK) return s;
    return nhwc_enqueue(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations, g, in_dtype,
                        out_dtype, act, alpha, static_cast<cudaStream_t>(stream), R);
}

MMACT_EXPORT mmact_status mmact_conv2d_split(const void *x, const void *w, const float *bias,
                                             void *y, int64_t N, int64_t C, int64_t H, int64_t W,
                                             int64_t Co, int64_t kh, int64_t kw,
                                             const int32_t strides[2], const int32_t pads[4],
                                             const int32_t dilations[2], mmact_dtype in_dtype,
                                             mmact_dtype out_dtype, mmact_act act, float alpha,
                                             float *workspace, void *stream)
{
    ConvGeom g;
    mmact_status s = conv_check(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations,
                                in_dtype, out_dtype, act, &g);
    if (s != MMACT_OK) return s;
    if (workspace == nullptr) return MMACT_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return MMACT_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = conv_enqueue(x, w, bias, workspace, N, C, H, W, Co, kh, kw, strides, pads, dilations, g,
                     in_dtype, MMACT_F32, MMACT_ACT_NONE, 0.0f, st);
    if (s != MMACT_OK) return s;
    DeviceInfo *dev = nullptr;
    if ((s = device_info(&dev)) != MMACT_OK) return s;
    return launch_act(workspace, y, N * Co * g.Ho * g.Wo, out_kind(out_dtype), (int)act, alpha,
                      act_grid(dev), st) == cudaSuccess
               ? MMACT_OK
               : MMACT_ERR_CUDA;
}

MMACT_EXPORT mmact_status mmact_conv2d_nhwc(const void *x, const void *w, const float *bias, void *y,
                                            int64_t N, int64_t C, int64_t H, int64_t W, int64_t Co,
                                            int64_t kh, int64_t kw, const int32_t strides[2],
                                            const int32_t pads[4], const int32_t dilations[2],
                                            mmact_dtype in_dtype, mmact_dtype out_dtype,
                                            mmact_act act, float alpha, void *stream)
{
    ConvGeom g;
    mmact_status s = conv_check(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations,
                                in_dtype, out_dtype, act, &g, true);
    if (s != MMACT_OK) return s;
    // 16-byte pitches: channel rows of x and w, output rows of y
    if ((C * elem_bytes(in_dtype)) % 16 != 0 || Co % 8 != 0) return MMACT_ERR_UNSUPPORTED;
    if (N * g.Ho * g.Wo > MAX_DIM) return MMACT_ERR_UNSUPPORTED;
    return nhwc_enqueue(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations, g, in_dtype,
                        out_dtype, act, alpha, static_cast<cudaStream_t>(stream));
}

MMACT_EXPORT mmact_status mmact_conv2d_auto_choice(int64_t N, int64_t C, int64_t H, int64_t W, int64_t Co,
                                                   int64_t kh, int64_t kw, const int32_t strides[2],
                                                   const int32_t pads[4], const int32_t dilations[2],
                                                   mmact_dtype in_dtype, mmact_dtype out_dtype, mmact_act act,
                                                   int *split)
{
    if (split == nullptr || N < 0 || C < 0 || Co < 0) return MMACT_ERR_INVALID_ARG;
    const bool in_ok = valid_in(in_dtype) || in_dtype == MMACT_F32;
    if (!in_ok || !valid_out(out_dtype) || !valid_act(act)) return MMACT_ERR_INVALID_ARG;
    ConvGeom g;
    mmact_status s = conv_geom(H, W, kh, kw, strides, pads, dilations, &g);
    if (s != MMACT_OK) return s;
    if (C * H * W > MAX_DIM || Co * g.Ho * g.Wo > MAX_DIM || C * kh * kw > MAX_DIM) return MMACT_ERR_UNSUPPORTED;
    *split = conv_prefers_split(N, C, H, W, Co, kh, kw, strides, pads, dilations, g, in_dtype, out_dtype, act)
                 ? 1 : 0;
    return MMACT_OK;
}

MMACT_EXPORT mmact_status mmact_conv2d_auto(const void *x, const void *w, const float *bias, void *y,
                                            int64_t N, int64_t C, int64_t H, int64_t W, int64_t Co,
                                            int64_t kh, int64_t kw, const int32_t strides[2],
                                            const int32_t pads[4], const int32_t dilations[2],
                                            mmact_dtype in_dtype, mmact_dtype out_dtype, mmact_act act,
                                            float alpha, float *workspace, void *stream)
{
    ConvGeom g;
    mmact_status s = conv_check(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations,
                                in_dtype, out_dtype, act, &g);
    if (s != MMACT_OK) return s;
    if (workspace != nullptr && !aligned16(workspace)) return MMACT_ERR_UNSUPPORTED;
    if (workspace != nullptr &&
        conv_prefers_split(N, C, H, W, Co, kh, kw, strides, pads, dilations, g, in_dtype, out_dtype, act))
        return mmact_conv2d_split(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations, in_dtype,
                                  out_dtype, act, alpha, workspace, stream);
    return mmact_conv2d(x, w, bias, y, N, C, H, W, Co, kh, kw, strides, pads, dilations, in_dtype, out_dtype,
                        act, alpha, stream);
}

MMACT_EXPORT mmact_status mmact_conv2d_out_shape(int64_t H, int64_t W, int64_t kh, int64_t kw,
                                                 const int32_t strides[2], const int32_t pads[4],
                                                 const int32_t dilations[2], int64_t *Ho,
                                                 int64_t *Wo)
{
    if (Ho == nullptr || Wo == nullptr) return MMACT_ERR_INVALID_ARG;
    ConvGeom g;
    mmact_status s = conv_geom(H, W, kh, kw, strides, pads, dilations, &g);
    if (s != MMACT_OK) return s;
    *Ho = g.Ho;
    *Wo = g.Wo;
    return MMACT_OK;
}

MMACT_EXPORT int mmact_conv2d_producer(int64_t N, int64_t C, int64_t H, int64_t W, int64_t Co,
                                       int64_t kh, int64_t kw, const int32_t strides[2],
                                       const int32_t pads[4], const int32_t dilations[2],
                                       mmact_dtype in_dtype, mmact_dtype out_dtype)
{
    ConvGeom g;
    if (N < 0 || C <= 0 || Co < 0 || !(valid_in(in_dtype) || in_dtype == MMACT_F32) || !valid_out(out_dtype))
        return -1;
    if (conv_geom(H, W, kh, kw, strides, pads, dilations, &g) != MMACT_OK) return -1;
    if (C * H * W > MAX_DIM || Co * g.Ho * g.Wo > MAX_DIM || C * kh * kw > MAX_DIM) return -1;
    if (use_tconv()) {
        TmemConvArgs tp;
        int bn = 0;
        if (tconv_plan(N, C, H, W, Co, kh, kw, strides, pads, dilations, g, in_dtype, tp, bn))
            return MMACT_CONV_TMEM;
    }
    ConvArgs a;
    conv_plan(N, C, H, W, Co, kh, kw, strides, pads, dilations, g, in_dtype, out_dtype, a);
    return a.win ? MMACT_CONV_WINDOW : a.vec ? MMACT_CONV_VECTOR : MMACT_CONV_GATHER;
}

MMACT_EXPORT mmact_status mmact_get_last_error(void *stream)
{
    DeviceInfo *dev = nullptr;
    mmact_status s = device_info(&dev);
    if (s != MMACT_OK) return s;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MMACT_ERR_CUDA;
    unsigned int word = 0;
    const unsigned int zero = 0;
    if (cudaMemcpy(&word, dev->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return MMACT_ERR_CUDA;
    if (word & ST_TIMEOUT) return MMACT_ERR_TIMEOUT;
    if (word != 0) return MMACT_ERR_CUDA;
    return MMACT_OK;
}

MMACT_EXPORT void mmact_set_wait_timeout_ns(uint64_t ns)
{
    g_wait_ns.store(ns == 0 ? DEFAULT_WAIT_NS : ns);
}

MMACT_EXPORT mmact_status mmact_selftest_wait_timeout(uint64_t timeout_ns, void *stream)
{
    DeviceInfo *dev = nullptr;
    mmact_status s = device_info(&dev);
    if (s != MMACT_OK) return s;
    return launch_wait_selftest(dev->status, timeout_ns, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? MMACT_OK
               : MMACT_ERR_CUDA;
}

MMACT_EXPORT mmact_status mmact_set_gemm_tile_n(int tile_n)
{
    if (tile_n != 0 && tile_n != 64 && tile_n != 128 && tile_n != 192 && tile_n != 224 &&
        tile_n != 256)
        return MMACT_ERR_INVALID_ARG;
    g_tile_n.store(tile_n);
    return MMACT_OK;
}

MMACT_EXPORT mmact_status mmact_gemm_split_k_choice(int64_t M, int64_t N, int64_t K, int *split_k)
{
    if (split_k == nullptr || M < 0 || N < 0 || K < 0) return MMACT_ERR_INVALID_ARG;
    DeviceInfo *dev = nullptr;
    mmact_status st = device_info(&dev);
    if (st != MMACT_OK) return st;
    *split_k = (M == 0 || N == 0 || K == 0)
                   ? 0
                   : choose_split_k(*dev, (M + 127) / 128, N, (K + 63) / 64);
    return MMACT_OK;
}

MMACT_EXPORT mmact_status mmact_gemm_kernel_choice(int64_t M, int64_t N, int64_t K, int has_residual,
                                                   int *kernel)
{
    if (kernel == nullptr || M < 0 || N < 0 || K < 0) return MMACT_ERR_INVALID_ARG;
    DeviceInfo *dev = nullptr;
    mmact_status st = device_info(&dev);
    if (st != MMACT_OK) return st;
    if (M == 0 || N == 0 || K == 0) {
        *kernel = MMACT_GEMM_KERNEL_NONE;
    } else if (choose_split_k(*dev, (M + 127) / 128, N, (K + 63) / 64) != 0) {
        *kernel = MMACT_GEMM_KERNEL_SPLIT_K;
    } else {
        *kernel = choose_pair(*dev, M, N, (K + 63) / 64, has_residual != 0) ? MMACT_GEMM_KERNEL_PAIR
                                                                            : MMACT_GEMM_KERNEL_PERSISTENT;
    }
    return MMACT_OK;
}

MMACT_EXPORT mmact_status mmact_set_gemm_pair(int mode)
{
    if (mode != 0 && mode != 1 && mode != 2) return MMACT_ERR_INVALID_ARG;
    g_pair.store(mode);
    return MMACT_OK;
}

MMACT_EXPORT mmact_status mmact_set_conv_tmem(int mode)
{
    if (mode != 0 && mode != 1) return MMACT_ERR_INVALID_ARG;
    g_conv_tmem.store(mode);
    return MMACT_OK;
}

MMACT_EXPORT mmact_status mmact_set_gemm_l2_policy(int mode)
{
    if (mode != 0 && mode != 1) return MMACT_ERR_INVALID_ARG;
    g_l2_policy.store(mode);
    return MMACT_OK;
}

MMACT_EXPORT mmact_status mmact_tensor_map_cache_stats(uint64_t *hits, uint64_t *encodes)
{
    if (hits != nullptr) *hits = g_tmap_hits.load();
    if (encodes != nullptr) *encodes = g_tmap_encodes.load();
    return MMACT_OK;
}

MMACT_EXPORT mmact_status mmact_set_gemm_split_k(int split_k)
{
    if (split_k != 0 && split_k != 1 && split_k != 2 && split_k != 4) return MMACT_ERR_INVALID_ARG;
    g_split_k.store(split_k);
    return MMACT_OK;
}

MMACT_EXPORT const char *mmact_status_string(mmact_status status)
{
    switch (status) {
    case MMACT_OK: return "MMACT_OK";
    case MMACT_ERR_INVALID_ARG: return "MMACT_ERR_INVALID_ARG: invalid argument";
    case MMACT_ERR_UNSUPPORTED: return "MMACT_ERR_UNSUPPORTED: alignment or dtype combination not supported";
    case MMACT_ERR_CUDA: return "MMACT_ERR_CUDA: a CUDA call failed";
    case MMACT_ERR_TIMEOUT: return "MMACT_ERR_TIMEOUT: a bounded wait inside a kernel ran out";
    default: return "unknown mmact_status";
    }
}

MMACT_EXPORT int mmact_version(void) { return 1; }
