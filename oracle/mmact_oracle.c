/*
 * mmact_oracle.c -- plain, slow, obviously-correct CPU oracle for the fused
 * GEMM / implicit-GEMM-conv + bias + activation path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load it.  It shares no code,
 * header, table or helper with the CUDA path; the two meet only through the
 * seeded input bytes that both consume.
 *
 * What it computes (fp64 throughout, over the exact input values: fp16 / bf16
 * codes, or fp32 values for the fp32-input variants):
 *
 *   GEMM   z[i][j] = (sum_{t<K} A[i][t] * B[t][j]) + bias[j]
 *          C[i][j] = act(z[i][j])
 *     -- "MatmulLeakyRelu fusion walkthrough" (pyasc examples/05_matmul_leakyrelu),
 *        overview: C = A x B + Bias, then LeakyReLU element-wise; its sample
 *        spec table (a [M,K] and b [K,N] fp16 row-major, not transposed; bias
 *        fp32 [1,N]; c fp32); and its precision check, which multiplies in fp32
 *        and adds the bias after the product.
 *
 *   CONV   z[n][co][oh][ow] = bias[co] + sum_{ci<C} sum_{r<kh} sum_{q<kw}
 *                 w[co][ci][r][q] * x[n][ci][oh*sh - pt + r*dh][ow*sw - pl + q*dw]
 *          (x is 0 outside [0,H) x [0,W)),  y = act(z)
 *          Ho = floor((H + pt + pb - dh*(kh-1) - 1) / sh) + 1, Wo likewise.
 *     -- "multimodal-ops Fused ConvTanh" article, section "what the operator
 *        computes": y = tanh(conv2d(x, filter, bias)) with strides / pads /
 *        dilations attributes; the output-shape rule is the standard
 *        (H + 2p - d(k-1) - 1)/s + 1 extended to asymmetric pads.
 *
 *   act    NONE: z;  RELU: z > 0 ? z : 0;  LEAKY_RELU: z > 0 ? z : alpha*z;
 *          TANH: (e^z - e^-z) / (e^z + e^-z);  SIGMOID: 1 / (1 + e^-z);
 *          GELU: z/2 * (1 + erf(z / sqrt(2)))
 *     -- LeakyReLU: MatmulLeakyRelu walkthrough, overview formula and its
 *        interface table (the comparison operator was lost when the page was
 *        extracted; read as '>').  ReLU: "ops-nn fused_matmul_relu" article,
 *        the naive fused loop (tmp > 0 ? tmp : 0).  tanh: Fused ConvTanh
 *        article, section "K2: the Vector engine computes tanh" (exp(z),
 *        exp(-z), difference over sum).  For |z| > 20 the ratio equals
 *        sign(z) to within fp64 rounding (1 - tanh(20) < 1e-17), so the
 *        oracle returns +-1 there instead of forming inf/inf.
 *          SIGMOID: 1 / (1 + e^-z)  -- the Fused ConvTanh article's twin operator,
 *        Fused ConvSigmoid (sigmoid(conv2d)), and the fused_matmul_relu article's
 *        first fusion family (matmul + ReLU / GELU / Sigmoid / Tanh).
 *          GELU: z * Phi(z) = z/2 * (1 + erf(z / sqrt(2))) -- same family; the pages
 *        print no formula, so this is the exact (erf) form, with C's erf() as
 *        the library step.
 *
 *   RESIDUAL (optional, both operators)
 *          z += R[same index],   then act(z)
 *     -- "ops-nn fused_matmul_relu" article, section on the fusion families
 *        (the element-wise "math" family): matmul + add + bias fused so that a
 *        residual path is accumulated on chip instead of through HBM.  The page
 *        gives no formula; the plain reading, in the order residual networks
 *        use, adds R to the pre-activation: act(A x B + bias + R).  R has the
 *        output's shape and dtype (fp16 / bf16 codes or fp32 values).
 *
 * Input decoding follows the IEEE 754 binary16 definition (1 sign, 5 exponent
 * bits with bias 15, 10 fraction bits) and the bfloat16 definition (the upper
 * 16 bits of an IEEE binary32); fp32 inputs are widened to fp64 exactly.  The
 * fp32 variants (the Fused ConvTanh article's evaluation covers fp32 cases
 * beside fp16 and bf16) are still defined on the exact fp32 values: any
 * reduced-precision arithmetic on the GPU side is the GPU's error.
 *
 * Each output element is computed on its own, from the definition, with the
 * sum over t (GEMM) or (ci, r, q) (conv) taken in ascending order.  Callers
 * may ask for all outputs or for a list of flat output indices; the value of
 * an element does not depend on which other elements are requested.
 *
 * Build: plain C99, -O2 -ffp-contract=off (no fused multiply-add, so the
 * x86 and Arm builds round identically), no vector intrinsics, no OpenMP.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { OR_F16 = 0, OR_BF16 = 1, OR_F32 = 2 };
enum { OR_ACT_NONE = 0, OR_ACT_RELU = 1, OR_ACT_LEAKY_RELU = 2, OR_ACT_TANH = 3,
       OR_ACT_SIGMOID = 4, OR_ACT_GELU = 5 };

/* IEEE 754 binary16 -> double, from the format's definition. */
double oracle_decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -24);            /* subnormal: f * 2^-10 * 2^-14 */
    } else if (e == 31) {
        mag = f ? NAN : INFINITY;
    } else {
        mag = ldexp(1.0 + (double)f / 1024.0, e - 15);
    }
    return sign ? -mag : mag;
}

/* bfloat16 -> double: the 16 bits are the top half of an IEEE binary32. */
double oracle_decode_bf16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -133);           /* subnormal: f * 2^-7 * 2^-126 */
    } else if (e == 255) {
        mag = f ? NAN : INFINITY;
    } else {
        mag = ldexp(1.0 + (double)f / 128.0, e - 127);
    }
    return sign ? -mag : mag;
}

static double decode(uint16_t code, int dtype)
{
    return dtype == OR_BF16 ? oracle_decode_bf16(code) : oracle_decode_f16(code);
}

/* Element idx of an input tensor: 16-bit codes (OR_F16 / OR_BF16) or fp32 values (OR_F32). */
static double in_value(const void *p, int dtype, int64_t idx)
{
    if (dtype == OR_F32) return (double)((const float *)p)[idx];
    return decode(((const uint16_t *)p)[idx], dtype);
}

static int valid_in_dtype(int dtype)
{
    return dtype == OR_F16 || dtype == OR_BF16 || dtype == OR_F32;
}

/* Element idx of a residual tensor of dtype rdtype (16-bit codes or fp32). */
static double residual_value(const void *R, int rdtype, int64_t idx)
{
    return in_value(R, rdtype, idx);
}

/* z plus residual element idx (z itself when there is no residual). */
static double add_residual(double z, const void *R, int rdtype, int64_t idx)
{
    return R ? z + residual_value(R, rdtype, idx) : z;
}

/* tanh written out as the ratio of exponentials. */
double oracle_tanh(double z)
{
    if (z > 20.0) return 1.0;
    if (z < -20.0) return -1.0;
    double ep = exp(z);
    double em = exp(-z);
    return (ep - em) / (ep + em);
}

double oracle_sigmoid(double z)
{
    return 1.0 / (1.0 + exp(-z));
}

double oracle_gelu(double z)
{
    return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));
}

double oracle_act(double z, int act, double alpha)
{
    switch (act) {
    case OR_ACT_NONE:       return z;
    case OR_ACT_RELU:       return z > 0.0 ? z : 0.0;
    case OR_ACT_LEAKY_RELU: return z > 0.0 ? z : alpha * z;
    case OR_ACT_TANH:       return oracle_tanh(z);
    case OR_ACT_SIGMOID:    return oracle_sigmoid(z);
    case OR_ACT_GELU:       return oracle_gelu(z);
    default:                return NAN;
    }
}

/* One GEMM output element: the K-term dot product, then the bias. */
static double gemm_z(const void *A, const void *B, int dtype, const float *bias,
                     int64_t N, int64_t K, int64_t i, int64_t j)
{
    double s = 0.0;
    for (int64_t t = 0; t < K; ++t)
        s += in_value(A, dtype, i * K + t) * in_value(B, dtype, t * N + j);
    return s + (bias ? (double)bias[j] : 0.0);
}

/*
 * A: [M,K] row-major; B: [K,N] row-major (16-bit codes of dtype, or fp32
 * values when dtype == OR_F32); bias: [N] fp32 or NULL;
 * R: residual [M,N] of dtype rdtype (OR_F16 / OR_BF16 codes, OR_F32 floats) or NULL.
 * points == NULL: out[i*N + j] for every element.  Otherwise out[p] is the
 * element at flat index points[p] (= i*N + j).  Returns 0, or -1 on a bad
 * argument.
 */
int oracle_gemm_res(const void *A, const void *B, int dtype, const float *bias,
                    const void *R, int rdtype, int64_t M, int64_t N, int64_t K, int act,
                    double alpha, const int64_t *points, int64_t npoints, double *out)
{
    if (M < 0 || N < 0 || K < 0 || !valid_in_dtype(dtype)) return -1;
    if (R != NULL && !valid_in_dtype(rdtype)) return -1;
    int64_t count = points ? npoints : M * N;
    for (int64_t p = 0; p < count; ++p) {
        int64_t idx = points ? points[p] : p;
        if (idx < 0 || idx >= M * N) return -1;
        double z = gemm_z(A, B, dtype, bias, N, K, idx / N, idx % N);
        out[p] = oracle_act(add_residual(z, R, rdtype, idx), act, alpha);
    }
    return 0;
}

/* As oracle_gemm_res with no residual. */
int oracle_gemm(const void *A, const void *B, int dtype, const float *bias,
                int64_t M, int64_t N, int64_t K, int act, double alpha,
                const int64_t *points, int64_t npoints, double *out)
{
    return oracle_gemm_res(A, B, dtype, bias, NULL, 0, M, N, K, act, alpha, points, npoints, out);
}

/* Output extent of one spatial axis. */
int64_t oracle_conv_out_dim(int64_t in, int64_t k, int64_t stride, int64_t pad_lo,
                            int64_t pad_hi, int64_t dil)
{
    if (stride <= 0 || dil <= 0 || k <= 0) return -1;
    int64_t span = in + pad_lo + pad_hi - dil * (k - 1) - 1;
    if (span < 0) return 0;
    return span / stride + 1;
}

typedef struct {
    int64_t Nb, C, H, W, Co, kh, kw, sh, sw, pt, pb, pl, pr, dh, dw, Ho, Wo;
} conv_geom;

/* One conv output element, by direct summation over (ci, r, q). */
static double conv_z(const void *x, const void *w, int dtype, const float *bias,
                     const conv_geom *g, int64_t n, int64_t co, int64_t oh, int64_t ow)
{
    double s = 0.0;
    for (int64_t ci = 0; ci < g->C; ++ci)
        for (int64_t r = 0; r < g->kh; ++r)
            for (int64_t q = 0; q < g->kw; ++q) {
                int64_t ih = oh * g->sh - g->pt + r * g->dh;
                int64_t iw = ow * g->sw - g->pl + q * g->dw;
                if (ih < 0 || ih >= g->H || iw < 0 || iw >= g->W) continue;  /* zero padding */
                double xv = in_value(x, dtype, ((n * g->C + ci) * g->H + ih) * g->W + iw);
                double wv = in_value(w, dtype, ((co * g->C + ci) * g->kh + r) * g->kw + q);
                s += wv * xv;
            }
    return s + (bias ? (double)bias[co] : 0.0);
}

/*
 * x: [Nb,C,H,W]; w: [Co,C,kh,kw] (16-bit codes of dtype, or fp32 values
 * when dtype == OR_F32); bias: [Co] fp32 or NULL;
 * R: residual [Nb,Co,Ho,Wo] of dtype rdtype, or NULL.
 * pads = (top, bottom, left, right).  y is [Nb,Co,Ho,Wo]; points are flat
 * indices into y (NULL = all).  Returns 0, or -1 on a bad argument.
 */
int oracle_conv2d_res(const void *x, const void *w, int dtype, const float *bias,
                      const void *R, int rdtype,
                      int64_t Nb, int64_t C, int64_t H, int64_t W, int64_t Co, int64_t kh, int64_t kw,
                      int64_t sh, int64_t sw, int64_t pt, int64_t pb, int64_t pl, int64_t pr,
                      int64_t dh, int64_t dw, int act, double alpha,
                      const int64_t *points, int64_t npoints, double *out)
{
    if (!valid_in_dtype(dtype)) return -1;
    if (R != NULL && !valid_in_dtype(rdtype)) return -1;
    if (Nb < 0 || C < 0 || H < 0 || W < 0 || Co < 0 || kh <= 0 || kw <= 0) return -1;
    if (pt < 0 || pb < 0 || pl < 0 || pr < 0) return -1;
    conv_geom g = {Nb, C, H, W, Co, kh, kw, sh, sw, pt, pb, pl, pr, dh, dw, 0, 0};
    g.Ho = oracle_conv_out_dim(H, kh, sh, pt, pb, dh);
    g.Wo = oracle_conv_out_dim(W, kw, sw, pl, pr, dw);
    if (g.Ho < 0 || g.Wo < 0) return -1;
    int64_t total = Nb * Co * g.Ho * g.Wo;
    int64_t count = points ? npoints : total;
    for (int64_t p = 0; p < count; ++p) {
        int64_t idx = points ? points[p] : p;
        if (idx < 0 || idx >= total) return -1;
        int64_t ow = idx % g.Wo;
        int64_t oh = (idx / g.Wo) % g.Ho;
        int64_t co = (idx / (g.Wo * g.Ho)) % Co;
        int64_t n = idx / (g.Wo * g.Ho * Co);
        double z = conv_z(x, w, dtype, bias, &g, n, co, oh, ow);
        out[p] = oracle_act(add_residual(z, R, rdtype, idx), act, alpha);
    }
    return 0;
}

/* As oracle_conv2d_res with no residual. */
int oracle_conv2d(const void *x, const void *w, int dtype, const float *bias,
                  int64_t Nb, int64_t C, int64_t H, int64_t W, int64_t Co, int64_t kh, int64_t kw,
                  int64_t sh, int64_t sw, int64_t pt, int64_t pb, int64_t pl, int64_t pr,
                  int64_t dh, int64_t dw, int act, double alpha,
                  const int64_t *points, int64_t npoints, double *out)
{
    return oracle_conv2d_res(x, w, dtype, bias, NULL, 0, Nb, C, H, W, Co, kh, kw, sh, sw, pt, pb,
                             pl, pr, dh, dw, act, alpha, points, npoints, out);
}
