/*
 * oracle.c -- plain, slow CPU oracle for one KV-cache decode step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may load this library.  It shares no
 * source, header, table or helper with the GPU library; the two are compared
 * element by element on the same seeded inputs.
 *
 * Sources, cited by page title and section:
 *   [LEAN]    "用Lean4形式化验证滑动窗口KV Cache的正确性" (framerc.cn/news/4505248)
 *   [LOOP]    "KV Cache 自回归生成推理（增量更新与状态拼接）" (airsota.com/?p=549)
 *   [WITCERT] "WitCert: Sound Runtime Risk Observability and Gating for
 *             KV-Cache Quantization" (agifrontier.github.io tutorial)
 *
 * Arithmetic rules.  Attention is evaluated in fp64 from the exact stored
 * values.  The stored cache values (RoPE-rotated keys, bf16 rounding, INT8
 * codes, scales and witnesses) are integer or IEEE-rounded results that the
 * GPU must reproduce bit for bit, so they are computed here with the IEEE
 * operations their definition names, one rounding per operation.  Build with
 * -ffp-contract=off -frounding-math and without -ffast-math so that the
 * compiler neither fuses nor reorders them.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#pragma STDC FENV_ACCESS ON

#define ORC_VERSION 1

int orc_version(void) { return ORC_VERSION; }

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the upper half of an fp32 bit pattern, so widening is exact. */
float orc_bf16_to_f32(uint16_t b) { return bits_to_f32((uint32_t)b << 16); }

/* Round an fp32 value to bf16, to nearest, ties to the even neighbour.
 * The two candidates are the truncation `lo` (toward zero) and the next bf16
 * away from zero `hi`; the discarded low half decides between them. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u = f32_to_bits(f);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);           /* NaN stays a quiet NaN */
    uint32_t lo = u >> 16;
    uint32_t hi = lo + 1u;                                 /* may carry into inf: correct */
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u) return (uint16_t)hi;
    if (rest < 0x8000u) return (uint16_t)lo;
    return (uint16_t)((lo & 1u) ? hi : lo);
}

void orc_f32_to_bf16_array(const float* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_bf16(x[i]);
}

void orc_bf16_to_f32_array(const uint16_t* x, float* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = orc_bf16_to_f32(x[i]);
}

/* Value of an IEEE binary16 bit pattern. */
double orc_f16_value(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(m + 1024), e - 25);            /* (1 + m/1024) * 2^(e-15) */
    return s ? -v : v;
}

/* The smallest binary16 value that is >= x (rounding toward +infinity).
 * For x >= 0 the patterns 0x0000..0x7bff are the finite values in increasing
 * order, so a binary search over them finds it; beyond 65504 it is +inf. */
uint16_t orc_f32_to_f16_up(float xf)
{
    double x = (double)xf;
    if (isnan(x)) return 0x7e00u;
    if (x > 65504.0) return 0x7c00u;
    if (x <= 0.0) {
        /* smallest fp16 >= x <= 0 is minus the largest magnitude <= |x| */
        if (x == 0.0) return 0x0000u;
        double ax = -x;
        if (ax >= 65504.0) return 0xfbffu;
        int lo = 0, hi = 0x7bff;                           /* largest bits with value <= ax */
        while (lo < hi) {
            int mid = (lo + hi + 1) / 2;
            if (orc_f16_value((uint16_t)mid) <= ax) lo = mid; else hi = mid - 1;
        }
        return lo == 0 ? 0x0000u : (uint16_t)(0x8000u | (unsigned)lo);
    }
    int lo = 0, hi = 0x7bff;                               /* smallest bits with value >= x */
    while (lo < hi) {
        int mid = (lo + hi) / 2;
        if (orc_f16_value((uint16_t)mid) >= x) hi = mid; else lo = mid + 1;
    }
    return (uint16_t)lo;
}

/* ------------------------------------------------------------------------ */
/* Rotary position embedding of cached keys and of the query                */
/* ------------------------------------------------------------------------ */
/*
 * The pages require keys to be stored RoPE-rotated at their absolute position
 * and rely on RoPE acting as an orthogonal rotation on whole frequency pairs
 * ([WITCERT] "频带酉性与双层证书", band unitarity); they print no formula.
 * Reading taken: interleaved pairs (2i, 2i+1); frequency theta_i =
 * base^(-(2i)/d); angle = p * theta_i in double; cos and sin of the angle in
 * double, each rounded once to fp32.
 *
 * cs receives n rows (positions p0 .. p0+n-1) of d/2 {cos, sin} pairs.
 */
void orc_rope_cos_sin(double base, int d, int64_t p0, int64_t n, float* cs)
{
    int half = d / 2;
    for (int64_t r = 0; r < n; ++r) {
        double p = (double)(p0 + r);
        for (int i = 0; i < half; ++i) {
            double expo = (double)(-2 * i) / (double)d;
            double theta = pow(base, expo);
            double ang = p * theta;
            cs[(r * half + i) * 2 + 0] = (float)cos(ang);
            cs[(r * half + i) * 2 + 1] = (float)sin(ang);
        }
    }
}

/* Rotate rows of d fp32 values; row r uses the {cos, sin} row cs[r].
 * Per pair, in fp32 with each product and the sum rounded separately:
 *   y0 = (x0*c) - (x1*s),   y1 = (x1*c) + (x0*s).                         */
void orc_rope_rotate(const float* x, const float* cs, int64_t rows, int d, float* y)
{
    int half = d / 2;
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * d;
        const float* cr = cs + r * half * 2;
        float* yr = y + r * d;
        for (int i = 0; i < half; ++i) {
            float c = cr[2 * i], s = cr[2 * i + 1];
            float x0 = xr[2 * i], x1 = xr[2 * i + 1];
            float a = x0 * c;
            float b = x1 * s;
            float e = x1 * c;
            float f = x0 * s;
            yr[2 * i] = a - b;
            yr[2 * i + 1] = e + f;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Attention by definition                                                  */
/* ------------------------------------------------------------------------ */
/*
 * Reference attention with the full cache plus window and causal masks
 * ([LEAN] §2.1):  out = softmax(q K^T / sqrt(d) + mask_window + mask_causal) V.
 * Row j of the history holds absolute position p0 + j.  A row is visible to
 * the query at position t iff pos <= t (causal mask) and, when a window W > 0
 * is given, pos >= t - W + 1 (window mask).  Signed 64-bit positions keep
 * t - W + 1 from wrapping ([LEAN] §5.2).  The softmax subtracts the maximum
 * visible logit before exponentiating ([LOOP] §三).  Everything is fp64.
 *
 * kind: 0 = fp32 values, 1 = bf16 bit patterns, 2 = fp64 values.
 * Returns the number of visible rows (0 leaves out[] zero).
 */
static double elem(int kind, const void* base, int64_t idx)
{
    if (kind == 0) return (double)((const float*)base)[idx];
    if (kind == 1) return (double)orc_bf16_to_f32(((const uint16_t*)base)[idx]);
    return ((const double*)base)[idx];
}

static int64_t attend_one(int d, const double* q, int64_t n, int kind, const void* K,
                          const void* V, int64_t p0, int64_t t, int64_t window, double* out)
{
    double* logit = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    double mx = -INFINITY;
    int64_t visible = 0;
    for (int64_t j = 0; j < n; ++j) {
        int64_t pos = p0 + j;
        int vis = (pos <= t) && (window <= 0 || pos >= t - window + 1);
        if (!vis) { logit[j] = -INFINITY; continue; }
        double s = 0.0;
        for (int i = 0; i < d; ++i) s += q[i] * elem(kind, K, j * d + i);
        logit[j] = s / sqrt((double)d);
        if (logit[j] > mx) mx = logit[j];
        ++visible;
    }
    for (int i = 0; i < d; ++i) out[i] = 0.0;
    if (visible == 0) { free(logit); return 0; }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        if (logit[j] == -INFINITY) continue;
        double p = exp(logit[j] - mx);
        l += p;
        for (int i = 0; i < d; ++i) out[i] += p * elem(kind, V, j * d + i);
    }
    for (int i = 0; i < d; ++i) out[i] /= l;
    free(logit);
    return visible;
}

/* Independent problems, each: nq query rows sharing one history (the query
 * heads of one KV head).  q: [nprob][nq][d]; K[i], V[i]: n[i] rows of d;
 * out: [nprob][nq][d].  Problems are distributed over nthreads threads. */
void orc_attend_batch(int nprob, int nq, int d, int kind, int64_t window, const double* q,
                      const void* const* K, const void* const* V, const int64_t* n,
                      const int64_t* p0, const int64_t* t, double* out, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int pi = 0; pi < nprob; ++pi)
        for (int h = 0; h < nq; ++h)
            attend_one(d, q + ((int64_t)pi * nq + h) * d, n[pi], kind, K[pi], V[pi], p0[pi],
                       t[pi], window, out + ((int64_t)pi * nq + h) * d);
}

/* Softmax weights of one query over one history, same masks as above, fp64.
 * Used for the total-variation check of the quantized tier. */
int64_t orc_softmax_weights(int d, const double* q, int64_t n, int kind, const void* K,
                            int64_t p0, int64_t t, int64_t window, double* p)
{
    double mx = -INFINITY;
    int64_t visible = 0;
    for (int64_t j = 0; j < n; ++j) {
        int64_t pos = p0 + j;
        int vis = (pos <= t) && (window <= 0 || pos >= t - window + 1);
        if (!vis) { p[j] = -INFINITY; continue; }
        double s = 0.0;
        for (int i = 0; i < d; ++i) s += q[i] * elem(kind, K, j * d + i);
        p[j] = s / sqrt((double)d);
        if (p[j] > mx) mx = p[j];
        ++visible;
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        p[j] = (p[j] == -INFINITY) ? 0.0 : exp(p[j] - mx);
        l += p[j];
    }
    if (visible) for (int64_t j = 0; j < n; ++j) p[j] /= l;
    return visible;
}

/* ------------------------------------------------------------------------ */
/* INT8 tier: block quantizer, residual, witness                            */
/* ------------------------------------------------------------------------ */
/*
 * Symmetric INT8 quantization with one fp32 scale per 16-token block
 * ([WITCERT] "SGLang 生产级落地与闭环门控修复": per-block scale factors).
 * Reading taken: s = amax / 127 (one fp32 division), code =
 * clamp(rint(x / s), -127, 127) with x / s one fp32 division and rint rounding
 * half to even; amax = 0 gives s = 0 and all codes 0.
 * x holds `count` fp32 values (the exact bf16 cache values of the block).
 * Returns s.
 */
float orc_quantize_block(const float* x, int64_t count, int8_t* codes)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < count; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    for (int64_t i = 0; i < count; ++i) {
        if (s == 0.0f) { codes[i] = 0; continue; }
        float y = x[i] / s;
        float r = rintf(y);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        codes[i] = (int8_t)r;
    }
    return s;
}

/*
 * Philox4x32-10 (J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
 * Random Numbers: As Easy as 1, 2, 3", SC 2011): a counter of four 32-bit words
 * and a key of two go through ten rounds; each round multiplies counter words 0
 * and 2 by the round multipliers (64-bit products split into high and low
 * halves), and recombines them with words 1 and 3 and the key by xor, after
 * which the key is bumped by the Weyl constants.
 */
void orc_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out)
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        c0 = n0; c1 = (uint32_t)p1; c2 = n2; c3 = (uint32_t)p0;
        k0 += 0x9E3779B9u; k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/*
 * Key dither bytes of n rows at positions p0 .. p0+n-1 of one (request, layer, KV
 * head), out[n][d].  One Philox call per (position, group of 16 channels) with the
 * five-tuple counter (position, group, KV head + 65536 layer, request); byte i of the
 * call (word i/4, least significant byte first) is the dither of channel 16 group + i.
 */
void orc_dither_rows(const uint32_t* key, uint32_t request, uint32_t layer, uint32_t kv_head, int64_t p0,
                     int64_t n, int d, uint8_t* out)
{
    const uint32_t c2 = kv_head + 65536u * layer;
    for (int64_t r = 0; r < n; ++r) {
        uint8_t* row = out + r * d;
        for (int j = 0; j < d / 16; ++j) {
            const uint32_t ctr[4] = {(uint32_t)(p0 + r), (uint32_t)j, c2, request};
            uint32_t w[4];
            orc_philox4x32_10(ctr, key, w);
            for (int i = 0; i < 16; ++i) row[16 * j + i] = (uint8_t)(w[i / 4] >> (8 * (i % 4)));
        }
    }
}

/*
 * Block quantization with a subtractive dither ([WITCERT] "为了进一步压榨显存极限"
 * paragraph, Tier B): the dither u (one per element, multiples of 2^-8 in
 * [-1/2, 1/2)) is added before rounding and removed again on reading:
 *   s = amax/127,  code = clamp(rint(x/s + u), -127, 127),  x_hat = (code - u) s.
 * x/s and the addition are IEEE fp32 operations (the GPU does the same); s = 0
 * gives codes 0.  Returns s.
 */
float orc_quantize_block_dither(const float* x, const float* u, int64_t count, int8_t* codes)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < count; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    for (int64_t i = 0; i < count; ++i) {
        if (s == 0.0f) { codes[i] = 0; continue; }
        volatile float y = x[i] / s;
        volatile float z = y + u[i];
        float r = rintf(z);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        codes[i] = (int8_t)r;
    }
    return s;
}

/*
 * Witness of one key row ([WITCERT] "频带酉性与双层证书": w_{t,b} = ||r_{t,b}||
 * for 16 bands, fp16, 32 bytes per token and head).
 * r = x - code*s is exact in fp64 and also representable in fp32 (|r| <= s/2
 * and r is a multiple of 2^-23 ulp(s)); this is checked and -1 is returned if
 * it ever fails.  The band norm is then evaluated in fp32 with every operation
 * rounded toward +infinity, squares summed in index order from zero, and the
 * result stored as the smallest fp16 not below it, so the stored witness is
 * never below the exact norm.  The band b covers dims [b*d/nb, (b+1)*d/nb).
 */
int orc_witness_row(const float* x, const int8_t* codes, float s, int d, int nb, uint16_t* w)
{
    int bw = d / nb;
    float r[1024];
    if (d > 1024) return -2;
    for (int i = 0; i < d; ++i) {
        double r64 = (double)x[i] - (double)codes[i] * (double)s;
        r[i] = (float)r64;
        if ((double)r[i] != r64) return -1;
    }
    for (int b = 0; b < nb; ++b) {
        int old = fegetround();
        fesetround(FE_UPWARD);
        volatile float acc = 0.0f;
        for (int i = b * bw; i < (b + 1) * bw; ++i) {
            volatile float sq = r[i] * r[i];
            acc = acc + sq;
        }
        volatile float nrm = sqrtf(acc);
        fesetround(old);
        w[b] = orc_f32_to_f16_up(nrm);
    }
    return 0;
}

/* Residual of one row as fp32 (exact), for the soundness checks. */
void orc_residual_row(const float* x, const int8_t* codes, float s, int d, float* r)
{
    for (int i = 0; i < d; ++i) r[i] = (float)((double)x[i] - (double)codes[i] * (double)s);
}
