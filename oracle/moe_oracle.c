/*
 * CPU oracle for the routed mixture-of-experts FFN over NVFP4 weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant generator with the CUDA path.
 *
 * This file holds the parts of the oracle whose result must be bit-exact:
 * the E2M1 / E4M3 codecs, the NVFP4 block quantiser (fp32 arithmetic in a
 * fixed order), the router logits in a fixed fp32 summation order, top-k
 * selection and the grouping of (token, slot) pairs by expert.  The FFN
 * itself (FP64) lives in oracle/__init__.py.
 *
 * Sources (page title, section):
 *  - "NVIDIA FP4-Local checkpoints on DGX Spark ... #565", section 4 Round 1:
 *    NVFP4 weights are U8 codes (two E2M1 values a byte) with F8_E4M3 scales
 *    held as stored (#489) and one FP32 tensor scale per weight (#517, #545);
 *    routed experts are grouped so each is read once (#740); router logits are
 *    fp32 (#763).
 *  - "bloomery 0.3.9", From our contributors: the router's normalisation
 *    policy is a named choice (#772).
 *  The E2M1 and E4M3 bit layouts are the OCP Microscaling ones (the pages
 *  name the formats but never print them).  Every other open point is the
 *  plain reading listed in the design notes: block of 16, tensor scale
 *  amax/(6*448), element 2i in the low nibble, canonical logit order below.
 *
 * Build: gcc -O2 -ffp-contract=off (no implicit fused multiply-adds; the only
 * fused operations are the explicit fmaf() calls of the router).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- codecs */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: value = mantissa * 0.5. */
double oracle_e2m1_value(int code)
{
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return (code & 8) ? -v : v;
}

/* E4M3 ("FN" variant): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa, no infinities, S.1111.111 is NaN, exponent field 0 subnormal. */
double oracle_e4m3_value(int byte)
{
    int e = (byte >> 3) & 15;
    int m = byte & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return (byte & 0x80) ? -v : v;
}

void oracle_e2m1_table(double *out16)
{
    for (int c = 0; c < 16; ++c) out16[c] = oracle_e2m1_value(c);
}

void oracle_e4m3_table(double *out256)
{
    for (int b = 0; b < 256; ++b) out256[b] = oracle_e4m3_value(b);
}

/* fp32 -> E4M3 with round-to-nearest-even and saturation to +-448.
 * The magnitude is split as 2^e * (1 + q/8) (or q * 2^-9 below 2^-6) and q is
 * rounded with rint(), which rounds halves to even; an even q is an even code. */
uint8_t oracle_e4m3_from_f32(float f)
{
    int neg = signbit(f) ? 1 : 0;
    double v = fabs((double)f);
    int code;
    if (isnan(f))
        return (uint8_t)(0x7F | (neg << 7));
    if (v >= 448.0) {
        code = 0x7E;
    } else if (v < ldexp(1.0, -6)) {
        code = (int)rint(ldexp(v, 9));            /* 0..8; 8 is 2^-6 */
    } else {
        int E;
        frexp(v, &E);
        int e = E - 1;                            /* v in [2^e, 2^(e+1)) */
        double q = rint((ldexp(v, -e) - 1.0) * 8.0);
        if (q >= 8.0) { q = 0.0; e += 1; }
        code = ((e + 7) << 3) | (int)q;
        if (code > 0x7E) code = 0x7E;
    }
    return (uint8_t)(code | (neg << 7));
}

/* fp32 -> E2M1 with round-to-nearest-even and saturation to +-6.  A negative
 * value keeps its sign bit even when it rounds to zero (code 8 is -0). */
uint8_t oracle_e2m1_from_f32(float f)
{
    int neg = signbit(f) ? 1 : 0;
    double v = fabs((double)f);
    int code;
    if (isnan(f) || v >= 6.0) {
        code = 7;
    } else if (v < 1.0) {
        code = (int)rint(v * 2.0);                 /* 0, 0.5, 1.0 -> codes 0,1,2 */
    } else {
        int E;
        frexp(v, &E);
        int e = E - 1;                             /* 0..2 */
        double q = rint((ldexp(v, -e) - 1.0) * 2.0);
        if (q >= 2.0) { q = 0.0; e += 1; }
        code = ((e + 1) << 1) | (int)q;
        if (code > 7) code = 7;
    }
    return (uint8_t)(code | (neg << 3));
}

float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* FP64 -> bf16 with one round-to-nearest-even (never through fp32). */
uint16_t oracle_f64_to_bf16(double d)
{
    if (isnan(d))
        return 0x7FC0;
    int neg = signbit(d) ? 1 : 0;
    double a = fabs(d), q;
    if (a == 0.0) {
        q = 0.0;
    } else if (a < ldexp(1.0, -126)) {
        q = ldexp(rint(ldexp(a, 133)), -133);      /* subnormal spacing 2^-133 */
    } else {
        int E;
        frexp(a, &E);
        int e = E - 1;                             /* a in [2^e, 2^(e+1)) */
        q = ldexp(rint(ldexp(a, 7 - e)), e - 7);   /* 8 significant bits */
    }
    float f = (float)q;                            /* exact, or +inf past the range */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)((u >> 16) | (neg ? 0x8000u : 0u));
}

void oracle_f64_to_bf16_array(const double *src, int64_t n, uint16_t *dst)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_f64_to_bf16(src[i]);
}

void oracle_e4m3_from_f32_array(const float *src, int64_t n, uint8_t *dst)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_e4m3_from_f32(src[i]);
}

void oracle_e2m1_from_f32_array(const float *src, int64_t n, uint8_t *dst)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_e2m1_from_f32(src[i]);
}

/* ------------------------------------------------------- NVFP4 quantiser */

/* Tensor scale of a whole tensor: amax / (6 * 448), in fp32. */
float oracle_nvfp4_tensor_scale(const float *x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    return amax / 2688.0f;
}

/* Quantise a row-major [rows][cols] fp32 matrix to NVFP4 with a given tensor
 * scale ts.  For every block of 16 consecutive values of a row:
 *   s    = E4M3_rne_sat((block_amax / 6) / ts)        (fp32 divisions)
 *   den  = E4M3_value(s) * ts                          (fp32 multiply)
 *   code = E2M1_rne_sat(x / den)                       (fp32 division)
 * A zero tensor scale gives scale byte 0; a zero den gives code 0.
 * codes: [rows][cols/2], element 2i in bits 0..3 and 2i+1 in bits 4..7.
 * scales: [rows][cols/16].  cols must be a multiple of 16. */
void oracle_nvfp4_quantize(const float *x, int64_t rows, int64_t cols, float ts,
                           uint8_t *codes, uint8_t *scales)
{
    int64_t nb = cols / 16;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *blk = x + r * cols + b * 16;
            float bamax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = fabsf(blk[i]);
                if (a > bamax) bamax = a;
            }
            uint8_t s = 0;
            if (ts != 0.0f) {
                float t = (bamax / 6.0f) / ts;
                s = oracle_e4m3_from_f32(t);
            }
            float den = (float)oracle_e4m3_value(s) * ts;
            uint8_t q[16];
            for (int i = 0; i < 16; ++i)
                q[i] = (den == 0.0f) ? 0 : oracle_e2m1_from_f32(blk[i] / den);
            scales[r * nb + b] = s;
            uint8_t *dst = codes + r * (cols / 2) + b * 8;
            for (int i = 0; i < 8; ++i)
                dst[i] = (uint8_t)(q[2 * i] | (q[2 * i + 1] << 4));
        }
    }
}

/* ----------------------------------------------------- MXFP4 (OCP MX) */

/* E8M0: an unsigned power of two, value 2^(byte - 127); 0xFF is NaN. */
double oracle_e8m0_value(int byte)
{
    return byte == 255 ? NAN : ldexp(1.0, byte - 127);
}

void oracle_e8m0_table(double *out256)
{
    for (int b = 0; b < 256; ++b) out256[b] = oracle_e8m0_value(b);
}

/* MXFP4 quantiser, following the OCP Microscaling (MX) v1.0 conversion: for
 * every block of 32 consecutive values of a row,
 *   amax  = max |x|;
 *   E     = floor(log2(amax)) - 2       (2: exponent of E2M1's largest value, 6 = 1.5 * 2^2)
 *   scale = E + 127, clamped to [0, 254] (an all-zero block: 0)
 *   code  = E2M1_rne_sat(x / 2^(scale - 127))   (fp32 division by a power of two)
 * codes: [rows][cols/2], element 2i in bits 0..3; scales: [rows][cols/32].
 * cols must be a multiple of 32. */
void oracle_mxfp4_quantize(const float *x, int64_t rows, int64_t cols, uint8_t *codes, uint8_t *scales)
{
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *blk = x + r * cols + b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(blk[i]);
                if (a > amax) amax = a;
            }
            int s = 0;
            if (amax > 0.0f) {
                int e2;
                frexp((double)amax, &e2);           /* amax = m * 2^e2, m in [0.5, 1) */
                int e = (e2 - 1) - 2;               /* floor(log2(amax)) - 2 */
                s = e + 127;
                if (s < 0) s = 0;
                if (s > 254) s = 254;
            }
            const float X = ldexpf(1.0f, s - 127);
            uint8_t q[32];
            for (int i = 0; i < 32; ++i) q[i] = oracle_e2m1_from_f32(blk[i] / X);
            scales[r * nb + b] = (uint8_t)s;
            uint8_t *dst = codes + r * (cols / 2) + b * 16;
            for (int i = 0; i < 16; ++i) dst[i] = (uint8_t)(q[2 * i] | (q[2 * i + 1] << 4));
        }
    }
}

/* ------------------------------------------------------------------ router */

/* Router logits l[t][e] = x[t] . Wr[e] (+ bias[e]) in fp32, in a fixed order
 * that a warp can reproduce exactly:
 *   - the H positions are dealt to 32 lanes one at a time: position h
 *     belongs to lane h mod 32;
 *   - each lane sums fmaf(x[h], w[h], acc) over its positions in increasing h,
 *     starting from +0;
 *   - the 32 partial sums are combined by a butterfly: for offset 16, 8, 4,
 *     2, 1 every lane adds the partial of lane (lane xor offset);
 *   - the bias, when given, is added last in fp32.
 * x is bf16 (uint16 bit patterns) [T][H], Wr is fp32 [E][H]. */
void oracle_router_logits(const uint16_t *x, int32_t T, int32_t H, const float *Wr, int32_t E,
                          const float *bias, float *logits)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t t = 0; t < T; ++t) {
        float *xf = (float *)malloc(sizeof(float) * (size_t)H);
        for (int32_t h = 0; h < H; ++h) xf[h] = oracle_bf16_to_f32(x[(int64_t)t * H + h]);
        for (int32_t e = 0; e < E; ++e) {
            const float *w = Wr + (int64_t)e * H;
            float part[32], next[32];
            for (int l = 0; l < 32; ++l) part[l] = 0.0f;
            for (int32_t h = 0; h < H; ++h) {
                int l = h & 31;
                part[l] = fmaf(xf[h], w[h], part[l]);
            }
            for (int off = 16; off >= 1; off >>= 1) {
                for (int l = 0; l < 32; ++l) next[l] = part[l] + part[l ^ off];
                memcpy(part, next, sizeof(part));
            }
            float v = part[0];
            if (bias) v = v + bias[e];
            logits[(int64_t)t * E + e] = v;
        }
        free(xf);
    }
}

/* Top-k by logit, larger first, equal logits broken toward the lower expert
 * id; then the routing weights in FP64:
 *   softmax (kind 0): p = exp(l - max_l); w_j = p_j / sum over the selected
 *                     (renormalise) or over all E (no renormalise);
 *   sigmoid (kind 1): s = 1 / (1 + exp(-l)); w_j = s_j / sum over the
 *                     selected (renormalise) or s_j.
 * Selecting by logit selects by score: both maps are increasing. */
void oracle_topk(const float *logits, int32_t T, int32_t E, int32_t k, int32_t kind,
                 int32_t renormalize, int32_t *ids, double *weights)
{
    char *taken = (char *)malloc((size_t)E);
    for (int32_t t = 0; t < T; ++t) {
        const float *l = logits + (int64_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;   /* strict: ties keep the lower id */
            }
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
        }
        double sel[64];
        double denom = 0.0;
        if (kind == 0) {
            double m = -INFINITY;
            for (int32_t e = 0; e < E; ++e) if ((double)l[e] > m) m = l[e];
            for (int32_t j = 0; j < k; ++j) {
                sel[j] = exp((double)l[ids[(int64_t)t * k + j]] - m);
                denom += sel[j];
            }
            if (!renormalize) {
                denom = 0.0;
                for (int32_t e = 0; e < E; ++e) denom += exp((double)l[e] - m);
            }
        } else {
            for (int32_t j = 0; j < k; ++j) {
                sel[j] = 1.0 / (1.0 + exp(-(double)l[ids[(int64_t)t * k + j]]));
                denom += sel[j];
            }
            if (!renormalize) denom = 1.0;
        }
        for (int32_t j = 0; j < k; ++j) weights[(int64_t)t * k + j] = sel[j] / denom;
    }
    free(taken);
}

/* Group (token, slot) pairs by expert with a stable counting sort.
 * Pair p = t*k + j has expert ids[p].  offsets[e] = number of pairs with an
 * expert below e (offsets[E] = P); sorted_rows lists the pair indices expert
 * by expert, each expert's pairs in increasing p. */
void oracle_group(const int32_t *ids, int64_t P, int32_t E, int32_t *offsets, int32_t *sorted_rows)
{
    int64_t *count = (int64_t *)calloc((size_t)E + 1, sizeof(int64_t));
    for (int64_t p = 0; p < P; ++p) count[ids[p]] += 1;
    int64_t run = 0;
    for (int32_t e = 0; e < E; ++e) {
        offsets[e] = (int32_t)run;
        run += count[e];
    }
    offsets[E] = (int32_t)run;
    int64_t *fill = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    for (int64_t p = 0; p < P; ++p) {
        int32_t e = ids[p];
        sorted_rows[offsets[e] + fill[e]] = (int32_t)p;
        fill[e] += 1;
    }
    free(fill);
    free(count);
}
