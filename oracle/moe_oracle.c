/*
 * moe_oracle.c -- CPU oracle for the routed MoE expert FFN with the live-row
 * (aligned prefix-sum endpoint) layout, and for the sparse decode GEMV path.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the test suite, the smoke check and the
 * benchmark's CPU-baseline leg, never by the CUDA library. It shares no code,
 * header, table or constant generator with the GPU path.
 *
 * Sources, cited below by the tag in brackets and the page's own section:
 *  [LR] "Blackwell FP4 MoE：把 live-row 边界贯穿整个 FFN" (lab.ttaoai.cn)
 *  [DG] "Blackwell 上的 DeepGEMM FusedMoE（sglang）" (dingfen.github.io)
 *  [SD] "Phase 20: Sparse MoE Decode — 只算被路由到的专家" (xserv docs)
 *  [KM] "kimi3_pro6000_sglang_sm120_flashinfer_mxfp4" experiment log (sskj)
 *
 * Precision: GEMM-like sums are accumulated in fp64 and rounded once. The
 * quantisation steps follow the fp32 recipe the pages fix (amax/448 in fp32,
 * round the scale up to a power of two, scale and round to e4m3). The combine
 * accumulates in fp32 in slot order because the page's kernel does ([DG] §2.6.1).
 *
 * Build with -O2 -ffp-contract=off (no fast-math) so every float operation is
 * a single IEEE operation and fmaf() is the only fused one.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static long align_up_l(long x, long a) { return (x + a - 1) / a * a; }

/* ------------------------------------------------------------------ bf16 */

float orc_bf16_to_float(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* Round-to-nearest-even from fp32 to bf16 (keep the high 16 bits). */
uint16_t orc_bf16_from_float(float f) {
    uint32_t u = f32_bits(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Round-to-nearest-even from fp64 straight to bf16. Rounding to fp32 first is
 * exact here unless the fp32 value lands on a bf16 midpoint that the fp64
 * value is not on; then the tie is broken toward the fp64 value. */
uint16_t orc_bf16_from_double(double d) {
    if (isnan(d)) return 0x7FC0;
    float f = (float)d;
    uint32_t u = f32_bits(f);
    if ((u & 0xFFFFu) == 0x8000u && (double)f != d) {
        if (fabs(d) > fabs((double)f)) u += 0x8000u; else u -= 0x8000u;
        return (uint16_t)(u >> 16);
    }
    return orc_bf16_from_float(f);
}

/* ------------------------------------------------------------ fp8 / fp4 */

/* e4m3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; S.1111.111 is NaN;
 * largest finite 448 ([DG] §2.4.1: the 448 in ceil(amax/448)). */
double orc_e4m3_value(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return s ? -v : v;
}

/* fp32 -> e4m3 with round-to-nearest-even and saturation to the largest
 * finite value; NaN -> 0x7F. */
uint8_t orc_e4m3_from_float(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {                 /* subnormal: steps of 2^-9 */
        double q = nearbyint(a * 512.0);      /* q == 8 is the smallest normal */
        return sign | (uint8_t)q;
    }
    int e2;
    frexp(a, &e2);                            /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;
    double q = nearbyint(ldexp(a, 3 - E));    /* 8 + mantissa, in [8, 16] */
    if (q == 16.0) { q = 8.0; E += 1; }
    return sign | (uint8_t)(((E + 7) << 3) | ((int)q - 8));
}

/* e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit. */
double orc_e2m1_value(uint8_t nib) {
    int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

double orc_ue8m0_value(uint8_t b) { return b == 0xFF ? NAN : ldexp(1.0, (int)b - 127); }

/* Smallest power of two >= s, as its biased exponent byte. This is the bit
 * recipe of [DG] 附录 A (_cast_to_e8m0_with_rounding_up): take the fp32
 * exponent field, add one when the mantissa is non-zero, except at 0xFE and
 * for subnormals not above 2^-127. */
uint8_t orc_ue8m0_ceil(float s) {
    uint32_t bits = f32_bits(s);
    uint32_t e = (bits >> 23) & 0xFFu;
    uint32_t m = bits & 0x7FFFFFu;
    int ru = (m > 0 && e != 0xFE) && !(e == 0 && m <= 0x400000u);
    return (uint8_t)((e + (uint32_t)ru) & 0xFFu);
}

/* 2^k as fp32 for k in [-127, 127] (2^-127 is subnormal). */
static float pow2f(int k) {
    if (k >= -126) return bits_f32((uint32_t)(k + 127) << 23);
    return bits_f32(0x00400000u);
}

/* ------------------------------------------------------- exp specification
 * The pages give no exp; both sides of the parity check implement this one
 * definition independently (Cody & Waite argument reduction, Taylor series):
 *   n  = rint(x * fl(log2 e))
 *   r  = fma(-n, L_hi, x);  r = fma(-n, L_lo, r)
 *        L_hi = fl(ln 2) with its 12 low significand bits cleared, so n*L_hi
 *        is exact for |n| < 2^12;  L_lo = fl(ln 2 - L_hi)
 *   p  = Horner over 1 + r + r^2/2! + ... + r^7/7!, coefficients fl(1/k!),
 *        each step one fma
 *   result = (p * 2^(n/2)) * 2^(n - n/2)      (n/2 truncates toward zero)
 * with x >= 128 -> +inf, x <= -150 -> +0, NaN -> NaN. */
static float g_log2e, g_ln2_hi, g_ln2_lo, g_c[8];

__attribute__((constructor)) static void exp_spec_init(void) {
    g_log2e = (float)1.44269504088896340736;
    const double ln2 = 0.693147180559945309417232121458;
    g_ln2_hi = bits_f32(f32_bits((float)ln2) & ~0xFFFu);
    g_ln2_lo = (float)(ln2 - (double)g_ln2_hi);
    double fact = 1.0;
    for (int k = 0; k < 8; k++) {
        if (k > 0) fact *= k;
        g_c[k] = (float)(1.0 / fact);
    }
}

float orc_exp_spec(float x) {
    if (isnan(x)) return x;
    if (x >= 128.0f) return INFINITY;
    if (x <= -150.0f) return 0.0f;
    float t = x * g_log2e;
    int n = (int)rintf(t);
    float fn = (float)n;
    float r = fmaf(-fn, g_ln2_hi, x);
    r = fmaf(-fn, g_ln2_lo, r);
    float p = g_c[7];
    for (int k = 6; k >= 0; k--) p = fmaf(p, r, g_c[k]);
    int n1 = n / 2, n2 = n - n1;
    float y = p * pow2f(n1);
    return y * pow2f(n2);
}

/* silu(g) = g / (1 + exp(-g)): one add, one IEEE division. */
float orc_silu_spec(float g) {
    float e = orc_exp_spec(-g);
    float d = 1.0f + e;
    return g / d;
}

float orc_sigmoid_spec(float x) {
    float e = orc_exp_spec(-x);
    float d = 1.0f + e;
    return 1.0f / d;
}

/* ------------------------------------------------------- tanh specification
 * The pages use tanh in SiTU without defining it; both sides implement this
 * one definition independently:
 *   |y| < 2^-12          y  (tanh y = y (1 - y^2/3 + ...), the correction is
 *                        below half an fp32 ulp)
 *   |y| < 1/4            y + (y y^2) P(y^2), P the Taylor series of
 *                        (tanh y - y) / y^3 to the y^8 term: coefficients
 *                        fl(-1/3), fl(2/15), fl(-17/315), fl(62/2835),
 *                        fl(-1382/155925), Horner with one fma per step,
 *                        the last step fma(y y^2, P, y)
 *   |y| >= 9             sign(y)
 *   otherwise            sign(y) (1 - e) / (1 + e), e = exp_spec(-2|y|)
 *   NaN                  NaN */
static float g_tanh_c[5];

__attribute__((constructor)) static void tanh_spec_init(void) {
    g_tanh_c[0] = (float)(-1.0 / 3.0);
    g_tanh_c[1] = (float)(2.0 / 15.0);
    g_tanh_c[2] = (float)(-17.0 / 315.0);
    g_tanh_c[3] = (float)(62.0 / 2835.0);
    g_tanh_c[4] = (float)(-1382.0 / 155925.0);
}

float orc_tanh_spec(float y) {
    if (isnan(y)) return y;
    float a = fabsf(y);
    if (a < 0x1p-12f) return y;
    if (a < 0.25f) {
        float z = y * y;
        float p = g_tanh_c[4];
        for (int i = 3; i >= 0; i--) p = fmaf(p, z, g_tanh_c[i]);
        return fmaf(y * z, p, y);
    }
    if (a >= 9.0f) return copysignf(1.0f, y);
    float e = orc_exp_spec(-2.0f * a);
    float t = (1.0f - e) / (1.0f + e);
    return copysignf(t, y);
}

/* SiTU ([KM] reference formula and the [DG] §2.4.1 situ branch; the LaTeX
 * there prints tan, the code tanh -- tanh is taken):
 *   gate' = (beta_s * tanh(g / beta_s)) * sigmoid(g)
 *   up'   = beta_l * tanh(u / beta_l)
 * each operation one IEEE fp32 operation, in this order. */
float orc_situ_gate_spec(float g, float beta_s) {
    float t = orc_tanh_spec(g / beta_s);
    return (beta_s * t) * orc_sigmoid_spec(g);
}

float orc_situ_up_spec(float u, float beta_l) { return beta_l * orc_tanh_spec(u / beta_l); }

/* ------------------------------------------------ group quantisation
 * Per 128-column group ([DG] §2.4.1, DeepGEMM convention, and §2.2.4
 * "per-token-group quant"): amax = max |v| (NaN ignored, like IEEE maxNum);
 * s = amax / 448 in fp32; b = ceil-to-power-of-two exponent of s; codes =
 * e4m3(v * 2^(127-b)). A non-finite amax stores b = 0xFE: UE8M0 0xFF is NaN
 * and the scale must stay finite ([KM] "NaN/Inf 决策记录"). */
void orc_group_quant_row(const float* v, int K, int group, uint8_t* codes, uint8_t* scales) {
    int G = (K + group - 1) / group;
    for (int g = 0; g < G; g++) {
        int lo = g * group, hi = lo + group < K ? lo + group : K;
        float amax = 0.0f;
        for (int i = lo; i < hi; i++) {
            float a = fabsf(v[i]);
            if (a > amax) amax = a;
        }
        uint8_t b = isinf(amax) ? (uint8_t)0xFE : orc_ue8m0_ceil(amax / 448.0f);
        float scale = pow2f(127 - (int)b);
        for (int i = lo; i < hi; i++) codes[i] = orc_e4m3_from_float(v[i] * scale);
        scales[g] = b;
    }
}

static void pack_scales(const uint8_t* sf, int G, int32_t* dst_words, long ld, long row) {
    int G4 = (G + 3) / 4;
    for (int w = 0; w < G4; w++) {
        uint32_t word = 0;
        for (int i = 0; i < 4; i++) {
            int g = 4 * w + i;
            if (g < G) word |= (uint32_t)sf[g] << (8 * i);
        }
        dst_words[(long)w * ld + row] = (int32_t)word;
    }
}

static uint8_t unpack_scale(const int32_t* words, long ld, long row, int g) {
    uint32_t w = (uint32_t)words[(long)(g / 4) * ld + row];
    return (uint8_t)((w >> (8 * (g % 4))) & 0xFFu);
}

/* ----------------------------------------------------------------- routing
 * Softmax top-k with renormalisation ([DG] §2.2.1 TopK; [SD] §1 topk_softmax):
 * softmax is monotone, so selection compares raw logits; ties go to the lower
 * expert index (+0 and -0 tie); NaN ranks last; slots are in selection order. Weights are
 * exp(l_j - l_max) / sum over the selected slots (slot order, fp32), which is
 * softmax followed by top-k and renormalisation. */
/* a ranks strictly above b. The pages do not say how a NaN score ranks; here
 * it ranks below every number (and NaNs tie), so a NaN router output can only
 * fill slots that no number is left for. */
static int ranks_above(float a, float b) {
    if (a != a) return 0;
    if (b != b) return 1;
    return a > b;
}

static void select_topk(const float* score, int E, int k, unsigned char* taken, int32_t* ids) {
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; j++) {
        int best = -1;
        for (int e = 0; e < E; e++)
            if (!taken[e] && (best < 0 || ranks_above(score[e], score[best]))) best = e;
        taken[best] = 1;
        ids[j] = best;
    }
}

void orc_route_softmax_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w) {
#pragma omp parallel
    {
        unsigned char* taken = (unsigned char*)malloc((size_t)E);
        float* ex = (float*)malloc(sizeof(float) * (size_t)k);
#pragma omp for
        for (int t = 0; t < T; t++) {
            const float* l = logits + (long)t * E;
            int32_t* id = ids + (long)t * k;
            select_topk(l, E, k, taken, id);
            float m = l[id[0]];
            float s = 0.0f;
            for (int j = 0; j < k; j++) { ex[j] = orc_exp_spec(l[id[j]] - m); s = s + ex[j]; }
            for (int j = 0; j < k; j++) w[(long)t * k + j] = ex[j] / s;
        }
        free(taken); free(ex);
    }
}

/* Sigmoid scores plus a correction bias select the experts; the weights are
 * the unbiased sigmoid scores of the selected experts, renormalised
 * ([KM] Phase 1 table, topk.py row). */
void orc_route_sigmoid_bias_topk(const float* logits, const float* bias, int T, int E, int k,
                                 int32_t* ids, float* w) {
#pragma omp parallel
    {
        unsigned char* taken = (unsigned char*)malloc((size_t)E);
        float* sig = (float*)malloc(sizeof(float) * (size_t)E);
        float* score = (float*)malloc(sizeof(float) * (size_t)E);
#pragma omp for
        for (int t = 0; t < T; t++) {
            const float* l = logits + (long)t * E;
            int32_t* id = ids + (long)t * k;
            for (int e = 0; e < E; e++) { sig[e] = orc_sigmoid_spec(l[e]); score[e] = sig[e] + bias[e]; }
            select_topk(score, E, k, taken, id);
            float s = 0.0f;
            for (int j = 0; j < k; j++) s = s + sig[id[j]];
            for (int j = 0; j < k; j++) w[(long)t * k + j] = sig[id[j]] / s;
        }
        free(taken); free(sig); free(score);
    }
}

/* ---------------------------------------------------- endpoints / scatter */

void orc_expert_counts(const int32_t* ids, long R, int E, int32_t* counts) {
    for (int e = 0; e < E; e++) counts[e] = 0;
    for (long i = 0; i < R; i++)
        if (ids[i] >= 0 && ids[i] < E) counts[ids[i]]++;
}

/* [LR] §2: start[0] = 0, start[e] = align_up(end[e-1], A), end[e] = start[e] + count[e]. */
void orc_endpoints(const int32_t* counts, int E, int A, int32_t* start, int32_t* end) {
    for (int e = 0; e < E; e++) {
        long s = (e == 0) ? 0 : align_up_l(end[e - 1], A);
        start[e] = (int32_t)s;
        end[e] = (int32_t)(s + counts[e]);
    }
}

static void starts_from_ends(const int32_t* ends, int E, int A, int32_t* start) {
    for (int e = 0; e < E; e++) start[e] = (e == 0) ? 0 : (int32_t)align_up_l(ends[e - 1], A);
}

/* Token scatter ([LR] §2 "scatter → endpoint[E]"; [DG] 附录 C ep_scatter):
 * routes are walked in row-major (token, slot) order, so rows inside an
 * expert segment keep token order; route (t, j) of expert e lands on row
 * start[e] + (number of earlier routes to e). Ids outside [0, E) are skipped
 * (src2dst = -1). Each token row is quantised once and copied to its rows.
 * Only live rows of a_fp8 / a_sf are written. Returns -1 if end[E-1] > cap. */
int orc_scatter(const int32_t* ids, const uint16_t* x, int T, int k, int E, int H, int A, int cap,
                int ld_sf, int group, int32_t* expert_ends, int32_t* src2dst, uint8_t* a_fp8, int32_t* a_sf) {
    long R = (long)T * k;
    int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    int32_t* start = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    orc_expert_counts(ids, R, E, counts);
    orc_endpoints(counts, E, A, start, expert_ends);
    if (E > 0 && expert_ends[E - 1] > cap) { free(counts); free(start); free(fill); return -1; }
    for (long i = 0; i < R; i++) {
        int e = ids[i];
        if (e < 0 || e >= E) { src2dst[i] = -1; continue; }
        src2dst[i] = start[e] + fill[e]++;
    }
    int G = H / group;
#pragma omp parallel
    {
        float* v = (float*)malloc(sizeof(float) * (size_t)H);
        uint8_t* q = (uint8_t*)malloc((size_t)H);
        uint8_t* sf = (uint8_t*)malloc((size_t)G + 1);
#pragma omp for
        for (int t = 0; t < T; t++) {
            for (int h = 0; h < H; h++) v[h] = orc_bf16_to_float(x[(long)t * H + h]);
            orc_group_quant_row(v, H, group, q, sf);
            for (int j = 0; j < k; j++) {
                long dst = src2dst[(long)t * k + j];
                if (dst < 0) continue;
                memcpy(a_fp8 + dst * H, q, (size_t)H);
                pack_scales(sf, G, a_sf, ld_sf, dst);
            }
        }
        free(v); free(q); free(sf);
    }
    free(counts); free(start); free(fill);
    return 0;
}

/* ------------------------------------------------------------ grouped GEMM
 * out[r, n] = bf16( sum_k e4m3(a[r,k]) 2^(sa(r, k/128)-127)
 *                          * e2m1(w[e,n,k]) 2^(sw(e,n,k/32)-127) )
 * for every live row r of expert e ([LR] §2: FC1/FC2 use the same endpoint
 * layout; [DG] §2.1.3 recipes (1,128) for activations, (1,32) for MXFP4
 * weights). Weights: w[e][n][k/2] packed, low nibble = even k; scales
 * w_sf[e][n][k/32]. Rows outside [start[e], end[e]) are not written. */
static double dq_w(const uint8_t* w, const uint8_t* w_sf, int wfmt, int N, int K, int e, int n, int kk) {
    const double s = orc_ue8m0_value(w_sf[((long)e * N + n) * (K / 32) + kk / 32]);
    if (wfmt == 1) return orc_e4m3_value(w[((long)e * N + n) * K + kk]) * s;
    uint8_t byte = w[((long)e * N + n) * (K / 2) + kk / 2];
    uint8_t nib = (kk & 1) ? (byte >> 4) : (byte & 0xF);
    return orc_e2m1_value(nib) * s;
}

static void gemm_row(const double* a_deq, int K, int e, const uint8_t* w, const uint8_t* w_sf, int wfmt, int N,
                     uint16_t* out_row) {
    for (int n = 0; n < N; n++) {
        double acc = 0.0;
        for (int kk = 0; kk < K; kk++) acc += a_deq[kk] * dq_w(w, w_sf, wfmt, N, K, e, n, kk);
        out_row[n] = orc_bf16_from_double(acc);
    }
}

/* FP8-block128 weight scales ([DG] §6 "FP8 block128": one UE8M0 scale per
 * 128 x 128 weight block, sf_blk[e][n/128][k/128]) as per-(row, 32-K) bytes:
 * sf32[e][n][j] = sf_blk[e][n/128][j/4]. */
void orc_expand_block_scales(const uint8_t* sf_blk, int E, int N, int K, uint8_t* sf32) {
    for (int e = 0; e < E; e++)
        for (int n = 0; n < N; n++)
            for (int j = 0; j < K / 32; j++)
                sf32[((long)e * N + n) * (K / 32) + j] =
                    sf_blk[((long)e * ((N + 127) / 128) + n / 128) * (K / 128) + j / 4];
}

void orc_grouped_gemm(const uint8_t* a, const int32_t* a_sf, int ld_sf, int K, int a_group,
                      const int32_t* expert_ends, int E, int A,
                      const uint8_t* w, const uint8_t* w_sf, int wfmt, int N, uint16_t* out) {
    int32_t* start = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    starts_from_ends(expert_ends, E, A, start);
    for (int e = 0; e < E; e++) {
        int r0 = start[e], r1 = expert_ends[e];
#pragma omp parallel
        {
            double* ad = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for
            for (int r = r0; r < r1; r++) {
                for (int kk = 0; kk < K; kk++)
                    ad[kk] = orc_e4m3_value(a[(long)r * K + kk]) *
                             orc_ue8m0_value(unpack_scale(a_sf, ld_sf, r, kk / a_group));
                gemm_row(ad, K, e, w, w_sf, wfmt, N, out + (long)r * N);
            }
            free(ad);
        }
    }
    free(start);
}

/* ---------------------------------------------------------- act + quant
 * For each live row ([LR] §2-3: rows [start[e], end[e]) only; with no
 * endpoints every row, the dense launch): gate = gateup[r, j],
 * up = gateup[r, I + j] ([DG] §2.4.1, [gate; up] halves); with a clamp limit
 * L the gate is clamped from above and up on both sides ([DG] §2.4.1 default
 * branch: "up 双向钳、gate 只钳上限"); h = silu(gate) * up kept in fp32
 * (silu_mul_keep_fp32), or with SiTU h = gate'(gate) * up'(up) (the situ
 * branch of [DG] §2.4.1); then group-128 quantisation with
 * packed UE8M0 scales. */
/* min(a, b) and max(a, b) in which a NaN operand, quiet or signalling, yields
 * the other operand (IEEE minNum / maxNum): the reading taken for the pages'
 * min(gate, L) and clamp(up, -L, L). Written out because the C library's
 * min/max treat a signalling NaN differently from one platform to the next. */
static float min_num(float a, float b) {
    if (a != a) return b;
    if (b != b) return a;
    return b < a ? b : a;
}

static float max_num(float a, float b) {
    if (a != a) return b;
    if (b != b) return a;
    return b > a ? b : a;
}

/* h for one (gate, up) pair: kind 0 SiLU, 1 SiLU with the clamp, 2 SiTU. */
static float act_value(float g, float u, const orc_act* act) {
    if (act->kind == 2) return orc_situ_gate_spec(g, act->beta_s) * orc_situ_up_spec(u, act->beta_l);
    if (act->kind == 1) { g = min_num(g, act->limit); u = min_num(max_num(u, -act->limit), act->limit); }
    return orc_silu_spec(g) * u;
}

static void act_quant_row(const uint16_t* row, int I, const orc_act* act, float* h, uint8_t* q, uint8_t* sf) {
    for (int j = 0; j < I; j++)
        h[j] = act_value(orc_bf16_to_float(row[j]), orc_bf16_to_float(row[I + j]), act);
    orc_group_quant_row(h, I, act->group, q, sf);
}

void orc_act_quant(const uint16_t* gateup, int M_alloc, int I, const int32_t* expert_ends, int E,
                   int A, int act_kind, float limit, float beta_s, float beta_l, int group, uint8_t* out,
                   int32_t* out_sf, int ld_sf) {
    const orc_act act = {act_kind, limit, beta_s, beta_l, group};
    int G = (I + group - 1) / group;
    int nseg = expert_ends ? E : 1;
    int32_t* start = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    if (expert_ends) starts_from_ends(expert_ends, E, A, start);
    for (int s = 0; s < nseg; s++) {
        int r0 = expert_ends ? start[s] : 0;
        int r1 = expert_ends ? expert_ends[s] : M_alloc;
#pragma omp parallel
        {
            float* h = (float*)malloc(sizeof(float) * (size_t)I);
            uint8_t* sf = (uint8_t*)malloc((size_t)G + 1);
#pragma omp for
            for (int r = r0; r < r1; r++) {
                act_quant_row(gateup + (long)r * 2 * I, I, &act, h, out + (long)r * I, sf);
                pack_scales(sf, G, out_sf, ld_sf, r);
            }
            free(h); free(sf);
        }
    }
    free(start);
}

/* --------------------------------------------------------------- combine
 * [DG] §2.6.1 post_reorder: out[t] = rsf * sum over slots j in order with
 * src2dst[t, j] >= 0 of w[t, j] * down[src2dst[t, j]], accumulated in fp32
 * (one fused multiply-add per slot), then rounded to bf16. */
void orc_combine(const uint16_t* down, int H, const float* topk_w, const int32_t* src2dst, int T,
                 int k, float rsf, uint16_t* out) {
#pragma omp parallel for
    for (int t = 0; t < T; t++) {
        for (int h = 0; h < H; h++) {
            float acc = 0.0f;
            for (int j = 0; j < k; j++) {
                long dst = src2dst[(long)t * k + j];
                if (dst < 0) continue;
                acc = fmaf(topk_w[(long)t * k + j], orc_bf16_to_float(down[dst * H + h]), acc);
            }
            acc = acc * rsf;
            out[(long)t * H + h] = orc_bf16_from_float(acc);
        }
    }
}

/* ------------------------------------------------- whole layer per token
 * The same arithmetic as scatter -> GEMM1 -> act-quant -> GEMM2 -> combine,
 * restricted to one token's selected experts (every row of the grouped
 * layout depends only on its own token). Used to check samples of large
 * configurations, and pinned against the layout path on small ones. */
static void expert_chain(const double* a_deq, int H, int I, int e, const uint8_t* w13,
                         const uint8_t* w13_sf, const uint8_t* w2, const uint8_t* w2_sf, int wfmt,
                         const orc_act* act, uint16_t* gu, float* h, uint8_t* q, uint8_t* sf, double* act_deq,
                         uint16_t* down_row) {
    gemm_row(a_deq, H, e, w13, w13_sf, wfmt, 2 * I, gu);
    act_quant_row(gu, I, act, h, q, sf);
    for (int i = 0; i < I; i++) act_deq[i] = orc_e4m3_value(q[i]) * orc_ue8m0_value(sf[i / act->group]);
    gemm_row(act_deq, I, e, w2, w2_sf, wfmt, H, down_row);
}

static void token_input(const uint16_t* xrow, int H, int group, float* v, uint8_t* q, uint8_t* sf,
                        double* a_deq) {
    for (int i = 0; i < H; i++) v[i] = orc_bf16_to_float(xrow[i]);
    orc_group_quant_row(v, H, group, q, sf);
    for (int i = 0; i < H; i++) a_deq[i] = orc_e4m3_value(q[i]) * orc_ue8m0_value(sf[i / group]);
}

void orc_ffn_tokens(const uint16_t* x, int H, int I, const int32_t* ids, const float* topk_w, int k,
                    int E, const uint8_t* w13, const uint8_t* w13_sf, const uint8_t* w2,
                    const uint8_t* w2_sf, int wfmt, int group, int act_kind, float limit, float beta_s,
                    float beta_l, float rsf, const int32_t* tokens, int n_tokens, uint16_t* out) {
    const orc_act act = {act_kind, limit, beta_s, beta_l, group};
    int maxd = H > 2 * I ? H : 2 * I;
#pragma omp parallel
    {
        float* v = (float*)malloc(sizeof(float) * (size_t)maxd);
        uint8_t* q = (uint8_t*)malloc((size_t)maxd);
        uint8_t* sf = (uint8_t*)malloc((size_t)maxd / 32 + 2);
        double* a_deq = (double*)malloc(sizeof(double) * (size_t)H);
        double* act_deq = (double*)malloc(sizeof(double) * (size_t)I);
        uint16_t* gu = (uint16_t*)malloc(sizeof(uint16_t) * 2 * (size_t)I);
        uint16_t* down = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)k * H);
        int* valid = (int*)malloc(sizeof(int) * (size_t)k);
#pragma omp for schedule(dynamic, 1)
        for (int s = 0; s < n_tokens; s++) {
            int t = tokens[s];
            token_input(x + (long)t * H, H, group, v, q, sf, a_deq);
            for (int j = 0; j < k; j++) {
                int e = ids[(long)t * k + j];
                valid[j] = (e >= 0 && e < E);
                if (!valid[j]) continue;
                expert_chain(a_deq, H, I, e, w13, w13_sf, w2, w2_sf, wfmt, &act, gu, v, q, sf,
                             act_deq, down + (long)j * H);
            }
            for (int hh = 0; hh < H; hh++) {
                float acc = 0.0f;
                for (int j = 0; j < k; j++)
                    if (valid[j])
                        acc = fmaf(topk_w[(long)t * k + j], orc_bf16_to_float(down[(long)j * H + hh]), acc);
                acc = acc * rsf;
                out[(long)s * H + hh] = orc_bf16_from_float(acc);
            }
        }
        free(v); free(q); free(sf); free(a_deq); free(act_deq); free(gu); free(down); free(valid);
    }
}

/* Dense twin ([SD] §3: the dense path computes every expert for every token
 * and the weighted sum picks the routed ones; the sparse path must be
 * equivalent bit for bit). */
void orc_ffn_dense(const uint16_t* x, int T, int H, int I, const int32_t* ids, const float* topk_w,
                   int k, int E, const uint8_t* w13, const uint8_t* w13_sf, const uint8_t* w2,
                   const uint8_t* w2_sf, int wfmt, int group, int act_kind, float limit, float beta_s,
                   float beta_l, float rsf, uint16_t* out) {
    const orc_act act = {act_kind, limit, beta_s, beta_l, group};
    int maxd = H > 2 * I ? H : 2 * I;
    uint16_t* all_down = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)T * E * H);
#pragma omp parallel
    {
        float* v = (float*)malloc(sizeof(float) * (size_t)maxd);
        uint8_t* q = (uint8_t*)malloc((size_t)maxd);
        uint8_t* sf = (uint8_t*)malloc((size_t)maxd / 32 + 2);
        double* a_deq = (double*)malloc(sizeof(double) * (size_t)H);
        double* act_deq = (double*)malloc(sizeof(double) * (size_t)I);
        uint16_t* gu = (uint16_t*)malloc(sizeof(uint16_t) * 2 * (size_t)I);
#pragma omp for
        for (int t = 0; t < T; t++) {
            token_input(x + (long)t * H, H, group, v, q, sf, a_deq);
            for (int e = 0; e < E; e++)
                expert_chain(a_deq, H, I, e, w13, w13_sf, w2, w2_sf, wfmt, &act, gu, v, q, sf,
                             act_deq, all_down + ((long)t * E + e) * H);
        }
        free(v); free(q); free(sf); free(a_deq); free(act_deq); free(gu);
    }
    for (int t = 0; t < T; t++)
        for (int hh = 0; hh < H; hh++) {
            float acc = 0.0f;
            for (int j = 0; j < k; j++) {
                int e = ids[(long)t * k + j];
                if (e < 0 || e >= E) continue;
                acc = fmaf(topk_w[(long)t * k + j],
                           orc_bf16_to_float(all_down[((long)t * E + e) * H + hh]), acc);
            }
            acc = acc * rsf;
            out[(long)t * H + hh] = orc_bf16_from_float(acc);
        }
    free(all_down);
}

/* ---------------------------------------------------------------- decode
 * [SD] §3: per (token, slot) whose expert is local, y1 = W_gu[e] x (+bias),
 * GLU, y2 = W_d[e] act (+bias); out[t] = sum over local slots of w * y2.
 * Non-local slots are skipped, never multiplied by zero. Epilogue
 * y = acc * scale + bias ([SD] §3 "epilogue"). wfmt 0: e4m3 weights [E,N,K]
 * with one fp32 scale per expert; wfmt 1: MXFP4 [E,N,K/2] with UE8M0
 * group-32 scales [E,N,K/32]. Intermediates y1, act, y2 are bf16.
 *
 * GLU (parameters alpha=1.702, beta=1, limit=7 and the interleaved layout,
 * [KM] Phase 1 差异矩阵). [DG] §2.4.1 clamps up on both sides and the gate
 * from above only; [DG] §2.1.3 makes alpha the scale of the SiLU part. Where
 * beta enters is a reading (parity unpinned for that part):
 *   g = min(g, L); u = clamp(u, -L, L); act = (g * sigmoid(alpha g)) * (u + beta). */
float orc_glu_oai(float g, float u, float alpha, float beta, float limit) {
    if (limit > 0.0f) { g = min_num(g, limit); u = min_num(max_num(u, -limit), limit); }
    float s = orc_sigmoid_spec(alpha * g);
    return (g * s) * (u + beta);
}

static double dec_w(int wfmt, const uint8_t* w, const float* scale, const uint8_t* sf, int N, int K,
                    int lid, int n, int kk) {
    if (wfmt == 0) return orc_e4m3_value(w[((long)lid * N + n) * K + kk]);
    uint8_t byte = w[((long)lid * N + n) * (K / 2) + kk / 2];
    uint8_t nib = (kk & 1) ? (byte >> 4) : (byte & 0xF);
    (void)scale;
    return orc_e2m1_value(nib) * orc_ue8m0_value(sf[((long)lid * N + n) * (K / 32) + kk / 32]);
}

static void dec_gemv(int wfmt, const float* xin, int K, int N, int lid, const uint8_t* w,
                     const float* scale, const uint8_t* sf, const uint16_t* bias, uint16_t* y) {
    for (int n = 0; n < N; n++) {
        double acc = 0.0;
        for (int kk = 0; kk < K; kk++) acc += (double)xin[kk] * dec_w(wfmt, w, scale, sf, N, K, lid, n, kk);
        double s = (wfmt == 0) ? (double)scale[lid] : 1.0;
        y[n] = orc_bf16_from_double(acc * s + (double)orc_bf16_to_float(bias[(long)lid * N + n]));
    }
}

static void dec_glu(const uint16_t* y1, int I, int interleaved, float alpha, float beta, float limit,
                    uint16_t* act) {
    for (int i = 0; i < I; i++) {
        float g = orc_bf16_to_float(interleaved ? y1[2 * i] : y1[i]);
        float u = orc_bf16_to_float(interleaved ? y1[2 * i + 1] : y1[I + i]);
        act[i] = orc_bf16_from_float(orc_glu_oai(g, u, alpha, beta, limit));
    }
}

/* The four steps of the decode path, each over every (token, slot) whose
 * expert is local ([SD] §3 kernel flow). Each step takes the previous step's
 * bf16 output as its input, so a checker can run any step on another
 * implementation's intermediate. Slots of non-local experts are not written. */
static int dec_local(const int32_t* ids, long slot, int expert_start, int n_local) {
    int lid = ids[slot] - expert_start;
    return (lid < 0 || lid >= n_local) ? -1 : lid;
}

/* Step 1: y1[t, j] = bf16(W_gu[e] x[t] * scale + b_gu[e]). */
void orc_decode_gemv1(const uint16_t* x, int T, int H, int I, const int32_t* ids, int k, int expert_start,
                      int n_local, int wfmt, const uint8_t* w_gu, const float* gu_scale, const uint8_t* gu_sf,
                      const uint16_t* b_gu, uint16_t* y1) {
#pragma omp parallel
    {
        float* xin = (float*)malloc(sizeof(float) * (size_t)H);
#pragma omp for collapse(2)
        for (int t = 0; t < T; t++)
            for (int j = 0; j < k; j++) {
                long slot = (long)t * k + j;
                int lid = dec_local(ids, slot, expert_start, n_local);
                if (lid < 0) continue;
                for (int h = 0; h < H; h++) xin[h] = orc_bf16_to_float(x[(long)t * H + h]);
                dec_gemv(wfmt, xin, H, 2 * I, lid, w_gu, gu_scale, gu_sf, b_gu, y1 + slot * 2 * I);
            }
        free(xin);
    }
}

/* Step 2: act[t*k + j] = GLU(y1[t, j]). */
void orc_decode_glu(const uint16_t* y1, int T, int I, const int32_t* ids, int k, int expert_start, int n_local,
                    int glu_interleaved, float alpha, float beta, float limit, uint16_t* act) {
    for (long slot = 0; slot < (long)T * k; slot++) {
        if (dec_local(ids, slot, expert_start, n_local) < 0) continue;
        dec_glu(y1 + slot * 2 * I, I, glu_interleaved, alpha, beta, limit, act + slot * I);
    }
}

/* Step 3: y2[t, j] = bf16(W_d[e] act[t*k + j] * scale + b_d[e]). */
void orc_decode_gemv2(const uint16_t* act, int T, int H, int I, const int32_t* ids, int k, int expert_start,
                      int n_local, int wfmt, const uint8_t* w_d, const float* d_scale, const uint8_t* d_sf,
                      const uint16_t* b_d, uint16_t* y2) {
#pragma omp parallel
    {
        float* xin = (float*)malloc(sizeof(float) * (size_t)I);
#pragma omp for collapse(2)
        for (int t = 0; t < T; t++)
            for (int j = 0; j < k; j++) {
                long slot = (long)t * k + j;
                int lid = dec_local(ids, slot, expert_start, n_local);
                if (lid < 0) continue;
                for (int i = 0; i < I; i++) xin[i] = orc_bf16_to_float(act[slot * I + i]);
                dec_gemv(wfmt, xin, I, H, lid, w_d, d_scale, d_sf, b_d, y2 + slot * H);
            }
        free(xin);
    }
}

/* Step 4: out[t] = bf16(sum over local slots j, in slot order, of w[t, j] * y2[t, j]),
 * one fp32 fma per slot. */
void orc_decode_sum(const uint16_t* y2, int T, int H, const int32_t* ids, const float* topk_w, int k,
                    int expert_start, int n_local, uint16_t* out) {
    for (int t = 0; t < T; t++)
        for (int h = 0; h < H; h++) {
            float acc = 0.0f;
            for (int j = 0; j < k; j++) {
                long slot = (long)t * k + j;
                if (dec_local(ids, slot, expert_start, n_local) < 0) continue;
                acc = fmaf(topk_w[slot], orc_bf16_to_float(y2[slot * H + h]), acc);
            }
            out[(long)t * H + h] = orc_bf16_from_float(acc);
        }
}

void orc_decode(const uint16_t* x, int T, int H, int I, const int32_t* ids, const float* topk_w, int k,
                int expert_start, int n_local, int wfmt,
                const uint8_t* w_gu, const float* gu_scale, const uint8_t* gu_sf, const uint16_t* b_gu,
                const uint8_t* w_d, const float* d_scale, const uint8_t* d_sf, const uint16_t* b_d,
                int glu_interleaved, float alpha, float beta, float limit,
                uint16_t* y1, uint16_t* act, uint16_t* y2, uint16_t* out) {
    orc_decode_gemv1(x, T, H, I, ids, k, expert_start, n_local, wfmt, w_gu, gu_scale, gu_sf, b_gu, y1);
    orc_decode_glu(y1, T, I, ids, k, expert_start, n_local, glu_interleaved, alpha, beta, limit, act);
    orc_decode_gemv2(act, T, H, I, ids, k, expert_start, n_local, wfmt, w_d, d_scale, d_sf, b_d, y2);
    orc_decode_sum(y2, T, H, ids, topk_w, k, expert_start, n_local, out);
}

/* Dense twin of the decode path: every local expert on every token, then the
 * weighted sum over the routed local slots ([SD] §1 dense flow, steps 3-8). */
void orc_decode_dense(const uint16_t* x, int T, int H, int I, const int32_t* ids, const float* topk_w,
                      int k, int expert_start, int n_local, int wfmt,
                      const uint8_t* w_gu, const float* gu_scale, const uint8_t* gu_sf,
                      const uint16_t* b_gu, const uint8_t* w_d, const float* d_scale,
                      const uint8_t* d_sf, const uint16_t* b_d, int glu_interleaved, float alpha,
                      float beta, float limit, uint16_t* out) {
    uint16_t* all_y2 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)T * n_local * H);
#pragma omp parallel
    {
        float* xin = (float*)malloc(sizeof(float) * (size_t)(H > I ? H : I));
        uint16_t* y1 = (uint16_t*)malloc(sizeof(uint16_t) * 2 * (size_t)I);
        uint16_t* act = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
#pragma omp for collapse(2)
        for (int t = 0; t < T; t++)
            for (int lid = 0; lid < n_local; lid++) {
                for (int h = 0; h < H; h++) xin[h] = orc_bf16_to_float(x[(long)t * H + h]);
                dec_gemv(wfmt, xin, H, 2 * I, lid, w_gu, gu_scale, gu_sf, b_gu, y1);
                dec_glu(y1, I, glu_interleaved, alpha, beta, limit, act);
                for (int i = 0; i < I; i++) xin[i] = orc_bf16_to_float(act[i]);
                dec_gemv(wfmt, xin, I, H, lid, w_d, d_scale, d_sf, b_d,
                         all_y2 + ((long)t * n_local + lid) * H);
            }
        free(xin); free(y1); free(act);
    }
    for (int t = 0; t < T; t++)
        for (int h = 0; h < H; h++) {
            float acc = 0.0f;
            for (int j = 0; j < k; j++) {
                int lid = ids[(long)t * k + j] - expert_start;
                if (lid < 0 || lid >= n_local) continue;
                acc = fmaf(topk_w[(long)t * k + j],
                           orc_bf16_to_float(all_y2[((long)t * n_local + lid) * H + h]), acc);
            }
            out[(long)t * H + h] = orc_bf16_from_float(acc);
        }
    free(all_y2);
}
