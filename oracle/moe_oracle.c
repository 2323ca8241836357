/*
 * moe_oracle.c -- the ORACLE for the NVFP4 fused mixture-of-experts layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and its
 * Python binding) links, loads or calls this file; only the tests, the smoke check and
 * the CPU-baseline leg of the benchmark do.  It shares no code, header, table or
 * constant generator with the CUDA path.
 *
 * What it computes, in plain loops, with the pages it follows:
 *   - Layer shape: routed experts plus one always-on shared expert, top-k routing
 *     (Solar Open 2 on DGX Spark, "Solar Open 2 개요": 320 routed + 1 shared, top-8).
 *   - Expert parallelism: a contiguous shard [off, off+E_loc) of the experts; a global
 *     expert id e maps to e - off and pairs outside the shard are dropped; the result
 *     is the shard's partial sum (same page, "b12x에서의 Expert Parallelism 구현 추가").
 *   - NVFP4: packed FP4 codes, FP8 block scales clamped at 448, one FP32 global scale
 *     per tensor/expert (same page, "b12x 버전이 실제 NVFP4 체크포인트를 읽어들이도록
 *     만들기").  The element format is E2M1, the block is 16 elements, the block scale
 *     is E4M3 -- the NVFP4 format definition.
 *   - Expert MLP: fused gate/up projection (same section: "fused gate/up projection"),
 *     activation silu(gate) * up, down projection.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - routing: softmax over the selected top-k logits (= softmax over all experts then
 *     renormalised over the top-k); ties broken toward the lower expert id;
 *   - dropped (non-local) pairs are not renormalised, so shard partials add up to the
 *     full layer;
 *   - the shared expert has weight 1 and is added by the shard that sets add_shared;
 *   - dynamic activation scale: one FP32 scale for the whole [T,H] input,
 *     gs = 2688 / amax (2688 = 448 * 6);
 *   - the intermediate (post-SwiGLU) tensor is requantised with a static global scale,
 *     or, when the configured scale is <= 0, with the dynamic one 2688 / amax over every
 *     intermediate row the shard computes (two passes);
 *   - the permutation groups pairs by local expert and keeps ascending pair index
 *     p = t*k + j inside an expert.
 *
 * Precision: every quantisation decision is taken in fp32 with IEEE round-to-nearest
 * operations in the order written (build with -ffp-contract=off, no fast-math);
 * every contraction accumulates in fp64 over exactly dequantised values (an E2M1 code
 * times an E4M3 scale is exact in fp64, and so is the product of two such values).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* Element and scale formats                                                  */
/* ------------------------------------------------------------------------- */

/* E2M1 (4 bits): sign bit 3, exponent bits 2..1 with bias 1, mantissa bit 0.
 * Exponent field 0 is subnormal: m * 2^-1.  Otherwise (1 + m/2) * 2^(e-1).
 * No infinities, no NaN; largest magnitude 6. */
double orc_e2m1_value(int code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 (8 bits, the "fn" variant): sign bit 7, exponent bits 6..3 with bias 7,
 * mantissa bits 2..0.  Exponent field 0 is subnormal: (m/8) * 2^-6.  The pattern
 * exponent 15 / mantissa 7 is NaN; there are no infinities; largest magnitude 448. */
double orc_e4m3_value(int code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* The non-negative points of each format, by code, filled once at load from the value
 * functions above (a cache, so the encoders below need not recompute them). */
static double g_e2m1[8];
static double g_e4m3[127];

__attribute__((constructor)) static void grids_init(void)
{
    int c;
    for (c = 0; c < 8; c++) g_e2m1[c] = orc_e2m1_value(c);
    for (c = 0; c < 127; c++) g_e4m3[c] = orc_e4m3_value(c);
}

/* Round a >= 0 to the nearest point of the increasing grid g[0..n-1]; exact ties go
 * to the even code; anything at or above the top point saturates to it (satfinite). */
static int round_to_grid(double a, const double* g, int n)
{
    int c = 0;
    double mid;
    if (a >= g[n - 1]) return n - 1;
    while (c + 1 < n && g[c + 1] <= a) c++;
    if (a == g[c]) return c;
    mid = 0.5 * (g[c] + g[c + 1]);
    if (a < mid) return c;
    if (a > mid) return c + 1;
    return (c % 2 == 0) ? c : c + 1;
}

/* fp32 -> E2M1 code, round-to-nearest-even, saturating to +-6; the sign bit follows
 * the sign of x, so a negative value that rounds to zero gives -0 (code 8). */
int orc_e2m1_encode(float x)
{
    int mag = round_to_grid(fabs((double)x), g_e2m1, 8);
    return (signbit(x) ? 8 : 0) | mag;
}

/* fp32 -> E4M3 code, round-to-nearest-even, saturating to +-448 (never NaN). */
int orc_e4m3_encode(float x)
{
    int mag = round_to_grid(fabs((double)x), g_e4m3, 127);
    return (signbit(x) ? 0x80 : 0) | mag;
}

/* bf16 bit pattern -> value (exact). */
double orc_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* fp64 -> nearest bf16 (8 significant bits), ties to even, overflow to infinity.
 * Written from the definition: scale the significand to [128, 256), round, rescale. */
uint16_t orc_bf16_round(double d)
{
    int e;
    double m, r, v;
    float f;
    uint32_t u;
    if (d == 0.0 || isnan(d) || isinf(d)) {
        f = (float)d;
        memcpy(&u, &f, 4);
        return (uint16_t)(u >> 16);
    }
    m = frexp(fabs(d), &e);           /* |d| = m * 2^e, m in [0.5, 1) */
    if (e - 8 < -133) {               /* below the normal range: fixed quantum 2^-133 */
        r = nearbyint(ldexp(fabs(d), 133));
        v = ldexp(r, -133);
    } else {
        r = nearbyint(ldexp(m, 8));   /* default rounding mode: nearest, ties to even */
        v = ldexp(r, e - 8);
    }
    if (v > 3.3895313892515355e38) v = INFINITY;  /* above the largest finite bf16 */
    f = (float)v;                     /* exact: v has at most 8 significant bits */
    if (d < 0) f = -f;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------- */
/* NVFP4 quantisation                                                         */
/* ------------------------------------------------------------------------- */

/* Quantise one block of 16 fp32 values with global encode scale gs.
 *   m  = max |x|
 *   sf = E4M3(m * gs / 6)   (fp32 multiply, then fp32 divide by 6)
 *   sf == 0 -> every code is +0
 *   r  = gs / sf            (fp32 divide)
 *   code_i = E2M1(x_i * r)  (fp32 multiply)
 * Codes are returned one per byte (unpacked). */
static uint8_t quant_block16(const float* x, float gs, uint8_t* code)
{
    float m = 0.0f, t, q, sfv, r;
    int i, sf;
    for (i = 0; i < 16; i++) {
        float a = fabsf(x[i]);
        if (a > m) m = a;
    }
    t = m * gs;
    q = t / 6.0f;
    sf = orc_e4m3_encode(q);
    if (sf == 0) {
        for (i = 0; i < 16; i++) code[i] = 0;
        return 0;
    }
    sfv = (float)orc_e4m3_value(sf);
    r = gs / sfv;
    for (i = 0; i < 16; i++) code[i] = (uint8_t)orc_e2m1_encode(x[i] * r);
    return (uint8_t)sf;
}

/* amax over a whole tensor and the dynamic global scale 2688 / amax (1 if amax == 0). */
float orc_dynamic_global_scale(const float* X, long n)
{
    float amax = 0.0f;
    long i;
    for (i = 0; i < n; i++) {
        float a = fabsf(X[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) return 1.0f;
    return 2688.0f / amax;
}

/* X[R][K] fp32 row-major, K % 16 == 0.
 * codes[R][K/2]: element 2i in the low nibble, element 2i+1 in the high nibble.
 * sf[R][K/16]: E4M3 block scales.  gs is read (dynamic == 0) or computed (dynamic). */
void orc_quant_nvfp4(const float* X, long R, int K, int dynamic, float* gs_io,
                     uint8_t* codes, uint8_t* sf)
{
    float gs;
    long r;
    if (dynamic) *gs_io = orc_dynamic_global_scale(X, R * (long)K);
    gs = *gs_io;
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; r++) {
        uint8_t c[16];
        int b, i;
        for (b = 0; b < K / 16; b++) {
            sf[r * (K / 16) + b] = quant_block16(X + r * (long)K + b * 16, gs, c);
            for (i = 0; i < 8; i++)
                codes[r * (long)(K / 2) + b * 8 + i] = (uint8_t)(c[2 * i] | (c[2 * i + 1] << 4));
        }
    }
}

/* Value of element (r, k) without the global scale: E2M1(code) * E4M3(sf). */
static double nvfp4_elem(const uint8_t* codes, const uint8_t* sf, int K, long r, int k)
{
    uint8_t byte = codes[r * (long)(K / 2) + k / 2];
    int code = (k & 1) ? (byte >> 4) : (byte & 15);
    int s = sf[r * (long)(K / 16) + k / 16];
    double cv = (code & 8) ? -g_e2m1[code & 7] : g_e2m1[code & 7];
    double sv = ((s & 0x7f) == 0x7f) ? NAN : ((s & 0x80) ? -g_e4m3[s & 0x7f] : g_e4m3[s & 0x7f]);
    return cv * sv;
}

/* Dequantise R rows into out[R][K] = E2M1 * E4M3 / gs (fp64). */
void orc_dequant_nvfp4(const uint8_t* codes, const uint8_t* sf, float gs, long R, int K, double* out)
{
    long r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; r++) {
        int k;
        for (k = 0; k < K; k++) out[r * (long)K + k] = nvfp4_elem(codes, sf, K, r, k) / (double)gs;
    }
}

/* ------------------------------------------------------------------------- */
/* Routing                                                                    */
/* ------------------------------------------------------------------------- */

/* logits[t][e] = sum_h x[t][h] * Wr[e][h] (bf16 inputs, fp64 sum) + bias[e]. */
void orc_router_logits(const uint16_t* x, const uint16_t* wr, const float* bias,
                       long T, int H, int E, double* logits)
{
    long t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; t++) {
        int e, h;
        for (e = 0; e < E; e++) {
            double acc = 0.0;
            for (h = 0; h < H; h++)
                acc += orc_bf16_value(x[t * (long)H + h]) * orc_bf16_value(wr[(long)e * H + h]);
            logits[t * (long)E + e] = acc + (bias ? (double)bias[e] : 0.0);
        }
    }
}

typedef struct { double l; int e; } orc_cand;

static int cand_cmp(const void* a, const void* b)
{
    const orc_cand* x = (const orc_cand*)a;
    const orc_cand* y = (const orc_cand*)b;
    if (x->l > y->l) return -1;  /* larger logit first */
    if (x->l < y->l) return 1;
    return (x->e < y->e) ? -1 : (x->e > y->e);  /* equal logits: lower id first */
}

/* Top-k experts of each token by logit (ties to the lower id), in that order, and the
 * softmax of the selected logits: w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max). */
void orc_topk(const double* logits, long T, int E, int k, int32_t* ids, double* w)
{
    long t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; t++) {
        orc_cand* c = (orc_cand*)malloc(sizeof(orc_cand) * E);
        double z = 0.0;
        int e, j;
        for (e = 0; e < E; e++) {
            c[e].l = logits[t * (long)E + e];
            c[e].e = e;
        }
        qsort(c, E, sizeof(orc_cand), cand_cmp);
        for (j = 0; j < k; j++) z += exp(c[j].l - c[0].l);
        for (j = 0; j < k; j++) {
            ids[t * k + j] = c[j].e;
            w[t * k + j] = exp(c[j].l - c[0].l) / z;
        }
        free(c);
    }
}

/* Local map and grouping.  Pair p = t*k + j is local iff 0 <= ids[p] - off < E_loc.
 * counts[e'] = number of local pairs of local expert e'; sorted_pairs lists the local
 * pairs grouped by e' (ascending), ascending p inside a group.  Returns their number. */
long orc_permute(const int32_t* ids, long T, int k, int E_loc, int off,
                 int32_t* counts, int32_t* sorted_pairs)
{
    long p, n = 0;
    int e;
    for (e = 0; e < E_loc; e++) counts[e] = 0;
    for (p = 0; p < T * k; p++) {
        int le = ids[p] - off;
        if (le >= 0 && le < E_loc) counts[le]++;
    }
    for (e = 0; e < E_loc; e++)
        for (p = 0; p < T * k; p++)
            if (ids[p] - off == e) sorted_pairs[n++] = (int32_t)p;
    return n;
}

/* ------------------------------------------------------------------------- */
/* Expert MLP                                                                 */
/* ------------------------------------------------------------------------- */

typedef struct {
    int T, H, I, E, k;
    int E_loc, off;
    int has_shared, add_shared;
    int act_mode;        /* 0: W4A4 dynamic activation scale, 1: W4A4 static, 2: W4A16 */
    float act_gs;        /* static activation global scale (act_mode 1) */
    float inter_gs;      /* intermediate global scale (W4A4): static if > 0, else computed
                            per call from the intermediate's amax (dynamic) */
} orc_cfg;

/* One expert's weights, canonical layout (rows of the output dimension, K packed):
 *   w13: codes [2I][H/2], sf [2I][H/16], gs13   rows 0..I-1 gate, I..2I-1 up
 *   w2 : codes [H][I/2],  sf [H][I/16],  gs2 */
typedef struct {
    const uint8_t *w13, *w13_sf, *w2, *w2_sf;
    float gs13, gs2;
} orc_expert;

/* Dequantised (without global scale) weights of one expert, fp64. */
typedef struct {
    double* w13;   /* [2I][H] */
    double* w2;    /* [H][I] */
} orc_expert_f64;

static void expert_dequant(const orc_cfg* c, const orc_expert* x, orc_expert_f64* d)
{
    long n;
    int k;
    for (n = 0; n < 2L * c->I; n++)
        for (k = 0; k < c->H; k++) d->w13[n * c->H + k] = nvfp4_elem(x->w13, x->w13_sf, c->H, n, k);
    for (n = 0; n < c->H; n++)
        for (k = 0; k < c->I; k++) d->w2[n * c->I + k] = nvfp4_elem(x->w2, x->w2_sf, c->I, n, k);
}

/* silu(g) * u in fp64. */
static double swiglu(double g, double u) { return g / (1.0 + exp(-g)) * u; }

/* Gate/up projection of one input row (a: fp64 values without the activation global
 * scale, inv_a: 1/gs_a for W4A4 or 1 for W4A16):
 *   G[n] = (sum_k a[k] * w13[n][k]) * inv_a / gs13 */
static void row_gateup(const orc_cfg* c, const double* a, double a_div, const orc_expert* ex,
                       const orc_expert_f64* d, double* G)
{
    int n, k;
    for (n = 0; n < 2 * c->I; n++) {
        double acc = 0.0;
        const double* w = d->w13 + (long)n * c->H;
        for (k = 0; k < c->H; k++) acc += a[k] * w[k];
        G[n] = acc / (a_div * (double)ex->gs13);
    }
}

/* Intermediate activation of one row from its gate/up values and its down-projection
 * input (fp64 values without global scale plus the divisor that restores it):
 *   W4A4 : s = silu(g)*u rounded to fp32, NVFP4-quantised with the global scale gs_i
 *   W4A16: s rounded to bf16 */
static double row_inter(const orc_cfg* c, const double* G, float gs_i, double* s64, float* s32,
                        uint8_t* qc, uint8_t* qsf, double* aq)
{
    int i;
    for (i = 0; i < c->I; i++) s64[i] = swiglu(G[i], G[c->I + i]);
    if (c->act_mode == 2) {
        for (i = 0; i < c->I; i++) aq[i] = orc_bf16_value(orc_bf16_round(s64[i]));
        return 1.0;
    }
    for (i = 0; i < c->I; i++) s32[i] = (float)s64[i];
    orc_quant_nvfp4(s32, 1, c->I, 0, &gs_i, qc, qsf);
    for (i = 0; i < c->I; i++) aq[i] = nvfp4_elem(qc, qsf, c->I, 0, i);
    return (double)gs_i;
}

/* Down projection: Y[h] = (sum_i aq[i] * w2[h][i]) / (inter_div * gs2). */
static void row_down(const orc_cfg* c, const double* aq, double inter_div, const orc_expert* ex,
                     const orc_expert_f64* d, double* Y)
{
    int h, i;
    for (h = 0; h < c->H; h++) {
        double acc = 0.0;
        const double* w = d->w2 + (long)h * c->I;
        for (i = 0; i < c->I; i++) acc += aq[i] * w[i];
        Y[h] = acc / (inter_div * (double)ex->gs2);
    }
}

/* Input row of token t for the expert MLPs: W4A4 -> NVFP4 values without the global
 * scale (the divisor gs_a is applied after the contraction); W4A16 -> the bf16 value. */
static void input_row(const orc_cfg* c, const uint16_t* x, const uint8_t* xc, const uint8_t* xsf,
                      long t, double* a)
{
    int k;
    if (c->act_mode == 2) {
        for (k = 0; k < c->H; k++) a[k] = orc_bf16_value(x[t * (long)c->H + k]);
    } else {
        for (k = 0; k < c->H; k++) a[k] = nvfp4_elem(xc, xsf, c->H, t, k);
    }
}

/* Expert MLP for a set of rows (used by the unit tests): for each row r, token tok[r]
 * through expert ex.  Writes G[r][2I] (may be NULL), the intermediate codes/sf
 * (W4A4, may be NULL) and Y[r][H] (may be NULL). */
void orc_expert_rows(const orc_cfg* c, const orc_expert* ex, const uint16_t* x,
                     const uint8_t* xc, const uint8_t* xsf, float gs_a,
                     const int32_t* tok, long n_rows,
                     double* G_out, uint8_t* inter_codes, uint8_t* inter_sf, double* Y_out)
{
    orc_expert_f64 d;
    long r;
    d.w13 = (double*)malloc(sizeof(double) * 2L * c->I * c->H);
    d.w2 = (double*)malloc(sizeof(double) * (long)c->H * c->I);
    expert_dequant(c, ex, &d);
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < n_rows; r++) {
        double* a = (double*)malloc(sizeof(double) * c->H);
        double* G = (double*)malloc(sizeof(double) * 2 * c->I);
        double* s64 = (double*)malloc(sizeof(double) * c->I);
        float* s32 = (float*)malloc(sizeof(float) * c->I);
        uint8_t* qc = (uint8_t*)malloc(c->I / 2);
        uint8_t* qsf = (uint8_t*)malloc(c->I / 16);
        double* aq = (double*)malloc(sizeof(double) * c->I);
        double* Y = (double*)malloc(sizeof(double) * c->H);
        double a_div = (c->act_mode == 2) ? 1.0 : (double)gs_a;
        double i_div;
        input_row(c, x, xc, xsf, tok[r], a);
        row_gateup(c, a, a_div, ex, &d, G);
        if (G_out) memcpy(G_out + r * 2L * c->I, G, sizeof(double) * 2 * c->I);
        i_div = row_inter(c, G, c->inter_gs, s64, s32, qc, qsf, aq);
        if (inter_codes && c->act_mode != 2) {
            memcpy(inter_codes + r * (long)(c->I / 2), qc, c->I / 2);
            memcpy(inter_sf + r * (long)(c->I / 16), qsf, c->I / 16);
        }
        row_down(c, aq, i_div, ex, &d, Y);
        if (Y_out) memcpy(Y_out + r * (long)c->H, Y, sizeof(double) * c->H);
        free(a); free(G); free(s64); free(s32); free(qc); free(qsf); free(aq); free(Y);
    }
    free(d.w13);
    free(d.w2);
}

/* SwiGLU + NVFP4 requantisation of rows of fp32 gate/up values (gate = columns 0..I-1,
 * up = columns I..2I-1): s = silu(g)*u in fp64, rounded to fp32, quantised with the
 * static scale gs_i.  s_out (may be NULL) receives the fp64 s. */
void orc_swiglu_requant(const float* gu, long R, int I, float gs_i,
                        uint8_t* codes, uint8_t* sf, double* s_out)
{
    long r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; r++) {
        float* s32 = (float*)malloc(sizeof(float) * I);
        float g = gs_i;
        int i;
        for (i = 0; i < I; i++) {
            double s = swiglu((double)gu[r * 2L * I + i], (double)gu[r * 2L * I + I + i]);
            if (s_out) s_out[r * (long)I + i] = s;
            s32[i] = (float)s;
        }
        orc_quant_nvfp4(s32, 1, I, 0, &g, codes + r * (long)(I / 2), sf + r * (long)(I / 16));
        free(s32);
    }
}

/* ------------------------------------------------------------------------- */
/* Whole layer                                                                */
/* ------------------------------------------------------------------------- */

/* Dynamic intermediate global scale (W4A4 with inter_gs <= 0): 2688 / amax of the fp32
 * intermediate s = silu(g)*u over every row the shard computes -- its local pairs of all
 * T tokens and, with add_shared, every token's shared-expert row -- by the same formula as
 * the dynamic activation scale (1 if that amax is 0).  A first pass over the gate/up
 * projections; the forward then quantises each row's s with this scale. */
static float dynamic_inter_scale(const orc_cfg* c, const uint16_t* x, const uint8_t* xc,
                                 const uint8_t* xsf, float gs_a, const int32_t* ids,
                                 const orc_expert* ex)
{
    const long T = c->T;
    const int El = c->E_loc, k = c->k;
    float amax = 0.0f;
    int e;
#pragma omp parallel for schedule(dynamic, 1) reduction(max : amax)
    for (e = 0; e <= El; e++) {
        orc_expert_f64 d;
        double *a, *G;
        long p, n_rows = (e == El) ? T : T * k;
        int used = 0, i;
        if (e == El && !(c->has_shared && c->add_shared)) continue;
        if (e == El) used = T > 0;
        for (p = 0; p < T * k && !used; p++)
            if (ids[p] - c->off == e) used = 1;
        if (!used) continue;
        d.w13 = (double*)malloc(sizeof(double) * 2L * c->I * c->H);
        d.w2 = (double*)malloc(sizeof(double) * (long)c->H * c->I);
        expert_dequant(c, &ex[e], &d);
        a = (double*)malloc(sizeof(double) * c->H);
        G = (double*)malloc(sizeof(double) * 2 * c->I);
        for (p = 0; p < n_rows; p++) {
            const long tt = (e == El) ? p : p / k;
            if (e != El && ids[p] - c->off != e) continue;
            input_row(c, x, xc, xsf, tt, a);
            row_gateup(c, a, (double)gs_a, &ex[e], &d, G);
            for (i = 0; i < c->I; i++) {
                const float v = fabsf((float)swiglu(G[i], G[c->I + i]));
                if (v > amax) amax = v;
            }
        }
        free(a); free(G);
        free(d.w13);
        free(d.w2);
    }
    return orc_dynamic_global_scale(&amax, 1);
}

/* Forward of the layer (or of one expert shard of it).
 *
 * Inputs: x bf16 [T][H]; the router either from x (router_w bf16 [E][H]) or from given
 * fp32 logits (logits_in [T][E]); optional fp32 logit bias [E]; the local experts'
 * weights ex[0..E_loc-1] (ex[E_loc] is the shared expert when has_shared).
 * Outputs for every token: logits (fp64, may be NULL), top-k ids and weights, the local
 * counts and grouped pair list (may be NULL), the activation codes/sf/gs (W4A4, may be
 * NULL), the intermediate global scale used (W4A4; the static one, or the dynamic one of
 * dynamic_inter_scale when cfg.inter_gs <= 0; may be NULL).  Outputs for the tokens listed in tok[0..n_tok-1] (all tokens when tok is
 * NULL): out[n_tok][H] in fp64 and out_bf16 (may be NULL), the final values rounded to
 * bf16.
 *
 *   out[t] = sum_{j: pair (t,j) local} w[t][j] * MLP_{ids[t][j]-off}(x_t)
 *            + add_shared * MLP_shared(x_t)
 * with the sum in ascending j, then the shared term. */
int orc_moe_forward(const orc_cfg* c, const uint16_t* x, const uint16_t* router_w,
                    const float* logit_bias, const float* logits_in, const orc_expert* ex,
                    const int32_t* tok, long n_tok,
                    double* logits_out, int32_t* topk_ids, double* topk_w,
                    int32_t* counts, int32_t* sorted_pairs, long* n_local,
                    uint8_t* x_codes, uint8_t* x_sf, float* gs_a_out, float* gs_i_out,
                    double* out, uint16_t* out_bf16)
{
    const long T = c->T;
    const int H = c->H, k = c->k, E = c->E, El = c->E_loc;
    double* logits = (double*)malloc(sizeof(double) * T * E);
    double* w = topk_w;
    int32_t* ids = topk_ids;
    uint8_t* xc = NULL;
    uint8_t* xsf = NULL;
    float gs_a = 1.0f;
    float gs_i = c->inter_gs;
    long t, i, nt = tok ? n_tok : T;
    int* row_of_tok = (int*)malloc(sizeof(int) * T);
    double* Yr;   /* [nt][k][H] routed outputs (unweighted) */
    double* Ys;   /* [nt][H] shared outputs */
    int* have;    /* [nt][k] pair is local */
    int e;

    /* a1/a2: logits and top-k */
    if (logits_in) {
        for (t = 0; t < T; t++)
            for (e = 0; e < E; e++)
                logits[t * E + e] = (double)logits_in[t * E + e] + (logit_bias ? (double)logit_bias[e] : 0.0);
    } else {
        orc_router_logits(x, router_w, logit_bias, T, H, E, logits);
    }
    if (logits_out) memcpy(logits_out, logits, sizeof(double) * T * E);
    orc_topk(logits, T, E, k, ids, w);

    /* a3: local map + grouping */
    if (counts && sorted_pairs) {
        long n = orc_permute(ids, T, k, El, c->off, counts, sorted_pairs);
        if (n_local) *n_local = n;
    }

    /* a4: activation quantisation (W4A4) over all tokens */
    if (c->act_mode != 2) {
        float* xf = (float*)malloc(sizeof(float) * T * H);
        for (i = 0; i < T * H; i++) xf[i] = (float)orc_bf16_value(x[i]);
        xc = x_codes ? x_codes : (uint8_t*)malloc(T * (long)(H / 2));
        xsf = x_sf ? x_sf : (uint8_t*)malloc(T * (long)(H / 16));
        gs_a = c->act_gs;
        orc_quant_nvfp4(xf, T, H, c->act_mode == 0, &gs_a, xc, xsf);
        if (gs_a_out) *gs_a_out = gs_a;
        free(xf);
        if (!(c->inter_gs > 0.0f)) gs_i = dynamic_inter_scale(c, x, xc, xsf, gs_a, ids, ex);
    }
    if (gs_i_out) *gs_i_out = gs_i;

    /* a5..a8: expert MLPs for the requested tokens */
    for (t = 0; t < T; t++) row_of_tok[t] = -1;
    for (i = 0; i < nt; i++) row_of_tok[tok ? tok[i] : i] = (int)i;
    Yr = (double*)calloc((size_t)nt * k * H, sizeof(double));
    Ys = (double*)calloc((size_t)nt * H, sizeof(double));
    have = (int*)calloc((size_t)nt * k, sizeof(int));

#pragma omp parallel for schedule(dynamic, 1)
    for (e = 0; e <= El; e++) {
        orc_expert_f64 d;
        double *a, *G, *s64, *aq;
        float* s32;
        uint8_t *qc, *qsf;
        long p;
        int used = 0;
        if (e == El && !(c->has_shared && c->add_shared)) continue;
        /* does any requested row use this expert? */
        if (e == El) used = nt > 0;
        for (p = 0; p < T * k && !used; p++)
            if (ids[p] - c->off == e && row_of_tok[p / k] >= 0) used = 1;
        if (!used) continue;
        d.w13 = (double*)malloc(sizeof(double) * 2L * c->I * H);
        d.w2 = (double*)malloc(sizeof(double) * (long)H * c->I);
        expert_dequant(c, &ex[e], &d);
        a = (double*)malloc(sizeof(double) * H);
        G = (double*)malloc(sizeof(double) * 2 * c->I);
        s64 = (double*)malloc(sizeof(double) * c->I);
        s32 = (float*)malloc(sizeof(float) * c->I);
        qc = (uint8_t*)malloc(c->I / 2);
        qsf = (uint8_t*)malloc(c->I / 16);
        aq = (double*)malloc(sizeof(double) * c->I);
        for (p = 0; p < (e == El ? T : T * k); p++) {
            long tt = (e == El) ? p : p / k;
            long r = row_of_tok[tt];
            double i_div;
            double* Y;
            if (r < 0) continue;
            if (e != El && ids[p] - c->off != e) continue;
            input_row(c, x, xc, xsf, tt, a);
            row_gateup(c, a, c->act_mode == 2 ? 1.0 : (double)gs_a, &ex[e], &d, G);
            i_div = row_inter(c, G, gs_i, s64, s32, qc, qsf, aq);
            Y = (e == El) ? Ys + r * (long)H : Yr + (r * k + p % k) * (long)H;
            row_down(c, aq, i_div, &ex[e], &d, Y);
            if (e != El) have[r * k + p % k] = 1;
        }
        free(a); free(G); free(s64); free(s32); free(qc); free(qsf); free(aq);
        free(d.w13);
        free(d.w2);
    }

    /* a9: combine, ascending j then the shared term, then round to bf16 */
    for (i = 0; i < nt; i++) {
        long tt = tok ? tok[i] : i;
        int h, j;
        for (h = 0; h < H; h++) {
            double acc = 0.0;
            for (j = 0; j < k; j++)
                if (have[i * k + j]) acc += w[tt * k + j] * Yr[(i * k + j) * (long)H + h];
            if (c->has_shared && c->add_shared) acc += Ys[i * (long)H + h];
            if (out) out[i * (long)H + h] = acc;
            if (out_bf16) out_bf16[i * (long)H + h] = orc_bf16_round(acc);
        }
    }

    if (c->act_mode != 2) {
        if (!x_codes) free(xc);
        if (!x_sf) free(xsf);
    }
    free(logits);
    free(row_of_tok);
    free(Yr);
    free(Ys);
    free(have);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Checkpoint-convention weight preparation                                   */
/* ------------------------------------------------------------------------- */

/* One weight matrix type of a checkpoint (E_total experts of N x K NVFP4, canonical:
 * codes [E][N][K/2], E4M3 block scales [E][N][K/16], one global value per expert) ->
 * the library's convention for the experts off..off+count-1:
 *   - global: convention 0 gives the encode scale gs (dequantised value = code*sf/gs,
 *     the reciprocal form), convention 1 the dequantisation multiplier m (value =
 *     code*sf*m), turned into gs = 1/m in fp32;
 *   - fold_target > 0: the expert's global is folded into its block scales relative to
 *     the common scale gs_t = fold_target: r = gs_t / gs (fp32), sf' = E4M3(sf * r)
 *     rounded to nearest even and saturated at 448 (re-rounding), and gs' = gs_t for every
 *     expert (gs_t = 1 folds the global away completely);
 *   - swap_halves: rows N/2..N-1 come first (a fused gate/up matrix stored up-then-gate
 *     becomes gate-then-up).
 * Codes are copied unchanged. */
void orc_prepare_weights(const uint8_t* codes, const uint8_t* sf, const float* glob,
                         int N, int K, int convention, float fold_target, int swap_halves,
                         int off, int count, uint8_t* codes_out, uint8_t* sf_out,
                         float* gs_out)
{
    long e;
    for (e = 0; e < count; e++) {
        const long src_e = off + e;
        float gs = convention == 1 ? 1.0f / glob[src_e] : glob[src_e];
        float r = 1.0f;
        long n;
        if (fold_target > 0.0f) {
            r = fold_target / gs;
            gs = fold_target;
        }
        gs_out[e] = gs;
        for (n = 0; n < N; n++) {
            const long src_n = swap_halves ? (n + N / 2) % N : n;
            const long src_row = src_e * N + src_n, dst_row = e * N + n;
            int b;
            memcpy(codes_out + dst_row * (K / 2), codes + src_row * (K / 2), K / 2);
            for (b = 0; b < K / 16; b++) {
                const uint8_t v = sf[src_row * (K / 16) + b];
                if (fold_target > 0.0f) {
                    const float x = (float)orc_e4m3_value(v) * r;
                    sf_out[dst_row * (K / 16) + b] = (uint8_t)orc_e4m3_encode(x);
                } else {
                    sf_out[dst_row * (K / 16) + b] = v;
                }
            }
        }
    }
}

/* Threads the parallel loops use. */
int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
