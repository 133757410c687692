/*
 * moe_oracle.c -- CPU oracle for the fused MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product path.  It shares no
 * code with the CUDA library.  See moe_oracle.h for what each function
 * follows.  Build with -ffp-contract=off and without -ffast-math: every
 * fp32 operation here is meant to round once, as written.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ======================================================================
 * Element codecs (OCP 8-bit float "e4m3fn", OCP MX v1.0 e2m1 and e8m0,
 * bfloat16).  Encoders pick the nearest representable value; an exact
 * midpoint goes to the code whose last mantissa bit is 0 (ties to even);
 * magnitudes beyond the largest finite value saturate to it.
 * ====================================================================== */

float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t orc_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if (isnan(x))
        return (uint16_t)((u >> 16) | 0x0040);  /* quiet NaN, sign kept */
    /* round to nearest even on the 16 discarded bits */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* e4m3fn: s eeee mmm, bias 7, no infinities, s1111111 is NaN.
 * exponent field 0: subnormal m/8 * 2^-6.                               */
static double e4m3_mag(int c)   /* c in 0..0x7E, non-negative values */
{
    int e = (c >> 3) & 15, m = c & 7;
    if (e == 0)
        return ldexp((double)m, -9);
    return ldexp(8.0 + m, e - 10);   /* (1 + m/8) * 2^(e-7) */
}

float orc_e4m3_to_f32(uint8_t c)
{
    if ((c & 0x7F) == 0x7F)
        return NAN;
    double v = e4m3_mag(c & 0x7F);
    return (float)((c & 0x80) ? -v : v);
}

/* e2m1 (low nibble): s ee m, bias 1; exponent 0 is subnormal m * 0.5.  */
static double e2m1_mag(int c)   /* c in 0..7 */
{
    int e = (c >> 1) & 3, m = c & 1;
    if (e == 0)
        return 0.5 * m;
    return ldexp(2.0 + m, e - 2);    /* (1 + m/2) * 2^(e-1) */
}

float orc_e2m1_to_f32(uint8_t c)
{
    double v = e2m1_mag(c & 7);
    return (float)((c & 8) ? -v : v);
}

float orc_e8m0_to_f32(uint8_t c)
{
    if (c == 0xFF)
        return NAN;
    return (float)ldexp(1.0, (int)c - 127);
}

/* Nearest non-negative code to a >= 0 among codes 0..maxcode, whose
 * magnitudes mag(0) = 0 < mag(1) < ... are increasing.  Ties go to the even
 * code; a >= mag(maxcode) saturates.  The midpoint of two neighbouring
 * codes is exact in double, so the comparison is exact.                 */
static int nearest_code(double a, int maxcode, double (*mag)(int))
{
    if (a >= mag(maxcode))
        return maxcode;
    int lo = 0, hi = maxcode;        /* mag(lo) <= a < mag(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (mag(mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double mid = 0.5 * (mag(lo) + mag(hi));
    if (a < mid)
        return lo;
    if (a > mid)
        return hi;
    return (lo % 2 == 0) ? lo : hi;
}

static uint8_t enc_e4m3_d(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    return (uint8_t)(sign | nearest_code(fabs(x), 0x7E, e4m3_mag));
}

uint8_t orc_f32_to_e4m3(float x) { return enc_e4m3_d((double)x); }

uint8_t orc_f32_to_e2m1(float x)
{
    uint8_t sign = signbit(x) ? 0x8 : 0x0;
    return (uint8_t)(sign | nearest_code(fabs((double)x), 7, e2m1_mag));
}

/* ======================================================================
 * Block quantisers.
 * NVFP4 (block 16, e4m3 scale, activation global scale 1): the scale is
 * amax / 6 (6 = largest e2m1 magnitude) rounded to e4m3, and every element
 * is divided by the *quantised* scale before rounding to e2m1.
 * MXFP8 (block 32, e8m0 scale): OCP MX v1.0 shared exponent
 * X = floor(log2 amax) - 8 (8 = exponent of the largest e4m3 normal), and
 * elements x * 2^-X rounded to e4m3 with saturation.
 * ====================================================================== */

void orc_quant_nvfp4_block16(const float *x, uint8_t *codes, uint8_t *sf)
{
    float amax = 0.0f;
    for (int i = 0; i < 16; i++) {
        float a = fabsf(x[i]);
        if (a > amax)
            amax = a;
    }
    float s = amax / 6.0f;                 /* fp32, correctly rounded */
    uint8_t c = orc_f32_to_e4m3(s);
    float sv = orc_e4m3_to_f32(c);
    *sf = c;
    for (int i = 0; i < 16; i++)
        codes[i] = (sv == 0.0f) ? 0 : orc_f32_to_e2m1(x[i] / sv);
}

void orc_quant_mxfp8_block32(const float *x, uint8_t *codes, uint8_t *sf)
{
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(x[i]);
        if (a > amax)
            amax = a;
    }
    if (amax == 0.0f) {
        *sf = 127;
        for (int i = 0; i < 32; i++)
            codes[i] = 0;
        return;
    }
    int e;
    frexp((double)amax, &e);               /* amax = f * 2^e, f in [0.5,1) */
    int X = (e - 1) - 8;                   /* floor(log2 amax) - emax(e4m3) */
    if (X < -127)
        X = -127;
    if (X > 127)
        X = 127;
    *sf = (uint8_t)(X + 127);
    for (int i = 0; i < 32; i++)
        codes[i] = enc_e4m3_d(ldexp((double)x[i], -X));   /* exact scaling */
}

int orc_quant_row(int fmt, const float *x, int n, uint8_t *codes, uint8_t *sf)
{
    if (fmt == ORC_FMT_NVFP4) {
        if (n % 16)
            return -1;
        for (int b = 0; b < n / 16; b++) {
            uint8_t q[16];
            orc_quant_nvfp4_block16(x + 16 * b, q, sf + b);
            for (int j = 0; j < 8; j++)
                codes[8 * b + j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
        }
        return 0;
    }
    if (fmt == ORC_FMT_MXFP8) {
        if (n % 32)
            return -1;
        for (int b = 0; b < n / 32; b++)
            orc_quant_mxfp8_block32(x + 32 * b, codes + 32 * b, sf + b);
        return 0;
    }
    return -1;
}

int orc_dequant_row(int fmt, const uint8_t *codes, const uint8_t *sf, int n,
                    float *out)
{
    if (fmt == ORC_FMT_NVFP4) {
        if (n % 16)
            return -1;
        for (int i = 0; i < n; i++) {
            uint8_t byte = codes[i / 2];
            uint8_t q = (i % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            out[i] = orc_e2m1_to_f32(q) * orc_e4m3_to_f32(sf[i / 16]);
        }
        return 0;
    }
    if (fmt == ORC_FMT_MXFP8) {
        if (n % 32)
            return -1;
        for (int i = 0; i < n; i++)
            out[i] = orc_e4m3_to_f32(codes[i]) * orc_e8m0_to_f32(sf[i / 32]);
        return 0;
    }
    return -1;
}

void orc_fold_scales(const uint8_t *sf, int64_t n, float gs, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++) {
        float p = orc_e4m3_to_f32(sf[i]) * gs;    /* fp32 product */
        out[i] = orc_f32_to_e4m3(p);
    }
}

/* ======================================================================
 * Routing: the K largest logits (value descending, lower expert index first
 * on equal values), then a softmax over the K selected logits, which equals
 * the full softmax restricted to the top K and renormalised.
 * ====================================================================== */

void orc_route(const float *logits, int T, int E, int K, int32_t *ids,
               float *w)
{
    char *taken = (char *)malloc((size_t)E);
    for (int t = 0; t < T; t++) {
        const float *l = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int k = 0; k < K; k++) {
            int best = -1;
            for (int e = 0; e < E; e++) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best])
                    best = e;       /* strict: equal values keep lower e */
            }
            taken[best] = 1;
            ids[(size_t)t * K + k] = best;
        }
        double m = (double)l[ids[(size_t)t * K]];
        double den = 0.0;
        for (int k = 0; k < K; k++)
            den += exp((double)l[ids[(size_t)t * K + k]] - m);
        for (int k = 0; k < K; k++)
            w[(size_t)t * K + k] =
                (float)(exp((double)l[ids[(size_t)t * K + k]] - m) / den);
    }
    free(taken);
}

/* Counting sort, stable in the slot index s = t*K + k.                  */
void orc_permute(const int32_t *ids, int T, int K, int E, int32_t *offsets,
                 int32_t *perm, int32_t *inv)
{
    int R = T * K;
    int32_t *seen = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int e = 0; e <= E; e++)
        offsets[e] = 0;
    for (int s = 0; s < R; s++)
        offsets[ids[s] + 1]++;
    for (int e = 0; e < E; e++)
        offsets[e + 1] += offsets[e];
    for (int s = 0; s < R; s++) {
        int e = ids[s];
        int row = offsets[e] + seen[e]++;
        perm[row] = s;
        if (inv)
            inv[s] = row;
    }
    free(seen);
}

/* ======================================================================
 * The layer, row by row.
 * ====================================================================== */

static int bytes_per_row(int fmt, int n)   /* canonical code bytes */
{
    return fmt == ORC_FMT_NVFP4 ? n / 2 : fmt == ORC_FMT_MXFP8 ? n : 2 * n;
}

static int sf_per_row(int fmt, int n)
{
    return fmt == ORC_FMT_NVFP4 ? n / 16 : fmt == ORC_FMT_MXFP8 ? n / 32 : 0;
}

/* GEMM1 input for one token: bf16 as is, or quantised per block and
 * dequantised (activation global scale 1).                              */
static void act_row(const orc_cfg *c, const uint16_t *hid, float *a,
                    uint8_t *codes, uint8_t *sf)
{
    int H = c->H;
    for (int i = 0; i < H; i++)
        a[i] = orc_bf16_to_f32(hid[i]);
    if (c->fmt == ORC_FMT_BF16)
        return;
    orc_quant_row(c->fmt, a, H, codes, sf);
    orc_dequant_row(c->fmt, codes, sf, H, a);
}

/* Rows of W13: gate and up (SwiGLU) or up only (ReLU^2). */
static int w13_rows(const orc_cfg *c)
{
    return c->act == ORC_ACT_RELU2 ? c->I : 2 * c->I;
}

/* One dequantised weight row (exact in fp32).  which = 13: row n of W13_e
 * (reduction length H); which = 2: row n of W2_e (reduction length I).
 * NVFP4 block scales are first folded with the expert's global scale.   */
static void weight_row(const orc_cfg *c, const orc_weights *wt, int which,
                       int e, int n, float *out, uint8_t *sf_tmp)
{
    int N = which == 13 ? w13_rows(c) : c->H;
    int Kd = which == 13 ? c->H : c->I;
    size_t row = (size_t)e * N + n;
    const void *w = which == 13 ? wt->w13 : wt->w2;
    if (c->fmt == ORC_FMT_BF16) {
        const uint16_t *p = (const uint16_t *)w + row * Kd;
        for (int i = 0; i < Kd; i++)
            out[i] = orc_bf16_to_f32(p[i]);
        return;
    }
    const uint8_t *codes = (const uint8_t *)w + row * bytes_per_row(c->fmt, Kd);
    const uint8_t *sf = (which == 13 ? wt->w13_sf : wt->w2_sf) +
                        row * sf_per_row(c->fmt, Kd);
    if (c->fmt == ORC_FMT_NVFP4) {
        float gs = (which == 13 ? wt->w13_gs : wt->w2_gs)[e];
        orc_fold_scales(sf, sf_per_row(c->fmt, Kd), gs, sf_tmp);
        sf = sf_tmp;
    }
    orc_dequant_row(c->fmt, codes, sf, Kd, out);
}

static float dot(const float *a, const float *b, int n)
{
    double s = 0.0;
    for (int i = 0; i < n; i++)
        s += (double)a[i] * (double)b[i];
    return (float)s;
}

static int clamp_on(const orc_cfg *c)
{
    return c->clamp > 0.0f && isfinite(c->clamp);
}

/* The activation on one GEMM1 output row.  SwiGLU: G[0..2I), gate =
 * G[0..I), up = G[I..2I), optional symmetric clamp of both, h = silu(gate)
 * * up.  ReLU^2: G[0..I), h = max(G, 0)^2.  Both in double, rounded to
 * fp32.  Then the GEMM2 input: bf16-rounded (BF16) or re-quantised per
 * block from fp32 h.                                                    */
static void swiglu_requant(const orc_cfg *c, const float *G, float *hq,
                           uint8_t *codes, uint8_t *sf)
{
    int I = c->I;
    for (int i = 0; i < I && c->act == ORC_ACT_RELU2; i++) {
        /* non-gated squared ReLU of the single projection */
        double g = G[i] > 0.0f ? (double)G[i] : 0.0;
        hq[i] = (float)(g * g);
    }
    for (int i = 0; i < I && c->act == ORC_ACT_SWIGLU; i++) {
        float g = G[i], u = G[I + i];
        if (clamp_on(c)) {
            float L = c->clamp;
            g = g < -L ? -L : (g > L ? L : g);
            u = u < -L ? -L : (u > L ? L : u);
        }
        double gd = g, ud = u;
        hq[i] = (float)(gd / (1.0 + exp(-gd)) * ud);
    }
    if (c->fmt == ORC_FMT_BF16) {
        for (int i = 0; i < I; i++)
            hq[i] = orc_bf16_to_f32(orc_f32_to_bf16(hq[i]));
        return;
    }
    orc_quant_row(c->fmt, hq, I, codes, sf);
    orc_dequant_row(c->fmt, codes, sf, I, hq);
}

static int check_cfg(const orc_cfg *c)
{
    if (c->H <= 0 || c->I <= 0 || c->E <= 0 || c->K <= 0 || c->K > c->E)
        return -1;
    if (c->fmt < ORC_FMT_BF16 || c->fmt > ORC_FMT_NVFP4)
        return -1;
    if (c->fmt == ORC_FMT_NVFP4 && (c->H % 16 || c->I % 16))
        return -1;
    if (c->fmt == ORC_FMT_MXFP8 && (c->H % 32 || c->I % 32))
        return -1;
    if (c->act != ORC_ACT_SWIGLU && c->act != ORC_ACT_RELU2)
        return -1;
    if (c->act == ORC_ACT_RELU2 && clamp_on(c))
        return -1;
    return 0;
}

int orc_forward(const orc_cfg *c, const orc_weights *wt,
                const uint16_t *hidden, const float *logits, int T,
                uint16_t *out, int32_t *ids_o, float *w_o, int32_t *off_o,
                int32_t *perm_o, uint8_t *xq_codes, uint8_t *xq_sf,
                float *h_o, float *y_o)
{
    if (check_cfg(c) || T < 0)
        return -1;
    if (T == 0)
        return 0;
    const int H = c->H, I = c->I, E = c->E, K = c->K, fmt = c->fmt;
    const int R = T * K;
    const int xb = bytes_per_row(fmt, H), xs = sf_per_row(fmt, H);
    const int hb = bytes_per_row(fmt, I), hs = sf_per_row(fmt, I);

    int32_t *ids = ids_o ? ids_o : (int32_t *)malloc(sizeof(int32_t) * R);
    float *w = w_o ? w_o : (float *)malloc(sizeof(float) * R);
    int32_t *off = off_o ? off_o : (int32_t *)malloc(sizeof(int32_t) * (E + 1));
    int32_t *perm = perm_o ? perm_o : (int32_t *)malloc(sizeof(int32_t) * R);
    int32_t *inv = (int32_t *)malloc(sizeof(int32_t) * R);
    float *A = (float *)malloc(sizeof(float) * (size_t)T * H);
    uint8_t *xc = (uint8_t *)malloc((size_t)T * (xb + xs) + 1);
    float *Hq = h_o ? h_o : (float *)malloc(sizeof(float) * (size_t)R * I);
    float *Y = y_o ? y_o : (float *)malloc(sizeof(float) * (size_t)R * H);
    int maxrows = 0;
    float *G = NULL;

    /* 1. routing, 2. permutation */
    orc_route(logits, T, E, K, ids, w);
    orc_permute(ids, T, K, E, off, perm, inv);

    /* 3. GEMM1 input, once per token */
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++)
        act_row(c, hidden + (size_t)t * H, A + (size_t)t * H,
                xc + (size_t)t * (xb + xs), xc + (size_t)t * (xb + xs) + xb);
    if (fmt != ORC_FMT_BF16) {
        for (int t = 0; t < T; t++) {
            if (xq_codes)
                memcpy(xq_codes + (size_t)t * xb, xc + (size_t)t * (xb + xs), xb);
            if (xq_sf)
                memcpy(xq_sf + (size_t)t * xs, xc + (size_t)t * (xb + xs) + xb, xs);
        }
    }

    for (int e = 0; e < E; e++)
        if (off[e + 1] - off[e] > maxrows)
            maxrows = off[e + 1] - off[e];
    const int N1 = w13_rows(c);
    G = (float *)malloc(sizeof(float) * (size_t)maxrows * N1 + 1);

    /* 4. expert by expert: GEMM1, SwiGLU + re-quantisation, GEMM2 */
    for (int e = 0; e < E; e++) {
        int r0 = off[e], nr = off[e + 1] - off[e];
        if (nr == 0)
            continue;
#pragma omp parallel
        {
            float *wrow = (float *)malloc(sizeof(float) * (H > I ? H : I));
            uint8_t *sft = (uint8_t *)malloc((size_t)(H > I ? H : I) / 16 + 1);
            uint8_t *qc = (uint8_t *)malloc((size_t)hb + hs + 1);
#pragma omp for schedule(static)
            for (int n = 0; n < N1; n++) {
                weight_row(c, wt, 13, e, n, wrow, sft);
                for (int r = 0; r < nr; r++) {
                    int t = perm[r0 + r] / K;
                    G[(size_t)r * N1 + n] = dot(A + (size_t)t * H, wrow, H);
                }
            }
#pragma omp for schedule(static)
            for (int r = 0; r < nr; r++)
                swiglu_requant(c, G + (size_t)r * N1,
                               Hq + (size_t)(r0 + r) * I, qc, qc + hb);
#pragma omp for schedule(static)
            for (int j = 0; j < H; j++) {
                weight_row(c, wt, 2, e, j, wrow, sft);
                for (int r = 0; r < nr; r++)
                    Y[(size_t)(r0 + r) * H + j] =
                        dot(Hq + (size_t)(r0 + r) * I, wrow, I);
            }
            free(wrow);
            free(sft);
            free(qc);
        }
    }

    /* 5. combine: out[t] = bf16( sum_k w[t,k] * Y[row(t,k)] ), k ascending */
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        for (int j = 0; j < H; j++) {
            double acc = 0.0;
            for (int k = 0; k < K; k++)
                acc += (double)w[(size_t)t * K + k] *
                       (double)Y[(size_t)inv[(size_t)t * K + k] * H + j];
            out[(size_t)t * H + j] = orc_f32_to_bf16((float)acc);
        }
    }

    free(G);
    free(A);
    free(xc);
    free(inv);
    if (!ids_o) free(ids);
    if (!w_o) free(w);
    if (!off_o) free(off);
    if (!perm_o) free(perm);
    if (!h_o) free(Hq);
    if (!y_o) free(Y);
    return 0;
}

int orc_token_forward(const orc_cfg *c, const orc_weights *wt,
                      const uint16_t *hidden_row, const float *logits_row,
                      float *out_f32, uint16_t *out)
{
    if (check_cfg(c))
        return -1;
    const int H = c->H, I = c->I, K = c->K, fmt = c->fmt;
    const int hb = bytes_per_row(fmt, I), hs = sf_per_row(fmt, I);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * K);
    float *w = (float *)malloc(sizeof(float) * K);
    float *a = (float *)malloc(sizeof(float) * H);
    uint8_t *xc = (uint8_t *)malloc((size_t)H + H / 16 + 1);
    float *G = (float *)malloc(sizeof(float) * 2 * I);
    float *hq = (float *)malloc(sizeof(float) * I);
    double *acc = (double *)calloc((size_t)H, sizeof(double));
    uint8_t *qc = (uint8_t *)malloc((size_t)hb + hs + 1);

    orc_route(logits_row, 1, c->E, K, ids, w);
    act_row(c, hidden_row, a, xc, xc + H);
    for (int k = 0; k < K; k++) {
        int e = ids[k];
#pragma omp parallel
        {
            float *wrow = (float *)malloc(sizeof(float) * (H > I ? H : I));
            uint8_t *sft = (uint8_t *)malloc((size_t)(H > I ? H : I) / 16 + 1);
#pragma omp for schedule(static)
            for (int n = 0; n < w13_rows(c); n++) {
                weight_row(c, wt, 13, e, n, wrow, sft);
                G[n] = dot(a, wrow, H);
            }
#pragma omp single
            swiglu_requant(c, G, hq, qc, qc + hb);
#pragma omp for schedule(static)
            for (int j = 0; j < H; j++) {
                weight_row(c, wt, 2, e, j, wrow, sft);
                acc[j] += (double)w[k] * (double)dot(hq, wrow, I);
            }
            free(wrow);
            free(sft);
        }
    }
    for (int j = 0; j < H; j++) {
        float v = (float)acc[j];
        if (out_f32)
            out_f32[j] = v;
        if (out)
            out[j] = orc_f32_to_bf16(v);
    }
    free(ids);
    free(w);
    free(a);
    free(xc);
    free(G);
    free(hq);
    free(acc);
    free(qc);
    return 0;
}

int orc_forward_batched(const orc_cfg *c, const orc_weights *wt,
                        const uint16_t *hidden, const int32_t *counts, int M,
                        uint16_t *out, float *y)
{
    if (check_cfg(c) || M < 0)
        return -1;
    const int H = c->H, I = c->I, E = c->E, fmt = c->fmt, N1 = w13_rows(c);
    const int xb = bytes_per_row(fmt, H), hb = bytes_per_row(fmt, I);
    const int hs = sf_per_row(fmt, I);
    for (int e = 0; e < E; e++)
        if (counts[e] < 0 || counts[e] > M)
            return -1;
    for (int e = 0; e < E; e++) {
        const int nr = counts[e];
        if (nr == 0)
            continue;
        float *A = (float *)malloc(sizeof(float) * (size_t)nr * H);
        float *G = (float *)malloc(sizeof(float) * (size_t)nr * N1);
        float *Hq = (float *)malloc(sizeof(float) * (size_t)nr * I);
#pragma omp parallel
        {
            float *wrow = (float *)malloc(sizeof(float) * (H > I ? H : I));
            uint8_t *sft = (uint8_t *)malloc((size_t)(H > I ? H : I) / 16 + 1);
            uint8_t *qc = (uint8_t *)malloc((size_t)(xb > hb ? xb : hb) + H / 16 + hs + 1);
#pragma omp for schedule(static)
            for (int r = 0; r < nr; r++)
                act_row(c, hidden + ((size_t)e * M + r) * H, A + (size_t)r * H, qc,
                        qc + xb);
#pragma omp for schedule(static)
            for (int n = 0; n < N1; n++) {
                weight_row(c, wt, 13, e, n, wrow, sft);
                for (int r = 0; r < nr; r++)
                    G[(size_t)r * N1 + n] = dot(A + (size_t)r * H, wrow, H);
            }
#pragma omp for schedule(static)
            for (int r = 0; r < nr; r++)
                swiglu_requant(c, G + (size_t)r * N1, Hq + (size_t)r * I, qc, qc + hb);
#pragma omp for schedule(static)
            for (int j = 0; j < H; j++) {
                weight_row(c, wt, 2, e, j, wrow, sft);
                for (int r = 0; r < nr; r++) {
                    const float v = dot(Hq + (size_t)r * I, wrow, I);
                    const size_t o = ((size_t)e * M + r) * H + j;
                    out[o] = orc_f32_to_bf16(v);
                    if (y)
                        y[o] = v;
                }
            }
            free(wrow);
            free(sft);
            free(qc);
        }
        free(A);
        free(G);
        free(Hq);
    }
    return 0;
}

int orc_encode_n(int kind, const float *x, int64_t n, void *codes)
{
    for (int64_t i = 0; i < n; i++) {
        switch (kind) {
        case 0: ((uint16_t *)codes)[i] = orc_f32_to_bf16(x[i]); break;
        case 1: ((uint8_t *)codes)[i] = orc_f32_to_e4m3(x[i]); break;
        case 2: ((uint8_t *)codes)[i] = orc_f32_to_e2m1(x[i]); break;
        default: return -1;
        }
    }
    return 0;
}

int orc_decode_n(int kind, const void *codes, int64_t n, float *x)
{
    for (int64_t i = 0; i < n; i++) {
        switch (kind) {
        case 0: x[i] = orc_bf16_to_f32(((const uint16_t *)codes)[i]); break;
        case 1: x[i] = orc_e4m3_to_f32(((const uint8_t *)codes)[i]); break;
        case 2: x[i] = orc_e2m1_to_f32(((const uint8_t *)codes)[i]); break;
        case 3: x[i] = orc_e8m0_to_f32(((const uint8_t *)codes)[i]); break;
        default: return -1;
        }
    }
    return 0;
}

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
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
