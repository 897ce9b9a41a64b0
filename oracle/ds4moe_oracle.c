/*
 * CPU oracle for the routed mixture-of-experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * execute this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code with the CUDA library.
 *
 * It is a plain, slow, obviously correct restatement of what the layer
 * computes, in IEEE binary64 throughout:
 *
 *   logits   L[t,e] = sum_h x[t,h] * Wr[e,h]
 *   scores   s = sigmoid(L),  selection score sel = s + b_e  (b = 0 without a bias)
 *   routing  the top_k experts by sel (descending; equal scores -> lower index),
 *            weights w_k = s_{e_k} / sum_j s_{e_j}
 *   experts  g = Wg[e] x,  u = Wu[e] x,  h = silu(g) * u,  ye = Wd[e] h
 *   shared   ysh = Wd_sh (silu(Wg_sh x) * (Wu_sh x))
 *   output   y[t] = sum_k w_k * ye_k + ysh
 *
 * Sources. The block sum "y = sum_k rw_k (s_e * ye_k) + ysh" with an unweighted
 * shared expert is the engine's MoE sum in "YoungAi - DeepSeek V4.1 Flash on
 * one DGX Spark", section 4.2 ("The objective"); without a sidecar s_e = 1.
 * The bias enters the selection score only and leaves the mixing weights
 * untouched (same page, section 3 and section 4.2, "The router bias").
 * 384 experts with 6 chosen per token: same page, section 2.2. Only routed
 * experts are 2-bit; the shared expert stays 8-bit ("Running DeepSeek V4
 * Flash on an RTX 5080 ...", model list: "up/gate at IQ2_XXS, down at Q2_K",
 * shared experts left untouched; the quant recipe "...-SExpQ8-..." on the
 * txtmix.com ds4 teardown, section 3). Sigmoid scoring with renormalised
 * weights, SwiGLU experts and the exact block formats are part of the layer's
 * workload definition; the pages do not spell them out.
 *
 * Precision of decisions: the expert choice is an integer decided by floating
 * point, so it is taken on the fp32 rounding of the exact selection score, the
 * precision the CUDA kernels decide in. The gap between the k-th and (k+1)-th
 * fp32 selection score is reported so callers can flag near-ties.
 *
 * Storage formats (little-endian):
 *   2-bit block, 84 bytes per 256 consecutive weights of one row:
 *     scales[16] (low nibble = scale sc_j, high nibble = min m_j of sub-block j
 *     of 16 weights), qs[64] (code q_i of weight i at byte i/4, bits 2*(i%4)),
 *     d (binary16), dmin (binary16);   w_i = d * sc_j * q_i - dmin * m_j.
 *   8-bit block, 34 bytes per 32 consecutive weights: d (binary16), 32 int8
 *     codes;   w_i = d * q_i.
 *   Routed gate/up [E][I][H/256] blocks, down [E][H][I/256]; shared gate/up
 *   [I_sh][H/32], shared down [H][I_sh/32]; router fp32 [E][H]; x bf16 [T][H].
 *
 * Optional per-expert down gains (the sidecar and post-training files of
 * "YoungAi - DeepSeek V4.1 Flash on one DGX Spark", sections 3 and 4.2: one
 * multiplicative gain per output channel of each expert's down projection,
 * g_eff = g_base * s_sidecar * s_posttrain, stored as FP4 E2M1 with one scale
 * per 32 channels in 17-byte blocks that encode s - 1):
 *   gain block, 17 bytes per 32 consecutive output channels of one expert:
 *     16 bytes of E2M1 codes (channel i at byte i/2, low nibble first), then the
 *     block scale X as E8M0 (2^(byte - 127));   s_i = 1 + X * e2m1(code_i).
 *   Table [E][H/32] blocks; with gains the output is
 *     y[t] = sum_k w_k * (s1_{e_k} * s2_{e_k}) * ye_k + ysh.
 *
 * MXFP4 routed experts ("Running DeepSeek V4 Flash on an RTX 5080 ...", model
 * list: the MXFP4 GGUF keeps DeepSeek's released MXFP4 routed-expert weights;
 * Blackwell devices run batched expert work with FP4 activations on native FP4
 * matrix instructions, decode uses Q8 activations). Element and scale types are
 * the OCP microscaling ones (E2M1 elements, one E8M0 scale per 32):
 *   MXFP4 block, 17 bytes per 32 consecutive weights of one row: 16 bytes of
 *     E2M1 codes (weight i at byte i/2, low nibble for even i), then the E8M0
 *     scale X;   w_i = X * e2m1(code_i). Routed gate/up [E][I][H/32] blocks,
 *     down [E][H][I/32]; router and shared expert as above.
 *   Activations of each routed-expert matrix product are quantised first:
 *     Q8 (decode): per 32 values, d = amax / 127 and q_i = x_i / d rounded to
 *       the nearest integer (ties to even), in binary32; the product uses d*q_i.
 *     MXFP4 (prefill): per 32 values, the OCP conversion: X = 2^(floor(log2
 *       amax) - 2), element = E2M1 nearest to x_i / X (ties to even, magnitude
 *       saturating at 6); the product uses X*e2m1.
 *   The input x (bf16) is exact in binary32; the SwiGLU output h is rounded to
 *   binary32 (the kernels' precision) before it is quantised.
 *
 * VQ routed experts ("YoungAi - DeepSeek V4.1 Flash on one DGX Spark",
 * section 4.1): every 8 consecutive weights of a row are one codeword of a
 * per-layer codebook (shared by all experts and all three matrices) times one
 * gain per row:  w[r, 8j .. 8j+7] = g_r * C[idx[r, j]].
 *   codebook C: 2^bits x 8 codeword values as OCP FP8 E4M3 bytes (bits = 12
 *     or 13), entry n at bytes 8n .. 8n+7;
 *   index stream of one expert matrix: the rows' indices back to back (row r,
 *     group j at position r * K/8 + j), 12 bits each, packed least significant
 *     bit first (index k at bits 12k .. 12k+11 of the byte string), so every
 *     256 indices fill one 384-byte block;
 *   13-bit layers add a bit plane: bit k (least significant first) is bit 12
 *     of index k;
 *   gains: one binary16 g_r per row.
 *   Matrices [E] streams of rows = I (gate, up; K = H) or H (down; K = I).
 *   Activations are not quantised.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t hidden;       /* H */
    int32_t inter;        /* I, routed intermediate */
    int32_t n_experts;    /* E */
    int32_t top_k;        /* K */
    int32_t shared_inter; /* I_sh, 0 = no shared expert */
} oracle_shape;

enum { Q2_BYTES = 84, Q8_BYTES = 34, GAIN_BYTES = 17, MX4_BYTES = 17 };
enum { ACT_EXACT = 0, ACT_Q8 = 1, ACT_MX4 = 2 };

/* IEEE binary16 -> double: sign, 5-bit exponent (bias 15), 10-bit fraction. */
double oracle_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 -> double: sign, 8-bit exponent (bias 127), 7-bit fraction. */
double oracle_bf16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 255;
    int m = b & 127;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133); /* subnormal: m * 2^-133 */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + m), e - 134); /* (1 + m/128) * 2^(e-127) */
    return sign ? -v : v;
}

static uint16_t le16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* FP4 E2M1 (OCP microscaling element): sign bit 3, exponent bits 2-1 (bias 1),
 * mantissa bit 0; exponent 0 is subnormal (0 or 0.5). */
double oracle_e2m1(uint8_t code)
{
    const int sign = (code >> 3) & 1, ex = (code >> 1) & 3, man = code & 1;
    const double mag = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);
    return sign ? -mag : mag;
}

/* E8M0 block scale: 2^(x - 127); 0xFF is NaN. */
double oracle_e8m0(uint8_t x)
{
    return x == 0xFF ? NAN : ldexp(1.0, (int)x - 127);
}

/* The 32 gains of one 17-byte gain block: s_i = 1 + X * e2m1(code_i). */
void oracle_gain_block(const uint8_t *blk, double *s)
{
    const double X = oracle_e8m0(blk[16]);
    for (int i = 0; i < 32; i++)
        s[i] = 1.0 + X * oracle_e2m1((uint8_t)((blk[i / 2] >> (4 * (i % 2))) & 15));
}

/* One MXFP4 block -> 32 weights: w_i = X * e2m1(code_i). */
void oracle_dequant_mx4(const uint8_t *blk, double *w)
{
    const double X = oracle_e8m0(blk[16]);
    for (int i = 0; i < 32; i++)
        w[i] = X * oracle_e2m1((uint8_t)((blk[i / 2] >> (4 * (i % 2))) & 15));
}

/* One row of k weights in MXFP4 blocks. */
void oracle_dequant_mx4_row(const uint8_t *row, int64_t k, double *w)
{
    for (int64_t b = 0; b < k / 32; b++)
        oracle_dequant_mx4(row + b * MX4_BYTES, w + b * 32);
}

/* Q8 activation blocks: per 32 values d = amax / 127, q_i = nearest integer
 * to x_i / d (ties to even), in binary32 arithmetic; amax = 0 gives d = 0 and
 * q = 0. n is a multiple of 32. */
void oracle_act_q8(const float *x, int64_t n, float *d, int8_t *q)
{
    for (int64_t b = 0; b < n / 32; b++) {
        float amax = 0.0f;
        for (int i = 0; i < 32; i++) {
            const float a = fabsf(x[b * 32 + i]);
            if (a > amax)
                amax = a;
        }
        const float db = amax / 127.0f;
        d[b] = db;
        for (int i = 0; i < 32; i++) {
            const float r = db > 0.0f ? x[b * 32 + i] / db : 0.0f;
            q[b * 32 + i] = (int8_t)nearbyintf(r);
        }
    }
}

/* Nearest E2M1 code to r (ties to the even code, magnitude saturating at 6);
 * the sign bit follows the sign of r. */
uint8_t oracle_e2m1_nearest(double r)
{
    const double a = fabs(r);
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c < 8; c++) {
        const double dist = fabs(a - oracle_e2m1((uint8_t)c));
        if (dist < bd || (dist == bd && c % 2 == 0)) {
            bd = dist;
            best = c;
        }
    }
    return (uint8_t)(best | (signbit(r) ? 8 : 0));
}

/* MXFP4 activation blocks (OCP MX conversion): per 32 values the scale byte
 * of X = 2^(floor(log2 amax) - 2) (clamped to the E8M0 range; amax = 0 gives
 * byte 0) and one E2M1 code per value, the nearest to x_i / X. */
void oracle_act_mx4(const float *x, int64_t n, uint8_t *scale, uint8_t *codes)
{
    for (int64_t b = 0; b < n / 32; b++) {
        double amax = 0.0;
        for (int i = 0; i < 32; i++)
            if (fabs((double)x[b * 32 + i]) > amax)
                amax = fabs((double)x[b * 32 + i]);
        int sb = 0;
        if (amax > 0.0) {
            int e;
            frexp(amax, &e); /* amax = m 2^e, m in [0.5, 1): floor(log2 amax) = e - 1 */
            sb = (e - 1) - 2 + 127;
            sb = sb < 0 ? 0 : sb > 254 ? 254 : sb;
        }
        scale[b] = (uint8_t)sb;
        const double X = oracle_e8m0((uint8_t)sb);
        for (int i = 0; i < 32; i++)
            codes[b * 32 + i] = oracle_e2m1_nearest((double)x[b * 32 + i] / X);
    }
}

/* The values a routed-expert product sees for activations v[n]: v itself
 * (ACT_EXACT), or v rounded to binary32 and quantised (ACT_Q8, ACT_MX4). */
static void quantise_act(int act, const double *v, int64_t n, double *out)
{
    if (act == ACT_EXACT) {
        memcpy(out, v, sizeof(double) * (size_t)n);
        return;
    }
    float *f = (float *)malloc(sizeof(float) * (size_t)n);
    uint8_t *c = (uint8_t *)malloc((size_t)n);
    float *d = (float *)malloc(sizeof(float) * (size_t)(n / 32));
    uint8_t *sc = (uint8_t *)malloc((size_t)(n / 32));
    for (int64_t i = 0; i < n; i++)
        f[i] = (float)v[i];
    if (act == ACT_Q8) {
        oracle_act_q8(f, n, d, (int8_t *)c);
        for (int64_t i = 0; i < n; i++)
            out[i] = (double)d[i / 32] * (double)((int8_t *)c)[i];
    } else {
        oracle_act_mx4(f, n, sc, c);
        for (int64_t i = 0; i < n; i++)
            out[i] = oracle_e8m0(sc[i / 32]) * oracle_e2m1(c[i]);
    }
    free(f);
    free(c);
    free(d);
    free(sc);
}

/* OCP FP8 E4M3: sign bit 7, exponent bits 6-3 (bias 7), mantissa bits 2-0;
 * exponent 0 is subnormal; S.1111.111 is NaN (no infinities). */
double oracle_e4m3(uint8_t b)
{
    const int sign = b >> 7, ex = (b >> 3) & 15, man = b & 7;
    if (ex == 15 && man == 7)
        return NAN;
    const double mag = ex == 0 ? ldexp((double)man, -9) : ldexp(8.0 + man, ex - 10);
    return sign ? -mag : mag;
}

/* Index k of a VQ index stream (12-bit, least significant bit first), with
 * bit 12 from the bit plane when plane is not NULL. */
int32_t oracle_vq_index(const uint8_t *stream, const uint8_t *plane, int64_t k)
{
    int32_t v = 0;
    for (int i = 0; i < 12; i++) {
        const int64_t bit = 12 * k + i;
        v |= ((stream[bit / 8] >> (bit % 8)) & 1) << i;
    }
    if (plane)
        v |= ((plane[k / 8] >> (k % 8)) & 1) << 12;
    return v;
}

/* Row r (k weights) of a VQ matrix: w = g_r * C[idx]. */
void oracle_dequant_vq_row(const uint8_t *codebook, const uint8_t *stream, const uint8_t *plane,
                           const uint16_t *gains, int64_t r, int64_t k, double *w)
{
    const double g = oracle_f16(gains[r]);
    for (int64_t j = 0; j < k / 8; j++) {
        const int32_t n = oracle_vq_index(stream, plane, r * (k / 8) + j);
        for (int i = 0; i < 8; i++)
            w[8 * j + i] = g * oracle_e4m3(codebook[8 * n + i]);
    }
}

/* One 2-bit block -> 256 weights. */
void oracle_dequant_q2(const uint8_t *blk, double *w)
{
    const uint8_t *scales = blk;
    const uint8_t *qs = blk + 16;
    double d = oracle_f16(le16(blk + 80));
    double dmin = oracle_f16(le16(blk + 82));
    for (int i = 0; i < 256; i++) {
        int j = i / 16;
        int sc = scales[j] & 15;
        int m = scales[j] >> 4;
        int q = (qs[i / 4] >> (2 * (i % 4))) & 3;
        w[i] = d * sc * q - dmin * m;
    }
}

/* One 8-bit block -> 32 weights. */
void oracle_dequant_q8(const uint8_t *blk, double *w)
{
    double d = oracle_f16(le16(blk));
    for (int i = 0; i < 32; i++)
        w[i] = d * (double)(int8_t)blk[2 + i];
}

/* A row of k weights stored as k/256 2-bit blocks (or k/32 8-bit blocks). */
void oracle_dequant_q2_row(const uint8_t *row, int64_t k, double *w)
{
    for (int64_t b = 0; b < k / 256; b++)
        oracle_dequant_q2(row + b * Q2_BYTES, w + b * 256);
}

void oracle_dequant_q8_row(const uint8_t *row, int64_t k, double *w)
{
    for (int64_t b = 0; b < k / 32; b++)
        oracle_dequant_q8(row + b * Q8_BYTES, w + b * 32);
}

static double dot(const double *a, const double *b, int64_t n)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; i++)
        acc += a[i] * b[i];
    return acc;
}

/* Threads the oracle uses when not told otherwise. */
int32_t oracle_max_threads(void) { return omp_get_max_threads(); }

double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

double oracle_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* ---- routing ------------------------------------------------------------ */

typedef struct {
    float sel;
    int32_t e;
} scored;

/* Descending selection score, equal scores by ascending expert index. A NaN
 * score is not a number to rank: it sorts after every number (including -inf),
 * NaNs among themselves by index, so a NaN expert is chosen only when fewer
 * than K experts have numeric scores. */
static int by_score_then_index(const void *pa, const void *pb)
{
    const scored *a = (const scored *)pa, *b = (const scored *)pb;
    const int a_nan = a->sel != a->sel, b_nan = b->sel != b->sel;
    if (a_nan != b_nan) return a_nan - b_nan;
    if (!a_nan) {
        if (a->sel > b->sel) return -1;
        if (a->sel < b->sel) return 1;
    }
    return (a->e > b->e) - (a->e < b->e);
}

/* Exact logits L[T][E] = x Wr^T (bf16 x, fp32 Wr, binary64 sums). */
int oracle_logits(const oracle_shape *s, const float *router_w, const uint16_t *x, int32_t T, double *logits)
{
    const int H = s->hidden, E = s->n_experts;
    if (H <= 0 || E <= 0 || T < 0)
        return -1;
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < T; t++) {
        double *xt = (double *)malloc(sizeof(double) * H);
        for (int h = 0; h < H; h++)
            xt[h] = oracle_bf16(x[(int64_t)t * H + h]);
        for (int e = 0; e < E; e++) {
            double L = 0.0;
            for (int h = 0; h < H; h++)
                L += xt[h] * (double)router_w[(int64_t)e * H + h];
            logits[(int64_t)t * E + e] = L;
        }
        free(xt);
    }
    return 0;
}

/*
 * Selection from exact logits. Outputs (any may be NULL except idx):
 *   idx[T][K]     chosen experts in descending selection score
 *   weights[T][K] renormalised sigmoid scores of the chosen experts
 *   gap[T]        fp32 score of the K-th minus the (K+1)-th choice (+inf if K == E)
 *   sel[T][E]     fp32 selection scores the decision was taken on
 */
int oracle_select(const oracle_shape *s, const double *logits, const float *router_bias, int32_t T,
                  int32_t *idx, double *weights, double *gap, float *sel_out)
{
    const int E = s->n_experts, K = s->top_k;
    if (E <= 0 || K <= 0 || K > E || T < 0)
        return -1;
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < T; t++) {
        double *score = (double *)malloc(sizeof(double) * E);
        scored *order = (scored *)malloc(sizeof(scored) * E);
        for (int e = 0; e < E; e++) {
            score[e] = oracle_sigmoid(logits[(int64_t)t * E + e]);
            double selection = score[e] + (router_bias ? (double)router_bias[e] : 0.0);
            order[e].sel = (float)selection;
            order[e].e = e;
            if (sel_out)
                sel_out[(int64_t)t * E + e] = order[e].sel;
        }
        qsort(order, (size_t)E, sizeof(scored), by_score_then_index);
        double total = 0.0;
        for (int k = 0; k < K; k++)
            total += score[order[k].e];
        for (int k = 0; k < K; k++) {
            idx[(int64_t)t * K + k] = order[k].e;
            if (weights)
                weights[(int64_t)t * K + k] = total > 0.0 ? score[order[k].e] / total : 1.0 / K;
        }
        if (gap)
            gap[t] = (K < E) ? (double)order[K - 1].sel - (double)order[K].sel : INFINITY;
        free(score);
        free(order);
    }
    return 0;
}

/* Route T tokens: logits, then selection. logits_out may be NULL. */
int oracle_route(const oracle_shape *s, const float *router_w, const float *router_bias,
                 const uint16_t *x, int32_t T, int32_t *idx, double *weights, double *gap,
                 double *logits_out, float *sel_out)
{
    const int E = s->n_experts, K = s->top_k;
    if (s->hidden <= 0 || E <= 0 || K <= 0 || K > E || T < 0)
        return -1;
    double *logits = logits_out ? logits_out : (double *)malloc(sizeof(double) * ((size_t)T * E + 1));
    int rc = oracle_logits(s, router_w, x, T, logits);
    if (rc == 0)
        rc = oracle_select(s, logits, router_bias, T, idx, weights, gap, sel_out);
    if (!logits_out)
        free(logits);
    return rc;
}

/* ---- experts ------------------------------------------------------------ */

/* One routed expert on one token: ye[H] = Wd (silu(Wg x) * (Wu x)).
 * rows_threads > 1 spreads the rows of each product over that many threads;
 * every row is still one thread's sequential dot product, so the result does
 * not depend on it. */
static void expert_q2_rows(const oracle_shape *s, const uint8_t *gate_e, const uint8_t *up_e,
                           const uint8_t *down_e, const double *xt, double *ye, int rows_threads)
{
    const int H = s->hidden, I = s->inter;
    const int64_t gate_row = (int64_t)(H / 256) * Q2_BYTES, down_row = (int64_t)(I / 256) * Q2_BYTES;
    double *h = (double *)malloc(sizeof(double) * I);
#pragma omp parallel num_threads(rows_threads > 1 ? rows_threads : 1) if (rows_threads > 1)
    {
        double *w = (double *)malloc(sizeof(double) * (H > I ? H : I));
#pragma omp for schedule(static)
        for (int i = 0; i < I; i++) {
            oracle_dequant_q2_row(gate_e + i * gate_row, H, w);
            double g = dot(w, xt, H);
            oracle_dequant_q2_row(up_e + i * gate_row, H, w);
            double u = dot(w, xt, H);
            h[i] = oracle_silu(g) * u;
        }
#pragma omp for schedule(static)
        for (int j = 0; j < H; j++) {
            oracle_dequant_q2_row(down_e + j * down_row, I, w);
            ye[j] = dot(w, h, I);
        }
        free(w);
    }
    free(h);
}

void oracle_expert_q2(const oracle_shape *s, const uint8_t *gate_e, const uint8_t *up_e,
                      const uint8_t *down_e, const double *xt, double *ye)
{
    expert_q2_rows(s, gate_e, up_e, down_e, xt, ye, 1);
}

/* The shared expert on one token: ysh[H]. */
/* One MXFP4 routed expert: ye = Wd (silu(Wg a) * (Wu a)) with a the quantised
 * activations of x (act: ACT_Q8 decode, ACT_MX4 prefill, ACT_EXACT none) and
 * the down product on the quantised SwiGLU output. */
static void expert_mx4_rows(const oracle_shape *s, int32_t act, const uint8_t *gate_e, const uint8_t *up_e,
                            const uint8_t *down_e, const double *xt, double *ye, int rows_threads)
{
    const int H = s->hidden, I = s->inter;
    const int64_t gate_row = (int64_t)(H / 32) * MX4_BYTES, down_row = (int64_t)(I / 32) * MX4_BYTES;
    double *a = (double *)malloc(sizeof(double) * H);
    double *h = (double *)malloc(sizeof(double) * I);
    double *hq = (double *)malloc(sizeof(double) * I);
    quantise_act(act, xt, H, a);
#pragma omp parallel num_threads(rows_threads > 1 ? rows_threads : 1) if (rows_threads > 1)
    {
        double *w = (double *)malloc(sizeof(double) * (H > I ? H : I));
#pragma omp for schedule(static)
        for (int i = 0; i < I; i++) {
            oracle_dequant_mx4_row(gate_e + i * gate_row, H, w);
            double g = dot(w, a, H);
            oracle_dequant_mx4_row(up_e + i * gate_row, H, w);
            double u = dot(w, a, H);
            h[i] = oracle_silu(g) * u;
        }
#pragma omp single
        quantise_act(act, h, I, hq);
#pragma omp for schedule(static)
        for (int j = 0; j < H; j++) {
            oracle_dequant_mx4_row(down_e + j * down_row, I, w);
            ye[j] = dot(w, hq, I);
        }
        free(w);
    }
    free(a);
    free(h);
    free(hq);
}

void oracle_expert_mx4(const oracle_shape *s, int32_t act, const uint8_t *gate_e, const uint8_t *up_e,
                       const uint8_t *down_e, const double *xt, double *ye)
{
    expert_mx4_rows(s, act, gate_e, up_e, down_e, xt, ye, 1);
}

/* One VQ matrix of a layer: the expert's index stream, bit plane (13-bit
 * layers; NULL for 12-bit) and row gains are at expert e of these arrays. */
typedef struct {
    const uint8_t *stream; /* [E][rows * K/8 * 12/8] */
    const uint8_t *plane;  /* [E][rows * K/8 / 8] or NULL */
    const uint16_t *gains; /* [E][rows] binary16 */
} oracle_vq_mat;

static void vq_row(const uint8_t *codebook, const oracle_vq_mat *m, int e, int64_t rows, int64_t r, int64_t k,
                   double *w)
{
    const int64_t n = rows * (k / 8);
    oracle_dequant_vq_row(codebook, m->stream + e * (n * 12 / 8), m->plane ? m->plane + e * (n / 8) : NULL,
                          m->gains + e * rows, r, k, w);
}

/* One VQ routed expert e: ye = Wd (silu(Wg x) * (Wu x)). */
static void expert_vq_rows(const oracle_shape *s, const uint8_t *codebook, const oracle_vq_mat *gate,
                           const oracle_vq_mat *up, const oracle_vq_mat *down, int32_t e, const double *xt,
                           double *ye, int rows_threads)
{
    const int H = s->hidden, I = s->inter;
    double *h = (double *)malloc(sizeof(double) * I);
#pragma omp parallel num_threads(rows_threads > 1 ? rows_threads : 1) if (rows_threads > 1)
    {
        double *w = (double *)malloc(sizeof(double) * (H > I ? H : I));
#pragma omp for schedule(static)
        for (int i = 0; i < I; i++) {
            vq_row(codebook, gate, e, I, i, H, w);
            double g = dot(w, xt, H);
            vq_row(codebook, up, e, I, i, H, w);
            double u = dot(w, xt, H);
            h[i] = oracle_silu(g) * u;
        }
#pragma omp for schedule(static)
        for (int j = 0; j < H; j++) {
            vq_row(codebook, down, e, H, j, I, w);
            ye[j] = dot(w, h, I);
        }
        free(w);
    }
    free(h);
}

void oracle_expert_vq(const oracle_shape *s, const uint8_t *codebook, const oracle_vq_mat *gate,
                      const oracle_vq_mat *up, const oracle_vq_mat *down, int32_t e, const double *xt, double *ye)
{
    expert_vq_rows(s, codebook, gate, up, down, e, xt, ye, 1);
}

static void shared_q8_rows(const oracle_shape *s, const uint8_t *sh_gate, const uint8_t *sh_up,
                           const uint8_t *sh_down, const double *xt, double *ysh, int rows_threads)
{
    const int H = s->hidden, I = s->shared_inter;
    const int64_t gate_row = (int64_t)(H / 32) * Q8_BYTES, down_row = (int64_t)(I / 32) * Q8_BYTES;
    double *h = (double *)malloc(sizeof(double) * I);
#pragma omp parallel num_threads(rows_threads > 1 ? rows_threads : 1) if (rows_threads > 1)
    {
        double *w = (double *)malloc(sizeof(double) * (H > I ? H : I));
#pragma omp for schedule(static)
        for (int i = 0; i < I; i++) {
            oracle_dequant_q8_row(sh_gate + i * gate_row, H, w);
            double g = dot(w, xt, H);
            oracle_dequant_q8_row(sh_up + i * gate_row, H, w);
            double u = dot(w, xt, H);
            h[i] = oracle_silu(g) * u;
        }
#pragma omp for schedule(static)
        for (int j = 0; j < H; j++) {
            oracle_dequant_q8_row(sh_down + j * down_row, I, w);
            ysh[j] = dot(w, h, I);
        }
        free(w);
    }
    free(h);
}

/* The shared expert on one token: ysh[H]. */
void oracle_shared_q8(const oracle_shape *s, const uint8_t *sh_gate, const uint8_t *sh_up,
                      const uint8_t *sh_down, const double *xt, double *ysh)
{
    shared_q8_rows(s, sh_gate, sh_up, sh_down, xt, ysh, 1);
}

/*
 * The layer output for given routing: y[T][H] = sum_k weights[t,k] (s1 s2)_{e} ye_{idx[t,k]} + ysh,
 * s1 and s2 the down gains of the gain tables gain1 and gain2 (1 where NULL).
 * ysh is skipped when shared_inter == 0 or the shared pointers are NULL.
 * Tokens are independent and each row is computed by one thread in a fixed
 * order, so the result does not depend on nthreads (<= 0: library default).
 * With at least as many tokens as threads the threads take whole tokens;
 * with fewer, the tokens run one after another and the threads share the
 * rows of each product.
 */
static int forward_routed_any(const oracle_shape *s, int mx4, int32_t act, const uint8_t *codebook,
                              const oracle_vq_mat *vq, const uint8_t *gate, const uint8_t *up, const uint8_t *down, const uint8_t *sh_gate, const uint8_t *sh_up,
                              const uint8_t *sh_down, const uint8_t *gain1, const uint8_t *gain2,
                              const uint16_t *x, int32_t T, const int32_t *idx, const double *weights,
                              double *y, int32_t nthreads)
{
    const int H = s->hidden, I = s->inter, E = s->n_experts, K = s->top_k;
    if (H <= 0 || I <= 0 || H % 256 || I % 256 || K <= 0 || K > E || T < 0)
        return -1;
    if (act < ACT_EXACT || act > ACT_MX4 || (!mx4 && act != ACT_EXACT) || (vq && !codebook))
        return -1;
    const int has_shared = s->shared_inter > 0 && sh_gate && sh_up && sh_down;
    if (has_shared && s->shared_inter % 32)
        return -1;
    for (int64_t p = 0; p < (int64_t)T * K; p++)
        if (idx[p] < 0 || idx[p] >= E)
            return -1;
    const int64_t expert_gate = mx4 ? (int64_t)I * (H / 32) * MX4_BYTES : (int64_t)I * (H / 256) * Q2_BYTES;
    const int64_t expert_down = mx4 ? (int64_t)H * (I / 32) * MX4_BYTES : (int64_t)H * (I / 256) * Q2_BYTES;
    const int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
    const int rows_threads = T < nt ? nt : 1; /* too few tokens to occupy the threads */
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) if (rows_threads == 1)
    for (int32_t t = 0; t < T; t++) {
        double *xt = (double *)malloc(sizeof(double) * H);
        double *ye = (double *)malloc(sizeof(double) * H);
        double *acc = (double *)calloc((size_t)H, sizeof(double));
        for (int h = 0; h < H; h++)
            xt[h] = oracle_bf16(x[(int64_t)t * H + h]);
        for (int k = 0; k < K; k++) {
            int e = idx[(int64_t)t * K + k];
            if (vq)
                expert_vq_rows(s, codebook, &vq[0], &vq[1], &vq[2], e, xt, ye, rows_threads);
            else if (mx4)
                expert_mx4_rows(s, act, gate + e * expert_gate, up + e * expert_gate, down + e * expert_down, xt,
                                ye, rows_threads);
            else
                expert_q2_rows(s, gate + e * expert_gate, up + e * expert_gate, down + e * expert_down, xt, ye,
                               rows_threads);
            double wk = weights[(int64_t)t * K + k];
            for (int j0 = 0; j0 < H; j0 += 32) {
                double s1[32], s2[32];
                for (int i = 0; i < 32; i++)
                    s1[i] = s2[i] = 1.0;
                if (gain1)
                    oracle_gain_block(gain1 + ((int64_t)e * (H / 32) + j0 / 32) * GAIN_BYTES, s1);
                if (gain2)
                    oracle_gain_block(gain2 + ((int64_t)e * (H / 32) + j0 / 32) * GAIN_BYTES, s2);
                for (int i = 0; i < 32; i++)
                    acc[j0 + i] += wk * (s1[i] * s2[i] * ye[j0 + i]);
            }
        }
        if (has_shared) {
            shared_q8_rows(s, sh_gate, sh_up, sh_down, xt, ye, rows_threads);
            for (int j = 0; j < H; j++)
                acc[j] += ye[j];
        }
        memcpy(y + (int64_t)t * H, acc, sizeof(double) * H);
        free(xt);
        free(ye);
        free(acc);
    }
    return 0;
}

int oracle_forward_routed_gain(const oracle_shape *s, const uint8_t *gate, const uint8_t *up,
                               const uint8_t *down, const uint8_t *sh_gate, const uint8_t *sh_up,
                               const uint8_t *sh_down, const uint8_t *gain1, const uint8_t *gain2,
                               const uint16_t *x, int32_t T, const int32_t *idx, const double *weights,
                               double *y, int32_t nthreads)
{
    return forward_routed_any(s, 0, ACT_EXACT, NULL, NULL, gate, up, down, sh_gate, sh_up, sh_down, gain1, gain2, x,
                              T, idx, weights, y, nthreads);
}

/* The layer with MXFP4 routed experts and act-quantised expert activations. */
int oracle_forward_routed_mx4(const oracle_shape *s, int32_t act, const uint8_t *gate, const uint8_t *up,
                              const uint8_t *down, const uint8_t *sh_gate, const uint8_t *sh_up,
                              const uint8_t *sh_down, const uint8_t *gain1, const uint8_t *gain2,
                              const uint16_t *x, int32_t T, const int32_t *idx, const double *weights,
                              double *y, int32_t nthreads)
{
    return forward_routed_any(s, 1, act, NULL, NULL, gate, up, down, sh_gate, sh_up, sh_down, gain1, gain2, x, T, idx,
                              weights, y, nthreads);
}

/* The layer with VQ routed experts (codebook and the three matrices). */
int oracle_forward_routed_vq(const oracle_shape *s, const uint8_t *codebook, const oracle_vq_mat *gate,
                             const oracle_vq_mat *up, const oracle_vq_mat *down, const uint8_t *sh_gate,
                             const uint8_t *sh_up, const uint8_t *sh_down, const uint8_t *gain1,
                             const uint8_t *gain2, const uint16_t *x, int32_t T, const int32_t *idx,
                             const double *weights, double *y, int32_t nthreads)
{
    const oracle_vq_mat vq[3] = {*gate, *up, *down};
    return forward_routed_any(s, 0, ACT_EXACT, codebook, vq, NULL, NULL, NULL, sh_gate, sh_up, sh_down, gain1, gain2,
                              x, T, idx, weights, y, nthreads);
}

/* oracle_forward_routed_gain without down gains. */
int oracle_forward_routed(const oracle_shape *s, const uint8_t *gate, const uint8_t *up,
                          const uint8_t *down, const uint8_t *sh_gate, const uint8_t *sh_up,
                          const uint8_t *sh_down, const uint16_t *x, int32_t T, const int32_t *idx,
                          const double *weights, double *y, int32_t nthreads)
{
    return oracle_forward_routed_gain(s, gate, up, down, sh_gate, sh_up, sh_down, NULL, NULL, x, T, idx, weights,
                                      y, nthreads);
}

/* Route, then compute the layer. idx/weights/gap may be NULL. */
int oracle_forward(const oracle_shape *s, const float *router_w, const float *router_bias,
                   const uint8_t *gate, const uint8_t *up, const uint8_t *down, const uint8_t *sh_gate,
                   const uint8_t *sh_up, const uint8_t *sh_down, const uint16_t *x, int32_t T, double *y,
                   int32_t *idx_out, double *weights_out, double *gap_out, int32_t nthreads)
{
    const int K = s->top_k;
    int32_t *idx = idx_out ? idx_out : (int32_t *)malloc(sizeof(int32_t) * (size_t)T * K + 1);
    double *w = weights_out ? weights_out : (double *)malloc(sizeof(double) * (size_t)T * K + 1);
    int rc = oracle_route(s, router_w, router_bias, x, T, idx, w, gap_out, NULL, NULL);
    if (rc == 0)
        rc = oracle_forward_routed(s, gate, up, down, sh_gate, sh_up, sh_down, x, T, idx, w, y, nthreads);
    if (!idx_out) free(idx);
    if (!weights_out) free(w);
    return rc;
}
