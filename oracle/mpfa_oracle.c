/*
 * mpfa_oracle.c -- plain CPU oracle for the MpFA QK4PV8 attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Sources (cited by page title and section):
 *  [MpFA]  "MpFA: Hardware-Efficient Train-Free QK4V8 FlashAttention Kernels on
 *          Blackwell GPUs", abstract: QK in NVFP4, P and V in FP8 ("QK4PV8"),
 *          rank-one smoothing compensation issued as one extra MMA, adaptive
 *          partitioning across prefill and decode.
 *  [FMT]   "FlashAttention压到4位" explainer, section "FP4 只有约 15 个可表示的数":
 *          E2M1 = 1 sign, 2 exponent, 1 mantissa bit, magnitudes
 *          {0, 1/2, 1, 3/2, 2, 3, 4, 6}, x = q*s; NVFP4 = blocks of 16 with an
 *          FP8 E4M3 scale plus a per-tensor FP32 second-level scale.
 *  [FA2]   same explainer, section "注意力慢在哪儿": FlashAttention-2 tiling with
 *          an online softmax (running max m, running sum l, rescale of the
 *          output) that equals the full softmax exactly.
 *  [SHR]   same explainer, section "Direct-P 的绕行方案": the softmax
 *          denominator must consume the same rounded P codes as the PV product.
 *  [BLOG]  "Blackwell免训练4-bit注意力MpFA" blog, section 2.1:
 *          S = QK^T / sqrt(d), P = softmax(S), O = PV.
 *
 * Where the pages leave a step open, this file implements one stated reading;
 * every such reading is listed in the repository's design notes:
 *  - E2M1 / E4M3 rounding is round-to-nearest, ties to the even code,
 *    saturating at the largest finite magnitude (6 / 448); the sign bit
 *    follows the input, so a negative value that rounds to zero keeps its sign.
 *  - NVFP4 tensor scale s = fp32(amax / (6 * 448)), 1 when amax == 0.
 *    Block scale sb = E4M3(fp32(bamax / fp32(6 * s))); code = E2M1(fp32(x / fp32(sb * s))).
 *  - V: s_v = fp32(amax / 448), code = E4M3(fp32(v / s_v)).
 *  - Compensation (rank-one smoothing): per query block, qbar = fp32 mean of
 *    the block's rows; Q' = fp32(Q - qbar); Q' and qbar are quantized to
 *    NVFP4 with one shared tensor scale; the score is
 *    S = s_q s_k (deq(Q')deq(K)^T + 1 deq(qbar) deq(K)^T).
 *  - P is stored as E4M3(2^s p) with p = 2^(t - m) and s = 4, where m is the
 *    reference max of the row: set by the first tile and moved to a tile's
 *    max only when that max exceeds m by more than tau = 4 (log2 units), so
 *    p <= 2^tau and 2^s p <= 256 stays in E4M3 range.  The running sum adds
 *    the decoded rounded codes [SHR]; KV tiles of 128 keys are visited in
 *    ascending order; the output is s_v acc / l, LSE = ln2 (m + log2(l) - s).
 *
 * Build: plain C11, no fast-math, no FP contraction (gcc -O2 -std=c11
 * -ffp-contract=off), so every float operation below rounds once, as written.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* E2M1 value of a 4-bit code: bit 3 sign, bits 2..1 exponent (bias 1),
 * bit 0 mantissa; exponent 0 is subnormal (m * 0.5).  [FMT] */
double orc_e2m1_value(int code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* Nearest E2M1 code to y: argmin over the 8 magnitude codes, ties to the
 * code whose mantissa bit is 0, saturating at 6 (the nearest magnitude to any
 * |y| > 6 is 6).  The sign bit copies the sign of y. */
int orc_e2m1_encode(double y)
{
    double a = fabs(y);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c < 8; c++) {
        double d = fabs(a - orc_e2m1_value(c));
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return best | (signbit(y) ? 8 : 0);
}

/* OCP FP8 E4M3 value: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa; exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN; the
 * largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_value(int code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest finite E4M3 code to y (ties to the even code, saturating at 448).
 * The 127 non-negative finite codes 0x00..0x7E are increasing in value, so
 * a binary search finds the code at or just below |y|; the nearer of it and
 * its successor wins. */
int orc_e4m3_encode(double y)
{
    double a = fabs(y);
    int sign = signbit(y) ? 0x80 : 0;
    if (a >= orc_e4m3_value(0x7E))
        return 0x7E | sign;
    int lo = 0, hi = 0x7E; /* value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (orc_e4m3_value(mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dlo = a - orc_e4m3_value(lo), dhi = orc_e4m3_value(hi) - a;
    int c = (dlo < dhi) ? lo : (dhi < dlo) ? hi : ((lo & 1) == 0 ? lo : hi);
    return c | sign;
}

/* bf16 bits of the value nearest to x (ties to even); x finite. */
uint16_t orc_bf16_round(double x)
{
    if (x == 0.0)
        return signbit(x) ? 0x8000 : 0;
    int sign = signbit(x) ? 1 : 0;
    double a = fabs(x);
    int e;
    frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
    int ex = e - 1;  /* a = 1.xxx * 2^ex */
    if (ex < -126)
        ex = -126;   /* subnormal range: fixed spacing 2^-133 */
    double ulp = ldexp(1.0, ex - 7);
    double q = a / ulp; /* exact: scaling by a power of two */
    double r = floor(q);
    double frac = q - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    double v = r * ulp;
    float vf = (float)v; /* exact: v has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &vf, 4);
    if (v > 3.3895313892515355e38) /* above the largest finite bf16 */
        bits = 0x7F800000u;
    return (uint16_t)((bits >> 16) | (sign ? 0x8000 : 0));
}

/* ------------------------------------------------------------------------ */
/* A tiny pthread parallel-for over [0, n)                                  */
/* ------------------------------------------------------------------------ */

typedef void (*orc_body_fn)(int64_t i, void *ctx);
typedef struct {
    orc_body_fn fn;
    void *ctx;
    int64_t n;
    int tid, nth;
} orc_job;

static void *orc_worker(void *arg)
{
    orc_job *j = (orc_job *)arg;
    for (int64_t i = j->tid; i < j->n; i += j->nth)
        j->fn(i, j->ctx);
    return NULL;
}

static int orc_threads(int requested)
{
    if (requested > 0)
        return requested;
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

static void orc_parallel_for(int64_t n, int nthreads, orc_body_fn fn, void *ctx)
{
    int nth = orc_threads(nthreads);
    if (nth > 256)
        nth = 256;
    if (n < nth)
        nth = (int)(n > 0 ? n : 1);
    pthread_t th[256];
    orc_job jobs[256];
    for (int t = 0; t < nth; t++) {
        jobs[t] = (orc_job){fn, ctx, n, t, nth};
        if (t > 0)
            pthread_create(&th[t], NULL, orc_worker, &jobs[t]);
    }
    orc_worker(&jobs[0]);
    for (int t = 1; t < nth; t++)
        pthread_join(th[t], NULL);
}

int orc_num_threads(int requested) { return orc_threads(requested); }

/* ------------------------------------------------------------------------ */
/* Quantizers                                                                */
/* ------------------------------------------------------------------------ */

/* Per-tensor FP32 scale: fp32(amax / qmax), 1 when amax is 0.  qmax is
 * 6 * 448 = 2688 for NVFP4 (so block scales land in E4M3 range) and 448 for
 * the FP8 V tensor. */
float orc_tensor_scale(float amax, float qmax)
{
    if (amax == 0.0f)
        return 1.0f;
    return amax / qmax;
}

typedef struct {
    const float *x;
    int64_t ld;
    int d;
    float s;
    uint8_t *codes, *scales;
} orc_nvfp4_ctx;

static void orc_nvfp4_row(int64_t r, void *vctx)
{
    orc_nvfp4_ctx *c = (orc_nvfp4_ctx *)vctx;
    const float *x = c->x + r * c->ld;
    int nb = c->d / 16;
    for (int b = 0; b < nb; b++) {
        float bamax = 0.0f;
        for (int i = 0; i < 16; i++) {
            float a = fabsf(x[16 * b + i]);
            if (a > bamax)
                bamax = a;
        }
        float six_s = 6.0f * c->s;
        float t = bamax / six_s;
        int sb = orc_e4m3_encode(t);
        c->scales[r * nb + b] = (uint8_t)sb;
        float denom = (float)orc_e4m3_value(sb) * c->s;
        for (int i = 0; i < 16; i += 2) {
            int lo = 0, hi = 0;
            if (sb != 0) {
                float y0 = x[16 * b + i] / denom;
                float y1 = x[16 * b + i + 1] / denom;
                lo = orc_e2m1_encode(y0);
                hi = orc_e2m1_encode(y1);
            }
            /* two codes per byte, the lower index in the low nibble */
            c->codes[r * (c->d / 2) + (16 * b + i) / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* NVFP4-quantize `rows` rows of d values (row stride ld floats) with tensor
 * scale s: codes [rows][d/2], block scales [rows][d/16] (E4M3 bytes). */
void orc_nvfp4_quantize(const float *x, int64_t rows, int64_t ld, int d, float s,
                        uint8_t *codes, uint8_t *scales, int nthreads)
{
    orc_nvfp4_ctx c = {x, ld, d, s, codes, scales};
    orc_parallel_for(rows, nthreads, orc_nvfp4_row, &c);
}

/* Dequantize NVFP4 rows without the tensor scale: out = code * sb. */
void orc_nvfp4_dequant(const uint8_t *codes, const uint8_t *scales, int64_t rows, int d,
                       double *out)
{
    for (int64_t r = 0; r < rows; r++)
        for (int k = 0; k < d; k++) {
            int byte = codes[r * (d / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            out[r * d + k] = orc_e2m1_value(code) * orc_e4m3_value(scales[r * (d / 16) + k / 16]);
        }
}

/* FP8 E4M3 quantization with a tensor scale: code = E4M3(fp32(x / s)). */
void orc_fp8_quantize(const float *x, int64_t n, float s, uint8_t *codes)
{
    for (int64_t i = 0; i < n; i++) {
        float y = x[i] / s;
        codes[i] = (uint8_t)orc_e4m3_encode(y);
    }
}

void orc_fp8_dequant(const uint8_t *codes, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_e4m3_value(codes[i]);
}

/* Rank-one smoothing inputs for one query block: qbar[c] = fp32 of the mean
 * of x[0..g)[c] (rows with stride ld), and xp = fp32(x - qbar).  The sum runs
 * in fp64 with a Neumaier correction term, so it is exact whenever the
 * correction is zero (always, for bf16 inputs of ordinary range); the mean
 * then rounds once to fp32. */
void orc_block_mean(const float *x, int g, int64_t ld, int d, float *qbar, float *xp)
{
    for (int c = 0; c < d; c++) {
        double s = 0.0, comp = 0.0;
        for (int r = 0; r < g; r++) {
            double v = x[r * ld + c];
            double t = s + v;
            if (fabs(s) >= fabs(v))
                comp += (s - t) + v;
            else
                comp += (v - t) + s;
            s = t;
        }
        qbar[c] = (float)((s + comp) / (double)g);
    }
    if (xp)
        for (int r = 0; r < g; r++)
            for (int c = 0; c < d; c++)
                xp[r * (int64_t)d + c] = x[r * ld + c] - qbar[c];
}

/* ------------------------------------------------------------------------ */
/* Attention                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * Tiled online-softmax attention for query rows `rows` of one head [FA2].
 *
 *   q    [nq][d]   query rows (dequantized codes * block scale, no tensor scale)
 *   qadd [nq][d]   or NULL: the compensation row added to every score,
 *                  S_ij = q_i.k_j + qadd_i.k_j  (qadd_i = the row's qbar)
 *   k, v [nk][d]
 *   t_ij = S_ij * score_scale (log2 domain); masked keys are -inf:
 *        causal: key j > query i;  any: key j >= kv_len.
 *   Keys are split into chunks of `chunk` keys (0: one chunk); each chunk is
 *   visited in tiles of 128 keys in ascending order with its own reference
 *   max m and sum l.  Per tile, with M = max_j t_ij:
 *        m' = M if m = -inf or M > m + tau, else m;  alpha = 2^(m - m')
 *        p_ij = 2^(t_ij - m'), and with x_ij = 2^s p_ij
 *          round_p = 0: P_ij = x_ij
 *          round_p = 1: P_ij = E4M3(x_ij)                (the method: FP8 P)
 *          round_p = 2: P_ij = NVFP4 of x_ij in fp32 (full-FP4 ablation):
 *            per block of 16 keys (key index / 16, so blocks never straddle
 *            a 128-key tile) the quantizer rule with tensor scale
 *            s_p = fp32(2^(s + tau) / 2688), the largest x a tile can
 *            produce mapped to 6 * 448; P_ij = code value * fp32(sb * s_p);
 *            masked keys count as 0
 *        l = alpha l + sum_j P_ij,  acc = alpha acc + sum_j P_ij v_j
 *   (tau = 0 is the FlashAttention-2 running max.)
 *   Chunk result: o_s = out_scale * acc / l, lse_s = ln2 (m + log2(l) - s).
 *   Chunks combine by weights w_s = e^(lse_s - max lse):
 *        o = sum_s w_s o_s / sum_s w_s,  lse = max lse + ln(sum_s w_s).
 *   A row with no visible key gets o = 0, lse = -inf.
 */
typedef struct {
    const double *q, *qadd, *k, *v;
    int64_t nq, nk;
    int d;
    double score_scale, out_scale;
    int causal;
    int64_t kv_len, chunk;
    int round_p;
    double p_shift, tau;
    const int64_t *rows;
    double *o, *lse;
} orc_attn_ctx;

static void orc_attn_row(int64_t ri, void *vctx)
{
    orc_attn_ctx *c = (orc_attn_ctx *)vctx;
    int d = c->d;
    int64_t i = c->rows[ri];
    const double *qi = c->q + i * d;
    const double *qa = c->qadd ? c->qadd + i * d : NULL;
    int64_t nkeys = c->kv_len < c->nk ? c->kv_len : c->nk;
    if (c->causal && i + 1 < nkeys)
        nkeys = i + 1;
    int64_t chunk = c->chunk > 0 ? c->chunk : (nkeys > 0 ? nkeys : 1);
    double *acc = (double *)calloc(d, sizeof(double));
    double *osum = (double *)calloc(d, sizeof(double));
    double t[128];
    int nsplit = 0;
    double lse_max = -INFINITY;
    /* first pass collects each chunk's (o_s, lse_s); kept small: store up to
     * all chunks in a heap array */
    int64_t nchunks = nkeys > 0 ? (nkeys + chunk - 1) / chunk : 0;
    double *os = (double *)calloc((size_t)(nchunks > 0 ? nchunks : 1) * d, sizeof(double));
    double *ls = (double *)calloc((size_t)(nchunks > 0 ? nchunks : 1), sizeof(double));
    for (int64_t cs = 0; cs < nkeys; cs += chunk) {
        int64_t ce = cs + chunk < nkeys ? cs + chunk : nkeys;
        double m = -INFINITY, l = 0.0;
        memset(acc, 0, sizeof(double) * d);
        for (int64_t ts = cs; ts < ce; ts += 128) {
            int64_t te = ts + 128 < ce ? ts + 128 : ce;
            double tmax = -INFINITY;
            for (int64_t j = ts; j < te; j++) {
                const double *kj = c->k + j * d;
                double s = 0.0;
                for (int x = 0; x < d; x++)
                    s += qi[x] * kj[x];
                if (qa)
                    for (int x = 0; x < d; x++)
                        s += qa[x] * kj[x];
                t[j - ts] = s * c->score_scale;
                if (t[j - ts] > tmax)
                    tmax = t[j - ts];
            }
            double mn = (m == -INFINITY || tmax > m + c->tau) ? tmax : m;
            double alpha = (m == -INFINITY) ? 0.0 : exp2(m - mn);
            l *= alpha;
            for (int x = 0; x < d; x++)
                acc[x] *= alpha;
            double pt[128];
            for (int64_t j = ts; j < te; j++) {
                double p = exp2(t[j - ts] - mn + c->p_shift);
                if (c->round_p == 1)
                    p = orc_e4m3_value(orc_e4m3_encode(p));
                pt[j - ts] = p;
            }
            if (c->round_p == 2) {
                /* NVFP4 per 16-key block of the tile, in fp32 */
                const float s_p = (float)(exp2(c->p_shift + c->tau) / 2688.0);
                for (int64_t b0 = ts; b0 < te; b0 += 16) {
                    int64_t b1 = b0 + 16 < te ? b0 + 16 : te;
                    float xb[16], bamax = 0.0f;
                    for (int64_t j = b0; j < b1; j++) {
                        xb[j - b0] = (float)pt[j - ts];
                        if (xb[j - b0] > bamax)
                            bamax = xb[j - b0];
                    }
                    int sb = orc_e4m3_encode((double)(bamax / (6.0f * s_p)));
                    float denom = (float)orc_e4m3_value(sb) * s_p;
                    for (int64_t j = b0; j < b1; j++)
                        pt[j - ts] = sb == 0 ? 0.0
                                             : orc_e2m1_value(orc_e2m1_encode(
                                                   (double)(xb[j - b0] / denom))) *
                                                   (double)denom;
                }
            }
            for (int64_t j = ts; j < te; j++) {
                double p = pt[j - ts];
                l += p;
                const double *vj = c->v + j * d;
                for (int x = 0; x < d; x++)
                    acc[x] += p * vj[x];
            }
            m = mn;
        }
        for (int x = 0; x < d; x++)
            os[nsplit * d + x] = c->out_scale * acc[x] / l;
        ls[nsplit] = M_LN2 * (m + log2(l) - c->p_shift);
        if (ls[nsplit] > lse_max)
            lse_max = ls[nsplit];
        nsplit++;
    }
    double *orow = c->o + ri * d;
    if (nsplit == 0) {
        for (int x = 0; x < d; x++)
            orow[x] = 0.0;
        c->lse[ri] = -INFINITY;
    } else {
        double wsum = 0.0;
        for (int s = 0; s < nsplit; s++) {
            double w = exp(ls[s] - lse_max);
            wsum += w;
            for (int x = 0; x < d; x++)
                osum[x] += w * os[s * d + x];
        }
        for (int x = 0; x < d; x++)
            orow[x] = osum[x] / wsum;
        c->lse[ri] = lse_max + log(wsum);
    }
    free(acc);
    free(osum);
    free(os);
    free(ls);
}

void orc_attn_online(const double *q, const double *qadd, const double *k, const double *v,
                     int64_t nq, int64_t nk, int d, double score_scale, double out_scale,
                     int causal, int64_t kv_len, int64_t chunk, int round_p, double p_shift,
                     double tau, const int64_t *rows, int64_t nrows, double *o, double *lse,
                     int nthreads)
{
    orc_attn_ctx c = {q, qadd, k, v, nq, nk, d, score_scale, out_scale, causal,
                      kv_len, chunk, round_p, p_shift, tau, rows, o, lse};
    orc_parallel_for(nrows, nthreads, orc_attn_row, &c);
}

/*
 * Exact attention in fp64 for query rows `rows` of one head [BLOG 2.1]:
 *   z_ij = (q_i . k_j) * score_scale_nat  over visible keys,
 *   lse_i = log sum_j e^(z_ij),  o_i = sum_j e^(z_ij - lse_i) v_j.
 * Visibility as in orc_attn_online.  No tiling, no quantization.
 */
typedef struct {
    const double *q, *k, *v;
    int64_t nq, nk;
    int d;
    double scale;
    int causal;
    int64_t kv_len;
    const int64_t *rows;
    double *o, *lse;
} orc_exact_ctx;

static void orc_exact_row(int64_t ri, void *vctx)
{
    orc_exact_ctx *c = (orc_exact_ctx *)vctx;
    int d = c->d;
    int64_t i = c->rows[ri];
    int64_t nkeys = c->kv_len < c->nk ? c->kv_len : c->nk;
    if (c->causal && i + 1 < nkeys)
        nkeys = i + 1;
    double *orow = c->o + ri * d;
    for (int x = 0; x < d; x++)
        orow[x] = 0.0;
    if (nkeys <= 0) {
        c->lse[ri] = -INFINITY;
        return;
    }
    double *z = (double *)malloc(sizeof(double) * nkeys);
    double zmax = -INFINITY;
    for (int64_t j = 0; j < nkeys; j++) {
        double s = 0.0;
        for (int x = 0; x < d; x++)
            s += c->q[i * d + x] * c->k[j * d + x];
        z[j] = s * c->scale;
        if (z[j] > zmax)
            zmax = z[j];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < nkeys; j++)
        sum += exp(z[j] - zmax);
    double lse = zmax + log(sum);
    for (int64_t j = 0; j < nkeys; j++) {
        double w = exp(z[j] - lse);
        for (int x = 0; x < d; x++)
            orow[x] += w * c->v[j * d + x];
    }
    c->lse[ri] = lse;
    free(z);
}

void orc_attn_exact(const double *q, const double *k, const double *v, int64_t nq, int64_t nk,
                    int d, double scale, int causal, int64_t kv_len, const int64_t *rows,
                    int64_t nrows, double *o, double *lse, int nthreads)
{
    orc_exact_ctx c = {q, k, v, nq, nk, d, scale, causal, kv_len, rows, o, lse};
    orc_parallel_for(nrows, nthreads, orc_exact_row, &c);
}

/* orc_block_mean over nblocks consecutive blocks of g rows (row stride ld):
 * block b starts at row b*g; qbar [nblocks][d], xp [nblocks*g][d] (or NULL). */
typedef struct {
    const float *x;
    int g;
    int64_t ld;
    int d;
    float *qbar, *xp;
} orc_mean_ctx;

static void orc_mean_block(int64_t b, void *vctx)
{
    orc_mean_ctx *c = (orc_mean_ctx *)vctx;
    orc_block_mean(c->x + b * c->g * c->ld, c->g, c->ld, c->d, c->qbar + b * c->d,
                   c->xp ? c->xp + b * c->g * (int64_t)c->d : NULL);
}

void orc_block_means(const float *x, int64_t nblocks, int g, int64_t ld, int d, float *qbar,
                     float *xp, int nthreads)
{
    orc_mean_ctx c = {x, g, ld, d, qbar, xp};
    orc_parallel_for(nblocks, nthreads, orc_mean_block, &c);
}

/* Vectorised helpers for tests: encode / decode arrays. */
void orc_e2m1_encode_array(const double *y, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = (uint8_t)orc_e2m1_encode(y[i]);
}

void orc_e4m3_encode_array(const double *y, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = (uint8_t)orc_e4m3_encode(y[i]);
}

void orc_bf16_round_array(const double *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_bf16_round(x[i]);
}
