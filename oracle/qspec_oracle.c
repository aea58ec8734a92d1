/*
 * qspec_oracle.c -- plain, slow CPU oracle for the QSPEC hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant generator
 * with the CUDA library; both are written separately from the same reading of
 * the pages.
 *
 * Sources (page title, section, equation):
 *   [QS-bg]   "QSPEC: Speculative Decoding with Complementary Quantization
 *             Schemes" summary (molayo1419.me), background terms: W4A16,
 *             W4A4, INT32 accumulation, dequantisation W^ = s(W_INT4 - z),
 *             speculative sampling a(x) = min(1, p/q), greedy acceptance,
 *             first-rejection cutoff, correction/bonus token, E[A], E[L].
 *   [QS-design] same page, "QSPEC structure": W4A4 draft, W4A16 verify on
 *             T<=i ++ T^_{i+1:i+gamma} giving gamma+1 distributions, one
 *             shared 4-bit weight set, KV overwrite for accepted tokens.
 *   [SK]      "SpecKV: compression-aware gamma selection" blog, architecture
 *             section: the controller's draft features, confidence (largest
 *             probability) and entropy -sum p log(p + 1e-9).
 *
 * Where the pages are silent the readings below are taken (each one is also
 * listed in the design notes of the repository):
 *   - weights: codes 0..15, group of 128 along K per output channel n,
 *     fp16 scale s and fp16 zero point z, z an integer 0..15;
 *   - packing: byte j of row n = code[2j] | code[2j+1] << 4;
 *     sz word = fp16 bits of s | fp16 bits of z << 16;
 *   - activations: symmetric INT4 per token and group of 128,
 *     sx = amax / 7 in fp32, q = rint(x / sx) clamped to [-7, 7], q = 0 when
 *     sx == 0, group sum qs = sum q; nibble = two's complement, same order;
 *   - W4A4: I_g = sum_{k in g} q (W - z) exactly (integer), then
 *     acc = fmaf((float) I_g, sx[m][g] * s[n][g], acc) for g ascending from
 *     acc = 0, y = bf16 round-to-nearest-even(acc);
 *   - W4A16: fp64 reference sum_k x * s * (W - z);
 *   - softmax in fixed point: E_v = rint(qexp(l_v - max) * 2^32), S = sum E;
 *   - acceptance: U * Eq_t * Sp < 2^24 * Ep_t * Sq with U a 24-bit uniform;
 *   - residual: R_v = max(0, Ep_v * Sq - Eq_v * Sp); if sum R == 0 the
 *     target row itself is used;
 *   - sampling from integer weights w: T = floor(U' * sum w / 2^24),
 *     v* = min { v : sum_{u<=v} w_u > T };
 *   - random numbers: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11),
 *     key = (seed lo, seed hi), counter = (slot, b, round lo, round hi),
 *     U = word0 >> 8; slot i-1 for the test at draft position i, slot gamma
 *     for the correction / bonus draw, slot 16 + i for drawing the draft
 *     token at position i (1 <= i <= 16) from the draft distribution;
 *   - draft statistics: confidence = largest fixed-point probability,
 *     (float)((double) max_v E_v / (double) S); entropy = -sum_v p_v
 *     log(p_v + 1e-9) with p_v = E_v / S, in fp64.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared
 * -fPIC.  fp-contract must stay off: every fused multiply-add below is an
 * explicit fmaf and every other operation is rounded on its own.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef unsigned __int128 u128;

/* status values returned by the oracle (same meaning as the library's) */
enum {
    ORC_OK = 0,
    ORC_ERR_RANGE = 6,
    ORC_ERR_ZERO_POINT = 7,
    ORC_ERR_NONFINITE = 8
};

#define GROUP 128

/* threads an OpenMP region of the oracle uses */
int orc_num_threads(void) { return omp_get_max_threads(); }

/* ------------------------------------------------------------------ */
/* number formats                                                       */
/* ------------------------------------------------------------------ */

/* IEEE binary16 -> double, written out from the format definition. */
static double fp16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-14 / 2^10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + (double)f, e - 25);   /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

static float bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* float -> bfloat16, round to nearest, ties to even. */
static uint16_t bf16_round(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x40);     /* keep NaN a quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* a1: weight pack                                                      */
/* ------------------------------------------------------------------ */

int orc_pack_weights(const uint8_t *codes, const uint16_t *s, const uint16_t *z,
                     int N, int K, uint8_t *packed, uint32_t *sz)
{
    int G = K / GROUP, st = ORC_OK;
    for (int n = 0; n < N; n++) {
        for (int j = 0; j < K / 2; j++) {
            uint8_t lo = codes[(size_t)n * K + 2 * j];
            uint8_t hi = codes[(size_t)n * K + 2 * j + 1];
            if (lo > 15 || hi > 15)
                st = st ? st : ORC_ERR_RANGE;
            packed[(size_t)n * (K / 2) + j] = (uint8_t)((lo & 15) | ((hi & 15) << 4));
        }
        for (int g = 0; g < G; g++) {
            uint16_t sb = s[(size_t)n * G + g], zb = z[(size_t)n * G + g];
            double sv = fp16_value(sb), zv = fp16_value(zb);
            if (!isfinite(sv))
                st = st ? st : ORC_ERR_NONFINITE;
            if (!(zv >= 0.0 && zv <= 15.0 && zv == floor(zv)))
                st = st ? st : ORC_ERR_ZERO_POINT;
            sz[(size_t)n * G + g] = (uint32_t)sb | ((uint32_t)zb << 16);
        }
    }
    return st;
}

/* ------------------------------------------------------------------ */
/* a2: activation quantiser, symmetric INT4 per token and group          */
/* ------------------------------------------------------------------ */

int orc_quant_act_int4(const uint16_t *x, int M, int K, int ldx,
                       uint8_t *xq, float *sx, int32_t *qs)
{
    int G = K / GROUP, st = ORC_OK;
    for (int m = 0; m < M; m++) {
        for (int g = 0; g < G; g++) {
            const uint16_t *row = x + (size_t)m * ldx + (size_t)g * GROUP;
            float amax = 0.0f;
            for (int k = 0; k < GROUP; k++) {
                float v = bf16_value(row[k]);
                if (!isfinite(v))
                    st = st ? st : ORC_ERR_NONFINITE;
                float a = fabsf(v);
                if (a > amax)
                    amax = a;
            }
            float scale = amax / 7.0f;
            int32_t sum = 0;
            int q[GROUP];
            for (int k = 0; k < GROUP; k++) {
                int v = 0;
                if (scale != 0.0f) {
                    float r = nearbyintf(bf16_value(row[k]) / scale);
                    if (r > 7.0f) r = 7.0f;
                    if (r < -7.0f) r = -7.0f;
                    v = (int)r;
                }
                q[k] = v;
                sum += v;
            }
            for (int k = 0; k < GROUP; k += 2)
                xq[(size_t)m * (K / 2) + (size_t)g * (GROUP / 2) + k / 2] =
                    (uint8_t)((q[k] & 15) | ((q[k + 1] & 15) << 4));
            sx[(size_t)m * G + g] = scale;
            qs[(size_t)m * G + g] = sum;
        }
    }
    return st;
}

/* ------------------------------------------------------------------ */
/* shared unpacking of the formats above (oracle-private)               */
/* ------------------------------------------------------------------ */

static int weight_code(const uint8_t *packed, int K, int n, int k)
{
    uint8_t b = packed[(size_t)n * (K / 2) + k / 2];
    return (k & 1) ? (b >> 4) : (b & 15);
}

static int act_code(const uint8_t *xq, int K, int m, int k)
{
    uint8_t b = xq[(size_t)m * (K / 2) + k / 2];
    int v = (k & 1) ? (b >> 4) : (b & 15);
    return v >= 8 ? v - 16 : v;                  /* two's complement nibble */
}

/* ------------------------------------------------------------------ */
/* a3: W4A4 linear                                                      */
/* ------------------------------------------------------------------ */

/* fp32 accumulator of output (m, n): the group integers folded in ascending g */
static float w4a4_acc(const uint8_t *xq, const float *sx, const uint8_t *packed,
                      const uint32_t *sz, int N, int K, int m, int n, int32_t *dbg_I)
{
    int G = K / GROUP;
    float acc = 0.0f;
    for (int g = 0; g < G; g++) {
        uint32_t w = sz[(size_t)n * G + g];
        float s = (float)fp16_value((uint16_t)(w & 0xffff));
        int z = (int)fp16_value((uint16_t)(w >> 16));
        int32_t I = 0;
        for (int k = g * GROUP; k < (g + 1) * GROUP; k++)
            I += act_code(xq, K, m, k) * (weight_code(packed, K, n, k) - z);
        if (dbg_I)
            dbg_I[((size_t)m * N + n) * G + g] = I;
        float c = sx[(size_t)m * G + g] * s;
        acc = fmaf((float)I, c, acc);
    }
    return acc;
}

void orc_linear_w4a4(const uint8_t *xq, const float *sx, const uint8_t *packed,
                     const uint32_t *sz, int M, int N, int K,
                     uint16_t *y, int ldy, int32_t *dbg_I, float *dbg_acc)
{
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        for (int m = 0; m < M; m++) {
            float acc = w4a4_acc(xq, sx, packed, sz, N, K, m, n, dbg_I);
            if (dbg_acc)
                dbg_acc[(size_t)m * N + n] = acc;
            y[(size_t)m * ldy + n] = bf16_round(acc);
        }
    }
}

/* W4A4 restricted to a list of (m, n) output elements (same arithmetic) */
void orc_linear_w4a4_points(const uint8_t *xq, const float *sx, const uint8_t *packed,
                            const uint32_t *sz, int N, int K, int P,
                            const int32_t *ms, const int32_t *ns, uint16_t *y)
{
#pragma omp parallel for schedule(static)
    for (int p = 0; p < P; p++)
        y[p] = bf16_round(w4a4_acc(xq, sx, packed, sz, N, K, ms[p], ns[p], NULL));
}

/* ------------------------------------------------------------------ */
/* a4: W4A16 linear, fp64 reference                                     */
/* ------------------------------------------------------------------ */

void orc_linear_w4a16(const uint16_t *x, int ldx, const uint8_t *packed,
                      const uint32_t *sz, int M, int N, int K, double *ref)
{
    int G = K / GROUP;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        for (int m = 0; m < M; m++) {
            double acc = 0.0;
            for (int k = 0; k < K; k++) {
                uint32_t w = sz[(size_t)n * G + k / GROUP];
                double s = fp16_value((uint16_t)(w & 0xffff));
                double z = fp16_value((uint16_t)(w >> 16));
                double what = s * ((double)weight_code(packed, K, n, k) - z);
                acc += (double)bf16_value(x[(size_t)m * ldx + k]) * what;
            }
            ref[(size_t)m * N + n] = acc;
        }
    }
}

/* same, restricted to a list of (m, n) output elements */
void orc_linear_w4a16_points(const uint16_t *x, int ldx, const uint8_t *packed,
                             const uint32_t *sz, int N, int K, int P,
                             const int32_t *ms, const int32_t *ns, double *ref)
{
    int G = K / GROUP;
    (void)N;
#pragma omp parallel for schedule(static)
    for (int p = 0; p < P; p++) {
        int m = ms[p], n = ns[p];
        double acc = 0.0;
        for (int k = 0; k < K; k++) {
            uint32_t w = sz[(size_t)n * G + k / GROUP];
            double s = fp16_value((uint16_t)(w & 0xffff));
            double z = fp16_value((uint16_t)(w >> 16));
            acc += (double)bf16_value(x[(size_t)m * ldx + k]) *
                   (s * ((double)weight_code(packed, K, n, k) - z));
        }
        ref[p] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* random numbers: Philox4x32-10 (Salmon et al., SC'11)                 */
/* ------------------------------------------------------------------ */

void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; r++) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* 24-bit uniform for (slot, sequence b) of a verification round */
uint32_t orc_uniform24(uint64_t seed, uint64_t round, uint32_t slot, uint32_t b)
{
    uint32_t ctr[4] = {slot, b, (uint32_t)round, (uint32_t)(round >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return out[0] >> 8;
}

/* ------------------------------------------------------------------ */
/* fixed-point softmax weights                                          */
/* ------------------------------------------------------------------ */

/*
 * qexp(x), x <= 0: Cody-Waite reduction x = n ln2 + r with ln2 split into a
 * 12-significant-bit head and a tail, then the degree-7 Taylor polynomial of
 * e^r in Horner form, then an exact scaling by 2^n.  Every step is one fp32
 * operation rounded to nearest (fmaf where a fused step is written).
 */
float orc_qexp(float x)
{
    const float log2e = 1.44269502925872802734375f;      /* 0x3FB8AA3B, log2(e) rounded */
    const float ln2_hi = 0.693145751953125f;             /* 0x3F317200 */
    const float ln2_lo = 1.428606765330187045037746429443359375e-6f; /* 0x35BFBE8E */
    if (x < -32.0f)
        return 0.0f;
    float n = nearbyintf(x * log2e);
    float r = fmaf(-n, ln2_hi, x);
    r = fmaf(-n, ln2_lo, r);
    float p = 1.0f / 5040.0f;
    p = fmaf(p, r, 1.0f / 720.0f);
    p = fmaf(p, r, 1.0f / 120.0f);
    p = fmaf(p, r, 1.0f / 24.0f);
    p = fmaf(p, r, 1.0f / 6.0f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int e = (int)n;                                      /* -47 <= e <= 0 here */
    uint32_t bits = (uint32_t)(e + 127) << 23;
    float two_e;
    memcpy(&two_e, &bits, 4);
    return p * two_e;
}

/* E = rint(qexp(l - m) * 2^32) as an unsigned 64-bit integer */
static uint64_t fixed_weight(float l, float m)
{
    float e = orc_qexp(l - m);
    return (uint64_t)nearbyintf(e * 4294967296.0f);
}

/* row statistics: max, fixed-point weights, their exact sum.
 * returns ORC_ERR_NONFINITE for a NaN or +inf logit or a row without mass. */
int orc_fixed_softmax_row(const uint16_t *logits, int V, uint64_t *E, uint64_t *S, float *mx)
{
    float m = -INFINITY;
    int st = ORC_OK;
    for (int v = 0; v < V; v++) {
        float l = bf16_value(logits[v]);
        if (isnan(l) || l == INFINITY)
            st = ORC_ERR_NONFINITE;
        if (l > m)
            m = l;
    }
    if (m == -INFINITY)
        st = ORC_ERR_NONFINITE;
    uint64_t sum = 0;
    for (int v = 0; v < V; v++) {
        uint64_t e = 0;
        if (st == ORC_OK)
            e = fixed_weight(bf16_value(logits[v]), m);
        if (E)
            E[v] = e;
        sum += e;
    }
    *S = sum;
    *mx = m;
    return st;
}

/* draw from integer weights w (as u128) with total W > 0 using U (24 bits) */
static int draw_index(const u128 *w, int V, u128 W, uint32_t U)
{
    u128 T = ((u128)U * W) >> 24;
    u128 c = 0;
    for (int v = 0; v < V; v++) {
        c += w[v];
        if (c > T)
            return v;
    }
    return V - 1;   /* not reached: c ends at W > T */
}

/* ------------------------------------------------------------------ */
/* a5: greedy verification                                              */
/* ------------------------------------------------------------------ */

/* status over the whole input: every logit of every row, every draft id */
static int verify_input_status(const uint16_t *P, const uint16_t *Q, const int32_t *draft,
                               int B, int gamma, int V, int sampled)
{
    int st = ORC_OK;
    size_t np = (size_t)B * (gamma + 1) * V, nq = sampled ? (size_t)B * gamma * V : 0;
    for (size_t i = 0; i < np + nq; i++) {
        float l = bf16_value(i < np ? P[i] : Q[i - np]);
        if (isnan(l) || (sampled && l == INFINITY))
            st = ORC_ERR_NONFINITE;
    }
    if (sampled && st == ORC_OK) {
        size_t rows = (size_t)B * (2 * gamma + 1);
        for (size_t r = 0; r < rows; r++) {
            const uint16_t *row = r < (size_t)B * (gamma + 1) ? P + r * V
                                                              : Q + (r - (size_t)B * (gamma + 1)) * V;
            int any = 0;
            for (int v = 0; v < V; v++)
                any |= bf16_value(row[v]) != -INFINITY;
            if (!any)
                st = ORC_ERR_NONFINITE;
        }
    }
    for (size_t i = 0; i < (size_t)B * gamma; i++)
        if (draft[i] < 0 || draft[i] >= V)
            st = st ? st : ORC_ERR_RANGE;
    return st;
}

int orc_verify_greedy(const uint16_t *P, const int32_t *draft, int B, int gamma, int V,
                      int32_t *n_acc, int32_t *out)
{
    int st = verify_input_status(P, NULL, draft, B, gamma, V, 0);
    for (int b = 0; b < B; b++) {
        int arg[64] = {0};
        for (int i = 0; i <= gamma; i++) {
            const uint16_t *row = P + ((size_t)b * (gamma + 1) + i) * V;
            int best = 0;
            float bv = bf16_value(row[0]);
            for (int v = 1; v < V; v++) {
                float l = bf16_value(row[v]);
                if (l > bv) {                         /* strict: lowest index wins ties */
                    bv = l;
                    best = v;
                }
            }
            arg[i] = best;
        }
        int A = gamma;
        for (int i = 0; i < gamma; i++) {
            if (draft[(size_t)b * gamma + i] != arg[i]) {
                A = i;
                break;
            }
        }
        for (int i = 0; i <= gamma; i++)
            out[(size_t)b * (gamma + 1) + i] = i < A ? draft[(size_t)b * gamma + i] : -1;
        out[(size_t)b * (gamma + 1) + A] = arg[A];
        n_acc[b] = A;
    }
    return st;
}

/* ------------------------------------------------------------------ */
/* a6: sampled verification (speculative sampling)                     */
/* ------------------------------------------------------------------ */

int orc_verify_sample(const uint16_t *P, const uint16_t *Q, const int32_t *draft,
                      int B, int gamma, int V, uint64_t seed, uint64_t round,
                      int32_t *n_acc, int32_t *out)
{
    int st = verify_input_status(P, Q, draft, B, gamma, V, 1);
    if (st != ORC_OK)
        return st;                                    /* outputs unspecified */
    uint64_t *Ep = malloc(sizeof(uint64_t) * 2 * (size_t)V), *Eq = Ep + V;
    u128 *w = malloc(sizeof(u128) * (size_t)V);
    for (int b = 0; b < B; b++) {
        uint64_t Sp, Sq;
        float mp, mq;
        int A = gamma;
        for (int i = 0; i < gamma; i++) {
            orc_fixed_softmax_row(P + ((size_t)b * (gamma + 1) + i) * V, V, Ep, &Sp, &mp);
            orc_fixed_softmax_row(Q + ((size_t)b * gamma + i) * V, V, Eq, &Sq, &mq);
            int t = draft[(size_t)b * gamma + i];
            uint32_t U = orc_uniform24(seed, round, (uint32_t)i, (uint32_t)b);
            u128 lhs = (u128)U * Sp * Eq[t];          /* u < p'(t) / q'(t), cross-multiplied */
            u128 rhs = ((u128)Ep[t] * Sq) << 24;
            if (!(lhs < rhs)) {
                A = i;
                break;
            }
        }
        uint32_t U2 = orc_uniform24(seed, round, (uint32_t)gamma, (uint32_t)b);
        orc_fixed_softmax_row(P + ((size_t)b * (gamma + 1) + A) * V, V, Ep, &Sp, &mp);
        u128 W = 0;
        if (A < gamma) {                              /* residual max(0, p' - q') * Sp * Sq */
            orc_fixed_softmax_row(Q + ((size_t)b * gamma + A) * V, V, Eq, &Sq, &mq);
            for (int v = 0; v < V; v++) {
                u128 a = (u128)Ep[v] * Sq, c = (u128)Eq[v] * Sp;
                w[v] = a > c ? a - c : 0;
                W += w[v];
            }
        }
        if (W == 0) {                                 /* bonus draw, or p' == q' */
            for (int v = 0; v < V; v++) {
                w[v] = Ep[v];
                W += Ep[v];
            }
        }
        int vstar = draw_index(w, V, W, U2);
        for (int i = 0; i <= gamma; i++)
            out[(size_t)b * (gamma + 1) + i] = i < A ? draft[(size_t)b * gamma + i] : -1;
        out[(size_t)b * (gamma + 1) + A] = vstar;
        n_acc[b] = A;
    }
    free(Ep);
    free(w);
    return st;
}

/* ------------------------------------------------------------------ */
/* draft-side sampling and the draft statistics                         */
/* ------------------------------------------------------------------ */

/*
 * [QS-bg] the draft model proposes x ~ q(x|h), the distribution the
 * acceptance test divides by.  [SK] "SpecKV: compression-aware gamma
 * selection" blog, architecture section (feature extraction step): the gamma
 * controller reads two statistics of the draft model's softmax over the
 * vocabulary, its confidence (the largest probability) and its entropy,
 * -sum_v p_v log(p_v + 1e-9).  Per row b of Q [B][V]: the fixed-point
 * weights E_v and S of the verification above; the token drawn from E with
 * the uniform of slot 16 + step; confidence and entropy of p_v = E_v / S.
 * Returns ORC_ERR_NONFINITE for a NaN or +inf logit or a row without mass
 * (that row's outputs are then unspecified).
 */
int orc_draft_sample(const uint16_t *Q, int B, int V, uint64_t seed, uint64_t round, int step,
                     int32_t *token, float *confidence, double *entropy)
{
    int st = ORC_OK;
    uint64_t *E = malloc(sizeof(uint64_t) * (size_t)V);
    u128 *w = malloc(sizeof(u128) * (size_t)V);
    for (int b = 0; b < B; b++) {
        uint64_t S;
        float m;
        int rs = orc_fixed_softmax_row(Q + (size_t)b * V, V, E, &S, &m);
        if (rs != ORC_OK) {
            st = rs;
            token[b] = -1;
            confidence[b] = 0.0f;
            entropy[b] = 0.0;
            continue;
        }
        uint64_t Emax = 0;
        u128 W = 0;
        for (int v = 0; v < V; v++) {
            w[v] = E[v];
            W += E[v];
            if (E[v] > Emax)
                Emax = E[v];
        }
        uint32_t U = orc_uniform24(seed, round, (uint32_t)(16 + step), (uint32_t)b);
        token[b] = draw_index(w, V, W, U);
        confidence[b] = (float)((double)Emax / (double)S);
        double h = 0.0;
        for (int v = 0; v < V; v++) {
            double p = (double)E[v] / (double)S;
            h += p * log(p + 1e-9);
        }
        entropy[b] = -h;
    }
    free(E);
    free(w);
    return st;
}

/* ------------------------------------------------------------------ */
/* a7: KV overwrite                                                     */
/* ------------------------------------------------------------------ */

int orc_kv_overwrite(uint16_t *kc, uint16_t *vc, const uint16_t *kn, const uint16_t *vn,
                     const int32_t *base_pos, const int32_t *n_acc,
                     int L, int B, int H, int T, int D, int gamma)
{
    int st = ORC_OK;
    for (int b = 0; b < B; b++) {
        int p0 = base_pos[b], a = n_acc[b];
        if (p0 < 0 || a < 0 || a > gamma || p0 + a >= T) {
            st = st ? st : ORC_ERR_RANGE;
            continue;
        }
        for (int l = 0; l < L; l++)
            for (int r = 0; r <= a; r++)
                for (int h = 0; h < H; h++) {
                    size_t dst = ((((size_t)l * B + b) * H + h) * T + (p0 + r)) * D;
                    size_t src = ((((size_t)l * B + b) * (gamma + 1) + r) * H + h) * D;
                    memcpy(kc + dst, kn + src, (size_t)D * 2);
                    memcpy(vc + dst, vn + src, (size_t)D * 2);
                }
    }
    return st;
}

/* ------------------------------------------------------------------ */
/* next-3: SpecQuant Q8 -- FP8 (E4M3) weights derived from the FP16     */
/* parent, and the FP8 linear of the Q8 (parent / verify) model         */
/* ------------------------------------------------------------------ */
/*
 * [SQ] "SpecQuant: Speculative Decoding with Multi-Parent Quantization for
 * Adaptive LLM Inference" summary (arxiv-wiki), contributions and approach:
 * Q4 (INT4), Q8 (FP8) and Q16 (FP16) variants derived post-training from one
 * FP16 parent with shared base weights; a draft proposes, the chosen parent
 * verifies.  Readings taken (the page names only "FP8"):
 *   - E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
 *     infinities, S.1111.111 is NaN, largest finite 448, subnormals m 2^-9;
 *   - conversion to E4M3: round to nearest, ties to the even code; finite
 *     values beyond 448 in magnitude saturate to +-448;
 *   - weights: per output channel n, s8 = amax_k |W[n][k]| / 448 (fp32, IEEE
 *     division), w8 = E4M3(W / s8) (fp32 quotient, IEEE division); an
 *     all-zero row has s8 = 0 and codes 0;
 *   - activations: the same per token m (bf16 input), scale sa[m];
 *   - linear: y[m][n] = sa[m] s8[n] sum_k E4M3(xq) E4M3(w8), fp64 reference
 *     (the GPU accumulates in fp32, compared within 1e-2 (1 + |ref|)).
 */

/* value of an E4M3 byte, from the format definition */
double orc_e4m3_value(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = (e == 0) ? ldexp((double)m, -9)             /* subnormal: m / 8 * 2^-6 */
                        : ldexp(8.0 + (double)m, e - 10);  /* (1 + m / 8) * 2^(e - 7) */
    return s ? -v : v;
}

/* float -> E4M3: the nearest representable value (ties to the even code),
 * magnitudes of 448 and above saturate to 448, NaN -> 0x7F.  The positive
 * codes 0x00..0x7E are ordered by value, so the neighbours are found by
 * search and compared exactly in fp64. */
uint8_t orc_e4m3_from_float(float f)
{
    if (isnan(f))
        return 0x7F;
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 448.0)
        return sign | 0x7E;
    int lo = 0;
    for (int c = 0; c <= 0x7E; ++c)
        if (orc_e4m3_value((uint8_t)c) <= a)
            lo = c;
    double dl = a - orc_e4m3_value((uint8_t)lo), dh = orc_e4m3_value((uint8_t)(lo + 1)) - a;
    int c = dl < dh ? lo : dh < dl ? lo + 1 : ((lo & 1) ? lo + 1 : lo);
    return sign | (uint8_t)c;
}

void orc_e4m3_from_float_array(const float *f, int n, uint8_t *out)
{
    for (int i = 0; i < n; ++i)
        out[i] = orc_e4m3_from_float(f[i]);
}

/* one row of n values (already as floats): scale amax / 448 and codes */
static int fp8_row(const float *v, int n, uint8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int k = 0; k < n; ++k) {
        if (!isfinite(v[k]))
            return ORC_ERR_NONFINITE;
        float a = fabsf(v[k]);
        if (a > amax)
            amax = a;
    }
    float s = amax / 448.0f;
    *scale = s;
    for (int k = 0; k < n; ++k)
        codes[k] = (s == 0.0f) ? 0 : orc_e4m3_from_float(v[k] / s);
    return ORC_OK;
}

/* Q8 weights from the fp16 parent W16 [N][K] -> w8 [N][K], s8 [N] */
int orc_quant_weights_fp8(const uint16_t *w16, int N, int K, uint8_t *w8, float *s8)
{
    int st = ORC_OK;
#pragma omp parallel for schedule(static) reduction(max : st)
    for (int n = 0; n < N; ++n) {
        float *row = (float *)malloc(sizeof(float) * (size_t)K);
        for (int k = 0; k < K; ++k)
            row[k] = (float)fp16_value(w16[(size_t)n * K + k]);
        int r = fp8_row(row, K, w8 + (size_t)n * K, &s8[n]);
        if (r > st)
            st = r;
        free(row);
    }
    return st;
}

/* per-token E4M3 activations from bf16 x [M][K] -> xq [M][K], sa [M] */
int orc_quant_act_fp8(const uint16_t *x, int M, int K, uint8_t *xq, float *sa)
{
    int st = ORC_OK;
    for (int m = 0; m < M; ++m) {
        float *row = (float *)malloc(sizeof(float) * (size_t)K);
        for (int k = 0; k < K; ++k)
            row[k] = bf16_value(x[(size_t)m * K + k]);
        int r = fp8_row(row, K, xq + (size_t)m * K, &sa[m]);
        if (r > st)
            st = r;
        free(row);
    }
    return st;
}

/* fp64 reference of the FP8 linear: ref[m][n] = sa s8 sum_k xq w8 */
void orc_linear_fp8(const uint8_t *xq, const float *sa, const uint8_t *w8, const float *s8, int M, int N, int K,
                    double *ref)
{
    double lut[256];
    for (int b = 0; b < 256; ++b)
        lut[b] = orc_e4m3_value((uint8_t)b);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += lut[xq[(size_t)m * K + k]] * lut[w8[(size_t)n * K + k]];
            ref[(size_t)m * N + n] = acc * (double)sa[m] * (double)s8[n];
        }
}

/* threads for the oracle's later OpenMP regions (the CPU baseline measures
 * all host cores and one) */
void orc_set_num_threads(int n)
{
    omp_set_num_threads(n > 0 ? n : 1);
}
