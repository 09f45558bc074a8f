/*
 * moe_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU definition of one Mixture-of-Experts layer
 * (route -> plan -> dispatch -> expert FFN -> combine, optionally split into two
 * micro-batches).  It is the yardstick the CUDA library is checked against.  Only
 * the tests, the smoke check and the benchmark's CPU-baseline leg may load it; the
 * library itself never links, loads or calls anything in this directory, and this
 * file includes no header and copies no helper, table or constant generator from
 * the CUDA path.
 *
 * Sources.  The pages this project follows describe the scheduling around an MoE
 * layer, not its arithmetic:
 *   - "[Core/DBO][1/N] Add Dual-Batch Overlap mechanism to VLLM", Purpose: the batch
 *     is split into two micro-batches whose dispatch/combine and expert compute are
 *     interleaved; the layer's result must not depend on that split.
 *   - "[Core/DBO][2/N] Dual-Batch Overlap add DeepEP High Throughput support and
 *     Prefill support", Purpose: one request (one prompt) may be split across the two
 *     micro-batches, i.e. any token split is legal.
 *   - "DeepEP HT: full decode CUDA graphs via worst-token dispatch (whole-step +
 *     graphed TBO)", description and commit messages: per-expert token counts kept
 *     in a device tensor, static worst-case receive shapes ("worst-token" capacity),
 *     the BatchedExperts (per-expert padded) vs Standard (contiguous) activation
 *     formats.
 * Everything the pages leave open (the gate formulas, tie-breaks, FFN shape, the
 * FP8 scale rule, the rounding points) is a stated reading; each reading is marked
 * "reading:" where it is used.
 *
 * Precision: sums and products in double; values are rounded to the storage type
 * (bf16 / fp8 e4m3 / fp32) only at the points where the layer stores them.
 * Build: gcc -O2 -ffp-contract=off (no FMA contraction: the specified exp below
 * must see exactly the fused/unfused operations it names).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_FP8 2

#define ORC_GATE_SOFTMAX 0
#define ORC_GATE_SIGMOID_GROUPED 1
#define ORC_GATE_SQRT_SOFTPLUS 2

#define ORC_OK 0
#define ORC_BAD_INDEX 1
#define ORC_CAPACITY 2

#define QG 128 /* FP8 quantisation group (1x128 activations, 128x128 weights) */

typedef struct {
    int32_t hidden, inter, num_experts, num_shared, top_k;
    int32_t gate, renormalize, n_group, topk_group;
    double routed_scale;
    int32_t dtype; /* ORC_F32 / ORC_BF16 / ORC_FP8 */
} orc_cfg;

/* ------------------------------------------------------------------------- */
/* Number formats                                                            */
/* ------------------------------------------------------------------------- */

/* bfloat16 = the upper 16 bits of an IEEE binary32; round to nearest, ties to
 * even.  Returned widened back to float. */
float orc_bf16_round(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7f800000u) == 0x7f800000u) { /* inf / nan: keep, quiet a nan */
        if (u & 0x007fffffu) u |= 0x00400000u;
        u &= 0xffff0000u;
    } else {
        uint32_t lsb = (u >> 16) & 1u;
        u += 0x7fffu + lsb;
        u &= 0xffff0000u;
    }
    float r;
    memcpy(&r, &u, 4);
    return r;
}

/* OCP 8-bit floating point, E4M3 ("fn" flavour): 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite
 * value 448, subnormal step 2^-9. */
double orc_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round to nearest E4M3, ties to even, saturating to +-448. */
uint8_t orc_e4m3_encode(double v) {
    if (isnan(v)) return 0x7f;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7e;
    if (a < ldexp(1.0, -6)) { /* subnormal range: multiples of 2^-9 */
        double m = nearbyint(ldexp(a, 9)); /* 0..8; 8 is the smallest normal */
        return sign | (uint8_t)m;
    }
    int e2;
    frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1; /* a = (1 + frac) * 2^E, E in [-6, 8] */
    double mant = nearbyint((ldexp(a, -E) - 1.0) * 8.0);
    if (mant >= 8.0) {
        mant = 0.0;
        E += 1;
    }
    if (E > 8) return sign | 0x7e;
    return sign | (uint8_t)(((E + 7) << 3) | (int)mant);
}

/* reading: a 1x128 activation group (or a 128x128 weight block) is scaled by the
 * power of two 2^s with s the smallest integer such that amax <= 448 * 2^s, so
 * that x / 2^s is exact and fits E4M3's range.  amax == 0 gives s = 0. */
int orc_fp8_scale_exp(float amax) {
    if (!(amax > 0.0f)) return 0;
    int e;
    float f = frexpf(amax, &e); /* amax = f * 2^e, f in [0.5, 1); 448 = 0.875 * 2^9 */
    return (f <= 0.875f) ? e - 9 : e - 8;
}

/* ------------------------------------------------------------------------- */
/* reading: the specified exponential and sigmoid used for the grouped-sigmoid */
/* gate's expert SELECTION.  Selection must be identical on every            */
/* implementation, so the value of sigma must be too; it is therefore defined */
/* operation by operation here (Cody and Waite's argument reduction with a    */
/* two-part ln 2, then the degree-7 Taylor polynomial of e^r in Horner form). */
/* Every operation is IEEE binary32 round-to-nearest; fmaf is a fused         */
/* multiply-add; nothing else may be fused.                                   */
/* ------------------------------------------------------------------------- */
static const float SPEC_LOG2E = 0x1.715476p+0f;
static const float SPEC_LN2_HI = 0x1.62e400p-1f;
static const float SPEC_LN2_LO = 0x1.7f7d1cp-20f;
static const float SPEC_C7 = 0x1.a01a02p-13f; /* 1/5040 */
static const float SPEC_C6 = 0x1.6c16c2p-10f; /* 1/720 */
static const float SPEC_C5 = 0x1.111112p-7f;  /* 1/120 */
static const float SPEC_C4 = 0x1.555556p-5f;  /* 1/24 */
static const float SPEC_C3 = 0x1.555556p-3f;  /* 1/6 */
static const float SPEC_C2 = 0x1.000000p-1f;  /* 1/2 */

/* e^x for |x| <= 87 (so that 2^n below stays a normal number). */
float orc_spec_exp(float x) {
    float t = x * SPEC_LOG2E;
    float n = rintf(t); /* nearest integer, ties to even */
    float r = fmaf(-n, SPEC_LN2_HI, x);
    r = fmaf(-n, SPEC_LN2_LO, r);
    float p = SPEC_C7;
    p = fmaf(p, r, SPEC_C6);
    p = fmaf(p, r, SPEC_C5);
    p = fmaf(p, r, SPEC_C4);
    p = fmaf(p, r, SPEC_C3);
    p = fmaf(p, r, SPEC_C2);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    uint32_t bits = (uint32_t)((int)n + 127) << 23; /* 2^n */
    float two_n;
    memcpy(&two_n, &bits, 4);
    return p * two_n;
}

/* sigma(x) = 1 / (1 + e^-x), input clamped to [-80, 80] first. */
float orc_spec_sigmoid(float x) {
    float c = x < -80.0f ? -80.0f : (x > 80.0f ? 80.0f : x);
    float e = orc_spec_exp(-c);
    float d = 1.0f + e;
    return 1.0f / d;
}

/* ------------------------------------------------------------------------- */
/* reading: the specified log1p and sqrt-softplus used by the DeepSeek-V4      */
/* shaped gate's expert SELECTION ("DeepEP HT: full decode CUDA graphs via    */
/* worst-token dispatch", file table and commit messages, name a              */
/* sqrt-softplus top-k op and give no formula).  The score is                 */
/* s(x) = sqrt(softplus(x)), softplus(x) = ln(1 + e^x), written as            */
/* max(x, 0) + log1p(e^-|x|) on x clamped to [-80, 80].  log1p(y), y in       */
/* [0, 1], is the series 2 atanh(z) = 2 (z + z^3/3 + ... + z^15/15) of        */
/* z = y / (2 + y) <= 1/3, in Horner form in z^2 with fused multiply-adds.     */
/* Every operation binary32 round-to-nearest; sqrt is the correctly rounded  */
/* IEEE square root.                                                          */
/* ------------------------------------------------------------------------- */
static const float SPEC_I3 = 0x1.555556p-2f;  /* 1/3 */
static const float SPEC_I5 = 0x1.99999ap-3f;  /* 1/5 */
static const float SPEC_I7 = 0x1.24924ap-3f;  /* 1/7 */
static const float SPEC_I9 = 0x1.c71c72p-4f;  /* 1/9 */
static const float SPEC_I11 = 0x1.745d18p-4f; /* 1/11 */
static const float SPEC_I13 = 0x1.3b13b2p-4f; /* 1/13 */
static const float SPEC_I15 = 0x1.111112p-4f; /* 1/15 */

float orc_spec_log1p(float y) {
    float z = y / (2.0f + y);
    float z2 = z * z;
    float p = SPEC_I15;
    p = fmaf(p, z2, SPEC_I13);
    p = fmaf(p, z2, SPEC_I11);
    p = fmaf(p, z2, SPEC_I9);
    p = fmaf(p, z2, SPEC_I7);
    p = fmaf(p, z2, SPEC_I5);
    p = fmaf(p, z2, SPEC_I3);
    p = fmaf(p, z2, 1.0f);
    return (2.0f * z) * p;
}

float orc_spec_sqrt_softplus(float x) {
    float c = x < -80.0f ? -80.0f : (x > 80.0f ? 80.0f : x);
    float e = orc_spec_exp(-fabsf(c));
    float sp = fmaxf(c, 0.0f) + orc_spec_log1p(e);
    return sqrtf(sp);
}

/* sqrt(softplus(x)) in double (the weights). */
static double sqrt_softplus_d(double x) { return sqrt(x > 30.0 ? x + log1p(exp(-x)) : log1p(exp(x))); }

/* ------------------------------------------------------------------------- */
/* Route                                                                     */
/* ------------------------------------------------------------------------- */

/* reading (softmax gate): the k experts with the largest logits, in descending
 * order, equal logits broken toward the lower expert id.  Weight of a chosen
 * expert = its softmax probability over all E experts; with renormalisation, the
 * softmax over the chosen k logits only (the same thing divided by its sum).
 * Logits are an input: the router projection x.W_g is an ordinary dense GEMM
 * upstream of the layer. */
void orc_route_softmax(int32_t T, int32_t E, int32_t k, int32_t renorm, const float* logits,
                       int32_t* ids, double* w) {
    char* chosen = (char*)malloc((size_t)E);
    for (int32_t t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E;
        memset(chosen, 0, (size_t)E);
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (!chosen[e] && (best < 0 || l[e] > l[best])) best = e;
            chosen[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        double m = -INFINITY;
        for (int32_t e = 0; e < E; ++e) m = fmax(m, (double)l[e]);
        double z = 0.0;
        if (renorm) {
            for (int32_t j = 0; j < k; ++j) z += exp((double)l[ids[(size_t)t * k + j]] - m);
        } else {
            for (int32_t e = 0; e < E; ++e) z += exp((double)l[e] - m);
        }
        for (int32_t j = 0; j < k; ++j)
            w[(size_t)t * k + j] = exp((double)l[ids[(size_t)t * k + j]] - m) / z;
    }
    free(chosen);
}

/* reading (grouped sigmoid gate, DeepSeek-V3 shaped): s_e = sigma(l_e) with the
 * specified sigma; choice score c_e = s_e + bias_e (binary32 add, bias 0 when
 * absent).  The E experts form n_group equal groups of consecutive ids; a group's
 * score is the sum of its two largest choice scores.  The topk_group best groups
 * are kept (equal scores -> lower group id), then the k best experts inside the
 * kept groups by choice score (equal -> lower id), in descending order.  Weight =
 * the plain sigmoid of the chosen logits (no bias), divided by their sum when
 * renormalising, times routed_scale. */
/* reading (DeepSeek-V4 shaped gate): the same group-limited selection with the score
 * s_e = the specified sqrt-softplus of l_e instead of sigma (n_group = 1: plain top-k);
 * weight = sqrt(softplus(l)) of the chosen (no bias), divided by their sum when
 * renormalising, times routed_scale.  sqrt_softplus = 1 selects it. */
static void route_grouped(int32_t T, int32_t E, int32_t k, int32_t n_group, int32_t topk_group, int32_t renorm,
                          double routed_scale, const float* logits, const float* bias, int32_t* ids, double* w,
                          int sqrt_softplus);

void orc_route_sigmoid_grouped(int32_t T, int32_t E, int32_t k, int32_t n_group,
                               int32_t topk_group, int32_t renorm, double routed_scale,
                               const float* logits, const float* bias, int32_t* ids, double* w) {
    route_grouped(T, E, k, n_group, topk_group, renorm, routed_scale, logits, bias, ids, w, 0);
}

void orc_route_sqrt_softplus(int32_t T, int32_t E, int32_t k, int32_t n_group, int32_t topk_group, int32_t renorm,
                             double routed_scale, const float* logits, const float* bias, int32_t* ids, double* w) {
    route_grouped(T, E, k, n_group, topk_group, renorm, routed_scale, logits, bias, ids, w, 1);
}

static void route_grouped(int32_t T, int32_t E, int32_t k, int32_t n_group, int32_t topk_group, int32_t renorm,
                          double routed_scale, const float* logits, const float* bias, int32_t* ids, double* w,
                          int sqrt_softplus) {
    int32_t gsz = E / n_group;
    float* s = (float*)malloc(sizeof(float) * (size_t)E);
    float* c = (float*)malloc(sizeof(float) * (size_t)E);
    float* gs = (float*)malloc(sizeof(float) * (size_t)n_group);
    char* gsel = (char*)malloc((size_t)n_group);
    char* chosen = (char*)malloc((size_t)E);
    for (int32_t t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E;
        for (int32_t e = 0; e < E; ++e) {
            s[e] = sqrt_softplus ? orc_spec_sqrt_softplus(l[e]) : orc_spec_sigmoid(l[e]);
            c[e] = s[e] + (bias ? bias[e] : 0.0f);
        }
        for (int32_t g = 0; g < n_group; ++g) {
            float m1 = -INFINITY, m2 = -INFINITY;
            for (int32_t i = 0; i < gsz; ++i) {
                float v = c[g * gsz + i];
                if (v > m1) {
                    m2 = m1;
                    m1 = v;
                } else if (v > m2) {
                    m2 = v;
                }
            }
            gs[g] = gsz >= 2 ? m1 + m2 : m1;
        }
        memset(gsel, 0, (size_t)n_group);
        for (int32_t j = 0; j < topk_group; ++j) {
            int32_t best = -1;
            for (int32_t g = 0; g < n_group; ++g)
                if (!gsel[g] && (best < 0 || gs[g] > gs[best])) best = g;
            gsel[best] = 1;
        }
        memset(chosen, 0, (size_t)E);
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (gsel[e / gsz] && !chosen[e] && (best < 0 || c[e] > c[best])) best = e;
            chosen[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        double sum = 0.0, sj[32];
        for (int32_t j = 0; j < k; ++j) {
            double x = (double)l[ids[(size_t)t * k + j]];
            sj[j] = sqrt_softplus ? sqrt_softplus_d(x) : 1.0 / (1.0 + exp(-x));
            sum += sj[j];
        }
        for (int32_t j = 0; j < k; ++j) w[(size_t)t * k + j] = (renorm ? sj[j] / sum : sj[j]) * routed_scale;
    }
    free(s);
    free(c);
    free(gs);
    free(gsel);
    free(chosen);
}

void orc_route(const orc_cfg* cfg, int32_t T, const float* logits, const float* bias,
               int32_t* ids, double* w) {
    if (cfg->gate == ORC_GATE_SOFTMAX)
        orc_route_softmax(T, cfg->num_experts, cfg->top_k, cfg->renormalize, logits, ids, w);
    else if (cfg->gate == ORC_GATE_SQRT_SOFTPLUS)
        orc_route_sqrt_softplus(T, cfg->num_experts, cfg->top_k, cfg->n_group, cfg->topk_group, cfg->renormalize,
                                cfg->routed_scale, logits, bias, ids, w);
    else
        orc_route_sigmoid_grouped(T, cfg->num_experts, cfg->top_k, cfg->n_group, cfg->topk_group,
                                  cfg->renormalize, cfg->routed_scale, logits, bias, ids, w);
}

/* reading (hash routing of the DeepSeek-V4 shaped layers; the pages name hash-routing
 * metadata of int32 expert ids passed to the sqrt-softplus top-k op and give no
 * formula): token t's k experts are row token_ids[t] of a fixed table [vocab][k]; the
 * weights are the sqrt-softplus gate's, sqrt(softplus(l)) of those experts divided by
 * their sum when renormalising, times routed_scale.  A token id outside [0, vocab)
 * gives ids -1 and weights 0; a table entry outside [0, E) is passed on (the plan
 * reports it) with weight 0. */
void orc_route_hash(const orc_cfg* cfg, int32_t T, const float* logits, const int32_t* token_ids,
                    const int32_t* table, int32_t vocab, int32_t* ids, double* w) {
    int32_t E = cfg->num_experts, k = cfg->top_k;
    for (int32_t t = 0; t < T; ++t) {
        int32_t tid = token_ids[t];
        double sj[32], sum = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = (tid >= 0 && tid < vocab) ? table[(size_t)tid * k + j] : -1;
            ids[(size_t)t * k + j] = e;
            sj[j] = (e >= 0 && e < E) ? sqrt_softplus_d((double)logits[(size_t)t * E + e]) : 0.0;
            sum += sj[j];
        }
        for (int32_t j = 0; j < k; ++j) {
            double v = (cfg->renormalize && sum > 0.0) ? sj[j] / sum : sj[j];
            w[(size_t)t * k + j] = v * cfg->routed_scale;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Plan: counting sort of the (token, choice) pairs by expert                */
/* ------------------------------------------------------------------------- */

/* Entry (t, j) for j < k is routed expert ids[t][j]; for k <= j < k+S it is shared
 * expert E + (j - k) (every token visits every shared expert, weight 1).
 * Within an expert, rows are ordered by (t, then j) -- a stable counting sort.
 *   exact mode (capacity == 0, the "Standard" contiguous format): expert e owns
 *     rows [offsets[e], offsets[e] + counts[e]); segment starts are aligned up to
 *     `align` rows; offsets[E+S] is the total row count;
 *   capacity mode (capacity C > 0, the "BatchedExperts" / worst-token format):
 *     expert e owns rows [e*C, e*C + C); counts[e] is the number of rows placed;
 *     an entry whose rank is >= C gets slot -1 and the call reports a capacity
 *     overflow (nothing is dropped silently).
 * token_of[row] = the token stored in a row, -1 for padding.  An id outside
 * [0, E) gets slot -1 and reports a bad index.  Returns ORC_OK or the first error
 * found in (t, j) order. */
int32_t orc_plan(int32_t T, int32_t k, int32_t E, int32_t S, const int32_t* ids, int32_t capacity,
                 int32_t align, int32_t* counts, int32_t* offsets, int32_t* slot_of,
                 int32_t* token_of) {
    int32_t NE = E + S, kk = k + S;
    int32_t status = ORC_OK;
    int32_t* fill = (int32_t*)calloc((size_t)NE, sizeof(int32_t));
    memset(counts, 0, sizeof(int32_t) * (size_t)NE);
    for (int32_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < kk; ++j) {
            int32_t e = j < k ? ids[(size_t)t * k + j] : E + (j - k);
            if (j < k && (e < 0 || e >= E)) continue;
            counts[e] += 1;
        }
    offsets[0] = 0;
    for (int32_t e = 0; e < NE; ++e) {
        if (capacity > 0) {
            offsets[e + 1] = (e + 1) * capacity;
        } else {
            int32_t padded = (counts[e] + align - 1) / align * align;
            offsets[e + 1] = offsets[e] + padded;
        }
    }
    if (capacity > 0)
        for (int32_t e = 0; e < NE; ++e)
            if (counts[e] > capacity) counts[e] = capacity;
    for (int32_t r = 0; r < offsets[NE]; ++r) token_of[r] = -1;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < kk; ++j) {
            int32_t e = j < k ? ids[(size_t)t * k + j] : E + (j - k);
            int32_t* out = &slot_of[(size_t)t * kk + j];
            if (j < k && (e < 0 || e >= E)) {
                *out = -1;
                if (status == ORC_OK) status = ORC_BAD_INDEX;
                continue;
            }
            int32_t rank = fill[e]++;
            if (capacity > 0 && rank >= capacity) {
                *out = -1;
                if (status == ORC_OK) status = ORC_CAPACITY;
                continue;
            }
            *out = offsets[e] + rank;
            token_of[*out] = t;
        }
    free(fill);
    return status;
}

/* ------------------------------------------------------------------------- */
/* Dispatch: gather token rows into expert-contiguous rows                   */
/* ------------------------------------------------------------------------- */

/* FP8: quantise one row of n values (n a multiple of 128) group by group. */
void orc_quant_row_fp8(int32_t n, const float* v, uint8_t* q, float* scales) {
    for (int32_t g = 0; g < n / QG; ++g) {
        float amax = 0.0f;
        for (int32_t i = 0; i < QG; ++i) amax = fmaxf(amax, fabsf(v[g * QG + i]));
        int32_t se = orc_fp8_scale_exp(amax);
        for (int32_t i = 0; i < QG; ++i) q[g * QG + i] = orc_e4m3_encode(ldexp((double)v[g * QG + i], -se));
        scales[g] = ldexpf(1.0f, se);
    }
}

/* xe[slot_of[t][j]] = x[t] for every placed entry.  x holds values already
 * representable in the input type (fp32, or bf16 for the bf16 / fp8 layers).
 * FP8 layers store codes in xe_q and one scale per 1x128 group in xe_s; other
 * layers store the values in xe.  Padding rows are left untouched. */
void orc_dispatch(const orc_cfg* cfg, int32_t T, const float* x, const int32_t* slot_of, float* xe,
                  uint8_t* xe_q, float* xe_s) {
    int32_t H = cfg->hidden, kk = cfg->top_k + cfg->num_shared;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < kk; ++j) {
            int32_t r = slot_of[(size_t)t * kk + j];
            if (r < 0) continue;
            if (cfg->dtype == ORC_FP8)
                orc_quant_row_fp8(H, x + (size_t)t * H, xe_q + (size_t)r * H, xe_s + (size_t)r * (H / QG));
            else
                memcpy(xe + (size_t)r * H, x + (size_t)t * H, sizeof(float) * (size_t)H);
        }
}

/* ------------------------------------------------------------------------- */
/* Expert FFN                                                                */
/* ------------------------------------------------------------------------- */

typedef struct {
    const float* w13;
    const uint8_t* w13_q;
    const float* w13_s;
    const float* w2;
    const uint8_t* w2_q;
    const float* w2_s;
} orc_weights;

static double g_e4m3_table[256];
static int g_e4m3_table_ready = 0;
static void e4m3_table_init(void) {
    if (g_e4m3_table_ready) return;
    for (int c = 0; c < 256; ++c) g_e4m3_table[c] = orc_e4m3_decode((uint8_t)c);
    g_e4m3_table_ready = 1;
}

/* Layout (reading): W13 is [E+S][2I][H] with rows 0..I-1 the gate projection and
 * rows I..2I-1 the up projection; W2 is [E+S][H][I]; both K-major (the reduced
 * index is contiguous).  FP8 weights carry one scale per 128x128 block:
 * W13_s[E+S][2I/128][H/128], W2_s[E+S][H/128][I/128]. */
static double w13_at(const orc_cfg* cfg, const orc_weights* W, int32_t e, int32_t n, int32_t kx) {
    int32_t H = cfg->hidden, I2 = 2 * cfg->inter;
    size_t idx = ((size_t)e * I2 + n) * H + kx;
    if (cfg->dtype != ORC_FP8) return (double)W->w13[idx];
    double s = W->w13_s[((size_t)e * (I2 / QG) + n / QG) * (H / QG) + kx / QG];
    return g_e4m3_table[W->w13_q[idx]] * s;
}

static double w2_at(const orc_cfg* cfg, const orc_weights* W, int32_t e, int32_t n, int32_t i) {
    int32_t H = cfg->hidden, I = cfg->inter;
    size_t idx = ((size_t)e * H + n) * I + i;
    if (cfg->dtype != ORC_FP8) return (double)W->w2[idx];
    double s = W->w2_s[((size_t)e * (H / QG) + n / QG) * (I / QG) + i / QG];
    return g_e4m3_table[W->w2_q[idx]] * s;
}

static float round_out(int32_t dtype, double v) {
    float f = (float)v;
    return dtype == ORC_F32 ? f : orc_bf16_round(f);
}

/* One row through expert e (reading: SwiGLU):
 *   g = a . W13[e][0:I]^T,  u = a . W13[e][I:2I]^T,  h = silu(g) * u,
 *   silu(g) = g / (1 + e^-g);
 *   h is stored in the activation type (fp32 / bf16 / fp8 with 1x128 scales);
 *   out = h . W2[e]^T, stored as fp32 (fp32 layer) or bf16. */
static void ffn_row(const orc_cfg* cfg, const orc_weights* W, int32_t e, const double* a, float* out) {
    int32_t H = cfg->hidden, I = cfg->inter;
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    for (int32_t n = 0; n < I; ++n) {
        double g = 0.0, u = 0.0;
        for (int32_t kx = 0; kx < H; ++kx) {
            g += a[kx] * w13_at(cfg, W, e, n, kx);
            u += a[kx] * w13_at(cfg, W, e, I + n, kx);
        }
        h[n] = g / (1.0 + exp(-g)) * u;
    }
    if (cfg->dtype == ORC_FP8) {
        float* hf = (float*)malloc(sizeof(float) * (size_t)I);
        uint8_t* hq = (uint8_t*)malloc((size_t)I);
        float* hs = (float*)malloc(sizeof(float) * (size_t)(I / QG));
        for (int32_t n = 0; n < I; ++n) hf[n] = (float)h[n];
        orc_quant_row_fp8(I, hf, hq, hs);
        for (int32_t n = 0; n < I; ++n) h[n] = g_e4m3_table[hq[n]] * hs[n / QG];
        free(hf);
        free(hq);
        free(hs);
    } else {
        for (int32_t n = 0; n < I; ++n) h[n] = (double)round_out(cfg->dtype, h[n]);
    }
    for (int32_t n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int32_t i = 0; i < I; ++i) acc += h[i] * w2_at(cfg, W, e, n, i);
        out[n] = round_out(cfg->dtype, acc);
    }
    free(h);
}

/* Dequantised dispatched row r. */
static void load_xe_row(const orc_cfg* cfg, int32_t r, const float* xe, const uint8_t* xe_q,
                        const float* xe_s, double* a) {
    int32_t H = cfg->hidden;
    for (int32_t kx = 0; kx < H; ++kx)
        a[kx] = cfg->dtype == ORC_FP8
                    ? g_e4m3_table[xe_q[(size_t)r * H + kx]] * xe_s[(size_t)r * (H / QG) + kx / QG]
                    : (double)xe[(size_t)r * H + kx];
}

/* ye[r] = FFN_e(xe[r]) for every row r of every expert's used range
 * [offsets[e], offsets[e] + counts[e]); other rows of ye are left untouched. */
void orc_expert_ffn(const orc_cfg* cfg, const int32_t* counts, const int32_t* offsets, const float* xe,
                    const uint8_t* xe_q, const float* xe_s, const float* w13, const uint8_t* w13_q,
                    const float* w13_s, const float* w2, const uint8_t* w2_q, const float* w2_s,
                    float* ye) {
    e4m3_table_init();
    orc_weights W = {w13, w13_q, w13_s, w2, w2_q, w2_s};
    int32_t H = cfg->hidden, NE = cfg->num_experts + cfg->num_shared;
    double* a = (double*)malloc(sizeof(double) * (size_t)H);
    for (int32_t e = 0; e < NE; ++e)
        for (int32_t r = offsets[e]; r < offsets[e] + counts[e]; ++r) {
            load_xe_row(cfg, r, xe, xe_q, xe_s, a);
            ffn_row(cfg, &W, e, a, ye + (size_t)r * H);
        }
    free(a);
}

/* ------------------------------------------------------------------------- */
/* Combine                                                                   */
/* ------------------------------------------------------------------------- */

/* y[t] = sum_j w[t][j] * ye[slot_of[t][j]] + sum_s ye[slot_of[t][k+s]], summed in
 * double in (j, then s) order and rounded once to the output type.  Entries with
 * slot -1 contribute nothing. */
/* The same with a residual: y[t] = resid[t] + sum ..., one rounding (resid may be
 * NULL).  This is the combine of a layer inside a stack of layers. */
void orc_combine_resid(const orc_cfg* cfg, int32_t T, const float* ye, const double* w,
                       const int32_t* slot_of, const float* resid, float* y) {
    int32_t H = cfg->hidden, k = cfg->top_k, kk = k + cfg->num_shared;
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t n = 0; n < H; ++n) acc[n] = resid ? (double)resid[(size_t)t * H + n] : 0.0;
        for (int32_t j = 0; j < kk; ++j) {
            int32_t r = slot_of[(size_t)t * kk + j];
            if (r < 0) continue;
            double wj = j < k ? w[(size_t)t * k + j] : 1.0;
            for (int32_t n = 0; n < H; ++n) acc[n] += wj * (double)ye[(size_t)r * H + n];
        }
        for (int32_t n = 0; n < H; ++n) y[(size_t)t * H + n] = round_out(cfg->dtype, acc[n]);
    }
    free(acc);
}

void orc_combine(const orc_cfg* cfg, int32_t T, const float* ye, const double* w,
                 const int32_t* slot_of, float* y) {
    orc_combine_resid(cfg, T, ye, w, slot_of, NULL, y);
}

/* ------------------------------------------------------------------------- */
/* Brute force: one token, no permutation                                    */
/* ------------------------------------------------------------------------- */

/* y_t = sum_j w_t[j] * FFN_{ids_t[j]}(q(x_t)) + sum_s FFN_{E+s}(q(x_t)), with the
 * same quantisation of x_t as dispatch and the same rounding of each expert's
 * output as the FFN.  A per-token loop over the chosen experts, independent of
 * the plan / dispatch / combine permutation. */
void orc_token_output(const orc_cfg* cfg, const float* x_t, const int32_t* ids_t, const double* w_t,
                      const float* w13, const uint8_t* w13_q, const float* w13_s, const float* w2,
                      const uint8_t* w2_q, const float* w2_s, float* y_t) {
    e4m3_table_init();
    orc_weights W = {w13, w13_q, w13_s, w2, w2_q, w2_s};
    int32_t H = cfg->hidden, k = cfg->top_k, S = cfg->num_shared, E = cfg->num_experts;
    double* a = (double*)malloc(sizeof(double) * (size_t)H);
    double* acc = (double*)calloc((size_t)H, sizeof(double));
    float* out = (float*)malloc(sizeof(float) * (size_t)H);
    if (cfg->dtype == ORC_FP8) {
        uint8_t* q = (uint8_t*)malloc((size_t)H);
        float* s = (float*)malloc(sizeof(float) * (size_t)(H / QG));
        orc_quant_row_fp8(H, x_t, q, s);
        for (int32_t kx = 0; kx < H; ++kx) a[kx] = g_e4m3_table[q[kx]] * s[kx / QG];
        free(q);
        free(s);
    } else {
        for (int32_t kx = 0; kx < H; ++kx) a[kx] = (double)x_t[kx];
    }
    for (int32_t j = 0; j < k + S; ++j) {
        int32_t e = j < k ? ids_t[j] : E + (j - k);
        if (e < 0 || e >= E + S) continue;
        double wj = j < k ? w_t[j] : 1.0;
        ffn_row(cfg, &W, e, a, out);
        for (int32_t n = 0; n < H; ++n) acc[n] += wj * (double)out[n];
    }
    for (int32_t n = 0; n < H; ++n) y_t[n] = round_out(cfg->dtype, acc[n]);
    free(a);
    free(acc);
    free(out);
}

/* ------------------------------------------------------------------------- */
/* The layer, optionally as two micro-batches                                */
/* ------------------------------------------------------------------------- */

/* Largest row count a plan can produce for T tokens. */
int64_t orc_max_rows(const orc_cfg* cfg, int32_t T, int32_t capacity, int32_t align) {
    int64_t NE = cfg->num_experts + cfg->num_shared;
    if (capacity > 0) return NE * capacity;
    return (int64_t)T * (cfg->top_k + cfg->num_shared) + NE * (align - 1);
}

/* route -> plan -> dispatch -> FFN -> combine on tokens [t0, t0 + T). */
static int32_t layer_range(const orc_cfg* cfg, int32_t t0, int32_t T, const float* logits,
                           const float* bias, const float* x, const orc_weights* W, int32_t capacity,
                           int32_t align, int32_t* ids, double* w, const float* resid, float* y) {
    int32_t H = cfg->hidden, k = cfg->top_k, E = cfg->num_experts, S = cfg->num_shared;
    int32_t NE = E + S, kk = k + S;
    int32_t cap = capacity;
    orc_route(cfg, T, logits + (size_t)t0 * E, bias, ids + (size_t)t0 * k, w + (size_t)t0 * k);
    int64_t rows = orc_max_rows(cfg, T, cap, align);
    int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * (size_t)NE);
    int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(NE + 1));
    int32_t* slot_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * kk);
    int32_t* token_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)rows);
    int32_t st = orc_plan(T, k, E, S, ids + (size_t)t0 * k, cap, align, counts, offsets, slot_of, token_of);
    float* xe = NULL;
    uint8_t* xe_q = NULL;
    float* xe_s = NULL;
    if (cfg->dtype == ORC_FP8) {
        xe_q = (uint8_t*)malloc((size_t)rows * H);
        xe_s = (float*)malloc(sizeof(float) * (size_t)rows * (H / QG));
    } else {
        xe = (float*)malloc(sizeof(float) * (size_t)rows * H);
    }
    float* ye = (float*)malloc(sizeof(float) * (size_t)rows * H);
    orc_dispatch(cfg, T, x + (size_t)t0 * H, slot_of, xe, xe_q, xe_s);
    orc_expert_ffn(cfg, counts, offsets, xe, xe_q, xe_s, W->w13, W->w13_q, W->w13_s, W->w2, W->w2_q,
                   W->w2_s, ye);
    orc_combine_resid(cfg, T, ye, w + (size_t)t0 * k, slot_of, resid ? resid + (size_t)t0 * H : NULL,
                      y + (size_t)t0 * H);
    free(counts);
    free(offsets);
    free(slot_of);
    free(token_of);
    free(xe);
    free(xe_q);
    free(xe_s);
    free(ye);
    return st;
}

/* The whole layer on T tokens.  split > 0 runs it as two micro-batches, tokens
 * [0, split) and [split, T), each routed, planned, dispatched, computed and
 * combined on its own (reading of the Dual-Batch Overlap pages: the split only
 * reorders work, so every token's output is the unsplit one).  With capacity
 * mode the capacity applies per micro-batch.  Returns the first error status. */
int32_t orc_moe_layer(const orc_cfg* cfg, int32_t T, int32_t split, const float* logits,
                      const float* bias, const float* x, const float* w13, const uint8_t* w13_q,
                      const float* w13_s, const float* w2, const uint8_t* w2_q, const float* w2_s,
                      int32_t capacity, int32_t align, int32_t* ids, double* w, float* y) {
    orc_weights W = {w13, w13_q, w13_s, w2, w2_q, w2_s};
    if (split <= 0 || split >= T)
        return layer_range(cfg, 0, T, logits, bias, x, &W, capacity, align, ids, w, NULL, y);
    int32_t s0 = layer_range(cfg, 0, split, logits, bias, x, &W, capacity, align, ids, w, NULL, y);
    int32_t s1 = layer_range(cfg, split, T - split, logits, bias, x, &W, capacity, align, ids, w, NULL, y);
    return s0 != ORC_OK ? s0 : s1;
}

/* ------------------------------------------------------------------------- */
/* A stack of layers                                                         */
/* ------------------------------------------------------------------------- */

/* The stand-in for a layer's non-MoE compute (reading: the pages overlap dispatch
 * and combine with "the other microbatch's non-MoE compute" -- attention and the
 * like -- whose content is outside this library; a dense projection with a residual
 * stands in for it):  a[t] = x[t] + x[t] . Wa^T,  Wa [H][H] K-major, summed in
 * double, rounded once to the activation storage type. */
void orc_standin(const orc_cfg* cfg, int32_t T, const float* x, const float* wa, float* a) {
    int32_t H = cfg->hidden;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int32_t kx = 0; kx < H; ++kx) acc += (double)x[(size_t)t * H + kx] * (double)wa[(size_t)n * H + kx];
            a[(size_t)t * H + n] = round_out(cfg->dtype, (double)x[(size_t)t * H + n] + acc);
        }
}

/* L layers; layer l:  a = x_l + x_l . Wa_l^T (stand-in),  x_{l+1} = a + MoE_l(a), the
 * MoE part routed by the given logits_l and combined onto the residual a with one
 * rounding.  Weights / logits of layer l are at the given per-layer pointers.  Each
 * layer runs as two micro-batches when split > 0, like the layer above. */
int32_t orc_moe_stack(const orc_cfg* cfg, int32_t L, int32_t T, int32_t split, const float* x0,
                      const float* const* wa, const float* const* logits, const float* bias,
                      const float* const* w13, const uint8_t* const* w13_q, const float* const* w13_s,
                      const float* const* w2, const uint8_t* const* w2_q, const float* const* w2_s,
                      int32_t capacity, int32_t align, float* out) {
    int32_t H = cfg->hidden, k = cfg->top_k;
    size_t n = (size_t)T * H;
    float* x = (float*)malloc(sizeof(float) * n);
    float* a = (float*)malloc(sizeof(float) * n);
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
    double* w = (double*)malloc(sizeof(double) * (size_t)T * k);
    int32_t st = ORC_OK;
    memcpy(x, x0, sizeof(float) * n);
    for (int32_t l = 0; l < L; ++l) {
        orc_weights W = {w13 ? w13[l] : NULL, w13_q ? w13_q[l] : NULL, w13_s ? w13_s[l] : NULL,
                         w2 ? w2[l] : NULL,   w2_q ? w2_q[l] : NULL,   w2_s ? w2_s[l] : NULL};
        orc_standin(cfg, T, x, wa[l], a);
        int32_t r;
        if (split <= 0 || split >= T) {
            r = layer_range(cfg, 0, T, logits[l], bias, a, &W, capacity, align, ids, w, a, x);
        } else {
            r = layer_range(cfg, 0, split, logits[l], bias, a, &W, capacity, align, ids, w, a, x);
            int32_t r1 = layer_range(cfg, split, T - split, logits[l], bias, a, &W, capacity, align, ids, w, a, x);
            if (r == ORC_OK) r = r1;
        }
        if (st == ORC_OK) st = r;
    }
    memcpy(out, x, sizeof(float) * n);
    free(x);
    free(a);
    free(ids);
    free(w);
    return st;
}
