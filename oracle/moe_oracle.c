/*
 * CPU oracle for one mixture-of-experts FFN layer forward.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke entry and the
 * benchmark's CPU-baseline leg may load this library. The product path (the
 * CUDA library and its Python binding) never calls it and shares no code with
 * it.
 *
 * What it computes is the plain definition of the layer, one token at a time,
 * one selected expert at a time, with no blocking, fusion or reordering:
 *
 *   spark_model/layers/moe/forward_prefill.rs, MoeLayer::forward_prefill, the
 *   pipeline in its doc comment: gate -> topK -> sort -> grouped gate/up GEMM
 *   -> SiLU -> grouped down GEMM -> unpermute + weighted reduce -> shared
 *   expert blend.  Grouping and sorting only reorder work, so per token:
 *
 *     L[e]   = sum_h x[h] * Wr[e,h] (+ bias[e])                  (step 1)
 *     ids    = the k largest L, descending, ties to the lower index
 *     w[j]   = softmax over the k selected logits (renormalised)  (step 2)
 *     g[i]   = sum_h x[h] W1[e,i,h];  u[i] = sum_h x[h] W3[e,i,h]
 *     a[i]   = silu(g[i]) * u[i],  silu(g) = g / (1 + exp(-g))   (steps 4-5)
 *     y[o]   = sum_i a[i] W2[e,o,i]                               (step 6)
 *     out    = sum_j w[j] y_j  (+ shared expert, weight 1)        (steps 7-8)
 *
 * with two variants of the same page: the sigmoid + correction-bias router
 * of step 2 (oracle_topk_sigmoid) and the sigmoid-gated shared expert of
 * step 8, out += sigmoid(dot(x, gate)) * shared.
 *
 * The accumulation type is float (the default build) or double (the build
 * with ORACLE_FP64 defined, used to bound the float build's own rounding).
 * Every sum runs in ascending index order.  Routing weights are formed in
 * double and rounded to float in both builds.
 *
 * fp8 weights (e4m3, 128x128 fp32 block scales) and fp8 activations (e4m3,
 * one fp32 scale per token per 128 contiguous elements) follow the block-scaled
 * fp8 layer shape: activation scale s = amax / 448 in float, code =
 * e4m3(round-to-nearest-even, saturating to +-448)(x / s), value = decode(code)
 * * s; an all-zero block takes s = 1 and codes 0.  The e4m3 codec here is
 * written from the format's definition (1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448).
 *
 * NVFP4 weights and activations (the "NVFP4 W4A4 block-scaled MMA MoE" of
 * span-02 gpu_model/forward.rs's module comment; the page names the format
 * and nothing more, so the format's usual definition is taken): each value is
 * an e2m1 code (1 sign, 2 exponent bits with bias 1, 1 mantissa bit: the
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) times an e4m3 scale shared by 16
 * contiguous inputs, times one fp32 scale per tensor.  A weight tensor is one
 * expert's matrix; an activation tensor is one row (a token's x, a pair's h),
 * which keeps tokens independent.  Activation rows are quantised as:
 *   g  = amax(row) / (6 * 448)           (g = 1 for an all-zero row)
 *   sb = e4m3(RNE, saturating)(amax(block) / (6 * g))
 *   code = e2m1(RNE, saturating to +-6)(v / (decode(sb) * g))  (0 when that scale is 0)
 *   value = decode(code) * decode(sb) * g
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifdef ORACLE_FP64
typedef double acc_t;
#define ACC_EXP(v) exp(v)
#else
typedef float acc_t;
#define ACC_EXP(v) expf(v)
#endif

#define EXPORT __attribute__((visibility("default")))

/* ---------------------------------------------------------------- codecs */

/* bf16 bit pattern -> float: the bf16 value is the top half of an IEEE float. */
static float bf16_to_float(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* e4m3 code -> float, from the format definition. */
static float e4m3_decode_one(uint8_t c) {
    int sign = (c >> 7) & 1;
    int expo = (c >> 3) & 0xF;
    int mant = c & 0x7;
    float v;
    if (expo == 0xF && mant == 0x7) {
        v = NAN;
    } else if (expo == 0) {
        v = ldexpf((float)mant, -9); /* subnormal: mant/8 * 2^(1-7) */
    } else {
        v = ldexpf(1.0f + (float)mant / 8.0f, expo - 7);
    }
    return sign ? -v : v;
}

/*
 * float -> e4m3 code, round to nearest, ties to even, saturating to +-448.
 * Exhaustive: the code whose value is nearest; on an exact tie the code with
 * an even mantissa (lowest bit 0).  Searching the 127 non-negative finite codes
 * keeps this obviously correct; speed does not matter here.
 */
static uint8_t e4m3_encode_one(float x) {
    if (isnan(x)) return 0x7F;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)((neg << 7) | 0x7E);
    int best = 0;
    double best_err = a; /* code 0 has value 0 */
    for (int c = 1; c <= 0x7E; ++c) {
        double v = (double)e4m3_decode_one((uint8_t)c);
        double err = fabs(v - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    if (best == 0) return (uint8_t)(neg << 7); /* keep the sign of zero */
    return (uint8_t)((neg << 7) | best);
}

/* decode table, filled from e4m3_decode_one before any parallel region */
static float g_e4m3[256];
static int g_e4m3_ready = 0;
static void e4m3_table_init(void) {
    if (g_e4m3_ready) return;
    for (int c = 0; c < 256; ++c) g_e4m3[c] = e4m3_decode_one((uint8_t)c);
    g_e4m3_ready = 1;
}

EXPORT void oracle_e4m3_decode(const uint8_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_decode_one(in[i]);
}

EXPORT void oracle_e4m3_encode(const float* in, uint8_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode_one(in[i]);
}

/*
 * Per-block activation quantisation, one block = 128 contiguous elements (the
 * last block of a row may be shorter).  v: [n] floats; q: [n] codes;
 * s: [ceil(n/128)] scales.  deq (optional): decode(q) * s.
 */
EXPORT void oracle_act_quant(const float* v, int64_t n, uint8_t* q, float* s, float* deq) {
    for (int64_t b0 = 0; b0 < n; b0 += 128) {
        int64_t b1 = b0 + 128 < n ? b0 + 128 : n;
        float amax = 0.0f;
        for (int64_t i = b0; i < b1; ++i) {
            float a = fabsf(v[i]);
            if (a > amax) amax = a;
        }
        float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        s[b0 / 128] = sc;
        for (int64_t i = b0; i < b1; ++i) {
            q[i] = amax > 0.0f ? e4m3_encode_one(v[i] / sc) : 0;
            if (deq) deq[i] = e4m3_decode_one(q[i]) * sc;
        }
    }
}

/* e2m1 code (low 4 bits) -> float, from the format definition. */
static float e2m1_decode_one(uint8_t c) {
    int sign = (c >> 3) & 1;
    int expo = (c >> 1) & 0x3;
    int mant = c & 0x1;
    float v = expo == 0 ? 0.5f * (float)mant : ldexpf(1.0f + 0.5f * (float)mant, expo - 1);
    return sign ? -v : v;
}

/* float -> e2m1 code, nearest, ties to the even code, saturating to +-6;
 * exhaustive over the 8 magnitudes, like e4m3_encode_one. */
static uint8_t e2m1_encode_one(float x) {
    int neg = signbit(x) ? 1 : 0;
    double a = fabs((double)x);
    if (isnan(x)) return 0;
    if (a >= 6.0) return (uint8_t)((neg << 3) | 0x7);
    int best = 0;
    double best_err = a;
    for (int c = 1; c <= 7; ++c) {
        double err = fabs((double)e2m1_decode_one((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)((neg << 3) | best);
}

EXPORT void oracle_e2m1_decode(const uint8_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = e2m1_decode_one(in[i] & 0xF);
}

EXPORT void oracle_e2m1_encode(const float* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = e2m1_encode_one(in[i]);
}

/* Element i of an NVFP4 vector: two codes per byte, element 2j in the low
 * nibble of byte j. */
static uint8_t nibble_at(const uint8_t* q, int64_t i) {
    uint8_t b = q[i >> 1];
    return (i & 1) ? (uint8_t)(b >> 4) : (uint8_t)(b & 0xF);
}

/*
 * NVFP4 quantisation of one activation row of n elements (n a multiple of 16),
 * per the recipe in the header comment.  q: [n/2] packed codes; sb: [n/16]
 * e4m3 block-scale codes; g: the row's fp32 scale; deq (optional): the values
 * decode(code) * decode(sb) * g.
 */
EXPORT void oracle_nvfp4_quant(const float* v, int64_t n, uint8_t* q, uint8_t* sb, float* g, float* deq) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    const float gs = amax > 0.0f ? amax / 2688.0f : 1.0f;
    *g = gs;
    for (int64_t i = 0; i < n / 2; ++i) q[i] = 0;
    for (int64_t b0 = 0; b0 < n; b0 += 16) {
        float bmax = 0.0f;
        for (int64_t i = b0; i < b0 + 16; ++i) {
            float a = fabsf(v[i]);
            if (a > bmax) bmax = a;
        }
        const float six_g = 6.0f * gs;
        const uint8_t sc = e4m3_encode_one(bmax / six_g);
        sb[b0 / 16] = sc;
        const float scale = e4m3_decode_one(sc) * gs;
        for (int64_t i = b0; i < b0 + 16; ++i) {
            const uint8_t c = scale != 0.0f ? e2m1_encode_one(v[i] / scale) : 0;
            q[i >> 1] |= (uint8_t)((i & 1) ? (c << 4) : c);
            if (deq) deq[i] = e2m1_decode_one(c) * e4m3_decode_one(sc) * gs;
        }
    }
}

/* ---------------------------------------------------------------- routing */

/*
 * Step "1. Gate GEMM" of forward_prefill (and "10. Router gemv" of
 * qwen3_moe/forward_layer.rs): logits[t,e] = sum_h x[t,h] * Wr[e,h] + bias[e].
 * x: [m,H] bf16 bits; Wr: [E,H] float; bias: [E] or NULL; L: [m,E].
 */
EXPORT void oracle_router_logits(const uint16_t* x, int64_t m, int H, const float* Wr,
                                 const float* bias, int E, float* L) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < m; ++t) {
        const uint16_t* xt = x + t * (int64_t)H;
        for (int e = 0; e < E; ++e) {
            const float* we = Wr + (int64_t)e * H;
            acc_t acc = 0;
            for (int h = 0; h < H; ++h) acc += (acc_t)bf16_to_float(xt[h]) * (acc_t)we[h];
            float l = (float)acc;
            if (bias) l = l + bias[e];
            L[t * (int64_t)E + e] = l;
        }
    }
}

/*
 * Step "2. Batched topK dispatch", the softmax branch with norm_topk_prob set:
 * ids = the k largest logits in descending order, equal logits ordered by the
 * lower expert index; w[j] = exp(L[ids[j]] - L[ids[0]]) / sum over the k
 * selected of exp(L[ids[i]] - L[ids[0]]), in double, rounded to float.
 * margin[t] (optional) = L of the k-th pick minus the best unpicked logit
 * (+inf when k == E).
 */
EXPORT void oracle_topk_softmax(const float* L, int64_t m, int E, int k, int32_t* ids, float* w,
                                float* margin) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < m; ++t) {
        const float* lt = L + t * (int64_t)E;
        unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
        int32_t* it = ids + t * (int64_t)k;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || lt[e] > lt[best]) best = e; /* strict: ties keep the lower index */
            }
            taken[best] = 1;
            it[j] = best;
        }
        double l0 = (double)lt[it[0]];
        double den = 0.0;
        for (int j = 0; j < k; ++j) den += exp((double)lt[it[j]] - l0);
        for (int j = 0; j < k; ++j) w[t * (int64_t)k + j] = (float)(exp((double)lt[it[j]] - l0) / den);
        if (margin) {
            if (k >= E) {
                margin[t] = INFINITY;
            } else {
                int best = -1;
                for (int e = 0; e < E; ++e)
                    if (!taken[e] && (best < 0 || lt[e] > lt[best])) best = e;
                margin[t] = lt[it[k - 1]] - lt[best];
            }
        }
        free(taken);
    }
}

/*
 * Step "2. Batched topK dispatch", the sigmoid + correction-bias branch
 * (DeepSeek-V3-style scoring): score s[e] = 1 / (1 + exp(-L[e])); the experts
 * are chosen by s[e] + bias[e] (bias may be NULL), the k largest in
 * descending order with ties to the lower index -- the bias selects experts,
 * the weights gather the pre-bias scores: w[j] = s[ids[j]], divided by their
 * sum when norm is set, then multiplied by scale (routed_scaling_factor).
 * The selection keys are formed in float, the precision the GPU decides in;
 * the weights in double, rounded to float.  margin[t] (optional) = key of the
 * k-th pick minus the best unpicked key (+inf when k == E).
 */
EXPORT void oracle_topk_sigmoid(const float* L, int64_t m, int E, int k, const float* bias, int norm,
                                float scale, int32_t* ids, float* w, float* margin) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < m; ++t) {
        const float* lt = L + t * (int64_t)E;
        float* key = (float*)malloc(sizeof(float) * (size_t)E);
        unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
        for (int e = 0; e < E; ++e) {
            const float sf = 1.0f / (1.0f + expf(-lt[e]));
            key[e] = bias ? sf + bias[e] : sf;
        }
        int32_t* it = ids + t * (int64_t)k;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || key[e] > key[best]) best = e; /* strict: ties keep the lower index */
            }
            taken[best] = 1;
            it[j] = best;
        }
        double sum = 0.0;
        for (int j = 0; j < k; ++j) sum += 1.0 / (1.0 + exp(-(double)lt[it[j]]));
        for (int j = 0; j < k; ++j) {
            double v = 1.0 / (1.0 + exp(-(double)lt[it[j]]));
            if (norm) v /= sum;
            w[t * (int64_t)k + j] = (float)(v * (double)scale);
        }
        if (margin) {
            if (k >= E) {
                margin[t] = INFINITY;
            } else {
                int best = -1;
                for (int e = 0; e < E; ++e)
                    if (!taken[e] && (best < 0 || key[e] > key[best])) best = e;
                margin[t] = key[it[k - 1]] - key[best];
            }
        }
        free(key);
        free(taken);
    }
}

/*
 * Step "3. Sort tokens by expert": a stable counting sort of the pairs
 * p = t*k + j by their expert ids[p].  offsets[E+1] is the exclusive prefix
 * sum of the per-expert counts; sorted_pair[s] is the pair at sorted slot s
 * (pairs ascending within an expert); slot_of_pair[p] is its inverse.
 */
/* Routing weights for a GIVEN selection (the forced-ids mode): the weight
 * half of forward_prefill.rs step "2. Batched topK dispatch" applied to ids
 * chosen elsewhere, e.g. by the GPU where a near-tie let it pick differently.
 * scoring 0 (softmax, renormalised): w_j = exp(L_j - L_max) / sum_i exp(L_i -
 * L_max) over the k given ids, L_max their largest logit; scoring 1 (sigmoid):
 * w_j = sigmoid(L_j), divided by their sum when norm, times scale.  Formed in
 * double and rounded to float, as in oracle_topk_softmax/_sigmoid. */
EXPORT void oracle_route_weights(const float* L, int64_t m, int E, int k, const int32_t* ids, int scoring,
                                 int norm, float scale, float* w) {
    for (int64_t t = 0; t < m; ++t) {
        const float* lt = L + t * (int64_t)E;
        const int32_t* it = ids + t * (int64_t)k;
        if (scoring == 0) {
            double lmax = (double)lt[it[0]];
            for (int j = 1; j < k; ++j)
                if ((double)lt[it[j]] > lmax) lmax = (double)lt[it[j]];
            double den = 0.0;
            for (int j = 0; j < k; ++j) den += exp((double)lt[it[j]] - lmax);
            for (int j = 0; j < k; ++j) w[t * (int64_t)k + j] = (float)(exp((double)lt[it[j]] - lmax) / den);
        } else {
            double sum = 0.0;
            for (int j = 0; j < k; ++j) sum += 1.0 / (1.0 + exp(-(double)lt[it[j]]));
            for (int j = 0; j < k; ++j) {
                double v = 1.0 / (1.0 + exp(-(double)lt[it[j]]));
                if (norm) v /= sum;
                w[t * (int64_t)k + j] = (float)(v * (double)scale);
            }
        }
    }
}

EXPORT void oracle_permute(const int32_t* ids, int64_t m, int k, int E, int32_t* offsets,
                           int32_t* sorted_pair, int32_t* slot_of_pair) {
    int64_t P = m * (int64_t)k;
    int32_t* cursor = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
    for (int e = 0; e <= E; ++e) offsets[e] = 0;
    for (int64_t p = 0; p < P; ++p) offsets[ids[p] + 1] += 1;
    for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    for (int64_t p = 0; p < P; ++p) {
        int e = ids[p];
        int32_t s = offsets[e] + cursor[e]++;
        sorted_pair[s] = (int32_t)p;
        slot_of_pair[p] = s;
    }
    free(cursor);
}

/* ---------------------------------------------------------------- experts */

#define FMT_BF16 0
#define FMT_FP8 1
#define FMT_NVFP4 2

typedef struct {
    int32_t hidden, num_experts, top_k, inter, shared_inter;
    int32_t wfmt;              /* FMT_BF16, FMT_FP8 or FMT_NVFP4 */
    const void *w1, *w3, *w2;  /* [E,I,H], [E,I,H], [E,H,I]: bf16 bits, e4m3 codes or packed e2m1 codes */
    /* fp8: block scales [E,I/128,H/128], [E,I/128,H/128], [E,H/128,I/128];
     * nvfp4: the per-matrix fp32 scale, [E] each */
    const float *s1, *s3, *s2;
    const void *ws1, *ws3, *ws2; /* shared expert, [Is,H], [Is,H], [H,Is] */
    const float *ss1, *ss3, *ss2; /* fp8: its block scales; nvfp4: [1] each */
    const float* shared_gate;    /* [H] or NULL: shared expert scaled by sigmoid(dot(x, gate)) */
    /* nvfp4 only: e4m3 block-scale codes, one per 16 inputs: [E,I,H/16],
     * [E,I,H/16], [E,H,I/16]; the shared expert's [Is,H/16], [Is,H/16], [H,Is/16] */
    const uint8_t *sb1, *sb3, *sb2;
    const uint8_t *ssb1, *ssb3, *ssb2;
} oracle_layer;

/* One expert's [R, C] weight matrix: its codes, and its scales. */
typedef struct {
    const void* w;      /* this expert's codes (element (0,0)) */
    const float* sc;    /* fp8: its 128x128 block scales; nvfp4: its fp32 matrix scale */
    const uint8_t* sb;  /* nvfp4: its [R, C/16] e4m3 block-scale codes */
} wmat;

/* Element (r, c) of one expert's [R, C] weight matrix, dequantised. */
static acc_t weight_at(const wmat* W, int fmt, int C, int r, int c) {
    const int64_t i = (int64_t)r * C + c;
    if (fmt == FMT_BF16) return (acc_t)bf16_to_float(((const uint16_t*)W->w)[i]);
    if (fmt == FMT_FP8) {
        int cb = (C + 127) / 128;
        float code = g_e4m3[((const uint8_t*)W->w)[i]];
        return (acc_t)(code * W->sc[(int64_t)(r / 128) * cb + (c / 128)]);
    }
    const float q = e2m1_decode_one(nibble_at((const uint8_t*)W->w, i));
    const float sb = g_e4m3[W->sb[(int64_t)r * (C / 16) + c / 16]];
    return (acc_t)(q * sb) * (acc_t)W->sc[0];
}

/* Quantise a float row in place to its fp8 or nvfp4 activation values. */
static void act_emulate(int fmt, float* v, int64_t n) {
    float* d = (float*)malloc(sizeof(float) * (size_t)n);
    uint8_t* q = (uint8_t*)malloc((size_t)n);
    float* s = (float*)malloc(sizeof(float) * (size_t)((n + 127) / 128));
    if (fmt == FMT_FP8) {
        oracle_act_quant(v, n, q, s, d);
    } else {
        uint8_t* sb = (uint8_t*)malloc((size_t)(n / 16));
        float g;
        oracle_nvfp4_quant(v, n, q, sb, &g, d);
        free(sb);
    }
    for (int64_t i = 0; i < n; ++i) v[i] = d[i];
    free(d); free(q); free(s);
}

/*
 * One expert's SwiGLU FFN on one input row (metrale moe_v41 forward.rs, the
 * swiglu launch, without its clamp; the routing weight is applied by the
 * caller after the down projection, as in forward_prefill step 7).
 *   xin: [H] (already quantisation-emulated for fp8 / nvfp4); y: [H] out.
 */
static void expert_ffn(const oracle_layer* Lr, int I, const wmat* W1, const wmat* W3, const wmat* W2,
                       const acc_t* xin, acc_t* a, acc_t* y) {
    int H = Lr->hidden;
    int fmt = Lr->wfmt;
    if (I <= 0 || H <= 0) return;
    for (int i = 0; i < I; ++i) {
        acc_t g = 0, u = 0;
        for (int h = 0; h < H; ++h) {
            g += xin[h] * weight_at(W1, fmt, H, i, h);
            u += xin[h] * weight_at(W3, fmt, H, i, h);
        }
        acc_t silu = g / ((acc_t)1 + ACC_EXP(-g));
        a[i] = silu * u;
    }
    if (fmt != FMT_BF16) {
        /* the down projection's input is quantised along I: per 128 elements
         * (fp8) or per 16 elements with a per-row scale (nvfp4) */
        float* af = (float*)malloc(sizeof(float) * (size_t)I);
        for (int i = 0; i < I; ++i) af[i] = (float)a[i];
        act_emulate(fmt, af, I);
        for (int i = 0; i < I; ++i) a[i] = (acc_t)af[i];
        free(af);
    }
    for (int o = 0; o < H; ++o) {
        acc_t acc = 0;
        for (int i = 0; i < I; ++i) acc += a[i] * weight_at(W2, fmt, I, o, i);
        y[o] = acc;
    }
}

/* Expert e's three matrices (e = -1: the shared expert, Is rows). */
static void expert_mats(const oracle_layer* Lr, int e, wmat* W1, wmat* W3, wmat* W2) {
    const int H = Lr->hidden, I = e < 0 ? Lr->shared_inter : Lr->inter;
    const int fmt = Lr->wfmt;
    const int64_t n = e < 0 ? 0 : (int64_t)e * I * H; /* elements before this expert */
    const size_t esz = fmt == FMT_BF16 ? 2 : 1;
    const int64_t wofs = fmt == FMT_NVFP4 ? n / 2 : n;
    W1->w = (const char*)(e < 0 ? Lr->ws1 : Lr->w1) + wofs * esz;
    W3->w = (const char*)(e < 0 ? Lr->ws3 : Lr->w3) + wofs * esz;
    W2->w = (const char*)(e < 0 ? Lr->ws2 : Lr->w2) + wofs * esz;
    W1->sb = W3->sb = W2->sb = 0;
    W1->sc = W3->sc = W2->sc = 0;
    if (fmt == FMT_FP8) {
        const int hb = (H + 127) / 128, ib = (I + 127) / 128;
        const int64_t so = e < 0 ? 0 : (int64_t)e * ib * hb;
        W1->sc = (e < 0 ? Lr->ss1 : Lr->s1) + so;
        W3->sc = (e < 0 ? Lr->ss3 : Lr->s3) + so;
        W2->sc = (e < 0 ? Lr->ss2 : Lr->s2) + so;
    } else if (fmt == FMT_NVFP4) {
        const int64_t bo = n / 16, so = e < 0 ? 0 : e;
        W1->sc = (e < 0 ? Lr->ss1 : Lr->s1) + so;
        W3->sc = (e < 0 ? Lr->ss3 : Lr->s3) + so;
        W2->sc = (e < 0 ? Lr->ss2 : Lr->s2) + so;
        W1->sb = (e < 0 ? Lr->ssb1 : Lr->sb1) + bo;
        W3->sb = (e < 0 ? Lr->ssb3 : Lr->sb3) + bo;
        W2->sb = (e < 0 ? Lr->ssb2 : Lr->sb2) + bo;
    }
}

/*
 * The layer output for the token rows listed in `rows` (all m tokens when
 * rows is NULL), given the routing (ids, w: [m,k]).  out: [nrows, H] float.
 * Per token: acc = sum_j w[j] * FFN_{ids[j]}(xin) (j ascending), then
 * acc += FFN_shared(xin) when a shared expert exists (metrale moe_v41
 * forward.rs, shared_expert_tail: acc += sd), or with a shared gate
 * acc += sigmoid(sum_h x[h] * gate[h]) * FFN_shared(xin) (forward_prefill
 * step "8. Blend shared expert"; x is the bf16 input, the sum in acc_t).
 * Returns 0, or -1 on a bad id.
 */
EXPORT int oracle_moe_forward(const oracle_layer* Lr, const uint16_t* x, int64_t m,
                              const int64_t* rows, int64_t nrows, const int32_t* ids,
                              const float* w, float* out) {
    int H = Lr->hidden, E = Lr->num_experts, k = Lr->top_k, I = Lr->inter;
    int Is = Lr->shared_inter;
    int64_t n = rows ? nrows : m;
    int bad = 0;
    e4m3_table_init();
    int Imax = I > Is ? I : Is;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < n; ++r) {
        int64_t t = rows ? rows[r] : r;
        if (t < 0 || t >= m) { bad |= 1; continue; }
        acc_t* xin = (acc_t*)malloc(sizeof(acc_t) * (size_t)H);
        acc_t* a = (acc_t*)malloc(sizeof(acc_t) * (size_t)Imax);
        acc_t* y = (acc_t*)malloc(sizeof(acc_t) * (size_t)H);
        acc_t* acc = (acc_t*)calloc((size_t)H, sizeof(acc_t));
        const uint16_t* xt = x + t * (int64_t)H;
        if (Lr->wfmt != FMT_BF16) {
            float* xf = (float*)malloc(sizeof(float) * (size_t)H);
            for (int h = 0; h < H; ++h) xf[h] = bf16_to_float(xt[h]);
            act_emulate(Lr->wfmt, xf, H);
            for (int h = 0; h < H; ++h) xin[h] = (acc_t)xf[h];
            free(xf);
        } else {
            for (int h = 0; h < H; ++h) xin[h] = (acc_t)bf16_to_float(xt[h]);
        }
        for (int j = 0; j < k; ++j) {
            int e = ids[t * (int64_t)k + j];
            if (e < 0 || e >= E) { bad |= 1; break; }
            wmat W1, W3, W2;
            expert_mats(Lr, e, &W1, &W3, &W2);
            expert_ffn(Lr, I, &W1, &W3, &W2, xin, a, y);
            acc_t wj = (acc_t)w[t * (int64_t)k + j];
            for (int h = 0; h < H; ++h) acc[h] += wj * y[h];
        }
        if (Is > 0) {
            wmat W1, W3, W2;
            expert_mats(Lr, -1, &W1, &W3, &W2);
            expert_ffn(Lr, Is, &W1, &W3, &W2, xin, a, y);
            acc_t gs = 1;
            if (Lr->shared_gate) {
                acc_t d = 0;
                for (int h = 0; h < H; ++h) d += (acc_t)bf16_to_float(xt[h]) * (acc_t)Lr->shared_gate[h];
                gs = (acc_t)1 / ((acc_t)1 + ACC_EXP(-d));
            }
            for (int h = 0; h < H; ++h) acc[h] += gs * y[h];
        }
        for (int h = 0; h < H; ++h) out[r * (int64_t)H + h] = (float)acc[h];
        free(xin); free(a); free(y); free(acc);
    }
    return bad ? -1 : 0;
}

/* bf16 bits of a float, round to nearest even (NaN kept quiet). */
static uint16_t float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/*
 * The layer tail folded into the combine (ferrum qwen3_moe/forward_layer.rs,
 * "weighted_sum_residual_norm": the weighted sum is written into the residual
 * stream and the next layer's rms_norm is taken of the result):
 *   residual[t,h] <- bf16(residual[t,h] + moe_out[t,h])
 *   r = the new residual's values; inv = 1 / sqrt(sum_h r^2 / H + eps)
 *   norm_out[t,h] = bf16(r[h] * inv * w[h])
 * moe_out fp32 [m,H] (the layer output before its bf16 rounding); residual and
 * norm_out bf16 bits [m,H]; w fp32 [H].  The sum of squares runs in acc_t in
 * ascending h, inv in double.
 */
EXPORT void oracle_residual_rmsnorm(const float* moe_out, int64_t m, int H, uint16_t* residual, const float* w,
                                    float eps, uint16_t* norm_out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < m; ++t) {
        uint16_t* rt = residual + t * (int64_t)H;
        const float* ot = moe_out + t * (int64_t)H;
        acc_t ss = 0;
        for (int h = 0; h < H; ++h) {
            rt[h] = float_to_bf16(bf16_to_float(rt[h]) + ot[h]);
            const acc_t r = (acc_t)bf16_to_float(rt[h]);
            ss += r * r;
        }
        const double inv = 1.0 / sqrt((double)ss / (double)H + (double)eps);
        for (int h = 0; h < H; ++h)
            norm_out[t * (int64_t)H + h] = float_to_bf16((float)((double)bf16_to_float(rt[h]) * inv * (double)w[h]));
    }
}

/* Threads the OpenMP loops use (0 leaves the runtime default). */
EXPORT int oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

EXPORT int oracle_acc_bits(void) { return (int)(8 * sizeof(acc_t)); }
