/*
 * oracle.c -- plain CPU reference of the MXFP4 routed MoE block.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): the tests, the smoke check and the
 * CPU-baseline leg of the benchmark are its only users.  Plain loops, double
 * arithmetic, no blocking, no fusion.  Every function names the passage of
 * the source pages it restates:
 *
 *   [gpt_oss.rs]  goosedump 0.12.31, src/engine/model/gpt_oss.rs
 *                 (constants block; `forward`; `mixture_of_experts`;
 *                  `mixture_of_experts_batch`; `mix_expert_outputs`;
 *                  `top_experts`; tensor validation of the expert tensors)
 *   [ds4.c]       antirez ds4, ds4.c (`dsv4_e2m1fn_value_cpu`;
 *                 `dsv4_e2m1fn_dequant_cpu`; `dsv4_fp4_act_quantize_row_inplace_cpu`;
 *                 `rms_norm_weight`; `DS4_SHAPE_FLASH` profile)
 *   [gptoss/mod]  turbospark-runtime 0.3.0, src/families/gptoss/mod.rs
 *                 (module doc comment: the per-layer formula)
 *
 * Parity pins: every function here is pinned by tests in tests/test_oracle_pins.py
 * except the exact form of the clamped SwiGLU, whose body no page prints (only
 * its name, alpha 1.702 and limit 7); its reading is pinned only by the
 * clamp/closed-form tests, so that formula is "parity unpinned" against the pages.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* [ds4.c] dsv4_e2m1fn_value_cpu: the eight E2M1 magnitudes indexed by the
 * low three bits; bit 3 of the nibble is the sign (MX E2M1 element format). */
double oracle_e2m1_value(int nibble) {
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[nibble & 7];
    return (nibble & 8) ? -v : v;
}

/* E8M0 block scale: a bare biased exponent, 2^(e-127); 0xFF encodes NaN. */
double oracle_e8m0_value(int e) {
    if (e == 255) return NAN;
    return ldexp(1.0, e - 127);
}

double oracle_mxfp4_element(const uint8_t *codes, const uint8_t *scales, int64_t cols, int64_t r,
                            int64_t c) {
    uint8_t byte = codes[r * (cols / 2) + c / 2];
    int nib = (c & 1) ? (byte >> 4) : (byte & 15);
    return oracle_e2m1_value(nib) * oracle_e8m0_value(scales[r * (cols / 32) + c / 32]);
}

void oracle_mxfp4_dequant(const uint8_t *codes, const uint8_t *scales, int64_t rows, int64_t cols,
                          double *out) {
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++)
            out[r * cols + c] = oracle_mxfp4_element(codes, scales, cols, r, c);
}

/* [ds4.c] dsv4_e2m1fn_dequant_cpu: the index of the E2M1 magnitude nearest to
 * |v| (|v| above 6, or NaN, is taken as 6), scanning the table upward and
 * letting an equally near entry replace the current best only when it has an
 * even index and the best so far has an odd one (ties to even). */
static int e2m1_nearest_index(double av) {
    if (!(av <= 6.0)) av = 6.0;
    int best = 0;
    double best_d = fabs(av - oracle_e2m1_value(0));
    for (int i = 1; i < 8; i++) {
        const double d = fabs(av - oracle_e2m1_value(i));
        if (d < best_d || (d == best_d && (i & 1) == 0 && (best & 1) == 1)) {
            best = i;
            best_d = d;
        }
    }
    return best;
}

/* [ds4.c] dsv4_fp4_act_quantize_row_inplace_cpu, returning the codes and the
 * block exponents instead of the round-tripped floats.  The page takes the
 * exponent as ceilf(log2f(amax / 6)); it is taken here exactly from q's
 * binary exponent (frexp), the plain meaning of ceil(log2 q) for every float
 * q, with no dependence on how a log2 routine rounds near powers of two. */
int oracle_mx_fp4_quantize(const float *x, int64_t rows, int64_t cols, uint8_t *codes,
                           uint8_t *scales) {
    if (!x || !codes || !scales || rows < 0 || cols <= 0 || cols % 32 != 0) return -1;
    const float amax_floor = 7.052966104933725e-38f; /* 6 * 2^-126: keeps q a normal float */
    const int64_t nblk = cols / 32;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < nblk; b++) {
            const float *xb = x + r * cols + 32 * b;
            float amax = 0.0f;
            for (int i = 0; i < 32; i++) {
                const float a = fabsf(xb[i]);
                if (a > amax) amax = a; /* false for NaN */
            }
            if (amax < amax_floor) amax = amax_floor;
            const float q = amax / 6.0f; /* one float rounding */
            int k;
            if (isinf(q)) {
                k = 127;
            } else {
                int ex;
                const float m = frexpf(q, &ex); /* q = m * 2^ex, m in [0.5, 1) */
                k = (m == 0.5f) ? ex - 1 : ex;
            }
            if (k > 127) k = 127;
            scales[r * nblk + b] = (uint8_t)(k + 127);
            const double scale = ldexp(1.0, k);
            for (int i = 0; i < 32; i++) {
                double v = (double)xb[i] / scale; /* exact: a power-of-two division in double */
                if (v > 6.0) v = 6.0;
                if (v < -6.0) v = -6.0;
                const int nib = ((xb[i] < 0.0f) ? 8 : 0) | e2m1_nearest_index(fabs(v));
                uint8_t *byte = codes + r * (cols / 2) + 16 * b + i / 2;
                if (i & 1)
                    *byte = (uint8_t)((*byte & 0x0F) | (nib << 4));
                else
                    *byte = (uint8_t)((*byte & 0xF0) | nib);
            }
        }
    }
    return 0;
}

/* bf16: 1 sign, 8 exponent, 7 fraction bits.  One rounding from double:
 * the quantum is 2^(e-8) for a value in [2^(e-1), 2^e) in the normal range and
 * 2^-133 below 2^-126; the scaled value is rounded to an integer with ties to
 * even (nearbyint in the default rounding mode), which is exact arithmetic. */
uint16_t oracle_bf16_rne(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int e;
    frexp(a, &e);
    int qexp = (e - 1 >= -126) ? (e - 8) : -133;
    double q = ldexp(1.0, qexp);
    double r = nearbyint(a / q) * q;
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
    float f = (float)r; /* exact: r is a bf16 value */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return (uint16_t)(sign | (bits >> 16));
}

double oracle_bf16_to_double(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* [ds4.c] rms_norm_weight (sum of squares accumulated in double, scale =
 * 1/sqrt(ss/n + eps), out = x * scale * weight) and [gpt_oss.rs] `forward`:
 * `rms_norm(hidden, HIDDEN, feed_forward_norm, EPSILON)` feeds both the router
 * and the experts.  Here every step is in double and the result is rounded
 * once to bf16 (the activation precision of the block's contract). */
void oracle_rmsnorm(const uint16_t *x, int64_t H, const float *gamma, double eps, uint16_t *xhat,
                    double *pre) {
    double ss = 0.0;
    for (int64_t i = 0; i < H; i++) {
        double xi = oracle_bf16_to_double(x[i]);
        ss += xi * xi;
    }
    double r = 1.0 / sqrt(ss / (double)H + eps);
    for (int64_t i = 0; i < H; i++) {
        double v = oracle_bf16_to_double(x[i]) * r * (double)gamma[i];
        if (pre) pre[i] = v;
        xhat[i] = oracle_bf16_rne(v);
    }
}

/* [gpt_oss.rs] `mixture_of_experts`: router matrix-vector product on the
 * normalised input, then `add_bias` with the router bias. */
void oracle_router_logits(const uint16_t *xhat, const uint16_t *router_w, const float *router_b,
                          int32_t E, int64_t H, double *logits) {
    for (int32_t e = 0; e < E; e++) {
        double acc = 0.0;
        for (int64_t i = 0; i < H; i++)
            acc += oracle_bf16_to_double(xhat[i]) * oracle_bf16_to_double(router_w[(int64_t)e * H + i]);
        logits[e] = acc + (double)router_b[e];
    }
}

/* [gpt_oss.rs] `top_experts`: slots start at -inf with index 0; scanning the
 * logits in index order, each value is inserted at the first slot holding a
 * strictly smaller value and the tail is shifted down by one. */
void oracle_topk(const double *logits, int32_t E, int32_t K, int32_t *ids, double *vals) {
    for (int32_t j = 0; j < K; j++) {
        ids[j] = 0;
        vals[j] = -INFINITY;
    }
    for (int32_t e = 0; e < E; e++) {
        double v = logits[e];
        int32_t pos = K;
        for (int32_t j = 0; j < K; j++) {
            if (v > vals[j]) {
                pos = j;
                break;
            }
        }
        if (pos < K) {
            for (int32_t j = K - 1; j > pos; j--) {
                vals[j] = vals[j - 1];
                ids[j] = ids[j - 1];
            }
            vals[pos] = v;
            ids[pos] = e;
        }
    }
}

/* [gpt_oss.rs] `mixture_of_experts`: `softmax(weights)` over the k selected raw
 * logits ([gptoss/mod]: "softmax_topk(...)[:4] on RAW logits"); the result is
 * multiplied by the block's expert weight scale ([ds4.c] expert_weight_scale,
 * 1.5 for the Flash profile; 1 for gpt-oss).  Max-subtracted, in double. */
void oracle_route_weights(const double *vals, int32_t K, double scale, double *w) {
    double m = -INFINITY;
    for (int32_t j = 0; j < K; j++)
        if (vals[j] > m) m = vals[j];
    if (m == -INFINITY) {
        for (int32_t j = 0; j < K; j++) w[j] = 0.0;
        return;
    }
    double s = 0.0;
    for (int32_t j = 0; j < K; j++) {
        w[j] = (vals[j] == -INFINITY) ? 0.0 : exp(vals[j] - m);
        s += w[j];
    }
    for (int32_t j = 0; j < K; j++) w[j] = scale * (w[j] / s);
}

/* [gpt_oss.rs] `swiglu_inplace(gate, up, SWIGLU_ALPHA = 1.702, SWIGLU_LIMIT = 7)`;
 * [gptoss/mod] "clamped SwiGLU".  The body is not printed on any page.  Reading
 * (gpt-oss form): the gate is clamped from above only, the up projection to
 * [-limit, limit]; glu = g * sigmoid(alpha * g); h = glu * (u + 1).
 * Comparisons are written so that a NaN input propagates. */
double oracle_swiglu(double g, double u, double alpha, double limit) {
    double gc = (g > limit) ? limit : g;
    double uc = (u > limit) ? limit : ((u < -limit) ? -limit : u);
    double glu = gc / (1.0 + exp(-alpha * gc));
    return glu * (uc + 1.0);
}

/* Row r of an MXFP4 matrix times a dense vector, in double. */
static double mxfp4_row_dot(const uint8_t *codes, const uint8_t *scales, int64_t cols, int64_t r,
                            const double *v) {
    double acc = 0.0;
    for (int64_t c = 0; c < cols; c++) acc += oracle_mxfp4_element(codes, scales, cols, r, c) * v[c];
    return acc;
}

/* [gpt_oss.rs] `mixture_of_experts` (per selected expert): `matrix_vector_pair`
 * of gate and up on the normalised input, `add_bias` to both, `swiglu_inplace`,
 * `matrix_vector` of down on the result, `add_bias`.  Expert tensors are
 * validated there as MXFP4; gate/up map hidden -> expert_hidden and down maps
 * back.  h is rounded to bf16 before the down projection (contract). */
/* The FP4 activation mode's round trip of a vector of n (a multiple of 32)
 * float values held in doubles: encode ([ds4.c] FP4 activation quantisation),
 * then decode each element as E2M1 x 2^(e - 127). */
static void fp4_round_trip(double *v, int64_t n) {
    float *f = (float *)malloc(sizeof(float) * (size_t)n);
    uint8_t *codes = (uint8_t *)calloc((size_t)n / 2, 1);
    uint8_t *scales = (uint8_t *)malloc((size_t)n / 32);
    for (int64_t i = 0; i < n; i++) f[i] = (float)v[i]; /* exact: v holds bf16 values */
    oracle_mx_fp4_quantize(f, 1, n, codes, scales);
    for (int64_t i = 0; i < n; i++) v[i] = oracle_mxfp4_element(codes, scales, n, 0, i);
    free(f);
    free(codes);
    free(scales);
}

void oracle_expert_ffn(const oracle_expert *ex, int64_t H, int64_t F, const uint16_t *xhat,
                       double alpha, double limit, double *y, uint16_t *h_out, double *gu_out) {
    oracle_expert_ffn_ex(ex, H, F, xhat, alpha, limit, 0, y, h_out, gu_out);
}

void oracle_expert_ffn_ex(const oracle_expert *ex, int64_t H, int64_t F, const uint16_t *xhat,
                          double alpha, double limit, int act_fp4, double *y, uint16_t *h_out,
                          double *gu_out) {
    double *xv = (double *)malloc(sizeof(double) * (size_t)H);
    double *hv = (double *)malloc(sizeof(double) * (size_t)F);
    for (int64_t i = 0; i < H; i++) xv[i] = oracle_bf16_to_double(xhat[i]);
    if (act_fp4) fp4_round_trip(xv, H);
    for (int64_t j = 0; j < F; j++) {
        double g = mxfp4_row_dot(ex->codes[0], ex->scales[0], H, j, xv) + (double)ex->bias[0][j];
        double u = mxfp4_row_dot(ex->codes[1], ex->scales[1], H, j, xv) + (double)ex->bias[1][j];
        if (gu_out) {
            gu_out[j] = g;
            gu_out[F + j] = u;
        }
        uint16_t hb = oracle_bf16_rne(oracle_swiglu(g, u, alpha, limit));
        if (h_out) h_out[j] = hb;
        hv[j] = oracle_bf16_to_double(hb);
    }
    if (act_fp4) fp4_round_trip(hv, F);
    for (int64_t i = 0; i < H; i++)
        y[i] = mxfp4_row_dot(ex->codes[2], ex->scales[2], F, i, hv) + (double)ex->bias[2][i];
    free(xv);
    free(hv);
}

/* [gpt_oss.rs] `mixture_of_experts_batch`: routes are appended to their
 * expert's list in token order, then slot order (`routes_by_expert[expert]
 * .push(ExpertRoute{token, slot, weight})`); `mix_expert_outputs` /
 * `route_output_index` give each (token, slot) exactly one location. */
void oracle_permutation(const int32_t *ids, int64_t T, int32_t K, int32_t E, int32_t *counts,
                        int32_t *offsets, int32_t *perm_token, int32_t *perm_slot, int32_t *loc) {
    for (int32_t e = 0; e < E; e++) counts[e] = 0;
    for (int64_t r = 0; r < T * K; r++) counts[ids[r]]++;
    offsets[0] = 0;
    for (int32_t e = 0; e < E; e++) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t t = 0; t < T; t++) {
        for (int32_t s = 0; s < K; s++) {
            int32_t e = ids[t * K + s];
            int32_t p = offsets[e] + fill[e]++;
            perm_token[p] = (int32_t)t;
            perm_slot[p] = s;
            loc[t * K + s] = p;
        }
    }
    free(fill);
}

static oracle_expert expert_at(const oracle_weights *w, const oracle_cfg *cfg, int32_t e) {
    oracle_expert ex;
    int64_t H = cfg->hidden, F = cfg->expert_hidden;
    int64_t rows[3] = {F, F, H}, cols[3] = {H, H, F};
    for (int m = 0; m < 3; m++) {
        ex.codes[m] = w->codes[m] + (int64_t)e * rows[m] * (cols[m] / 2);
        ex.scales[m] = w->scales[m] + (int64_t)e * rows[m] * (cols[m] / 32);
        ex.bias[m] = w->bias[m] + (int64_t)e * rows[m];
    }
    return ex;
}

/* One token of the block, [gptoss/mod] module doc comment:
 *   m = rms_norm(x); r = softmax_topk(m @ router + bias)[:k];
 *   x = x + sum(r_w * expert(m))
 * with [gpt_oss.rs] `mixture_of_experts` summing the weighted expert outputs in
 * slot order and `forward` adding the mixture to the residual (`vector_add`).
 * The always-on shared expert of the DeepSeek-V4 profile ([ds4.c] n_expert_shared
 * = 1) is added with weight 1. */
static void token_forward(const oracle_cfg *cfg, const oracle_weights *w, const uint16_t *x,
                          double *out, int32_t *ids, double *rw, uint16_t *xhat, double *logits) {
    int64_t H = cfg->hidden, F = cfg->expert_hidden;
    int32_t E = cfg->n_experts, K = cfg->top_k;
    double *vals = (double *)malloc(sizeof(double) * (size_t)K);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    double *mix = (double *)calloc((size_t)H, sizeof(double));
    oracle_rmsnorm(x, H, w->gamma, cfg->rms_eps, xhat, NULL);
    oracle_router_logits(xhat, w->router_w, w->router_b, E, H, logits);
    oracle_topk(logits, E, K, ids, vals);
    oracle_route_weights(vals, K, cfg->weight_scale, rw);
    for (int32_t j = 0; j < K; j++) {
        oracle_expert ex = expert_at(w, cfg, ids[j]);
        oracle_expert_ffn_ex(&ex, H, F, xhat, cfg->swiglu_alpha, cfg->swiglu_limit, cfg->act_fp4, y, NULL,
                             NULL);
        for (int64_t i = 0; i < H; i++) mix[i] += rw[j] * y[i];
    }
    if (cfg->n_shared) {
        oracle_expert sh;
        for (int m = 0; m < 3; m++) {
            sh.codes[m] = w->sh_codes[m];
            sh.scales[m] = w->sh_scales[m];
            sh.bias[m] = w->sh_bias[m];
        }
        oracle_expert_ffn_ex(&sh, H, F, xhat, cfg->swiglu_alpha, cfg->swiglu_limit, cfg->act_fp4, y, NULL,
                             NULL);
        for (int64_t i = 0; i < H; i++) mix[i] += y[i];
    }
    for (int64_t i = 0; i < H; i++) out[i] = oracle_bf16_to_double(x[i]) + mix[i];
    free(vals);
    free(y);
    free(mix);
}

int oracle_moe_forward(const oracle_cfg *cfg, const oracle_weights *w, const uint16_t *x, int64_t T,
                       double *out, int32_t *ids, double *route_w, uint16_t *xhat, double *logits,
                       int nthreads) {
    if (!cfg || !w || !x || !out || T < 0) return -1;
    int64_t H = cfg->hidden;
    int32_t E = cfg->n_experts, K = cfg->top_k;
    if (H <= 0 || H % 32 || cfg->expert_hidden <= 0 || cfg->expert_hidden % 32) return -1;
    if (K < 1 || K > E || K > 64) return -1;
    if (cfg->n_shared && !w->sh_codes[0]) return -1;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t t = 0; t < T; t++) {
        int32_t ids_l[64];
        double rw_l[64];
        uint16_t *xh = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)H);
        double *lg = (double *)malloc(sizeof(double) * (size_t)E);
        token_forward(cfg, w, x + t * H, out + t * H, ids_l, rw_l, xh, lg);
        if (ids) memcpy(ids + t * K, ids_l, sizeof(int32_t) * (size_t)K);
        if (route_w) memcpy(route_w + t * K, rw_l, sizeof(double) * (size_t)K);
        if (xhat) memcpy(xhat + t * H, xh, sizeof(uint16_t) * (size_t)H);
        if (logits) memcpy(logits + t * E, lg, sizeof(double) * (size_t)E);
        free(xh);
        free(lg);
    }
    return 0;
}
