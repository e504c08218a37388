/*
 * oracle.h -- plain, slow CPU reference of the MXFP4 routed mixture-of-experts
 * block (rms_norm -> router + bias -> top-k on raw logits -> softmax over the
 * k -> MXFP4 gate/up + bias -> clamped SwiGLU -> MXFP4 down + bias ->
 * route-weighted sum added to the residual).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this code: it exists to check the CUDA library.  Only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark use it.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * All floating-point arithmetic is done in double, with three contractual
 * rounding points to bf16 (round to nearest, ties to even):
 *   - the normalised activation x_hat,
 *   - the SwiGLU output h that enters the down projection,
 *   - (inputs) x, router weights are bf16 by definition.
 * Weights are dequantised exactly: value = E2M1(nibble) * 2^(e8m0 - 127).
 *
 * Canonical weight layout (the same the C-ABI of the CUDA library takes):
 *   codes  uint8 [E][rows][cols/2], element 2i in the low nibble of byte i,
 *          element 2i+1 in the high nibble; nibble bit 3 = sign, bits 0..2 =
 *          index into the E2M1 magnitude table {0,.5,1,1.5,2,3,4,6}
 *   scales uint8 E8M0 [E][rows][cols/32]
 *   bias   float [E][rows]
 *   gate, up: rows = F (expert_hidden), cols = H (hidden); down: rows = H, cols = F.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int64_t hidden;        /* H */
    int64_t expert_hidden; /* F */
    int32_t n_experts;     /* E */
    int32_t top_k;         /* K */
    int32_t n_shared;      /* 0 or 1 always-on shared experts (weight 1) */
    double swiglu_alpha;
    double swiglu_limit;
    double weight_scale;   /* route weights = weight_scale * softmax */
    double rms_eps;
    int32_t act_fp4;       /* 1: expert inputs pass through the FP4 activation encoding */
} oracle_cfg;

/* One expert's three matrices, already offset to that expert. */
typedef struct {
    const uint8_t *codes[3];  /* gate, up, down */
    const uint8_t *scales[3];
    const float *bias[3];
} oracle_expert;

typedef struct {
    const float *gamma;        /* [H] */
    const uint16_t *router_w;  /* bf16 bits [E][H] */
    const float *router_b;     /* [E] */
    const uint8_t *codes[3];   /* whole [E][rows][cols/2] tensors */
    const uint8_t *scales[3];
    const float *bias[3];
    const uint8_t *sh_codes[3];  /* shared expert, leading dim 1; NULL when n_shared == 0 */
    const uint8_t *sh_scales[3];
    const float *sh_bias[3];
} oracle_weights;

/* E2M1 value of a 4-bit code (sign in bit 3). */
double oracle_e2m1_value(int nibble);
/* E8M0 scale 2^(e-127); e = 255 is NaN. */
double oracle_e8m0_value(int e);
/* One dequantised element (row r, column c) of a [rows][cols] MXFP4 matrix. */
double oracle_mxfp4_element(const uint8_t *codes, const uint8_t *scales, int64_t cols,
                            int64_t r, int64_t c);
/* Dequantise a whole [rows][cols] matrix into doubles. */
void oracle_mxfp4_dequant(const uint8_t *codes, const uint8_t *scales, int64_t rows,
                          int64_t cols, double *out);

/* MX FP4 encoding of activations in 32-element blocks along each row
 * ([ds4.c] FP4 activation quantisation `dsv4_fp4_act_quantize_row_inplace_cpu`
 * with its nearest-E2M1 step `dsv4_e2m1fn_dequant_cpu`).  Per block:
 *   amax  = max |x_i| (NaN elements never raise it), at least 6 * 2^-126;
 *   q     = amax / 6 rounded once to float;
 *   k     = ceil(log2 q), taken exactly (q is a power of two -> its exponent);
 *           k = 127 when q is infinite;
 *   v_i   = x_i / 2^k clamped to [-6, 6]; NaN -> +6;
 *   code  = nearest E2M1 magnitude index, ties to the even index, sign bit
 *           set when x_i < 0 (so -0 and NaN encode as positive).
 * x float [rows][cols], cols % 32 == 0 -> codes [rows][cols/2] (element 2i in
 * the low nibble) and E8M0 scales [rows][cols/32] = k + 127, the canonical
 * weight layout; decoding them gives the page's round-tripped values.
 * Returns 0, or -1 on bad arguments. */
int oracle_mx_fp4_quantize(const float *x, int64_t rows, int64_t cols, uint8_t *codes,
                           uint8_t *scales);

/* Round a double to bf16 (nearest, ties to even; one rounding); bf16 -> double. */
uint16_t oracle_bf16_rne(double v);
double oracle_bf16_to_double(uint16_t b);

/* x_hat = bf16( x * 1/sqrt(mean(x^2) + eps) * gamma ); also returns the
 * un-rounded values when pre != NULL. */
void oracle_rmsnorm(const uint16_t *x, int64_t H, const float *gamma, double eps,
                    uint16_t *xhat, double *pre);
/* logits[e] = Σ_i x_hat[i] * W[e][i] + b[e] */
void oracle_router_logits(const uint16_t *xhat, const uint16_t *router_w, const float *router_b,
                          int32_t E, int64_t H, double *logits);
/* Insertion top-k: strict '>' so ties go to the lower index and NaN is never
 * selected; unfilled slots keep index 0 and value -inf. */
void oracle_topk(const double *logits, int32_t E, int32_t K, int32_t *ids, double *vals);
/* w_j = scale * softmax(vals)_j; -inf slots get 0; all -inf -> all 0. */
void oracle_route_weights(const double *vals, int32_t K, double scale, double *w);
/* Clamped SwiGLU: g clamped above at limit, u clamped to [-limit, limit],
 * h = g * sigmoid(alpha * g) * (u + 1). */
double oracle_swiglu(double g, double u, double alpha, double limit);
/* One expert: y = Wd * bf16(swiglu(Wg x_hat + bg, Wu x_hat + bu)) + bd.
 * y: [H]; h_out (optional): the bf16 bits of h, [F]; gu_out (optional): g then u, [2F]. */
void oracle_expert_ffn(const oracle_expert *ex, int64_t H, int64_t F, const uint16_t *xhat,
                       double alpha, double limit, double *y, uint16_t *h_out, double *gu_out);
/* oracle_expert_ffn with the FP4 activation mode: when act_fp4 is non-zero,
 * x_hat (before gate/up) and h (after its bf16 rounding, before down) are each
 * replaced by the decoded FP4 activation encoding of themselves, in 32-element
 * blocks along the contracted dimension; h_out still returns the bf16 h. */
void oracle_expert_ffn_ex(const oracle_expert *ex, int64_t H, int64_t F, const uint16_t *xhat,
                          double alpha, double limit, int act_fp4, double *y, uint16_t *h_out,
                          double *gu_out);
/* Token -> expert grouping: counts[E], offsets[E+1] (exclusive prefix sum),
 * routes of each expert in ascending (token, slot) order: perm_token / perm_slot [T*K],
 * and the inverse map loc[t*K + s] = position of route (t, s). */
void oracle_permutation(const int32_t *ids, int64_t T, int32_t K, int32_t E, int32_t *counts,
                        int32_t *offsets, int32_t *perm_token, int32_t *perm_slot, int32_t *loc);

/* Whole block for T tokens.  out [T][H] = x + Σ_slot w * y_slot (+ shared).
 * Optional outputs (NULL to skip): ids [T][K], route_w [T][K], xhat [T][H],
 * logits [T][E].  nthreads > 1 parallelises over tokens (each token's
 * arithmetic order is fixed, so results do not depend on nthreads).
 * Returns 0, or -1 on bad arguments. */
int oracle_moe_forward(const oracle_cfg *cfg, const oracle_weights *w, const uint16_t *x,
                       int64_t T, double *out, int32_t *ids, double *route_w, uint16_t *xhat,
                       double *logits, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
