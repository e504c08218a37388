/*
 * moe.h -- C-ABI of the GB300 (sm_103a) MXFP4 routed mixture-of-experts block.
 *
 * The block (turbospark-runtime gptoss/mod.rs, module doc comment; goosedump
 * gpt_oss.rs, `forward` and `mixture_of_experts`):
 *
 *     m   = rms_norm(x, gamma, eps)                     -- bf16 x_hat
 *     l   = m @ router_w^T + router_b                   -- raw logits
 *     ids = top_k(l)  (strict '>', ties to the lower index, NaN never chosen)
 *     w   = weight_scale * softmax(l[ids])
 *     out = x + Σ_slot w_slot * expert_{ids[slot]}(m)  (+ shared expert, weight 1)
 *     expert(m) = Wd * bf16(swiglu(Wg m + bg, Wu m + bu)) + bd
 *     swiglu(g, u) = min(g, L) * sigmoid(alpha * min(g, L)) * (clamp(u, -L, L) + 1)
 *
 * with MXFP4 expert weights (E2M1 nibbles in 32-element blocks with one E8M0
 * scale each; E2M1 table from ds4.c `dsv4_e2m1fn_value_cpu`).
 *
 * Conventions
 *  - All tensor pointers are DEVICE pointers unless a parameter says "host".
 *    The library never takes ownership: weights and workspace are borrowed
 *    and must outlive every forward call that uses them.
 *  - Every function returns MOE_OK (0) or a negative MOE_E* status; the
 *    thread-local text of the last failure is available from moe_last_error().
 *    Functions that return a pointer return NULL on failure.
 *  - moe_forward only enqueues kernels on the given CUDA stream: no host
 *    synchronisation, no allocation.  Errors found on the device (a bounded
 *    wait that timed out inside a kernel) set a device flag that
 *    moe_get_device_status() reads back.
 *  - bf16 values are passed as their 16-bit patterns.
 *
 * Canonical MXFP4 layout (per matrix, leading expert dimension E):
 *   codes  uint8 [E][rows][cols/2]: element 2i of a row in the low nibble of
 *          byte i, element 2i+1 in the high nibble; nibble bit 3 = sign,
 *          bits 0..2 = index into {0, 0.5, 1, 1.5, 2, 3, 4, 6}
 *   scales uint8 [E][rows][cols/32]: E8M0, value 2^(s-127); 0xFF (NaN) is rejected
 *   bias   float [E][rows]
 *   gate, up: rows = expert_hidden (F), cols = hidden (H)   (goosedump gpt_oss.rs
 *   down:     rows = H, cols = F                              tensor validation)
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    MOE_OK = 0,
    MOE_EINVAL = -1,    /* bad argument: NULL pointer, unknown key, bad value */
    MOE_ESHAPE = -2,    /* shape not supported (see moe_plan_create) */
    MOE_ENOTREADY = -3, /* weights or workspace missing */
    MOE_ECUDA = -4,     /* a CUDA runtime call failed */
    MOE_ENOMEM = -5,    /* workspace too small / token count above max_tokens */
    MOE_EDEVICE = -6    /* a kernel reported a device-side failure */
};

typedef struct moe_plan moe_plan;

/* One MXFP4 matrix of all experts (device pointers, canonical layout). */
typedef struct {
    const uint8_t *codes;
    const uint8_t *scales;
    const float *bias;
} moe_mxfp4_matrix;

typedef struct {
    const float *gamma;        /* rms_norm weight [H] */
    const uint16_t *router_w;  /* bf16 [E][H] */
    const float *router_b;     /* [E] */
    moe_mxfp4_matrix gate, up, down;            /* routed experts, leading dim E */
    moe_mxfp4_matrix sh_gate, sh_up, sh_down;   /* shared expert, leading dim 1;
                                                   read only when n_shared_experts = 1 */
} moe_weights;

/* Create a plan for one block shape (goosedump gpt_oss.rs, constants block:
 * HIDDEN, EXPERTS, EXPERTS_PER_TOKEN, EXPERT_HIDDEN, SWIGLU_ALPHA, SWIGLU_LIMIT;
 * ds4.c DS4_SHAPE_FLASH `expert_weight_scale` for weight_scale).
 * hidden (H) and expert_hidden (F) must be positive multiples of 32;
 * 1 <= top_k <= min(n_experts, 8); 1 <= n_experts <= 256; swiglu_limit > 0.
 * Defaults: rms_eps 1e-5 (goosedump gpt_oss.rs EPSILON), no shared expert,
 * max_tokens 4096.  Returns NULL (see moe_last_error) on bad arguments. */
moe_plan *moe_plan_create(int hidden, int expert_hidden, int n_experts, int top_k,
                          float swiglu_alpha, float swiglu_limit, float weight_scale);
/* Free the plan and the scale copy it owns (see moe_load_weights); borrowed
 * weights and workspace stay the caller's.  NULL is a no-op. */
void moe_plan_destroy(moe_plan *plan);

/* Integer options (no passage of the pages defines these knobs; each names
 * the passage its behaviour follows):
 *   "n_shared_experts"  0 or 1: an always-on expert added with weight 1
 *                       (ds4.c DS4_SHAPE_FLASH n_expert_shared)
 *   "max_tokens"        largest token count per forward (sizes the workspace),
 *                       1..65535
 *   "decode_max_tokens" forwards with tokens <= this use the GEMV decode path,
 *                       larger ones the tensor-core grouped-GEMM path; -1
 *                       (default): 60 for up to 64 experts, 8 above
 *                       (goosedump gpt_oss.rs: `mixture_of_experts` for one
 *                       token, `mixture_of_experts_batch` for a batch)
 *   "path"              0 auto, 1 force decode, 2 force prefill (testing)
 *   "router_exact"      1: compute every router logit in fp64 (testing)
 *   "act_fp4"           1: run both expert projections as block-scaled FP4
 *                       tensor-core GEMMs at every token count: the
 *                       normalised input x_hat and the SwiGLU output h are
 *                       themselves encoded as MXFP4 along the contracted
 *                       dimension (E2M1 codes, one E8M0 scale per 32 values,
 *                       ds4.c `dsv4_fp4_act_quantize_row_inplace_cpu`: scale
 *                       exponent ceil(log2(amax / 6)), codes rounded to
 *                       nearest even); needs H and F multiples of 64 and
 *                       H <= 4096 (else moe_load_weights leaves the plan
 *                       without this path and forwards fail with MOE_ESHAPE).
 *                       The result is the block with FP4 activations, not
 *                       the bf16 one: compare it with a reference that
 *                       encodes the activations the same way.  Must be set
 *                       before moe_set_workspace and before
 *                       moe_load_weights.  0 (default): off
 *   "expert_cache_slots" C in 1..n_experts: an expert cache (antirez ds4
 *                       ds4.c, the expert cache beside `ds4_expert_profile_record`;
 *                       goosedump gpt_oss.rs `ExpertStore`, a lease cache over
 *                       streamed expert bytes).  The expert matrices passed to
 *                       moe_load_weights become the store and may be pinned
 *                       (page-locked, device-mapped) host memory; the plan
 *                       allocates C device slots per matrix (and a device copy
 *                       of the shared expert) and, in every forward, right
 *                       after the routing and on the device: gives each routed
 *                       expert a slot (resident ones hit; a missing one takes
 *                       the least recently used slot this forward does not use,
 *                       the lowest slot on a tie) and copies the missing
 *                       experts' codes, scales and biases from the store into
 *                       their slots before the GEMVs read them.  Results are
 *                       those of the plan without the cache, bit for bit.
 *                       Serves the decode GEMVs only: a forward that would take
 *                       the grouped GEMM, or whose tokens x top_k (capped at
 *                       n_experts) exceed C, fails with MOE_ESHAPE; not with
 *                       act_fp4.  Set before moe_load_weights (which clears the
 *                       cache).  0 (default): off, the matrices read in place
 *   "test_stall_wait"   1: test hook: the decode gate/up kernel's consumer
 *                       warps first wait on a barrier nothing completes, so a
 *                       bounded wait (about 2 s) runs out: theirs (detail 59)
 *                       or the epilogue warp's wait for their partial sums
 *                       (detail 54), whichever expires first; the forward
 *                       then reports MOE_EDEVICE through
 *                       moe_get_device_status and its outputs are void.
 *                       0 (default): off
 *   "out_bf16"          1: the forwards write `out` as bf16 [T][hidden] --
 *                       x + the block's output rounded to nearest (ties to
 *                       even), exactly what moe_cast_f32_to_bf16 makes of
 *                       the fp32 output -- so that a stack of blocks passes
 *                       each block's out to the next as its x (the residual
 *                       stream between layers, goosedump gpt_oss.rs `forward`:
 *                       `vector_add(&mut hidden, &mixture)` per layer) with
 *                       no separate cast; `out` then needs T * hidden * 2
 *                       bytes.  0 (default): fp32 out
 *   "profile"           1: time each kernel launch with CUDA events (see
 *                       moe_profile_read); 0: off (default)
 * Options that change the workspace size must be set before moe_set_workspace. */
int moe_plan_set_i(moe_plan *plan, const char *key, long long value);
/* Floating options: "rms_eps" (goosedump gpt_oss.rs EPSILON; ds4.c
 * `rms_norm_weight` eps). */
int moe_plan_set_f(moe_plan *plan, const char *key, double value);
/* Which projection kernels a forward of `tokens` tokens would run: 1 the GEMV
 * decode path (goosedump gpt_oss.rs `mixture_of_experts`: one matvec pair per
 * selected expert), 2 the tensor-core grouped-GEMM path (`expert_batch_output`:
 * the routed rows of one expert as a matrix), 3 the block-scaled FP4 grouped
 * GEMM of the "act_fp4" option (the same grouping, FP4 activations) (the "path" and
 * "decode_max_tokens" options and the shape decide; the choice also needs
 * the weights loaded, since the grouped GEMM's tensor maps are built then).
 * Negative status on error (NULL plan, weights not loaded, no path for the
 * shape).  Host only; enqueues nothing. */
int moe_plan_path_for(const moe_plan *plan, int tokens);

/* Bytes of device workspace a forward of up to max_tokens tokens needs
 * (max_tokens <= 0: the plan's max_tokens; above 65535 refused).  0 on error.
 * No passage of the pages corresponds: the pages allocate per call on the
 * host; a caller-owned workspace keeps the forward allocation-free. */
size_t moe_workspace_bytes(const moe_plan *plan, int max_tokens);
/* Hand the plan a device buffer of at least moe_workspace_bytes() bytes,
 * 256-byte aligned.  The plan borrows it (the caller frees it).  No passage
 * of the pages corresponds (see moe_workspace_bytes).  Synchronises the
 * current device (it clears the status word and the routing tickets). */
int moe_set_workspace(moe_plan *plan, void *dev_ptr, size_t bytes);

/* Register the weights (device pointers, borrowed), as goosedump gpt_oss.rs's
 * expert tensor validation checks them (`ffn_{gate,up,down}_exps` Mxfp4 of
 * dims [EXPERT_HIDDEN, HIDDEN, EXPERTS], biases F32, router F32 + bias): here
 * pointer alignment (16 bytes) and every scale tensor scanned for the NaN
 * code 0xFF (this one call synchronises the current device).  It also builds
 * the plan's own copy of the scales repacked for the grouped GEMM (device
 * memory the plan owns until moe_plan_destroy).  Must precede moe_forward. */
int moe_load_weights(moe_plan *plan, const moe_weights *w);

/* The block (turbospark-runtime gptoss/mod.rs, module doc comment; goosedump
 * gpt_oss.rs `mixture_of_experts`, `mixture_of_experts_batch`,
 * `mix_expert_outputs`, `top_experts`):
 * out[T][H] (float; bf16 with the "out_bf16" option) = x + MoE(x) for x bf16
 * [T][H]; route_ids_out int32
 * [T][top_k] (may be NULL; 4-byte aligned) gets the selected experts of each
 * token in descending-logit order.  x and out (16-byte aligned) must not
 * alias.  tokens = 0 is a no-op.  MOE_EINVAL on NULL, misaligned or aliasing
 * pointers (checked before anything is enqueued).
 * Enqueue only; graph-capturable; stream is a cudaStream_t (NULL = legacy). */
int moe_forward(moe_plan *plan, const uint16_t *x, int tokens, float *out,
                int32_t *route_ids_out, void *stream);
/* As moe_forward (same passages), also writing the route weights
 * (goosedump gpt_oss.rs `softmax` over the selected logits) [T][top_k] (float, 4-byte
 * aligned) and the normalised activations x_hat [T][H] (bf16, 16-byte aligned,
 * not overlapping x) when those pointers are non-NULL. */
int moe_forward_ex(moe_plan *plan, const uint16_t *x, int tokens, float *out,
                   int32_t *route_ids_out, float *route_w_out, uint16_t *xhat_out, void *stream);

/* Per-expert token counts of the last moe_forward / moe_forward_ex on this
 * plan (goosedump gpt_oss.rs ExpertRouteProfile `counts`, the per-layer
 * selection histogram): int32 [n_experts] (device), enqueued.  Reads the
 * plan's workspace: moe_forward_noalloc calls are not seen (their counts
 * live in the shared static array and are not kept). */
int moe_get_expert_counts(const moe_plan *plan, int32_t *dev_counts_out, void *stream);
/* Token->expert grouping of the last moe_forward / moe_forward_ex (goosedump
 * gpt_oss.rs `mixture_of_experts_batch`: `routes_by_expert`, routes appended
 * per expert in token order; `route_output_index`: one location per route)
 * (device outputs, enqueued; moe_forward_noalloc calls are not seen, as for
 * moe_get_expert_counts): offsets [n_experts + n_shared + 1] (exclusive prefix
 * sums of the counts); perm_token / perm_slot: the routes of each expert in
 * ascending (token, slot) order, the shared expert last with slot top_k.
 * Both perm arrays must hold max_tokens * (top_k + n_shared) int32 entries
 * (the plan's largest route count: that extent is copied); entries from
 * offsets[n_experts + n_shared] on are unspecified. */
int moe_get_permutation(const moe_plan *plan, int32_t *offsets, int32_t *perm_token,
                        int32_t *perm_slot, void *stream);
/* Dequantise one expert matrix (ds4.c `dsv4_e2m1fn_value_cpu`: the E2M1 table,
 * times the block's E8M0 scale 2^(s-127)) (which: 0 gate, 1 up, 2 down; expert = n_experts
 * selects the shared expert) to float [rows][cols] on the device (dev_out
 * 4-byte aligned, rows x cols floats); with expert_cache_slots it reads the
 * store (the matrices as passed to moe_load_weights), not the slots.  Test
 * hook. */
int moe_debug_dequant(const moe_plan *plan, int expert, int which, float *dev_out, void *stream);

/* Expert cache state of a plan with expert_cache_slots (see the option):
 * slot_of [n_experts] (host int32, may be NULL) receives each expert's slot,
 * -1 for experts not resident; stats [3] (host, may be NULL) the cumulative
 * hits, misses and forwards (a hit or a miss is one routed expert of one
 * forward).  Synchronises the stream (device state after the forwards
 * enqueued on it).  MOE_ENOTREADY when the plan has no cache; MOE_ECUDA on a
 * CUDA error.  (antirez ds4 ds4.c, the expert profiler's cache statistics.) */
int moe_get_cache_state(const moe_plan *plan, int32_t *slot_of, long long *stats, void *stream);

/* Kernel timing for benchmarks (no passage of the pages corresponds; the
 * pages' own timers are turbospark-runtime gptoss/mod.rs's per-phase GPU
 * nanoseconds).  After moe_plan_set_i(plan, "profile", 1)
 * every forward records a CUDA event pair around each of its kernel launches,
 * on the forward's stream.  moe_profile_read synchronises on those events and
 * returns, per kernel slot (0 routing + permutation, 1 gate/up + SwiGLU,
 * 2 down + route weight, 3 combine + residual), the summed milliseconds and
 * the launch count since the previous read (at most 4096 forwards are kept),
 * then forgets them.  n_slots: length of the two output arrays (host). */
int moe_profile_read(moe_plan *plan, double *total_ms, int *launches, int n_slots);

/* Synchronises the stream and returns the device-side status of the plan's
 * kernels in *status (0 = fine; 1 = a bounded wait ran out, 2 = a route out
 * of range) and clears it: the plan's workspace word and, when this plan has
 * called moe_forward_noalloc on the current device, the static array's word
 * (shared by every no-alloc call on that device).  A status stays set until
 * read here, and outputs of forwards run while it is set are void.
 * MOE_EDEVICE when a word was set (message: status and detail), MOE_ENOTREADY
 * when the plan has neither a workspace nor a no-alloc call on this device.
 * (goosedump gpt_oss.rs `ensure!` checks: every violation is an error the
 * caller sees, here also those found on the device.) */
int moe_get_device_status(moe_plan *plan, int *status, void *stream);

/* moe_forward without any device allocation, for callers that may not
 * allocate device memory (a runtime that owns all device memory through its
 * own pool and forbids cudaMalloc, or code that must avoid the implicit
 * synchronisation an allocation can cause).  No passage of the source pages
 * corresponds to it: it is a deployment variant of moe_forward.
 *  - Scratch: a file-scope static device array of 16 MiB that every GPU
 *    loading this library holds until exit; no moe_set_workspace is needed.
 *    Token counts whose workspace (moe_workspace_bytes for that count) exceeds
 *    it are rejected with MOE_ENOMEM and a message.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls share the array and it keeps the last call's contents; each
 *    call clears the parts that must start at zero.  Calls that overlap on
 *    the GPU (other streams, other plans, other threads) race on it.
 *  - The kernels' status word is at the start of the array: read it with
 *    moe_get_device_status (on this plan, this device current).
 *    moe_get_expert_counts and moe_get_permutation do not see these calls.
 *  - tokens above 65535 are rejected with MOE_ENOMEM.
 *  - Calls no cudaMalloc, cudaFree or allocating library routine; weights,
 *    x, out and route_ids_out are as for moe_forward. */
int moe_forward_noalloc(moe_plan *plan, const uint16_t *x, int tokens, float *out,
                        int32_t *route_ids_out, void *stream);

/* dst[i] = src[i] rounded to bf16 (nearest, ties to even), i < n, enqueued on
 * `stream`: the residual stream between stacked blocks (a block's fp32 output
 * becomes the next block's bf16 input; goosedump gpt_oss.rs `forward`, the
 * layer loop's `vector_add` of the MoE output into the hidden state).  src fp32 and dst uint16 are device
 * pointers, 16-byte aligned, not overlapping.  NaN inputs give a quiet NaN.
 * MOE_EINVAL on NULL/misaligned pointers, MOE_ECUDA on a launch error. */
int moe_cast_f32_to_bf16(const float *src, uint16_t *dst, size_t n, void *stream);

/* FP4 activation encoding (ds4.c, FP4 activation quantisation
 * `dsv4_fp4_act_quantize_row_inplace_cpu` and its nearest-value step
 * `dsv4_e2m1fn_dequant_cpu`): x bf16 [rows][cols] -> codes uint8
 * [rows][cols/2] and E8M0 scales uint8 [rows][cols/32] in the canonical
 * MXFP4 layout above, enqueued on `stream`.  Per 32-element block:
 *   amax = max |x_i| over the block (NaN elements never raise it), at least
 *          6 * 2^-126;
 *   k    = ceil(log2(amax / 6)), the quotient rounded once to float and the
 *          ceiling taken exactly (127 when the quotient is infinite);
 *   scale byte = k + 127 (so 1..254: never the NaN code);
 *   code = the E2M1 value nearest to x_i / 2^k clamped to [-6, 6], ties to
 *          the even code; sign bit set when x_i < 0 (so -0 and NaN encode as
 *          positive; NaN becomes +6).
 * Decoding the result (E2M1 x 2^(scale-127)) gives the page's round-tripped
 * activations.  x and codes are device pointers, 16-byte aligned; scales a
 * device pointer; the three must not overlap.  rows = 0 is a no-op.
 * MOE_ESHAPE when cols is not a positive multiple of 32; MOE_EINVAL on NULL,
 * misaligned or overlapping pointers or a rows x cols beyond the address
 * space; MOE_ECUDA on a launch error. */
int moe_mx_quantize_fp4(const uint16_t *x, size_t rows, size_t cols, uint8_t *codes, uint8_t *scales,
                        void *stream);

/* ---------------------------------------------------------------------------
 * Expert-locality statistics (antirez ds4, ds4.c, the expert locality
 * profiler: `ds4_expert_profile_record`, `ds4_expert_profile_cache_use`,
 * `ds4_expert_profile_write_cache_summary`; its per-layer selection histogram
 * is goosedump gpt_oss.rs `ExpertRouteProfile::record`).  A profiler holds,
 * in device memory, per layer: the selections and the summed route weight of
 * each expert, the number of recorded tokens, the overlap of the expert sets
 * of tokens at consecutive positions, and for each cache capacity the hits
 * (and hit weight) a least-recently-used cache of that many of the layer's
 * experts would see.  Recording runs on the device, in stream order, after
 * the forward that produced the routes; one warp takes a layer's selections
 * in (token, slot) order for the cache statistics, so recording a batch of T
 * tokens costs about T * top_k dependent steps (microseconds for decode
 * batches, about half a millisecond for 12 K selections).
 */
typedef struct moe_locality moe_locality;

/* Host arrays a read fills (each may be NULL): hist and weight_hist
 * [n_layers][n_experts]; layer_records, adjacent_pairs, overlap_sum (sum over
 * adjacent pairs of intersection / top_k) and jaccard_sum (of intersection /
 * union) [n_layers]; cache_hits and cache_weight_hits [n_caps][n_layers];
 * caps [n_caps] the capacities kept.  n_caps is set by the read. */
typedef struct {
    uint64_t *hist;
    double *weight_hist;
    uint64_t *layer_records;
    uint64_t *adjacent_pairs;
    double *overlap_sum;
    double *jaccard_sum;
    uint64_t *cache_hits;
    double *cache_weight_hits;
    int *caps;
    int n_caps;
} moe_locality_stats;

/* A profiler for n_layers layers (1..4096) of n_experts experts (1..256) with
 * top_k slots (1..min(8, n_experts)) and up to 16 cache capacities; as the
 * page does, capacities outside 1..n_experts are left out.  Allocates its
 * device state (zeroed; this call synchronises).  NULL on bad arguments or
 * allocation failure (moe_last_error says which). */
moe_locality *moe_locality_create(int n_layers, int n_experts, int top_k, const int *caps, int n_caps);
/* Record `tokens` tokens of layer `layer` at sequence positions first_pos,
 * first_pos + 1, ...: ids int32 [tokens][top_k] and route_w float
 * [tokens][top_k], device pointers (4-byte aligned) as moe_forward_ex writes
 * them; experts outside [0, n_experts) are skipped, as on the page.  A token
 * is compared with the layer's previous recorded token when that one sat at
 * the position just before.  Enqueue only. */
int moe_locality_record(moe_locality *prof, int layer, const int32_t *ids, const float *route_w, int tokens,
                        long long first_pos, void *stream);
/* Record every later forward of `plan` (moe_forward, moe_forward_ex,
 * moe_forward_noalloc) into layer `layer` of prof, each forward's tokens at
 * the positions after the previous forward's, from 0 (goosedump gpt_oss.rs:
 * `forward` / `prefill` take an optional route profile).  prof NULL
 * detaches.  The profiler must outlive the attachment. */
int moe_locality_attach(moe_plan *plan, moe_locality *prof, int layer);
/* Synchronise the device and copy the statistics into *out. */
int moe_locality_read(const moe_locality *prof, moe_locality_stats *out);
/* Zero every statistic and forget every layer's previous token (synchronises stream). */
int moe_locality_reset(moe_locality *prof, void *stream);
/* Free the device state.  NULL is a no-op. */
void moe_locality_destroy(moe_locality *prof);

/* ---------------------------------------------------------------------------
 * The attention half of the gpt-oss layer, one decode step for a batch of
 * sequences (goosedump gpt_oss.rs `forward`: the attention norm, the query,
 * key and value projections with biases, `apply_rope` with `Rope::new`'s
 * YaRN tables, `LayerCache::append`, `causal_gqa` / `attention_head` with the
 * per-head sink logit and `attention_window`, the output projection with its
 * bias and the residual add; turbospark-runtime gptoss/mod.rs module doc
 * comment).  For each sequence b with its new token at position pos[b] (the
 * number of tokens its cache already holds):
 *   x_hat = bf16(rms_norm(x[b]) * gamma)              (as in the MoE block)
 *   q, k, v = Wq x_hat + bq, Wk x_hat + bk, Wv x_hat + bv   (fp32)
 *   q, k rotated per head: dims d and d + 32 form pair d, by the angle
 *     pos[b] * f_d, f_d the RoPE base frequency blended toward f_d / factor
 *     between the YaRN correction dimensions of beta_fast and beta_slow;
 *     cosine and sine scaled by 0.1 ln(factor) + 1
 *   k, v stored (fp16, nearest) at cache row pos[b] of sequence b
 *   per query head h (kv head h / (q_heads / kv_heads)): softmax over the
 *     scores q_h . k_t / 8 of the visible tokens (the last sliding_window of
 *     them, or all) and the head's sink logit; o_h = sum_t p_t v_t
 *   out[b] = x[b] + Wo bf16(o) + bo   (fp32, or bf16 with "out_bf16")
 * Weights: gamma f32 [H]; wq bf16 [q_heads * 64][H], wk and wv bf16
 * [kv_heads * 64][H], wo bf16 [H][q_heads * 64]; bq, bk, bv, bo f32 of the
 * matching lengths; sinks f32 [q_heads]; all device pointers, 16-byte
 * aligned, borrowed.  Caches: fp16 [max_seqs][max_ctx][kv_heads][64] for
 * keys and for values, device memory the caller owns.
 */
typedef struct moe_attn moe_attn;
typedef struct {
    const float *gamma;
    const uint16_t *wq, *wk, *wv, *wo;
    const float *bq, *bk, *bv, *bo;
    const float *sinks;
} moe_attn_weights;

/* A plan for one layer: hidden a multiple of 32 up to 4096, head_dim 64 (the
 * page's constant), q_heads a multiple of kv_heads with at most 16 per kv
 * head, up to 32 sequences per step, up to 65536 context tokens.  Defaults:
 * full attention, rms_eps 1e-5, the page's RoPE constants (base 150000,
 * factor 32, original context 4096, beta_fast 32, beta_slow 1).  NULL on bad
 * arguments. */
moe_attn *moe_attn_create(int hidden, int q_heads, int kv_heads, int head_dim, int max_seqs, int max_ctx);
/* "sliding_window": 0 (full attention) or the number of most recent tokens a
 * query sees (the page: 128 on even layers); "out_bf16": 1 writes out as bf16;
 * "prefill_rows": rows of one prefill block, 1..4096 (default and minimum:
 * max_seqs); it sizes the workspace, so set it before moe_attn_set_workspace
 * (setting it to a new value unsets the workspace). */
int moe_attn_set_i(moe_attn *plan, const char *key, long long value);
/* "rms_eps", "rope_base", "rope_factor", "rope_original_context",
 * "rope_beta_fast", "rope_beta_slow" (positive, finite). */
int moe_attn_set_f(moe_attn *plan, const char *key, double value);
/* Device workspace a step needs (the status word; x_hat; q, k, v before RoPE;
 * the RoPE table; the chunk partials; o): caller-owned, 256-byte aligned,
 * borrowed by moe_attn_set_workspace (which zeroes the status word). */
size_t moe_attn_workspace_bytes(const moe_attn *plan);
int moe_attn_set_workspace(moe_attn *plan, void *dev_ptr, size_t bytes);
/* The key and value caches (fp16, layout above; borrowed). */
int moe_attn_set_cache(moe_attn *plan, void *k_cache, void *v_cache);
int moe_attn_load_weights(moe_attn *plan, const moe_attn_weights *w);
/* One decode step for n_seqs sequences (0..max_seqs): x bf16 [n_seqs][H]
 * (16-byte aligned), positions int32 [n_seqs] on the device (each in
 * 0..max_ctx-1; a sequence whose position is outside is skipped and its out
 * row undefined), out [n_seqs][H] (16-byte aligned, not overlapping x).
 * Writes the new tokens' keys and values into the caches.  Enqueue only. */
int moe_attn_decode(moe_attn *plan, const uint16_t *x, int n_seqs, const int32_t *positions, void *out,
                    void *stream);
/* Prefill (goosedump gpt_oss.rs `prefill_attention_layer` / `causal_gqa_batch`):
 * n_tokens consecutive new tokens of cache sequence seq (0..max_seqs-1) at
 * positions pos0 .. pos0 + n_tokens - 1 (pos0 = the tokens its cache already
 * holds; the last position at most max_ctx - 1).  Token r sees the cached
 * tokens and the new tokens up to itself (the last sliding_window of them on
 * sliding layers), as a decode step at position pos0 + r would.  Processed in
 * blocks of max(max_seqs, prefill_rows) rows, each block's keys and values
 * appended before its attention.  x bf16 [n_tokens][H], out [n_tokens][H] (16-byte aligned, not
 * overlapping); writes cache rows pos0 .. pos0 + n_tokens - 1 of sequence
 * seq and no others.  Enqueue only. */
int moe_attn_prefill(moe_attn *plan, const uint16_t *x, int n_tokens, int seq, int pos0, void *out, void *stream);
/* Synchronises the stream and returns the device-side status of the plan's
 * kernels in *status (0 = fine; 1 = a bounded wait of the prefill's tensor-core
 * projections gave up), then clears it; MOE_EDEVICE when it was set (message:
 * status and detail). */
int moe_attn_get_device_status(moe_attn *plan, int *status, void *stream);
void moe_attn_destroy(moe_attn *plan);

/* Text of the last failure on this thread ("" if none) (goosedump gpt_oss.rs:
 * every `ensure!` carries a message). */
const char *moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif
