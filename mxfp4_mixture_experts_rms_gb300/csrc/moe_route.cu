// moe_route.cu -- fused rms_norm + router + top-k + softmax, then (in the last
// CTA to finish) the token->expert permutation: per-expert histogram,
// exclusive prefix sum, stable scatter, inverse map and the tile table.
//
// Page passages restated here:
//  * ds4.c `rms_norm_weight` and goosedump gpt_oss.rs `forward`
//    (`rms_norm(hidden, HIDDEN, feed_forward_norm, EPSILON)`): the norm;
//  * goosedump gpt_oss.rs `mixture_of_experts` / `mixture_of_experts_batch`:
//    router matvec + bias, `top_experts` (insertion with a strict '>', so ties
//    go to the lower index and NaN is never chosen), `softmax` over the k;
//  * goosedump gpt_oss.rs `mixture_of_experts_batch` / `mix_expert_outputs`:
//    routes appended per expert in token order, one output location per route.
//
// Two kernels.  Small batches (T <= 32, the decode regime): one thread-block
// cluster per token, its CTAs splitting the experts; every CTA normalises the
// token, computes its experts' logits with error bounds and writes them into
// the shared memory of the cluster's first CTA, which selects the top-k after
// a cluster barrier.  Larger batches: CTAs of 8 tokens x an expert chunk; the
// last CTA of a token group (atomic ticket) selects the top-k of its tokens.
// In both, the last token-owning CTA to finish (atomic ticket, never a wait)
// builds the permutation.
//
// Accuracy.  Σx² is summed from exact fp32 squares with error-free two-sums
// (relative error ~2^-44, the order of the reference's own double-sum
// rounding) and r = 1/sqrt(ms + eps) is evaluated in double.  x_hat = bf16(x * r * gamma) is computed in fp32 and recomputed
// in fp64 whenever the fp32 value lies within its error bound of a bf16
// rounding midpoint.  Router logits are accumulated in fp32 with a rigorous
// error bound; when the bounds cannot certify top-k membership and order, the
// candidate logits are recomputed in fp64 (exact for these operands) and the
// selection is redone on them.
#include "moe_common.cuh"

// Phase marker (no-op unless an instrumented build defines it).
#ifndef MOE_PHASE_MARK
#define MOE_PHASE_MARK(i)
#endif
#ifndef MOE_WARP_MARK
#define MOE_WARP_MARK(i)
#endif

namespace {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;

struct RouteArgs {
    BlockParams bp;
    Workspace ws;
    const uint16_t *x;
    const float *gamma;
    const uint16_t *router_w;
    const float *router_b;
    int T;
    int32_t *ids_out;   // user copy, may be null
    float *rw_out;      // user copy, may be null
    uint16_t *xhat_out; // user copy, may be null
    int tile_rows;
    int router_exact;
    int epc;        // experts per CTA (router rows staged in shared memory)
    int forms;      // x_hat copies the expert kernels read besides the natural one (kFormF16 | kFormMma)
    double inv_h;   // 1 / H
};

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// (value, index) order of `top_experts`: larger value first, equal values by lower index.
__device__ __forceinline__ bool better(float v, int i, float w, int j) { return v > w || (v == w && i < j); }
__device__ __forceinline__ bool better_d(double v, int i, double w, int j) { return v > w || (v == w && i < j); }

template <class V>
__device__ __forceinline__ void warp_best(V &v, int &i) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        V w = __shfl_xor_sync(0xffffffffu, v, o);
        int j = __shfl_xor_sync(0xffffffffu, i, o);
        if (w > v || (w == v && j < i)) {
            v = w;
            i = j;
        }
    }
}

// Exclusive scan by one warp over n <= 1024 ints (out[n] = total).
__device__ void warp_exclusive_scan(const int32_t *in, int32_t *out, int n, int lane) {
    int per = (n + 31) / 32;
    int lo = lane * per, hi = min(n, lo + per);
    int s = 0;
    for (int i = lo; i < hi; i++) s += in[i];
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - s;
    for (int i = lo; i < hi; i++) {
        int c = in[i];
        out[i] = run;
        run += c;
    }
    if (lane == 31) out[n] = incl;
}

constexpr int kXC = 2;  // 16-byte chunks of one x row per thread (H <= 8 * 256 * kXC)
constexpr int kRowChunks = kRouteThreads * kXC / 32;  // 16-byte chunks of one row per lane of a warp

// Σx² of a bf16 row, to ~2^-44 relative (the reference statistic is itself a
// double sum whose rounding is of that order).  Every value is scaled by
// 2^(127 - emax), emax the row's largest exponent field, which is exact and
// keeps the squares in fp32 range; squares of bf16 values are exact in fp32;
// they are summed with error-free two-sums (Knuth), the error terms carried
// alongside.
struct Comp {
    float s, c;
};
__device__ __forceinline__ void comp_add(Comp &a, float x) {
    const float t = __fadd_rn(a.s, x);
    const float z = __fadd_rn(t, -a.s);
    a.c = __fadd_rn(a.c, __fadd_rn(__fadd_rn(a.s, -__fadd_rn(t, -z)), __fadd_rn(x, -z)));
    a.s = t;
}
__device__ __forceinline__ void comp_merge(Comp &a, const Comp &b) {
    comp_add(a, b.s);
    a.c = __fadd_rn(a.c, b.c);
}
__device__ __forceinline__ Comp comp_warp(Comp a) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        Comp b;
        b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
        b.c = __shfl_xor_sync(0xffffffffu, a.c, o);
        comp_merge(a, b);
    }
    return a;
}
__device__ __forceinline__ int bf16_exp(uint32_t b) { return (int)((b >> 7) & 0xFFu); }
// 2^(127 - emax) as fp32 (subnormal for emax = 254: exact all the same)
__device__ __forceinline__ float exp_scale(int emax) {
    const int k = 127 - emax + 127;  // biased exponent of the scale
    return k >= 1 ? __uint_as_float((uint32_t)k << 23) : __uint_as_float(0x00400000u >> (-k));
}
__device__ __forceinline__ void comp_add_pair(Comp &a, uint32_t w2, float sc) {
    const float v0 = __fmul_rn(__uint_as_float(w2 << 16), sc), v1 = __fmul_rn(__uint_as_float(w2 & 0xFFFF0000u), sc);
    comp_add(a, __fmul_rn(v0, v0));
    comp_add(a, __fmul_rn(v1, v1));
}
__device__ __forceinline__ double comp_result(const Comp &a, int emax) {
    return ldexp((double)a.s + (double)a.c, 2 * (emax - 127));
}

// Router logit of expert e for an x_hat row in shared memory, by one warp, to
// ~2^-44 of Σ|products| (the reference's own double sum rounds at ~2^-50):
// products of two bf16 are exact in fp32 and are summed with error-free
// two-sums; equal rows give bit-identical results, so exact ties stay ties.
// Used where the fp32 bounds cannot decide the top-k (and in the exact mode).
__device__ double exact_logit(const uint16_t *xh, const uint16_t *router_w, const float *router_b, int e, int H,
                              int lane) {
    // the loads of both rows issued in two rounds of eight 16-byte chunks per
    // lane: two memory latencies per logit, not one per chunk
    constexpr int kRound = kRowChunks / 2;
    const int nch = H / 8;
    const uint4 *w = reinterpret_cast<const uint4 *>(router_w + (size_t)e * H);
    const uint4 *x = reinterpret_cast<const uint4 *>(xh);
    Comp acc[2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll 1
    for (int i0 = 0; i0 < kRowChunks && lane + 32 * i0 < nch; i0 += kRound) {
        uint4 wv[kRound], xv[kRound];
#pragma unroll
        for (int i = 0; i < kRound; i++) {
            const int c = lane + 32 * (i0 + i);
            wv[i] = c < nch ? __ldg(w + c) : make_uint4(0, 0, 0, 0);
            xv[i] = c < nch ? x[c] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kRound; i++) {
            if (lane + 32 * (i0 + i) >= nch) break;
            const uint32_t ww[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w}, xx[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
            for (int q = 0; q < 4; q++) {
                comp_add(acc[q & 1], __fmul_rn(__uint_as_float(xx[q] << 16), __uint_as_float(ww[q] << 16)));
                comp_add(acc[q & 1],
                         __fmul_rn(__uint_as_float(xx[q] & 0xFFFF0000u), __uint_as_float(ww[q] & 0xFFFF0000u)));
            }
        }
    }
    comp_merge(acc[0], acc[1]);
    const Comp t = comp_warp(acc[0]);
    return ((double)t.s + (double)t.c) + (double)router_b[e];
}

// Σx² of one bf16 row held in registers by the whole CTA of NTH threads (XC
// chunks of 8 per thread); every thread gets it.
template <int NTH, int XC>
__device__ double sumsq_block(const uint4 (&xv)[XC], int lane, int warp, int *s_maxexp, Comp *s_acc) {
    int mx = 1;
#pragma unroll
    for (int j = 0; j < XC; j++) {
        const uint32_t w[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
        for (int q = 0; q < 4; q++) mx = max(mx, max(bf16_exp(w[q]), bf16_exp(w[q] >> 16)));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_maxexp[warp] = mx;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < NTH / 32; w++) mx = max(mx, s_maxexp[w]);
    const float sc = exp_scale(mx);
    Comp acc{0.f, 0.f};
#pragma unroll
    for (int j = 0; j < XC; j++) {
        comp_add_pair(acc, xv[j].x, sc);
        comp_add_pair(acc, xv[j].y, sc);
        comp_add_pair(acc, xv[j].z, sc);
        comp_add_pair(acc, xv[j].w, sc);
    }
    acc = comp_warp(acc);
    if (lane == 0) s_acc[warp] = acc;
    __syncthreads();
    Comp tot = s_acc[0];
#pragma unroll
    for (int w = 1; w < NTH / 32; w++) comp_merge(tot, s_acc[w]);
    return comp_result(tot, mx);
}

// bf16(x * r * gamma) of one element: fp32 value, recomputed in fp64 when it
// lies within its error bound (3 fp32 ulps; 8 used) of a bf16 rounding midpoint.
// The fp64 evaluation sits in a function of its own: inlined, the compiler
// may evaluate it for every element (fp64 throughput is a small fraction of
// fp32 here) instead of branching to it for the rare uncertain one.
__device__ __noinline__ uint32_t norm_elem_fp64(uint32_t xb, float gf, double r) {
    return bf16_from_double_rne((double)__uint_as_float(xb << 16) * r * (double)gf);
}
__device__ __forceinline__ uint32_t norm_elem(uint32_t xb, float gf, float r32, double r) {
    const float xf = __uint_as_float(xb << 16);
    const float v32 = (xf * r32) * gf;
    const uint32_t low = __float_as_uint(v32) & 0xFFFFu;
    const bool safe =
        fabsf(v32) >= 0x1p-120f && fabsf(v32) < 0x1p126f && (low > 0x8000u + 8u || low + 8u < 0x8000u);
    if (__builtin_expect(safe, 1)) {
        __nv_bfloat16 bb = __float2bfloat16_rn(v32);
        return *reinterpret_cast<uint16_t *>(&bb);
    }
    return norm_elem_fp64(xb, gf, r);
}

// 1/sqrt(m) in double: Newton steps from the fp32 seed (two steps take its
// ~2^-22 error below double rounding), plain division outside the seed's range.
__device__ __forceinline__ double rsqrt_d(double m) {
    if (!(m >= 1e-30 && m <= 1e30)) return 1.0 / sqrt(m);
    double y = (double)rsqrtf((float)m);
    y = y * (1.5 - 0.5 * m * y * y);
    y = y * (1.5 - 0.5 * m * y * y);
    return y;
}

constexpr int kInvalid = 0x7fffffff;

// Top-k + softmax of one token by one warp (goosedump gpt_oss.rs
// `top_experts` and `softmax`), in three steps so that the exact logits a
// token may need are computed by every warp of the CTA at once:
//  * topk_select: the fp32 selection from the logits l[0..E) and their error
//    bounds (shared or global memory; lane j holds experts j, j+32, ...; the
//    r-th selection ends in lane r's registers).  It stands when consecutive
//    selected values are further apart than twice the largest bound;
//    otherwise every expert within reach of the k-th value is listed as a
//    candidate (cand[0..*ncand)) and exs[0..E) is set to -inf;
//  * exact_candidates: the listed candidates' exact logits into exs;
//  * topk_finish: the selection redone on the exact logits where needed, the
//    softmax over the selected raw logits times the weight scale, the stores.
template <bool GLOBAL>
__device__ bool topk_select(const float *l, const float *bd, const RouteArgs &a, int lane, float &my_v, int &my_i,
                            double *exs, uint16_t *cand, int *ncand) {
    const int E = a.bp.E, K = a.bp.K;
    const bool exact_mode = a.router_exact != 0;
    auto ld = [&](const float *p) { return GLOBAL ? __ldcg(p) : *p; };
    constexpr int NQ = MOE_MAX_EXPERTS / 32;
    float lv[NQ];
    float dmax = 0.f;
#pragma unroll
    for (int q = 0; q < NQ; q++) {
        const int j = lane + 32 * q;
        lv[q] = j < E ? ld(l + j) : -INFINITY;
        if (j < E) dmax = fmaxf(dmax, ld(bd + j));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
    uint32_t taken = 0;
    my_v = -INFINITY;
    my_i = kInvalid;
    if (E <= 32) {
        // one logit per lane: its rank among the selectable ones (NaN and -inf
        // never are) by 32 independent comparisons, then selection r moves to lane r
        const float v = lv[0];
        const bool ok_sel = lane < E && v > -INFINITY;
        const uint32_t okm = __ballot_sync(0xffffffffu, ok_sel);
        int rank = 0;
#pragma unroll
        for (int i = 0; i < 32; i++) {
            const float vi = __shfl_sync(0xffffffffu, v, i);
            rank += ((okm >> i) & 1u) && better(vi, i, v, lane);
        }
        for (int r = 0; r <= K; r++) {
            const uint32_t mr = __ballot_sync(0xffffffffu, ok_sel && rank == r);
            const int src = mr ? __ffs(mr) - 1 : 0;
            const float vv = __shfl_sync(0xffffffffu, v, src);
            if (lane == r && mr) {
                my_v = vv;
                my_i = src;
            }
        }
    } else {
        for (int r = 0; r <= K; r++) {
            float bv = -INFINITY;
            int bi = kInvalid;
#pragma unroll
            for (int q = 0; q < NQ; q++) {
                const int j = lane + 32 * q;
                const float v = lv[q];
                // NaN and -inf are never chosen
                if (j < E && v > -INFINITY && !(taken >> q & 1u) && better(v, j, bv, bi)) {
                    bv = v;
                    bi = j;
                }
            }
            warp_best(bv, bi);
            if (lane == r) {
                my_v = bv;
                my_i = bi;
            }
            if (bi != kInvalid && (bi & 31) == lane) taken |= 1u << (bi >> 5);
        }
    }
    // certification: selection r must beat selection r+1 by more than 2 dmax
    const float nx_v = __shfl_down_sync(0xffffffffu, my_v, 1);
    const int nx_i = __shfl_down_sync(0xffffffffu, my_i, 1);
    bool ok = true;
    if (lane < K && my_i != kInvalid) ok = my_v - (nx_i == kInvalid ? -INFINITY : nx_v) > 2.0f * dmax;
    if (!exact_mode && __all_sync(0xffffffffu, ok)) {
        if (lane == 0) *ncand = 0;
        return false;
    }
    const float kv = __shfl_sync(0xffffffffu, my_v, K - 1);
    const int ki = __shfl_sync(0xffffffffu, my_i, K - 1);
    const float thr = (exact_mode || ki == kInvalid) ? -INFINITY : kv - 2.0f * dmax;
    int n = 0;
    for (int base = 0; base < E; base += 32) {  // candidates listed in expert order
        const int j = base + lane;
        const float v = j < E ? ld(l + j) : -INFINITY;
        const bool c = v > -INFINITY && !(v < thr);
        const uint32_t m = __ballot_sync(0xffffffffu, c);
        if (c) cand[n + __popc(m & ((1u << lane) - 1u))] = (uint16_t)j;
        n += __popc(m);
        if (j < E) exs[j] = -INFINITY;
    }
    if (lane == 0) *ncand = n;
    return true;
}

// Exact logits of the candidates listed by topk_select for W tokens (token w:
// x_hat row xbase + w * xstride, candidates cand[w * E ..], count ncand[w],
// results into exs[w * E + j]), one candidate per warp of the CTA at a time.
__device__ void exact_candidates(const RouteArgs &a, const uint16_t *xbase, size_t xstride, const uint16_t *cand,
                                 const int *ncand, int W, double *exs, int warp, int nwarps, int lane) {
    const int E = a.bp.E;
    int total = 0;
    for (int w = 0; w < W; w++) total += ncand[w];
    for (int p = warp; p < total; p += nwarps) {
        int w = 0, q = p;
        while (q >= ncand[w]) {
            q -= ncand[w];
            w++;
        }
        const int j = cand[w * E + q];
        const double ex = exact_logit(xbase + (size_t)w * xstride, a.router_w, a.router_b, j, a.bp.H, lane);
        if (lane == 0) exs[w * E + j] = ex;
    }
}

__device__ int topk_finish(const RouteArgs &a, int t, int lane, bool need, const double *exs, float my_v, int my_i) {
    const int E = a.bp.E, K = a.bp.K;
    constexpr int NQ = MOE_MAX_EXPERTS / 32;
    double my_d = 0.0;
    if (need) {
        uint32_t taken = 0;
        my_i = kInvalid;
        my_d = -INFINITY;
        for (int r = 0; r < K; r++) {
            double bv = -INFINITY;
            int bi = kInvalid;
#pragma unroll
            for (int q = 0; q < NQ; q++) {
                const int j = lane + 32 * q;
                if (j < E && !(taken >> q & 1u)) {
                    const double v = exs[j];
                    if (v > -INFINITY && better_d(v, j, bv, bi)) {
                        bv = v;
                        bi = j;
                    }
                }
            }
            warp_best(bv, bi);
            if (lane == r) {
                my_d = bv;
                my_i = bi;
                my_v = (float)bv;
            }
            if (bi != kInvalid && (bi & 31) == lane) taken |= 1u << (bi >> 5);
        }
    }
    // softmax over the selected raw logits, times the weight scale; lane r owns slot r
    const float m = __shfl_sync(0xffffffffu, my_v, 0);
    const double md = __shfl_sync(0xffffffffu, my_d, 0);
    const bool valid = lane < K && my_i != kInvalid;
    float ew = 0.f;
    if (valid) ew = expf(need ? (float)(my_d - md) : (my_v - m));
    float ssum = ew;
#pragma unroll
    for (int o = 16; o; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    const int id = valid ? my_i : 0;  // unfilled slot: expert 0, weight 0
    if (lane < K) {
        const float w = (valid && ssum > 0.f) ? a.bp.wscale * (ew / ssum) : 0.f;
        a.ws.ids[t * K + lane] = id;
        a.ws.route_w[t * K + lane] = w;
        if (a.ids_out) a.ids_out[t * K + lane] = id;
        if (a.rw_out) a.rw_out[t * K + lane] = w;
    }
    return id;  // lane r: slot r's expert
}

// Bytes of shared memory the permutation needs (per-expert counters).
__host__ __device__ constexpr size_t perm_smem_bytes(int E, int warps = kRouteWarps) {
    return (size_t)(5 * 264 + warps * (E + 1)) * 4;
}

// The token->expert permutation (goosedump gpt_oss.rs `mixture_of_experts_batch`:
// routes appended per expert in token order): per-expert histogram, exclusive
// prefix sums of counts and of tiles, stable scatter of (token, slot, weight),
// the inverse map and the tile table.  Run by one CTA (any multiple of 32
// threads) once every token's ids are in global memory.
// CACHE: keep the first NTH routes' expert and weight in registers for the
// scatter pass (the small-batch kernel: decode batches have no more routes)
template <bool CACHE>
__device__ void build_permutation(const RouteArgs &a, unsigned char *smem) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NTH = blockDim.x, NW = NTH >> 5;
    const int E = a.bp.E, K = a.bp.K;
    const int ns = a.bp.n_shared;
    const int EE = E + ns;
    const int KK = K + ns;
    const int R = a.T * K;
    int32_t *cnt = reinterpret_cast<int32_t *>(smem);
    int32_t *offs = cnt + 264;
    int32_t *run = offs + 264;
    int32_t *tcnt = run + 264;
    int32_t *toff = tcnt + 264;
    int32_t *wcnt = toff + 264;  // [NW][EE]
    for (int e = tid; e < EE; e += NTH) {
        cnt[e] = 0;
        run[e] = 0;
    }
    __syncthreads();
    // with CACHE, the first NTH routes' expert and weight stay in registers for
    // the scatter pass, saving its round trips to L2
    int e_first = -1;
    float w_first = 0.f;
    if (CACHE && tid < R) w_first = __ldcg(a.ws.route_w + tid);
    for (int r = tid; r < R; r += NTH) {
        int e = __ldcg(a.ws.ids + r);
        if ((unsigned)e >= (unsigned)E) {
            set_device_error(a.ws.status, MOE_DEV_BAD_ROUTE, r);
            e = 0;
        }
        if (CACHE && r == tid) e_first = e;
        atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    if (ns && tid == 0) cnt[E] = a.T;
    __syncthreads();
    if (warp == 0) warp_exclusive_scan(cnt, offs, EE, lane);
    if (warp == 1) {
        for (int e = lane; e < EE; e += 32) tcnt[e] = (cnt[e] + a.tile_rows - 1) / a.tile_rows;
        __syncwarp();
        warp_exclusive_scan(tcnt, toff, EE, lane);
    }
    __syncthreads();
    for (int e = tid; e < EE; e += NTH) {
        if (e < E) a.ws.counts[e] = cnt[e];
        a.ws.offsets[e] = offs[e];
        const int n = tcnt[e], base = toff[e];
        for (int k = 0; k < n && base + k < a.ws.max_tiles; k++) {
            const int st = k * a.tile_rows;
            a.ws.tiles[base + k] = make_int4(e, offs[e] + st, min(a.tile_rows, cnt[e] - st), 0);
        }
    }
    if (tid == 0) {
        a.ws.offsets[EE] = offs[EE];
        *a.ws.n_tiles = min(toff[EE], a.ws.max_tiles);
        if (toff[EE] > a.ws.max_tiles) set_device_error(a.ws.status, MOE_DEV_BAD_ROUTE, -1);
    }
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = 0; base < R; base += NTH) {
        for (int i = tid; i < NW * EE; i += NTH) wcnt[i] = 0;
        __syncthreads();
        const int r = base + tid;
        int e = -1;
        if (r < R) {
            if (CACHE && base == 0) {
                e = e_first;
            } else {
                e = __ldcg(a.ws.ids + r);
                if ((unsigned)e >= (unsigned)E) e = 0;
            }
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank_w = __popc(peers & lt_mask);
        if (e >= 0 && rank_w == 0) wcnt[warp * EE + e] = __popc(peers);
        __syncthreads();
        if (e >= 0) {
            int rank = run[e] + rank_w;
            for (int w = 0; w < warp; w++) rank += wcnt[w * EE + e];
            const int pos = offs[e] + rank;
            const int t = r / K, s = r - t * K;
            a.ws.perm_token[pos] = t;
            a.ws.perm_slot[pos] = s;
            a.ws.perm_w[pos] = (CACHE && base == 0) ? w_first : __ldcg(a.ws.route_w + r);
            a.ws.loc[t * KK + s] = pos;
        }
        __syncthreads();
        for (int x = tid; x < EE; x += NTH) {
            int s = 0;
            for (int w = 0; w < NW; w++) s += wcnt[w * EE + x];
            run[x] += s;
        }
        __syncthreads();
    }
    if (ns) {
        for (int t = tid; t < a.T; t += NTH) {
            const int pos = offs[E] + t;
            a.ws.perm_token[pos] = t;
            a.ws.perm_slot[pos] = K;
            a.ws.perm_w[pos] = 1.0f;
            a.ws.loc[t * KK + K] = pos;
        }
    }
    if (tid == 0) a.ws.tickets[0] = 0u;  // re-arm for the next launch
}

// The same permutation by one warp, one lane per expert (E + n_shared <= 32,
// at most 256 routes: 8 per lane): each lane holds its routes' experts and
// weights in registers, ranks them within each 32-route chunk by matching
// lanes, and the counts, offsets, tile counts and tile offsets come from two
// warp scans; no shared-memory histogram and no block barrier.  Same tables
// as build_permutation, element for element.
constexpr int kWarpPermRoutes = 256;
__device__ void build_permutation_warp(const RouteArgs &a, int32_t *scr) {
    const int lane = threadIdx.x & 31;
    const int E = a.bp.E, K = a.bp.K, ns = a.bp.n_shared, EE = E + ns, KK = K + ns, T = a.T, R = T * K;
    const int TR = a.tile_rows;
    constexpr int RPL = kWarpPermRoutes / 32;
    const unsigned full = 0xffffffffu, lt = (1u << lane) - 1u;
    int ev[RPL];
    float wv[RPL];
#pragma unroll
    for (int i = 0; i < RPL; i++) {
        const int r = lane + 32 * i;
        ev[i] = r < R ? __ldcg(a.ws.ids + r) : -1;
        wv[i] = r < R ? __ldcg(a.ws.route_w + r) : 0.f;
    }
    // per 32-route chunk: each route's rank among the routes to its expert so
    // far; lane x counts expert x's routes
    int rk[RPL];
    int run = 0;
#pragma unroll
    for (int i = 0; i < RPL; i++) {
        rk[i] = 0;
        if (32 * i >= R) continue;
        if (lane + 32 * i < R && (unsigned)ev[i] >= (unsigned)E) {
            set_device_error(a.ws.status, MOE_DEV_BAD_ROUTE, lane + 32 * i);
            ev[i] = 0;
        }
        const unsigned peers = __match_any_sync(full, ev[i]);
        rk[i] = __shfl_sync(full, run, ev[i] & 31) + __popc(peers & lt);
        scr[lane] = 0;
        __syncwarp();
        if (ev[i] >= 0 && !(peers & lt)) scr[ev[i]] = __popc(peers);
        __syncwarp();
        run += scr[lane];
        __syncwarp();
    }
    const int c = lane < E ? run : (ns && lane == E) ? T : 0;
    const int tc = lane < EE ? (c + TR - 1) / TR : 0;
    int incl = c, inct = tc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(full, incl, o), u = __shfl_up_sync(full, inct, o);
        if (lane >= o) {
            incl += v;
            inct += u;
        }
    }
    const int offs = incl - c, toff = inct - tc;
    const int total = __shfl_sync(full, incl, 31), all_tiles = __shfl_sync(full, inct, 31);
    if (lane < E) a.ws.counts[lane] = c;
    if (lane < EE) a.ws.offsets[lane] = offs;
    for (int k = 0; k < tc && toff + k < a.ws.max_tiles; k++)
        a.ws.tiles[toff + k] = make_int4(lane, offs + k * TR, min(TR, c - k * TR), 0);
    if (lane == 0) {
        a.ws.offsets[EE] = total;
        *a.ws.n_tiles = min(all_tiles, a.ws.max_tiles);
        if (all_tiles > a.ws.max_tiles) set_device_error(a.ws.status, MOE_DEV_BAD_ROUTE, -1);
    }
#pragma unroll
    for (int i = 0; i < RPL; i++) {
        if (32 * i >= R) break;
        const int r = lane + 32 * i;
        const int pos = __shfl_sync(full, offs, ev[i] & 31) + rk[i];
        if (r < R) {
            const int t = r / K, s = r - t * K;
            a.ws.perm_token[pos] = t;
            a.ws.perm_slot[pos] = s;
            a.ws.perm_w[pos] = wv[i];
            a.ws.loc[t * KK + s] = pos;
        }
    }
    if (ns) {
        const int oE = __shfl_sync(full, offs, E & 31);
        for (int t = lane; t < T; t += 32) {
            a.ws.perm_token[oE + t] = t;
            a.ws.perm_slot[oE + t] = K;
            a.ws.perm_w[oE + t] = 1.0f;
            a.ws.loc[t * KK + K] = oE + t;
        }
    }
    if (lane == 0) a.ws.tickets[0] = 0u;  // re-arm for the next launch
}

// Normalise one token row held in registers (XC chunks of 8 per thread) into
// xh (shared memory; skipped when null) and, if `store`, into the workspace
// copies: bf16 natural order, and as a.forms asks, fp16 (the GEMV and the fp16
// grouped GEMM) and the grouped GEMM's pair order (its bf16 variant).  Returns
// this thread's sum of x_hat^2.
template <int NTH, int XC>
__device__ __forceinline__ float normalise_row(const RouteArgs &a, const uint4 (&xv)[XC], const float4 (&gm)[XC][2],
                                               int t, double r, uint16_t *xh, bool store) {
    const int H = a.bp.H, nchunk = H / 8;
    const float r32 = (float)r;
    float xs = 0.f;
#pragma unroll
    for (int j = 0; j < XC; j++) {
        const int c = threadIdx.x + NTH * j;
        if (c >= nchunk) continue;
        const uint32_t w4[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
        const float gg[8] = {gm[j][0].x, gm[j][0].y, gm[j][0].z, gm[j][0].w,
                             gm[j][1].x, gm[j][1].y, gm[j][1].z, gm[j][1].w};
        uint32_t hb[8];
#pragma unroll
        for (int q = 0; q < 8; q++) hb[q] = norm_elem((w4[q >> 1] >> (16 * (q & 1))) & 0xFFFFu, gg[q], r32, r);
#pragma unroll
        for (int q = 0; q < 8; q++) xs = fmaf(__uint_as_float(hb[q] << 16), __uint_as_float(hb[q] << 16), xs);
        const uint4 nat = make_uint4(hb[0] | hb[1] << 16, hb[2] | hb[3] << 16, hb[4] | hb[5] << 16,
                                     hb[6] | hb[7] << 16);
        if (xh) *reinterpret_cast<uint4 *>(xh + 8 * c) = nat;
        if (store) {
            const size_t go = (size_t)t * H + 8 * c;
            *reinterpret_cast<uint4 *>(a.ws.xhat + go) = nat;
            if (a.forms & kFormMma) {
                // pair order inside each 8-element chunk: (e0,e4),(e1,e5),(e2,e6),(e3,e7)
                *reinterpret_cast<uint4 *>(a.ws.xhat_mma + go) = make_uint4(
                    hb[0] | hb[4] << 16, hb[1] | hb[5] << 16, hb[2] | hb[6] << 16, hb[3] | hb[7] << 16);
            }
            if (a.forms & kFormF16) {
                uint32_t f[8];
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    __half hh = __float2half_rn(__uint_as_float(hb[q] << 16));  // exact for |x_hat| >= 2^-17
                    f[q] = *reinterpret_cast<uint16_t *>(&hh);
                }
                *reinterpret_cast<uint4 *>(a.ws.xhat16 + go) =
                    make_uint4(f[0] | f[1] << 16, f[2] | f[3] << 16, f[4] | f[5] << 16, f[6] | f[7] << 16);
            }
            if (a.xhat_out) *reinterpret_cast<uint4 *>(a.xhat_out + go) = nat;
        }
    }
    return xs;
}

// Router logit of expert e (row w, shared or global memory) for one x_hat row
// in shared memory, by one warp: products of two bf16 are exact in fp32 and
// enter the sums through FMA; each 8-product chunk is summed first (8
// roundings), chunk sums are accumulated per lane (per_lane roundings), then a
// 5-level butterfly and the bias: every partial sum is bounded by Σ|p|, so the
// error is <= gamma_n (Σ|p| + |b| + |l|) with n = 8 + per_lane + 6; the bound
// returned is doubled as a safety margin.
template <bool GLOBAL_ROW>
__device__ __forceinline__ void router_logit(const uint16_t *wrow, const uint16_t *xh, float b, int H, int lane,
                                             float &l, float &bound) {
    const int nchunk = H / 8, per_lane = (nchunk + 31) / 32, chain = 8 + per_lane + 6;
    float acc = 0.f, sab = 0.f;
    // global rows: the loads of four chunks are issued before their use
#pragma unroll 4
    for (int ch = lane; ch < nchunk; ch += 32) {
        const uint4 wv = GLOBAL_ROW ? __ldg(reinterpret_cast<const uint4 *>(wrow + 8 * ch))
                                    : *reinterpret_cast<const uint4 *>(wrow + 8 * ch);
        const uint4 xq = *reinterpret_cast<const uint4 *>(xh + 8 * ch);
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w}, xx[4] = {xq.x, xq.y, xq.z, xq.w};
        float cs = 0.f;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const float w0 = __uint_as_float(ww[q] << 16), w1 = __uint_as_float(ww[q] & 0xFFFF0000u);
            const float x0 = __uint_as_float(xx[q] << 16), x1 = __uint_as_float(xx[q] & 0xFFFF0000u);
            cs = fmaf(x0, w0, cs);
            cs = fmaf(x1, w1, cs);
            sab = fmaf(fabsf(x0), fabsf(w0), sab);
            sab = fmaf(fabsf(x1), fabsf(w1), sab);
        }
        acc += cs;
    }
    const float sm = warp_sum_f(acc), ab = warp_sum_f(sab);
    l = sm + b;
    bound = 2.0f * (float)chain * 0x1p-24f * (ab + fabsf(b) + fabsf(l)) + 1e-30f;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(const float *local, uint32_t rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Small batches: grid (T, C), cluster (1, C): CTA c of token t's cluster
// computes the logits of experts [c*epc, c*epc + epc) (router rows staged in
// shared memory by a bulk copy when STAGED, read from global memory
// otherwise) into CTA 0's shared memory; CTA 0 selects the top-k.
template <bool STAGED>
__global__ void __launch_bounds__(kRouteThreads) moe_route_small_kernel(RouteArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int H = a.bp.H, E = a.bp.E;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t = blockIdx.x;
    const uint32_t rank = cluster_ctarank();
    const int epc = a.epc, e0 = (int)rank * epc, ne = max(0, min(epc, E - e0));
    // the gate/up GEMV (one persistent CTA per SM, waiting for this grid's
    // results) may take the SMs this kernel leaves free and set itself up
    asm volatile("griddepcontrol.launch_dependents;");
    // layout: [router rows] [permutation counters] [x_hat row] [logits E] [bounds E] [exact logits E]
    // [candidates E]
    const size_t rows_b = STAGED ? (size_t)epc * H * 2 : 0;
    const size_t head = (rows_b + perm_smem_bytes(E) + 127) & ~(size_t)127;  // rows, then counters
    uint16_t *wsm = reinterpret_cast<uint16_t *>(smem);
    uint16_t *xh = reinterpret_cast<uint16_t *>(smem + head);
    float *lg = reinterpret_cast<float *>(smem + head + (size_t)H * 2);
    float *lb = lg + E;
    double *exs = reinterpret_cast<double *>(smem + ((head + (size_t)H * 2 + 8 * (size_t)E + 7) & ~(size_t)7));
    uint16_t *cand = reinterpret_cast<uint16_t *>(exs + E);
    __shared__ int s_ncand;
    __shared__ int s_maxexp[kRouteWarps];
    __shared__ Comp s_acc[kRouteWarps];
    __shared__ double s_r;
    __shared__ int s_flag;
    __shared__ __align__(8) uint64_t wbar;

    if (STAGED && tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&wbar)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const size_t bytes = (size_t)ne * H * 2;
        asm volatile("{ .reg .b64 t; mbarrier.arrive.expect_tx.shared::cta.b64 t, [%0], %1; }" ::"r"(smem_u32(&wbar)),
                     "r"((uint32_t)bytes)
                     : "memory");
        const unsigned char *src = reinterpret_cast<const unsigned char *>(a.router_w + (size_t)e0 * H);
        for (size_t off = 0; off < bytes; off += 32768) {
            const uint32_t n = (uint32_t)min((size_t)32768, bytes - off);
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(reinterpret_cast<unsigned char *>(wsm) + off)),
                "l"(src + off), "r"(n), "r"(smem_u32(&wbar))
                : "memory");
        }
    }
    // launched as a programmatic dependent of the previous forward's last
    // kernel: the router rows (constant) are on their way; x is its output
    asm volatile("griddepcontrol.wait;" ::: "memory");
    MOE_PHASE_MARK(0);
    // ---------------------------------------------------------------- norm
    const int nchunk = H / 8;
    float4 gm[kXC][2];
    uint4 xv[kXC];
    const uint4 *xr = reinterpret_cast<const uint4 *>(a.x + (size_t)t * H);
#pragma unroll
    for (int j = 0; j < kXC; j++) {
        const int c = tid + kRouteThreads * j;
        const float4 *g4 = reinterpret_cast<const float4 *>(a.gamma) + 2 * c;
        xv[j] = c < nchunk ? __ldg(xr + c) : make_uint4(0, 0, 0, 0);
        gm[j][0] = c < nchunk ? __ldg(g4) : make_float4(0.f, 0.f, 0.f, 0.f);
        gm[j][1] = c < nchunk ? __ldg(g4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const double ss = sumsq_block<kRouteThreads, kXC>(xv, lane, warp, s_maxexp, s_acc);
    MOE_PHASE_MARK(1);
    if (tid == 0) s_r = rsqrt_d(ss * a.inv_h + a.bp.eps);
    __syncthreads();
    MOE_PHASE_MARK(2);
    normalise_row<kRouteThreads, kXC>(a, xv, gm, t, s_r, xh, rank == 0);
    __syncthreads();
    MOE_PHASE_MARK(3);
    // -------------------------------------------------------------- router
    bool rows_ok = true;
    if (STAGED) {
        uint32_t ok = 0;
        uint64_t c0, c1;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(c0));
        for (;;) {
            asm volatile(
                "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0; selp.u32 %0, 1, 0, p; }"
                : "=r"(ok)
                : "r"(smem_u32(&wbar))
                : "memory");
            if (ok) break;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(c1));
            if (c1 - c0 > 2000000000ull) {
                set_device_error(a.ws.status, MOE_DEV_WAIT_TIMEOUT, 70);
                break;
            }
        }
        rows_ok = ok != 0;
    }
    if (rows_ok) {
        for (int el = warp; el < ne; el += kRouteWarps) {
            const int e = e0 + el;
            float l, bd;
            if (!a.router_exact) {
                if (STAGED)
                    router_logit<false>(wsm + (size_t)el * H, xh, a.router_b[e], H, lane, l, bd);
                else
                    router_logit<true>(a.router_w + (size_t)e * H, xh, a.router_b[e], H, lane, l, bd);
            } else {
                l = (float)exact_logit(xh, a.router_w, a.router_b, e, H, lane);
                bd = 0.f;
            }
            if (lane == 0) {
                st_cluster_f32(lg + e, 0, l);
                st_cluster_f32(lb + e, 0, bd);
            }
        }
    }
    // every CTA of the cluster arrives, whatever happened above
    cluster_sync();
    MOE_PHASE_MARK(4);
    if (rank != 0) return;
    // ---------------------------------------------------------- top-k + softmax
    // warp 0 selects; the candidates it cannot order are recomputed exactly by
    // all warps of the CTA
    float my_v = -INFINITY;
    int my_i = kInvalid;
    bool need = false;
    if (warp == 0) need = topk_select<false>(lg, lb, a, lane, my_v, my_i, exs, cand, &s_ncand);
    __syncthreads();
    if (s_ncand) exact_candidates(a, xh, 0, cand, &s_ncand, 1, exs, warp, kRouteWarps, lane);
    __syncthreads();
    if (warp == 0) topk_finish(a, t, lane, need, exs, my_v, my_i);
    MOE_PHASE_MARK(5);
    // ---------------------------------- last token to finish: permutation
    __threadfence();
    __syncthreads();
    if (tid == 0) s_flag = (atomicAdd(a.ws.tickets, 1u) == (unsigned)a.T - 1u);
    __syncthreads();
    if (!s_flag) return;
    __threadfence();
    MOE_PHASE_MARK(6);
    if (E + a.bp.n_shared <= 32 && a.T * a.bp.K <= kWarpPermRoutes) {
        if (warp == 0) build_permutation_warp(a, reinterpret_cast<int32_t *>(smem + rows_b));
    } else {
        build_permutation<true>(a, smem + rows_b);
    }
    MOE_PHASE_MARK(7);
}

// Larger batches (T > 32): four kernels chained by programmatic dependent
// launch.
//  * moe_route_norm_kernel: a CTA per token normalises it (x_hat in the forms
//    the expert kernels read) and records an upper bound of |x_hat|; a warp
//    per router row records an upper bound of |w|; the expert counts are
//    zeroed for the top-k kernel.
//  * moe_router_gemm_kernel: the logits over 64-token x 64-expert tiles on
//    the tensor cores, K split over grid.z when the tiles alone do not fill
//    the GPU.  Products of two bf16 are exact; each 32-element k-chunk is
//    summed by two MMAs into a zero accumulator (budgeted as 32 roundings of
//    the chunk's absolute product sum) and added to a compensated (Kahan)
//    running total, whose error stays within 2u of the sum of |chunk sums|
//    whatever the number of chunks; the K-split partials and the bias add
//    one rounding each.
//  * moe_route_topk_kernel: a warp per token sums the K-split partials in a
//    fixed order, adds the bias and the bound 2 gamma_n (|x_hat| |w| +
//    |b| + |l|) (Cauchy-Schwarz bounds sum |x_i w_i|), and selects the top-k,
//    recomputing exactly whatever the bounds cannot order; it adds its routes
//    to the expert counts.
//  * moe_permute_kernel: the token->expert permutation, a CTA per expert.
constexpr int kGT = 64, kGE = 64, kGK = 32;  // GEMM tile: tokens x experts, k-chunk
constexpr int kMaxKSplit = 16;               // K splits of the logits GEMM

// Roundings a product can pass through in the large-batch logits, with a
// margin: the chunk's FMAs, the compensated total (2, and its second-order
// term, counted as 4 more), the K-split partials, the bias.
__device__ __forceinline__ int router_chain(int ks) { return kGK + 6 + ks + 2; }

constexpr int kNormThreads = 128;                          // one token per CTA of the norm kernel
constexpr int kNormXC = kRouteThreads * kXC / kNormThreads;  // 16-byte chunks of the row per thread

__global__ void __launch_bounds__(kNormThreads) moe_route_norm_kernel(RouteArgs a) {
    const int H = a.bp.H, E = a.bp.E;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // launched as a programmatic dependent (rows only, no router: the
    // attention's norm) it waits for the previous kernel, whose output x is,
    // and lets its dependent launch at once (it prefetches weights meanwhile)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!a.router_w) asm volatile("griddepcontrol.launch_dependents;");
    if ((int)blockIdx.x >= a.T) {
        // |w| of router rows, a warp per row: a sum of squares (relative error
        // below 2e-6), one correctly rounded square root, then a margin well
        // above both
        const int e = ((int)blockIdx.x - a.T) * (kNormThreads / 32) + warp;
        if (e < E) {
            const uint4 *wr = reinterpret_cast<const uint4 *>(a.router_w + (size_t)e * H);
            uint4 wv[kRowChunks];  // the whole row's loads in flight at once
#pragma unroll
            for (int i = 0; i < kRowChunks; i++) {
                const int c = lane + 32 * i;
                wv[i] = c < H / 8 ? __ldg(wr + c) : make_uint4(0, 0, 0, 0);
            }
            float sw = 0.f;
#pragma unroll
            for (int i = 0; i < kRowChunks; i++) {
                const uint4 v = wv[i];
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const float lo = __uint_as_float(w4[q] << 16), hi = __uint_as_float(w4[q] & 0xFFFF0000u);
                    sw = fmaf(lo, lo, fmaf(hi, hi, sw));
                }
            }
            const float wn = sqrtf(warp_sum_f(sw)) * (1.0f + 0x1p-14f);
            if (lane == 0) a.ws.wnorm[e] = wn;
        }
        asm volatile("griddepcontrol.launch_dependents;");
        return;
    }
    // one token per CTA: the row and gamma in registers (kNormXC chunks of 8 per thread)
    __shared__ int s_maxexp[kNormThreads / 32];
    __shared__ Comp s_acc[kNormThreads / 32];
    __shared__ float s_xs[kNormThreads / 32];
    __shared__ double s_r;
    const int t = blockIdx.x, nchunk = H / 8;
    if (t == 0)  // expert counts start from zero; the top-k kernel adds its routes
        for (int e = tid; e <= E; e += kNormThreads) a.ws.counts[e] = 0;
    float4 gm[kNormXC][2];
    uint4 xv[kNormXC];
    const uint4 *xr = reinterpret_cast<const uint4 *>(a.x + (size_t)t * H);
#pragma unroll
    for (int j = 0; j < kNormXC; j++) {
        const int c = tid + kNormThreads * j;
        const float4 *g4 = reinterpret_cast<const float4 *>(a.gamma) + 2 * c;
        xv[j] = c < nchunk ? __ldg(xr + c) : make_uint4(0, 0, 0, 0);
        gm[j][0] = c < nchunk ? __ldg(g4) : make_float4(0.f, 0.f, 0.f, 0.f);
        gm[j][1] = c < nchunk ? __ldg(g4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const double ss = sumsq_block<kNormThreads, kNormXC>(xv, lane, warp, s_maxexp, s_acc);
    if (tid == 0) s_r = rsqrt_d(ss * a.inv_h + a.bp.eps);
    __syncthreads();
    const float xs = warp_sum_f(normalise_row<kNormThreads, kNormXC>(a, xv, gm, t, s_r, nullptr, true));
    if (lane == 0) s_xs[warp] = xs;
    __syncthreads();
    if (tid == 0) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kNormThreads / 32; w++) tot += s_xs[w];
        // |x_hat| with a margin above the error of the sum (positive terms) and of the root
        a.ws.xnorm[t] = sqrtf(tot) * (1.0f + 0x1p-14f);
    }
    // the logits GEMM may launch once every CTA is here: launched earlier, its
    // CTAs would take SM slots as the norm CTAs happen to leave them, not
    // evenly, and some SMs would run several of its equal-sized CTAs
    asm volatile("griddepcontrol.launch_dependents;");
}

// lpart[kz][t][e] = sum over the kz-th K range of x_hat[t][k] * W[e][k], on
// the tensor cores: each 32-element k-chunk is two bf16 mma.sync m16n8k16
// into a zero fp32 accumulator (the products of two bf16 are exact; the bound
// budgets 32 roundings of 2^-24 of the chunk's absolute product sum for the
// two MMAs, twice what an accumulation with 22 significant bits can lose), and
// the chunk sums are added to Kahan totals (compensated, as before).  A CTA's
// four warps own 32 tokens x 32 experts each of the 64 x 64 tile; each thread
// reads 16 contiguous bytes of a token row and of a router row per chunk and
// hands them to the two MMAs as if their k order were permuted (A and B see
// the same permutation; the dot product does not depend on the order).  The
// next chunk's rows are loaded while the current one is multiplied.
constexpr int kGThreads = 128;

__device__ __forceinline__ void rmma_bf16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1, bool zero) {
    if (zero)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%10,%10,%10};\n"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kGThreads) moe_router_gemm_kernel(const uint16_t *xhat, const uint16_t *w, int T,
                                                                    int E, int H, int kc_per_split, float *lpart) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t4 = lane & 3;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // x_hat comes from the norm kernel
    const int tb = blockIdx.x * kGT + 32 * (warp & 1), eb = blockIdx.y * kGE + 32 * (warp >> 1), kz = blockIdx.z;
    const int nkc = (H + kGK - 1) / kGK;
    const int kc0 = kz * kc_per_split, kc1 = min(nkc, kc0 + kc_per_split);
    // this thread's rows: tokens tb + 16 mi + g (+ 8), experts eb + 8 ni + g
    const uint16_t *xr[2][2];
    const uint16_t *wr[4];
#pragma unroll
    for (int mi = 0; mi < 2; mi++)
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int t = tb + 16 * mi + 8 * h + g;
            xr[mi][h] = t < T ? xhat + (size_t)t * H + 8 * t4 : nullptr;
        }
#pragma unroll
    for (int ni = 0; ni < 4; ni++) {
        const int e = eb + 8 * ni + g;
        wr[ni] = e < E ? w + (size_t)e * H + 8 * t4 : nullptr;
    }
    auto fetch = [&](int kc, uint4 (&a)[2][2], uint4 (&b)[4]) {
        const int k = kc * kGK;
#pragma unroll
        for (int mi = 0; mi < 2; mi++)
#pragma unroll
            for (int h = 0; h < 2; h++)
                a[mi][h] = xr[mi][h] ? __ldg(reinterpret_cast<const uint4 *>(xr[mi][h] + k)) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int ni = 0; ni < 4; ni++)
            b[ni] = wr[ni] ? __ldg(reinterpret_cast<const uint4 *>(wr[ni] + k)) : make_uint4(0, 0, 0, 0);
    };
    float tot[2][4][4], cmp[2][4][4];  // compensated running totals
#pragma unroll
    for (int mi = 0; mi < 2; mi++)
#pragma unroll
        for (int ni = 0; ni < 4; ni++)
#pragma unroll
            for (int q = 0; q < 4; q++) tot[mi][ni][q] = cmp[mi][ni][q] = 0.f;
    uint4 a[2][2], b[4], an[2][2], bn[4];
    if (kc0 < kc1) fetch(kc0, a, b);
    for (int kc = kc0; kc < kc1; kc++) {
        if (kc + 1 < kc1) fetch(kc + 1, an, bn);
#pragma unroll
        for (int mi = 0; mi < 2; mi++)
#pragma unroll
            for (int ni = 0; ni < 4; ni++) {
                float part[4];
                rmma_bf16(part, a[mi][0].x, a[mi][1].x, a[mi][0].y, a[mi][1].y, b[ni].x, b[ni].y, true);
                rmma_bf16(part, a[mi][0].z, a[mi][1].z, a[mi][0].w, a[mi][1].w, b[ni].z, b[ni].w, false);
#pragma unroll
                for (int q = 0; q < 4; q++) {  // Kahan: tot + cmp carries the sum of the chunk sums
                    const float y = part[q] - cmp[mi][ni][q];
                    const float tn = tot[mi][ni][q] + y;
                    cmp[mi][ni][q] = (tn - tot[mi][ni][q]) - y;
                    tot[mi][ni][q] = tn;
                }
            }
        if (kc + 1 < kc1) {
#pragma unroll
            for (int mi = 0; mi < 2; mi++) {
                a[mi][0] = an[mi][0];
                a[mi][1] = an[mi][1];
            }
#pragma unroll
            for (int ni = 0; ni < 4; ni++) b[ni] = bn[ni];
        }
    }
    // the top-k kernel may launch now (its CTAs then find the SMs free and spread evenly)
    asm volatile("griddepcontrol.launch_dependents;");
#pragma unroll
    for (int mi = 0; mi < 2; mi++)
#pragma unroll
        for (int ni = 0; ni < 4; ni++)
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int t = tb + 16 * mi + g + 8 * (q >> 1), e = eb + 8 * ni + 2 * t4 + (q & 1);
                if (t < T && e < E) lpart[((size_t)kz * T + t) * E + e] = tot[mi][ni][q];
            }
}

// A warp per token: logits and bounds into shared memory, then top-k + softmax
// (the exact logits of uncertain tokens by all warps of the CTA); the CTA's
// routes are counted per expert in shared memory and added to the expert
// counts.
__global__ void __launch_bounds__(kRouteThreads, 2) moe_route_topk_kernel(RouteArgs a, const float *lpart, int ks) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int E = a.bp.E, H = a.bp.H, K = a.bp.K;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    double *exs = reinterpret_cast<double *>(smem);                                    // [8][E]
    float *lg = reinterpret_cast<float *>(smem + (size_t)kRouteWarps * E * 8) + (size_t)warp * 2 * E;  // [8][2][E]
    float *lb = lg + E;
    uint16_t *cand = reinterpret_cast<uint16_t *>(smem + (size_t)kRouteWarps * E * 16);  // [8][E]
    __shared__ int s_ncand[kRouteWarps];
    __shared__ int s_hist[MOE_MAX_EXPERTS];
    for (int e = tid; e < E; e += kRouteThreads) s_hist[e] = 0;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // partials from the GEMM, norms from the norm kernel
    const int t0 = blockIdx.x * kRouteWarps, t = t0 + warp;
    float my_v = -INFINITY;
    int my_i = kInvalid;
    bool need = false;
    if (t < a.T) {
        const float chain = (float)router_chain(ks), xn = __ldcg(a.ws.xnorm + t);
        // the K-split partials of each logit summed in K order (into lg), their
        // loads issued ahead: all splits at once for up to 32 experts (one per
        // lane), 16-byte loads of eight splits at a time for wider rows
        if (E <= 32) {
            float pv[kMaxKSplit];
#pragma unroll
            for (int kz = 0; kz < kMaxKSplit; kz++)
                pv[kz] = (kz < ks && lane < E) ? __ldcg(lpart + ((size_t)kz * a.T + t) * E + lane) : 0.f;
            float sum = 0.f;
#pragma unroll
            for (int kz = 0; kz < kMaxKSplit; kz++)
                if (kz < ks) sum += pv[kz];
            if (lane < E) lg[lane] = sum;
        } else if (E % 4 == 0) {
            const int nv = E / 4;  // float4 per partial row: lane owns float4 lane and lane + 32
            float4 sum[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
            for (int k0 = 0; k0 < ks; k0 += 8) {
                float4 pv[8][2];
#pragma unroll
                for (int i = 0; i < 8; i++)
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const int v = lane + 32 * h;
                        pv[i][h] = (k0 + i < ks && v < nv)
                                       ? __ldcg(reinterpret_cast<const float4 *>(lpart + ((size_t)(k0 + i) * a.T + t) * E) + v)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                for (int i = 0; i < 8; i++)
                    if (k0 + i < ks)
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            sum[h].x += pv[i][h].x;
                            sum[h].y += pv[i][h].y;
                            sum[h].z += pv[i][h].z;
                            sum[h].w += pv[i][h].w;
                        }
            }
#pragma unroll
            for (int h = 0; h < 2; h++)
                if (lane + 32 * h < nv) reinterpret_cast<float4 *>(lg)[lane + 32 * h] = sum[h];
        } else {
            for (int e = lane; e < E; e += 32) {
                float sum = 0.f;
                for (int kz = 0; kz < ks; kz++) sum += __ldcg(lpart + ((size_t)kz * a.T + t) * E + e);
                lg[e] = sum;
            }
        }
        __syncwarp();
        for (int e = lane; e < E; e += 32) {
            const float b = a.router_b[e], l = lg[e] + b;
            lg[e] = l;
            lb[e] = 2.0f * chain * 0x1p-24f * (xn * __ldcg(a.ws.wnorm + e) + fabsf(b) + fabsf(l)) + 1e-30f;
        }
        __syncwarp();
        need = topk_select<false>(lg, lb, a, lane, my_v, my_i, exs + (size_t)warp * E, cand + (size_t)warp * E,
                                  &s_ncand[warp]);
    } else if (lane == 0) {
        s_ncand[warp] = 0;
    }
    __syncthreads();
    exact_candidates(a, a.ws.xhat + (size_t)t0 * H, (size_t)H, cand, s_ncand, kRouteWarps, exs, warp, kRouteWarps,
                     lane);
    __syncthreads();
    if (t < a.T) {
        const int id = topk_finish(a, t, lane, need, exs + (size_t)warp * E, my_v, my_i);
        if (lane < K) atomicAdd(&s_hist[id], 1);
    }
    __syncthreads();
    for (int e = tid; e < E; e += kRouteThreads)
        if (s_hist[e]) atomicAdd(a.ws.counts + e, s_hist[e]);
    asm volatile("griddepcontrol.launch_dependents;");
}

// The permutation of a large batch (the same result as build_permutation),
// one CTA per expert (and one for the shared expert).  Every CTA scans the
// expert counts (added up by the top-k kernel) and the tile counts, then
// collects its own expert's routes in route order: warp w owns the w-th
// contiguous segment of the routes; a first pass counts each warp's routes of
// the expert, a scan over warps places the segments, a second pass writes the
// entries (token, slot, weight), the inverse map and the expert's tiles.
constexpr int kPermThreads = 512;
constexpr int kPermWarps = kPermThreads / 32;
constexpr int kPermPer = 16;  // route ids per lane in flight
__host__ __device__ constexpr size_t perm_expert_smem_bytes(int EE) { return (size_t)(4 * (EE + 1) + 2 * 32) * 4; }

__global__ void __launch_bounds__(kPermThreads) moe_permute_kernel(RouteArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the routing result of the previous kernel
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.bp.E, K = a.bp.K, ns = a.bp.n_shared, EE = E + ns, KK = K + ns;
    const int R = a.T * K;
    const int me = blockIdx.x;  // this CTA's expert (E: the shared expert)
    int32_t *cnt = reinterpret_cast<int32_t *>(smem);  // [EE + 1]
    int32_t *offs = cnt + (EE + 1);                     // [EE + 1]
    int32_t *tcnt = offs + (EE + 1);                    // [EE + 1]
    int32_t *toff = tcnt + (EE + 1);                    // [EE + 1]
    int32_t *wn = toff + (EE + 1);                      // [32] this expert's routes per warp segment
    int32_t *wo = wn + 32;                              // [32] their exclusive prefix
    for (int e = tid; e < EE; e += kPermThreads) cnt[e] = e < E ? __ldcg(a.ws.counts + e) : a.T;
    const int seg = (R + kPermWarps - 1) / kPermWarps;
    const int r0 = min(R, warp * seg), r1 = min(R, r0 + seg);
    // pass 1: this warp's routes of `me` (ids out of range count as expert 0,
    // as the top-k kernel never writes one)
    int mine = 0;
    for (int b = r0; b < r1; b += 32 * kPermPer) {
        int ev[kPermPer];
#pragma unroll
        for (int i = 0; i < kPermPer; i++) {
            const int r = b + 32 * i + lane;
            ev[i] = r < r1 ? __ldcg(a.ws.ids + r) : -1;
        }
#pragma unroll
        for (int i = 0; i < kPermPer; i++) {
            const int r = b + 32 * i + lane;
            const int e = (r < r1 && (unsigned)ev[i] >= (unsigned)E) ? 0 : ev[i];
            mine += __popc(__ballot_sync(0xffffffffu, e == me));
        }
    }
    if (lane == 0) wn[warp] = mine;
    __syncthreads();
    if (warp == 0) warp_exclusive_scan(cnt, offs, EE, lane);
    if (warp == 1) {
        for (int e = lane; e < EE; e += 32) tcnt[e] = (cnt[e] + a.tile_rows - 1) / a.tile_rows;
        __syncwarp();
        warp_exclusive_scan(tcnt, toff, EE, lane);
    }
    if (warp == 2) {
        const int v = lane < kPermWarps ? wn[lane] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        wo[lane] = incl - v;
    }
    __syncthreads();
    // counts, offsets and tiles of this expert; the totals by CTA 0
    if (tid == 0) a.ws.offsets[me] = offs[me];
    {
        const int n = tcnt[me], base = toff[me];
        for (int k = tid; k < n && base + k < a.ws.max_tiles; k += kPermThreads) {
            const int st = k * a.tile_rows;
            a.ws.tiles[base + k] = make_int4(me, offs[me] + st, min(a.tile_rows, cnt[me] - st), 0);
        }
    }
    if (me == 0 && tid == 0) {
        a.ws.offsets[EE] = offs[EE];
        *a.ws.n_tiles = min(toff[EE], a.ws.max_tiles);
        if (toff[EE] > a.ws.max_tiles) set_device_error(a.ws.status, MOE_DEV_BAD_ROUTE, -1);
        a.ws.tickets[0] = 0u;  // kept re-armed for the small-batch kernel
    }
    if (me == E) {  // the shared expert: every token, slot K, weight 1
        for (int t = tid; t < a.T; t += kPermThreads) {
            const int pos = offs[E] + t;
            a.ws.perm_token[pos] = t;
            a.ws.perm_slot[pos] = K;
            a.ws.perm_w[pos] = 1.0f;
            a.ws.loc[t * KK + K] = pos;
        }
        return;
    }
    // pass 2: this expert's routes in route order (ids and weights loaded ahead)
    int pos = offs[me] + wo[warp];
    const uint32_t lt = (1u << lane) - 1u;
    for (int b = r0; b < r1; b += 32 * kPermPer) {
        int ev[kPermPer];
        float wv[kPermPer];
#pragma unroll
        for (int i = 0; i < kPermPer; i++) {
            const int r = b + 32 * i + lane;
            ev[i] = r < r1 ? __ldcg(a.ws.ids + r) : -1;
            wv[i] = r < r1 ? __ldcg(a.ws.route_w + r) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kPermPer; i++) {
            const int r = b + 32 * i + lane;
            int e = ev[i];
            if (r < r1 && (unsigned)e >= (unsigned)E) {
                if (me == 0) set_device_error(a.ws.status, MOE_DEV_BAD_ROUTE, r);
                e = 0;
            }
            const bool hit = r < r1 && e == me;
            const uint32_t m = __ballot_sync(0xffffffffu, hit);
            if (hit) {
                const int p = pos + __popc(m & lt);
                const int t = r / K, sl = r - t * K;
                a.ws.perm_token[p] = t;
                a.ws.perm_slot[p] = sl;
                a.ws.perm_w[p] = wv[i];
                a.ws.loc[t * KK + sl] = p;
            }
            pos += __popc(m);
        }
    }
}

// Small-batch geometry: C CTAs per token (a cluster, C <= cmax), epc experts each.
struct SmallGeo {
    int C, epc;
    bool staged;
    size_t smem;
};
SmallGeo small_geo(int H, int E, int cmax) {
    SmallGeo g;
    g.epc = E <= cmax * kRouteWarps ? kRouteWarps : (E + cmax - 1) / cmax;  // one expert per warp if possible
    g.C = (E + g.epc - 1) / g.epc;
    g.staged = (size_t)g.epc * H * 2 <= 160 * 1024;
    const size_t rows_b = g.staged ? (size_t)g.epc * H * 2 : 0;
    const size_t head = (rows_b + perm_smem_bytes(E) + 127) & ~(size_t)127;
    g.smem = ((head + (size_t)H * 2 + 8 * (size_t)E + 7) & ~(size_t)7) + 8 * (size_t)E + 2 * (size_t)E;
    return g;
}

template <bool STAGED>
cudaError_t launch_small(const RouteArgs &a, const SmallGeo &g, cudaStream_t st) {
    static PerDevice<bool> done, nonportable;
    MOE_CUDA_TRY(smem_optin_once(moe_route_small_kernel<STAGED>, done));
    int dev = 0;
    MOE_CUDA_TRY(current_device_slot(&dev));
    if (g.C > 8 && !nonportable.v[dev]) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(moe_route_small_kernel<STAGED>,
                                          cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
        nonportable.v[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.T, g.C);
    cfg.blockDim = dim3(kRouteThreads);
    cfg.dynamicSmemBytes = g.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = g.C;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, moe_route_small_kernel<STAGED>, a);
}

cudaError_t launch_small_geo(const RouteArgs &a, const SmallGeo &g, cudaStream_t st) {
    return g.staged ? launch_small<true>(a, g, st) : launch_small<false>(a, g, st);
}

}  // namespace

int route_ticket_count(int T) { return T + 1; }

// x_hat = bf16(rms_norm(x) * gamma) for T rows of H, by the routing's norm
// kernel alone (no router): the attention block's input norm.  xnorm_scratch
// [T] floats and count_scratch [1] int are the kernel's side outputs.
cudaError_t launch_rms_norm_rows(const uint16_t *x, const float *gamma, int T, int H, double eps, uint16_t *xhat,
                                 float *xnorm_scratch, int32_t *count_scratch, cudaStream_t st) {
    if (H <= 0 || H % 32 != 0 || H / 8 > kRouteThreads * kXC) return cudaErrorInvalidValue;
    BlockParams bp{};
    bp.H = H;
    bp.eps = eps;
    Workspace ws{};
    ws.xhat = xhat;
    ws.xnorm = xnorm_scratch;
    ws.counts = count_scratch;
    RouteArgs a{bp, ws, x, gamma, nullptr, nullptr, T, nullptr, nullptr, nullptr, 0, 0, 0, 0, 1.0 / (double)H};
    return launch_pdl(moe_route_norm_kernel, dim3(T), dim3(kNormThreads), 0, st, a);
}

cudaError_t launch_route(const BlockParams &bp, const Workspace &ws, const uint16_t *x, const float *gamma,
                         const uint16_t *router_w, const float *router_b, int T, int32_t *ids_out, float *rw_out,
                         uint16_t *xhat_out, int tile_rows, int router_exact, int forms, cudaStream_t st) {
    if (bp.H / 8 > kRouteThreads * kXC) return cudaErrorInvalidValue;
    RouteArgs a{bp, ws, x, gamma, router_w, router_b, T, ids_out, rw_out, xhat_out, tile_rows, router_exact, 0,
                forms, 1.0 / (double)bp.H};
    if (T <= 32) {
        // many experts: 16-CTA clusters (a non-portable size) keep every CTA's
        // router rows in shared memory; where such a cluster cannot be
        // launched, 8-CTA clusters read the rows from global memory
        static PerDevice<int> use16s;  // 0: not tried, 1: launches, 2: cannot launch here
        int dev = 0;
        MOE_CUDA_TRY(current_device_slot(&dev));
        int &use16 = use16s.v[dev];
        SmallGeo g = small_geo(bp.H, bp.E, 8);
        if (!g.staged && use16 != 2) {
            const SmallGeo g16 = small_geo(bp.H, bp.E, 16);
            if (g16.staged) {
                a.epc = g16.epc;
                const cudaError_t e = launch_small_geo(a, g16, st);
                if (e == cudaSuccess) {
                    use16 = 1;
                    return cudaSuccess;
                }
                cudaGetLastError();  // a launch-configuration error is not sticky
                use16 = 2;
            }
        }
        a.epc = g.epc;
        MOE_CUDA_TRY(launch_small_geo(a, g, st));
        return cudaGetLastError();
    }
    static PerDevice<bool> donet;
    int n_sm = 0, dev = 0;
    MOE_CUDA_TRY(current_device_slot(&dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
    // norm, a CTA per token (+ the router rows' norms, a warp per row)
    moe_route_norm_kernel<<<T + (bp.E + kNormThreads / 32 - 1) / (kNormThreads / 32), kNormThreads, 0, st>>>(a);
    MOE_CUDA_TRY(cudaGetLastError());
    // logits: K split so that the CTAs' waves times their chunks is least (the
    // partials live in y, which is free until the down projection; fewer
    // splits on a tie, since each split adds a rounding to the bound)
    static PerDevice<int> gemm_per_sms;
    int &gemm_per_sm = gemm_per_sms.v[dev];
    if (!gemm_per_sm) {
        MOE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&gemm_per_sm, moe_router_gemm_kernel, kGThreads, 0));
        if (gemm_per_sm < 1) gemm_per_sm = 1;
    }
    const int tiles = ((T + kGT - 1) / kGT) * ((bp.E + kGE - 1) / kGE);
    const int nkc = (bp.H + kGK - 1) / kGK;
    const long long slots = (long long)gemm_per_sm * n_sm;
    int ks = 1, kc_per = nkc;
    long long best = -1;
    for (int k = 1; k <= kMaxKSplit && k <= (nkc / 4 > 0 ? nkc / 4 : 1); k++) {
        const int per = (nkc + k - 1) / k, kk = (nkc + per - 1) / per;
        if (kk > 1 && (size_t)kk * bp.E > (size_t)(bp.K + bp.n_shared) * bp.H) break;
        const long long cost = ((tiles * (long long)kk + slots - 1) / slots) * per;
        if (best < 0 || cost < best) {
            best = cost;
            ks = kk;
            kc_per = per;
        }
    }
    MOE_CUDA_TRY(launch_pdl(moe_router_gemm_kernel, dim3((T + kGT - 1) / kGT, (bp.E + kGE - 1) / kGE, ks), dim3(kGThreads),
                            0, st, (const uint16_t *)ws.xhat, router_w, T, bp.E, bp.H, kc_per, ws.y));
    // top-k + softmax, a warp per token
    const size_t tsm = (size_t)kRouteWarps * bp.E * (8 + 8 + 2);
    MOE_CUDA_TRY(smem_optin_once(moe_route_topk_kernel, donet));
    MOE_CUDA_TRY(launch_pdl(moe_route_topk_kernel, dim3((T + kRouteWarps - 1) / kRouteWarps), dim3(kRouteThreads), tsm,
                            st, a, (const float *)ws.y, ks));
    return launch_pdl(moe_permute_kernel, dim3(bp.E + bp.n_shared), dim3(kPermThreads),
                      perm_expert_smem_bytes(bp.E + bp.n_shared), st, a);
}
