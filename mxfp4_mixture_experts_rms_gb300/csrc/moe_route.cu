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
// Grid: (token groups of G tokens) x (expert chunks of 8*EPW experts).  Every
// CTA normalises its tokens (chunk 0 also stores x_hat), computes the router
// logits of its experts and writes them with an error bound; the last CTA of a
// token group selects the top-k of its tokens; the last CTA of the grid builds
// the permutation.  "Last" is decided by atomic tickets, never by waiting.
//
// Exactness.  Σx² is accumulated exactly as a 128-bit fixed-point integer
// (bf16 squares have 16-bit significands), rounded once to double, and
// r = 1/sqrt(ms + eps) is evaluated in double, matching a plain double
// evaluation.  x_hat = bf16(x * r * gamma) is computed in fp32 and recomputed
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

namespace {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kMaxChunks = 16;  // router row chunks of 256 elements per lane held in registers (H <= 4096)

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
    int epc;  // experts per CTA (router rows staged in shared memory)
};

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
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

__device__ __forceinline__ void warp_best(float &v, int &i) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        float w = __shfl_xor_sync(0xffffffffu, v, o);
        int j = __shfl_xor_sync(0xffffffffu, i, o);
        if (better(w, j, v, i)) {
            v = w;
            i = j;
        }
    }
}

// Exact (fp64) router logit of expert e for an x_hat row in shared memory, by
// one warp: 16-byte loads of the router row, products of two bf16 values are
// exact in fp64, four independent accumulators per lane.
__device__ double exact_logit(const uint16_t *xh, const uint16_t *router_w, const float *router_b, int e, int H,
                              int lane) {
    double acc[4] = {0.0, 0.0, 0.0, 0.0};
    const uint4 *w = reinterpret_cast<const uint4 *>(router_w + (size_t)e * H);
    const uint4 *x = reinterpret_cast<const uint4 *>(xh);
    for (int c = lane; c < H / 8; c += 32) {
        const uint4 wv = __ldg(w + c), xv = x[c];
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w}, xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            acc[q] += (double)__uint_as_float(xx[q] << 16) * (double)__uint_as_float(ww[q] << 16);
            acc[q] += (double)__uint_as_float(xx[q] & 0xFFFF0000u) * (double)__uint_as_float(ww[q] & 0xFFFF0000u);
        }
    }
    double s = warp_sum_d((acc[0] + acc[1]) + (acc[2] + acc[3]));
    return s + (double)router_b[e];
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

// 128-bit unsigned accumulator (hi:lo)
struct U128 {
    unsigned long long lo, hi;
};
__device__ __forceinline__ void u128_add(U128 &a, const U128 &b) {
    unsigned long long lo = a.lo + b.lo;
    a.hi += b.hi + (lo < a.lo ? 1ull : 0ull);
    a.lo = lo;
}
__device__ __forceinline__ U128 u128_shfl_xor(const U128 &a, int o) {
    U128 r;
    r.lo = __shfl_xor_sync(0xffffffffu, a.lo, o);
    r.hi = __shfl_xor_sync(0xffffffffu, a.hi, o);
    return r;
}

constexpr int kXC = 2;  // 16-byte chunks of one x row per thread (H <= 8 * 256 * kXC)

// Exact Σx² of one bf16 row held in registers (kXC chunks of 8 per thread),
// rounded once to double.  Squares are placed on a fixed-point grid relative
// to the largest exponent of the row; a square more than 80 binary places
// below the largest one (|x| < 2^-40 max|x|) contributes less than 2^-60 of
// the sum and is dropped, far below double precision.
__device__ double sumsq_exact(const uint4 (&xv)[kXC], int lane, int warp, int *s_maxexp, U128 *s_acc) {
    int mx = 0;
#pragma unroll
    for (int j = 0; j < kXC; j++) {
        const uint32_t w4[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
        for (int q = 0; q < 4; q++) mx = max(mx, (int)max((w4[q] >> 7) & 0xFFu, (w4[q] >> 23) & 0xFFu));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_maxexp[warp] = mx;
    __syncthreads();
    int emax = 1;
#pragma unroll
    for (int w = 0; w < kRouteWarps; w++) emax = max(emax, s_maxexp[w]);
    // value = M * 2^(ex - 134) with M = 128 + mant (ex >= 1) or M = mant (ex == 0, exponent taken as 1)
    U128 acc{0ull, 0ull};
#pragma unroll
    for (int j = 0; j < kXC; j++) {
        const uint32_t w4[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
        for (int q = 0; q < 8; q++) {
            const uint32_t b = (w4[q >> 1] >> (16 * (q & 1))) & 0xFFFFu;
            const int ex = (b >> 7) & 0xFF;
            const uint32_t M = ex ? (128u + (b & 0x7Fu)) : (b & 0x7Fu);
            const int d = 2 * (emax - (ex ? ex : 1));
            if (M == 0 || d > 80) continue;
            const unsigned long long v = (unsigned long long)M * M;  // < 2^16
            const int sh = 80 - d;                                  // 0..80
            U128 t;
            if (sh == 0) {
                t.lo = v;
                t.hi = 0;
            } else if (sh < 64) {
                t.lo = v << sh;
                t.hi = v >> (64 - sh);
            } else {
                t.lo = 0;
                t.hi = v << (sh - 64);
            }
            u128_add(acc, t);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) u128_add(acc, u128_shfl_xor(acc, o));
    if (lane == 0) s_acc[warp] = acc;
    __syncthreads();
    U128 tot{0ull, 0ull};
#pragma unroll
    for (int w = 0; w < kRouteWarps; w++) u128_add(tot, s_acc[w]);
    if (tot.hi == 0 && tot.lo == 0) return 0.0;
    // value = tot * 2^(2*(emax - 134) - 80); take the top 64 significant bits and round to 53 (ties to even)
    const int lz = tot.hi ? __clzll((long long)tot.hi) : 64 + __clzll((long long)tot.lo);
    const int width = 128 - lz;  // significant bits of tot (<= 108)
    unsigned long long top;
    bool sticky;
    int shift;  // tot = top * 2^shift (+ sticky part)
    if (width > 64) {
        shift = width - 64;
        top = (tot.hi << (64 - shift)) | (tot.lo >> shift);
        sticky = (tot.lo << (64 - shift)) != 0ull;
    } else {
        shift = width - 64;  // <= 0
        top = (width == 64) ? tot.lo : (tot.lo << (-shift));
        sticky = false;
    }
    unsigned long long mant = top >> 11;
    const unsigned long long rem = top & 0x7FFull;
    if (rem > 0x400ull || (rem == 0x400ull && (sticky || (mant & 1ull)))) mant += 1ull;
    return ldexp((double)mant, 11 + shift + 2 * (emax - 134) - 80);
}

// bf16(x * r * gamma) of one element: fp32 value, recomputed in fp64 when it
// lies within its error bound (3 fp32 ulps; 8 used) of a bf16 rounding midpoint.
__device__ __forceinline__ uint32_t norm_elem(uint32_t xb, float gf, float r32, double r) {
    const float xf = __uint_as_float(xb << 16);
    const float v32 = (xf * r32) * gf;
    const uint32_t low = __float_as_uint(v32) & 0xFFFFu;
    const bool safe =
        fabsf(v32) >= 0x1p-120f && fabsf(v32) < 0x1p126f && (low > 0x8000u + 8u || low + 8u < 0x8000u);
    if (safe) {
        __nv_bfloat16 bb = __float2bfloat16_rn(v32);
        return *reinterpret_cast<uint16_t *>(&bb);
    }
    return bf16_from_double_rne((double)xf * r * (double)gf);
}

// Top-k + softmax of one token by one warp: fp32 selection certified by the
// error bounds, exact fp64 re-evaluation of the candidates when the bounds of
// consecutive selections overlap.  l / bd: the token's logits and bounds of
// experts [e0, e0 + ne) -- here always the whole [0, E).
__device__ void topk_token_warp(const float *l, const float *bd, bool global_src, const uint16_t *xh,
                                const RouteArgs &a, int t, int lane) {
    const int E = a.bp.E, K = a.bp.K, H = a.bp.H;
    const bool exact_mode = a.router_exact != 0;
    auto ld = [&](const float *p) { return global_src ? __ldcg(p) : *p; };
    int sel[MOE_MAX_TOPK + 1];
    float selv[MOE_MAX_TOPK + 1];
    float lv[MOE_MAX_EXPERTS / 32];
    uint32_t taken = 0;
    float dmax = 0.f;
#pragma unroll
    for (int q = 0; q < MOE_MAX_EXPERTS / 32; q++) {
        const int j = lane + 32 * q;
        lv[q] = j < E ? ld(l + j) : -INFINITY;
        if (j < E) dmax = fmaxf(dmax, ld(bd + j));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
    for (int r = 0; r <= K; r++) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int q = 0; q < MOE_MAX_EXPERTS / 32; q++) {
            const int j = lane + 32 * q;
            const float v = lv[q];
            if (j >= E || !(v > -INFINITY) || (taken >> q & 1u)) continue;  // NaN / -inf never chosen
            if (better(v, j, bv, bi)) {
                bv = v;
                bi = j;
            }
        }
        warp_best(bv, bi);
        sel[r] = bi;
        selv[r] = bv;
        if (bi != 0x7fffffff && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
    bool certain = !exact_mode;
    if (certain) {
        for (int r = 0; r < K; r++) {
            if (sel[r] == 0x7fffffff) break;
            const float nxt = (sel[r + 1] == 0x7fffffff) ? -INFINITY : selv[r + 1];
            if (!(selv[r] - nxt > 2.0f * dmax)) certain = false;
        }
    }
    double exactv[MOE_MAX_TOPK];
    bool have_exact = false;
    if (!certain) {
        const float thr =
            exact_mode ? -INFINITY : ((sel[K - 1] == 0x7fffffff) ? -INFINITY : selv[K - 1] - 2.0f * dmax);
        double bv_all[MOE_MAX_TOPK];
        int bi_all[MOE_MAX_TOPK];
        for (int r = 0; r < K; r++) {
            bv_all[r] = -INFINITY;
            bi_all[r] = 0x7fffffff;
        }
        for (int j = 0; j < E; j++) {  // warp-uniform
            const float v = ld(l + j);
            if (!(v > -INFINITY) || v < thr) continue;
            const double ex = exact_logit(xh, a.router_w, a.router_b, j, H, lane);
            if (!(ex > -INFINITY)) continue;
            int pos = K;
            for (int r = 0; r < K; r++)
                if (better_d(ex, j, bv_all[r], bi_all[r])) {
                    pos = r;
                    break;
                }
            if (pos < K) {
                for (int r = K - 1; r > pos; r--) {
                    bv_all[r] = bv_all[r - 1];
                    bi_all[r] = bi_all[r - 1];
                }
                bv_all[pos] = ex;
                bi_all[pos] = j;
            }
        }
        for (int r = 0; r < K; r++) {
            sel[r] = bi_all[r];
            exactv[r] = bv_all[r];
            selv[r] = (float)bv_all[r];
        }
        have_exact = true;
    }
    // softmax over the selected raw logits (lane 0), times the weight scale
    if (lane == 0) {
        float m = -INFINITY;
        for (int r = 0; r < K; r++)
            if (sel[r] != 0x7fffffff) m = fmaxf(m, selv[r]);
        float ew[MOE_MAX_TOPK], s = 0.f;
        for (int r = 0; r < K; r++) {
            const float d = have_exact ? (float)(exactv[r] - (double)m) : (selv[r] - m);
            ew[r] = (sel[r] == 0x7fffffff) ? 0.f : expf(d);
            s += ew[r];
        }
        for (int r = 0; r < K; r++) {
            const int id = (sel[r] == 0x7fffffff) ? 0 : sel[r];  // unfilled slot: expert 0, weight 0
            const float w = (s > 0.f) ? a.bp.wscale * (ew[r] / s) : 0.f;
            a.ws.ids[t * K + r] = id;
            a.ws.route_w[t * K + r] = w;
            if (a.ids_out) a.ids_out[t * K + r] = id;
            if (a.rw_out) a.rw_out[t * K + r] = w;
        }
    }
}

template <int G>
__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(RouteArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int H = a.bp.H, E = a.bp.E, K = a.bp.K;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int epc = a.epc;                                                        // experts per CTA
    uint16_t *wsm = reinterpret_cast<uint16_t *>(smem);                           // [epc][H] router rows
    uint16_t *xh = wsm + (size_t)epc * H;                                         // [G][H] x_hat
    float *lg = reinterpret_cast<float *>(xh + (size_t)G * H);                    // [G][epc] logits
    float *lb = lg + G * epc;                                                     // [G][epc] bounds
    __shared__ int s_maxexp[kRouteWarps];
    __shared__ U128 s_acc[kRouteWarps];
    __shared__ double s_r;
    __shared__ int s_flag;
    __shared__ __align__(8) uint64_t wbar;

    const int t0 = blockIdx.x * G;
    const int nt = min(G, a.T - t0);
    const int e0 = blockIdx.y * epc, ne = min(epc, E - e0);
    const int nchunk = H / 8;  // 16-byte chunks per row

    // router rows of this CTA's experts: one contiguous range, bulk-copied during the norm
    if (tid == 0) {
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

    MOE_PHASE_MARK(0);
    // ---------------------------------------------------------------- norm
    // x and gamma are read as 16-byte chunks held in registers: one round trip
    // per row, issued ahead of use.
    const bool store = blockIdx.y == 0;
    float4 gm[kXC][2];
#pragma unroll
    for (int j = 0; j < kXC; j++) {
        const int c = tid + kRouteThreads * j;
        const float4 *g4 = reinterpret_cast<const float4 *>(a.gamma) + 2 * c;
        gm[j][0] = c < nchunk ? __ldg(g4) : make_float4(0.f, 0.f, 0.f, 0.f);
        gm[j][1] = c < nchunk ? __ldg(g4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint4 xv[kXC], xnext[kXC];
    auto load_row = [&](int t, uint4(&dst)[kXC]) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(a.x + (size_t)t * H);
#pragma unroll
        for (int j = 0; j < kXC; j++) {
            const int c = tid + kRouteThreads * j;
            dst[j] = c < nchunk ? __ldg(xr + c) : make_uint4(0, 0, 0, 0);
        }
    };
    if (nt > 0) load_row(t0, xv);
    for (int g = 0; g < nt; g++) {
        const int t = t0 + g;
        if (g + 1 < nt) load_row(t + 1, xnext);
        const double ss = sumsq_exact(xv, lane, warp, s_maxexp, s_acc);
        MOE_PHASE_MARK(1);
        if (tid == 0) s_r = 1.0 / sqrt(ss / (double)H + a.bp.eps);
        __syncthreads();
        MOE_PHASE_MARK(2);
        const double r = s_r;
        const float r32 = (float)r;
#pragma unroll
        for (int j = 0; j < kXC; j++) {
            const int c = tid + kRouteThreads * j;
            if (c >= nchunk) continue;
            const uint32_t w4[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
            const float gg[8] = {gm[j][0].x, gm[j][0].y, gm[j][0].z, gm[j][0].w,
                                 gm[j][1].x, gm[j][1].y, gm[j][1].z, gm[j][1].w};
            uint32_t hb[8];
#pragma unroll
            for (int q = 0; q < 8; q++) hb[q] = norm_elem((w4[q >> 1] >> (16 * (q & 1))) & 0xFFFFu, gg[q], r32, r);
            const uint4 nat = make_uint4(hb[0] | hb[1] << 16, hb[2] | hb[3] << 16, hb[4] | hb[5] << 16,
                                         hb[6] | hb[7] << 16);
            *reinterpret_cast<uint4 *>(xh + g * H + 8 * c) = nat;
            if (store) {
                // prefill pair order inside each 8-element chunk: (e0,e4),(e1,e5),(e2,e6),(e3,e7)
                const uint4 prm = make_uint4(hb[0] | hb[4] << 16, hb[1] | hb[5] << 16, hb[2] | hb[6] << 16,
                                             hb[3] | hb[7] << 16);
                uint32_t f[8];
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    __half hh = __float2half_rn(__uint_as_float(hb[q] << 16));  // exact for |x_hat| >= 2^-14
                    f[q] = *reinterpret_cast<uint16_t *>(&hh);
                }
                const size_t go = (size_t)t * H + 8 * c;
                *reinterpret_cast<uint4 *>(a.ws.xhat + go) = nat;
                *reinterpret_cast<uint4 *>(a.ws.xhat_mma + go) = prm;
                *reinterpret_cast<uint4 *>(a.ws.xhat16 + go) =
                    make_uint4(f[0] | f[1] << 16, f[2] | f[3] << 16, f[4] | f[5] << 16, f[6] | f[7] << 16);
                if (a.xhat_out) *reinterpret_cast<uint4 *>(a.xhat_out + go) = nat;
            }
        }
#pragma unroll
        for (int j = 0; j < kXC; j++) xv[j] = xnext[j];
        __syncthreads();
    }

    MOE_PHASE_MARK(3);
    // -------------------------------------------------------------- router
    // Products of two bf16 are exact in fp32 and enter the sums through FMA.
    // Each 8-product chunk is summed first (8 roundings), chunk sums are
    // accumulated per lane (per_lane roundings), then a 5-level butterfly and
    // the bias: every partial sum is bounded by Σ|p|, so the error is
    // <= gamma_n * (Σ|p| + |b| + |l|) with n = 8 + per_lane + 6; the stored
    // bound is doubled as a safety margin.
    const int per_lane = (nchunk + 31) / 32;
    const int chain = 8 + per_lane + 6;
    {
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
        if (!ok) return;  // copies are reported lost; nothing else depends on this CTA
    }
    for (int el = warp; el < ne; el += kRouteWarps) {
        const int e = e0 + el;
        const uint16_t *wrow = wsm + (size_t)el * H;
        if (!a.router_exact) {
            float acc[G], sab[G];
#pragma unroll
            for (int g = 0; g < G; g++) acc[g] = sab[g] = 0.f;
            for (int ch = lane; ch < nchunk; ch += 32) {
                const uint4 wv = *reinterpret_cast<const uint4 *>(wrow + 8 * ch);
                const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
                float wf[8];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    wf[2 * q] = __uint_as_float(ww[q] << 16);
                    wf[2 * q + 1] = __uint_as_float(ww[q] & 0xFFFF0000u);
                }
#pragma unroll
                for (int g = 0; g < G; g++) {
                    if (g < nt) {
                        const uint4 xq = *reinterpret_cast<const uint4 *>(xh + g * H + ch * 8);
                        const uint32_t xx[4] = {xq.x, xq.y, xq.z, xq.w};
                        float cs = 0.f, ab = sab[g];
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            const float x0 = __uint_as_float(xx[q] << 16), x1 = __uint_as_float(xx[q] & 0xFFFF0000u);
                            cs = fmaf(x0, wf[2 * q], cs);
                            cs = fmaf(x1, wf[2 * q + 1], cs);
                            ab = fmaf(fabsf(x0), fabsf(wf[2 * q]), ab);
                            ab = fmaf(fabsf(x1), fabsf(wf[2 * q + 1]), ab);
                        }
                        acc[g] += cs;
                        sab[g] = ab;
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < G; g++) {
                const float sm = warp_sum_f(acc[g]);
                const float ab = warp_sum_f(sab[g]);
                if (lane == 0 && g < nt) {
                    const float b = a.router_b[e];
                    const float l = sm + b;
                    lg[g * epc + el] = l;
                    lb[g * epc + el] = 2.0f * (float)chain * 0x1p-24f * (ab + fabsf(b) + fabsf(l)) + 1e-30f;
                }
            }
        } else {
            for (int g = 0; g < nt; g++) {
                const double l = exact_logit(xh + g * H, a.router_w, a.router_b, e, H, lane);
                if (lane == 0) {
                    lg[g * epc + el] = (float)l;
                    lb[g * epc + el] = 0.f;
                }
            }
        }
    }
    __syncthreads();
    MOE_PHASE_MARK(4);

    // ---------------------------------------------------------- top-k + softmax
    if (gridDim.y == 1) {
        // this CTA holds every logit of its tokens
        for (int g = warp; g < nt; g += kRouteWarps)
            topk_token_warp(lg + g * epc, lb + g * epc, false, xh + g * H, a, t0 + g, lane);
    } else {
        for (int i = tid; i < nt * ne; i += kRouteThreads) {
            const int g = i / ne, el = i - g * ne;
            a.ws.logits[(size_t)(t0 + g) * E + e0 + el] = lg[g * epc + el];
            a.ws.lbound[(size_t)(t0 + g) * E + e0 + el] = lb[g * epc + el];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) s_flag = (atomicAdd(a.ws.tickets + 1 + blockIdx.x, 1u) == gridDim.y - 1);
        __syncthreads();
        if (!s_flag) return;
        __threadfence();
        for (int g = warp; g < nt; g += kRouteWarps)
            topk_token_warp(a.ws.logits + (size_t)(t0 + g) * E, a.ws.lbound + (size_t)(t0 + g) * E, true,
                            xh + g * H, a, t0 + g, lane);
        if (tid == 0) a.ws.tickets[1 + blockIdx.x] = 0u;  // re-arm the group ticket
    }
    MOE_PHASE_MARK(5);

    // --------------------------------------------- last CTA of the grid: permutation
    __threadfence();
    __syncthreads();
    if (tid == 0) s_flag = (atomicAdd(a.ws.tickets, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_flag) return;
    __threadfence();
    MOE_PHASE_MARK(6);

    const int ns = a.bp.n_shared;
    const int EE = E + ns;
    const int KK = K + ns;
    const int R = a.T * K;
    int32_t *cnt = reinterpret_cast<int32_t *>(smem);  // reuses the router-row area
    int32_t *offs = cnt + 264;
    int32_t *run = offs + 264;
    int32_t *tcnt = run + 264;
    int32_t *toff = tcnt + 264;
    int32_t *wcnt = toff + 264;  // [kRouteWarps][EE]
    for (int e = tid; e < EE; e += kRouteThreads) {
        cnt[e] = 0;
        run[e] = 0;
    }
    __syncthreads();
    for (int r = tid; r < R; r += kRouteThreads) {
        int e = __ldcg(a.ws.ids + r);
        if ((unsigned)e >= (unsigned)E) {
            set_device_error(a.ws.status, MOE_DEV_BAD_ROUTE, r);
            e = 0;
        }
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
    for (int e = tid; e < EE; e += kRouteThreads) {
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
    for (int base = 0; base < R; base += kRouteThreads) {
        for (int i = tid; i < kRouteWarps * EE; i += kRouteThreads) wcnt[i] = 0;
        __syncthreads();
        const int r = base + tid;
        int e = -1;
        if (r < R) {
            e = __ldcg(a.ws.ids + r);
            if ((unsigned)e >= (unsigned)E) e = 0;
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
            a.ws.perm_w[pos] = __ldcg(a.ws.route_w + r);
            a.ws.loc[t * KK + s] = pos;
        }
        __syncthreads();
        for (int x = tid; x < EE; x += kRouteThreads) {
            int s = 0;
            for (int w = 0; w < kRouteWarps; w++) s += wcnt[w * EE + x];
            run[x] += s;
        }
        __syncthreads();
    }
    if (ns) {
        for (int t = tid; t < a.T; t += kRouteThreads) {
            const int pos = offs[E] + t;
            a.ws.perm_token[pos] = t;
            a.ws.perm_slot[pos] = K;
            a.ws.perm_w[pos] = 1.0f;
            a.ws.loc[t * KK + K] = pos;
        }
    }
    if (tid == 0) a.ws.tickets[0] = 0u;  // re-arm for the next launch
    MOE_PHASE_MARK(7);
}

// Experts per CTA so that their router rows plus G x_hat rows fit in shared memory.
int route_epc(int G, int H, int E) {
    const size_t budget = 200 * 1024;
    const size_t xbytes = (size_t)G * H * 2;
    int epc = (int)((budget - xbytes) / ((size_t)H * 2 + 8 * G));
    if (epc > E) epc = E;
    if (epc < 1) epc = 1;
    return epc;
}

size_t route_smem_bytes(int G, int H, int E) {
    const int epc = route_epc(G, H, E);
    const size_t a = (size_t)epc * H * 2 + (size_t)G * H * 2 + (size_t)G * epc * 8;
    const size_t b = (size_t)(5 * 264 + kRouteWarps * (E + 1)) * 4;
    return a > b ? a : b;
}

}  // namespace

int route_ticket_count(int T) { return T + 1; }

cudaError_t launch_route(const BlockParams &bp, const Workspace &ws, const uint16_t *x, const float *gamma,
                         const uint16_t *router_w, const float *router_b, int T, int32_t *ids_out, float *rw_out,
                         uint16_t *xhat_out, int tile_rows, int router_exact, cudaStream_t st) {
    if (bp.H / 8 > kRouteThreads * kXC) return cudaErrorInvalidValue;
    static bool done1 = false, done8 = false;
    if (T <= 32) {
        RouteArgs a{bp, ws, x, gamma, router_w, router_b, T, ids_out, rw_out, xhat_out, tile_rows, router_exact,
                    route_epc(1, bp.H, bp.E)};
        MOE_CUDA_TRY(smem_optin_once(moe_route_kernel<1>, done1));
        dim3 grid(T, (bp.E + a.epc - 1) / a.epc);
        moe_route_kernel<1><<<grid, kRouteThreads, route_smem_bytes(1, bp.H, bp.E), st>>>(a);
    } else {
        RouteArgs a{bp, ws, x, gamma, router_w, router_b, T, ids_out, rw_out, xhat_out, tile_rows, router_exact,
                    route_epc(8, bp.H, bp.E)};
        MOE_CUDA_TRY(smem_optin_once(moe_route_kernel<8>, done8));
        dim3 grid((T + 7) / 8, (bp.E + a.epc - 1) / a.epc);
        moe_route_kernel<8><<<grid, kRouteThreads, route_smem_bytes(8, bp.H, bp.E), st>>>(a);
    }
    return cudaGetLastError();
}
