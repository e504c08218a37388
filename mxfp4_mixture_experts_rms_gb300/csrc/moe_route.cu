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
// Exactness.  The norm statistic is accumulated in fp64 from exact squares and
// x_hat is rounded once from fp64, so it matches a plain double evaluation
// bit for bit.  Router logits are accumulated in fp32 with a rigorous error
// bound per logit; when the bound cannot certify the top-k membership and
// order, the candidate logits are recomputed in fp64 (exact for these
// operands) and the selection is redone on them.
#include "moe_common.cuh"

namespace {

constexpr int kRouteThreads = 512;
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
    int write_mma;
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

// (value, index) order of `top_experts`: larger value first, equal values by
// lower index.  Candidates that can never beat an empty (-inf) slot are invalid.
__device__ __forceinline__ bool better(float v, int i, float w, int j) {
    return v > w || (v == w && i < j);
}
__device__ __forceinline__ bool better_d(double v, int i, double w, int j) {
    return v > w || (v == w && i < j);
}

// Warp-wide arg-best over per-lane candidates.
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
// Exact (fp64) router logit of expert e for the x_hat row in shared memory,
// computed by one warp.  Products of two bf16 values are exact in fp64.
__device__ double exact_logit(const uint16_t *xh, const uint16_t *router_w, const float *router_b,
                              int e, int H, int lane) {
    double acc = 0.0;
    const uint16_t *w = router_w + (size_t)e * H;
    for (int i = lane; i < H; i += 32) acc += (double)bf16_to_f32(xh[i]) * (double)bf16_to_f32(__ldg(w + i));
    acc = warp_sum_d(acc);
    return acc + (double)router_b[e];
}

// Exclusive scan by one warp over n <= 1024 ints in shared memory (in place
// into out[0..n], out[n] = total).
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

template <int G>
__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(RouteArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int H = a.bp.H, E = a.bp.E, K = a.bp.K;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint16_t *xh = reinterpret_cast<uint16_t *>(smem);                       // [G][H]
    float *lg = reinterpret_cast<float *>(smem + (size_t)G * H * 2);          // [G][E]
    float *bnd = lg + G * E;                                                  // [G][E]
    __shared__ double red[kRouteWarps];
    __shared__ int last_flag;

    const int t0 = blockIdx.x * G;
    // ---------------------------------------------------------------- norm
    for (int g = 0; g < G; g++) {
        int t = t0 + g;
        if (t >= a.T) break;  // uniform across the block
        const uint16_t *xr = a.x + (size_t)t * H;
        double ss = 0.0;
        for (int i = tid; i < H; i += kRouteThreads) {
            double xi = (double)bf16_to_f32(xr[i]);
            ss += xi * xi;
        }
        ss = warp_sum_d(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        double tot = 0.0;
#pragma unroll
        for (int w = 0; w < kRouteWarps; w++) tot += red[w];
        double r = 1.0 / sqrt(tot / (double)H + a.bp.eps);
        uint16_t *xo = a.ws.xhat + (size_t)t * H;
        for (int i = tid; i < H; i += kRouteThreads) {
            double v = (double)bf16_to_f32(xr[i]) * r;
            v = v * (double)a.gamma[i];
            uint16_t hb = bf16_from_double_rne(v);
            xh[g * H + i] = hb;
            xo[i] = hb;
            if (a.write_mma) a.ws.xhat_mma[(size_t)t * H + mma_perm_pos(i)] = hb;
            if (a.xhat_out) a.xhat_out[(size_t)t * H + i] = hb;
        }
        __syncthreads();
    }
    const int nt = min(G, a.T - t0);

    // -------------------------------------------------------------- router
    // Per (token, expert): fp32 FMA chain per lane over 8-element chunks, then
    // a 5-level butterfly.  Rounding error bound: gamma_{n+6} * (Σ|p| + |b|)
    // with n the per-lane chain length (products are exact in fp32).
    const int nchunk = H / 8;
    const int chain = 8 * ((nchunk + 31) / 32) + 6;
    for (int e = warp; e < E; e += kRouteWarps) {
        float acc[G], sab[G];
#pragma unroll
        for (int g = 0; g < G; g++) acc[g] = sab[g] = 0.f;
        if (!a.router_exact) {
            const uint4 *wr = reinterpret_cast<const uint4 *>(a.router_w + (size_t)e * H);
            for (int c = lane; c < nchunk; c += 32) {
                uint4 wv = __ldg(wr + c);
                const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int g = 0; g < G; g++) {
                    if (g < nt) {
                        uint4 xv = *reinterpret_cast<const uint4 *>(xh + g * H + c * 8);
                        const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                        for (int k = 0; k < 4; k++) {
                            float w0 = __uint_as_float(ww[k] << 16), w1 = __uint_as_float(ww[k] & 0xFFFF0000u);
                            float x0 = __uint_as_float(xx[k] << 16), x1 = __uint_as_float(xx[k] & 0xFFFF0000u);
                            float p0 = x0 * w0, p1 = x1 * w1;  // exact
                            acc[g] += p0;
                            acc[g] += p1;
                            sab[g] += fabsf(p0) + fabsf(p1);
                        }
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < G; g++) {
                float s = warp_sum_f(acc[g]);
                float ab = warp_sum_f(sab[g]);
                if (lane == 0 && g < nt) {
                    float b = a.router_b[e];
                    float l = s + b;
                    lg[g * E + e] = l;
                    bnd[g * E + e] = 2.0f * (float)chain * 0x1p-24f * (ab + fabsf(b) + fabsf(l)) + 1e-30f;
                }
            }
        } else {
            for (int g = 0; g < nt; g++) {
                double l = exact_logit(xh + g * H, a.router_w, a.router_b, e, H, lane);
                if (lane == 0) {
                    lg[g * E + e] = (float)l;
                    bnd[g * E + e] = -1.f;  // marks "exact requested"
                }
            }
        }
    }
    __syncthreads();

    // ---------------------------------------------------------- top-k + softmax
    for (int g = warp; g < nt; g += kRouteWarps) {
        const int t = t0 + g;
        const float *l = lg + g * E;
        const float *bd = bnd + g * E;
        const bool exact_mode = a.router_exact != 0;
        // K+1 best by (value, index) among valid candidates
        int sel[MOE_MAX_TOPK + 1];
        float selv[MOE_MAX_TOPK + 1];
        uint32_t taken = 0;  // per lane: bit j set if local candidate j was taken (E <= 256 -> 8 per lane)
        float dmax = 0.f;
        for (int j = lane; j < E; j += 32) dmax = fmaxf(dmax, bd[j]);
#pragma unroll
        for (int o = 16; o; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
        for (int r = 0; r <= K; r++) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int j = lane, q = 0; j < E; j += 32, q++) {
                float v = l[j];
                if (!(v > -INFINITY) || (taken >> q & 1u)) continue;  // NaN / -inf never chosen
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
        // certification: consecutive gaps among the K+1 best must exceed 2*dmax
        bool certain = !exact_mode;
        if (certain) {
            for (int r = 0; r < K; r++) {
                if (sel[r] == 0x7fffffff) break;
                float nxt = (sel[r + 1] == 0x7fffffff) ? -INFINITY : selv[r + 1];
                if (!(selv[r] - nxt > 2.0f * dmax)) certain = false;
            }
        }
        double exactv[MOE_MAX_TOPK];
        bool have_exact = false;
        if (!certain) {
            // candidates: every expert whose fp32 logit is within 2*dmax of the
            // K-th best (all of them in exact mode); recompute them in fp64
            float thr = exact_mode ? -INFINITY : ((sel[K - 1] == 0x7fffffff) ? -INFINITY : selv[K - 1] - 2.0f * dmax);
            double bv_all[MOE_MAX_TOPK];
            int bi_all[MOE_MAX_TOPK];
            for (int r = 0; r < K; r++) {
                bv_all[r] = -INFINITY;
                bi_all[r] = 0x7fffffff;
            }
            // insertion of candidates in index order (warp-uniform loop)
            for (int j = 0; j < E; j++) {
                float v = l[j];
                if (!(v > -INFINITY) || v < thr) continue;
                double ex = exact_logit(xh + g * H, a.router_w, a.router_b, j, H, lane);
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
        if (lane == 0) {
            // softmax over the selected raw logits, times the weight scale
            float m = -INFINITY;
            for (int r = 0; r < K; r++)
                if (sel[r] != 0x7fffffff) m = fmaxf(m, selv[r]);
            float ew[MOE_MAX_TOPK], s = 0.f;
            for (int r = 0; r < K; r++) {
                float d = have_exact ? (float)(exactv[r] - (double)m) : (selv[r] - m);
                ew[r] = (sel[r] == 0x7fffffff) ? 0.f : expf(d);
                s += ew[r];
            }
            for (int r = 0; r < K; r++) {
                int id = (sel[r] == 0x7fffffff) ? 0 : sel[r];  // unfilled slot: expert 0, weight 0
                float w = (s > 0.f) ? a.bp.wscale * (ew[r] / s) : 0.f;
                a.ws.ids[t * K + r] = id;
                a.ws.route_w[t * K + r] = w;
                if (a.ids_out) a.ids_out[t * K + r] = id;
                if (a.rw_out) a.rw_out[t * K + r] = w;
            }
        }
    }

    // --------------------------------------------- last CTA: permutation
    __threadfence();
    __syncthreads();
    if (tid == 0) last_flag = (atomicAdd(a.ws.ticket, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!last_flag) return;
    __threadfence();

    const int ns = a.bp.n_shared;
    const int EE = E + ns;            // experts incl. the shared one
    const int KK = K + ns;            // slots per token incl. the shared one
    const int R = a.T * K;            // routed routes
    int32_t *cnt = reinterpret_cast<int32_t *>(smem);   // [EE]      (reuses the x_hat area)
    int32_t *offs = cnt + 264;                            // [EE + 1]
    int32_t *run = offs + 264;                            // [EE]
    int32_t *tcnt = run + 264;                            // [EE]
    int32_t *toff = tcnt + 264;                           // [EE + 1]
    int32_t *wcnt = toff + 264;                           // [kRouteWarps][EE]
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
        a.ws.counts[e] = cnt[e];
        a.ws.offsets[e] = offs[e];
        int n = tcnt[e], base = toff[e];
        for (int k = 0; k < n && base + k < a.ws.max_tiles; k++) {
            int st = k * a.tile_rows;
            a.ws.tiles[base + k] = make_int4(e, offs[e] + st, min(a.tile_rows, cnt[e] - st), 0);
        }
    }
    if (tid == 0) {
        a.ws.offsets[EE] = offs[EE];
        *a.ws.n_tiles = min(toff[EE], a.ws.max_tiles);
        if (toff[EE] > a.ws.max_tiles) set_device_error(a.ws.status, MOE_DEV_BAD_ROUTE, -1);
    }
    // stable scatter of the routed routes, in token-major (token, slot) order
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = 0; base < R; base += kRouteThreads) {
        for (int i = tid; i < kRouteWarps * EE; i += kRouteThreads) wcnt[i] = 0;
        __syncthreads();
        int r = base + tid;
        int e = -1;
        if (r < R) {
            e = __ldcg(a.ws.ids + r);
            if ((unsigned)e >= (unsigned)E) e = 0;
        }
        unsigned peers = __match_any_sync(0xffffffffu, e);
        int rank_w = __popc(peers & lt_mask);
        if (e >= 0 && rank_w == 0) wcnt[warp * EE + e] = __popc(peers);
        __syncthreads();
        if (e >= 0) {
            int rank = run[e] + rank_w;
            for (int w = 0; w < warp; w++) rank += wcnt[w * EE + e];
            int pos = offs[e] + rank;
            int t = r / K, s = r - t * K;
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
            int pos = offs[E] + t;
            a.ws.perm_token[pos] = t;
            a.ws.perm_slot[pos] = K;
            a.ws.perm_w[pos] = 1.0f;
            a.ws.loc[t * KK + K] = pos;
        }
    }
    if (tid == 0) *a.ws.ticket = 0u;  // re-arm for the next launch
}

}  // namespace

size_t route_smem_bytes(int G, int H, int E) {
    size_t a = (size_t)G * H * 2 + (size_t)G * E * 8;
    size_t b = (size_t)(5 * 264 + kRouteWarps * (E + 1)) * 4;
    return a > b ? a : b;
}

cudaError_t launch_route(const BlockParams &bp, const Workspace &ws, const uint16_t *x,
                         const float *gamma, const uint16_t *router_w, const float *router_b, int T,
                         int32_t *ids_out, float *rw_out, uint16_t *xhat_out, int tile_rows,
                         int router_exact, int write_mma_layout, cudaStream_t st) {
    RouteArgs a{bp, ws, x, gamma, router_w, router_b, T, ids_out, rw_out, xhat_out, tile_rows,
                router_exact, write_mma_layout};
    static bool done1 = false, done8 = false;
    if (T <= 32) {
        MOE_CUDA_TRY(smem_optin_once(moe_route_kernel<1>, done1));
        moe_route_kernel<1><<<T, kRouteThreads, route_smem_bytes(1, bp.H, bp.E), st>>>(a);
    } else {
        MOE_CUDA_TRY(smem_optin_once(moe_route_kernel<8>, done8));
        moe_route_kernel<8><<<(T + 7) / 8, kRouteThreads, route_smem_bytes(8, bp.H, bp.E), st>>>(a);
    }
    return cudaGetLastError();
}
