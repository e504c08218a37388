// moe_attn.cu -- the attention half of the gpt-oss layer, one decode step for a
// batch of sequences (goosedump gpt_oss.rs `forward`: attention norm, the
// query/key/value projections with biases, `apply_rope` with `Rope::new`'s
// YaRN tables, `LayerCache::append` (fp16), `causal_gqa` / `attention_head`
// with the per-head sink logit and `attention_window`, the output projection
// with bias and the residual add; turbospark-runtime gptoss/mod.rs module doc
// comment).
//
// Kernels, in stream order:
//  * the routing's norm kernel: x_hat = bf16(rms_norm(x) * gamma), exact;
//  * moe_attn_qkv_kernel: the three projections as one GEMV over 16-row tiles
//    (mma.sync m16n8k16, bf16 weights and x_hat, fp32 accumulation; four
//    warps split K and add their partials in a fixed order).  A q or k tile
//    holds dims d and d + 32 of one head in its upper and lower eight rows, so
//    that each RoPE pair sits in one thread; biases, RoPE (cos and sin of the
//    exact angle, evaluated in double), then q to the workspace (fp32) and k,
//    v into the caller's fp16 cache at the token's position;
//  * moe_attn_chunk_kernel: one CTA per (256-token chunk of the visible
//    context, kv head, sequence): the scores of the kv head's query heads and
//    their weighted value sums on the tensor cores (mma.sync m16n8k16 f16,
//    the query heads as the MMA's rows; fp32 q and probabilities split into
//    fp16 high and low parts, keys and values fp16 as cached), the chunk's
//    softmax statistics;
//  * moe_attn_merge_kernel: the chunks and the head's sink logit combined
//    into o, rounded to bf16;
//  * moe_attn_out_kernel: out = x + Wo o + bo with the same GEMV core.
// In the GEMV core each thread reads 16 contiguous bytes of a weight row and
// of an activation row per 32-element block, and hands them to two MMAs as
// if their k order were permuted: the dot product does not depend on the
// order of k, and A and B see the same permutation.
#include "moe_common.cuh"
#include "../../include/moe.h"

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>

namespace {

constexpr int kHeadDim = 64;
constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kMaxSeqs = 32;      // tokens per decode step (4 MMA column tiles of 8)
constexpr int kChunk = 256;       // context tokens per attention CTA
constexpr int kMaxQPerKV = 16;    // query heads sharing one kv head (the attention MMA's 16 rows)

struct AttnDims {
    int H, QH, KVH;
    int window;       // 0: full causal attention; else the last `window` tokens
    int max_seq, max_ctx;
    double eps;
    double rope_af;   // attention factor 0.1 ln(factor) + 1
    double freq[kHeadDim / 2];
};

struct AttnWeights {
    const float *gamma;
    const uint16_t *wq, *wk, *wv, *wo;
    const float *bq, *bk, *bv, *bo, *sinks;
};

__device__ __forceinline__ void mma_bf16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// acc[nt][0..1]: row lo, tokens 8 nt + 2 t4, + 1; acc[nt][2..3]: row hi.
// Rows lo and hi (16-byte aligned row pointers, K elements each) against
// activation rows X[b] (K elements, 16-byte aligned rows, b < B), over the
// warp's share of the 32-element blocks; then the four warps' partials are
// added in warp order (result valid in warp 0).
template <int NT>
__device__ void gemv_tile(const uint16_t *wlo, const uint16_t *whi, const uint16_t *X, int B, int K, float (*red)[4],
                          float (&acc)[NT][4]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const int nblk = K / 32, per = (nblk + kGemvWarps - 1) / kGemvWarps;
    const int b0 = warp * per, b1 = min(nblk, b0 + per);
    const uint16_t *xrow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; nt++) xrow[nt] = (nt * 8 + g < B) ? X + (size_t)(nt * 8 + g) * K : nullptr;
#pragma unroll 4
    for (int kb = b0; kb < b1; kb++) {
        const int k = kb * 32 + 8 * t4;
        const uint4 alo = __ldg(reinterpret_cast<const uint4 *>(wlo + k));
        const uint4 ahi = __ldg(reinterpret_cast<const uint4 *>(whi + k));
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            const uint4 bv = xrow[nt] ? __ldg(reinterpret_cast<const uint4 *>(xrow[nt] + k)) : make_uint4(0, 0, 0, 0);
            mma_bf16(acc[nt], alo.x, ahi.x, alo.y, ahi.y, bv.x, bv.y);
            mma_bf16(acc[nt], alo.z, ahi.z, alo.w, ahi.w, bv.z, bv.w);
        }
    }
    // partials of warps 1..3 through shared memory, summed by warp 0 in order
    if (warp > 0)
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int q = 0; q < 4; q++) red[((warp - 1) * NT + nt) * 32 + lane][q] = acc[nt][q];
    __syncthreads();
    if (warp == 0)
        for (int w = 1; w < kGemvWarps; w++)
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
#pragma unroll
                for (int q = 0; q < 4; q++) acc[nt][q] += red[((w - 1) * NT + nt) * 32 + lane][q];
}

// Tiles 0 .. QH*4-1: q (head ti/4, dims 8(ti%4) + g and + 32); then KVH*4 k
// tiles the same way; then KVH*4 v tiles of 16 consecutive rows.
template <int NT>
__global__ void __launch_bounds__(kGemvThreads) moe_attn_qkv_kernel(AttnDims d, AttnWeights w, const uint16_t *xhat,
                                                                    int B, const int32_t *pos, float *q,
                                                                    __half *kc, __half *vc) {
    __shared__ float red[(kGemvWarps - 1) * NT * 32][4];
    const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
    const int ti = blockIdx.x, H = d.H;
    const int nq = d.QH * 4, nk = d.KVH * 4;
    int kind, head, sub;  // 0 q, 1 k, 2 v
    if (ti < nq) {
        kind = 0, head = ti / 4, sub = ti % 4;
    } else if (ti < nq + nk) {
        kind = 1, head = (ti - nq) / 4, sub = (ti - nq) % 4;
    } else {
        kind = 2, head = (ti - nq - nk) / 4, sub = (ti - nq - nk) % 4;
    }
    int rlo, rhi;  // rows within the matrix
    if (kind < 2) {
        rlo = head * kHeadDim + 8 * sub + g;
        rhi = rlo + 32;
    } else {
        rlo = head * kHeadDim + 16 * sub + g;
        rhi = rlo + 8;
    }
    const uint16_t *W = kind == 0 ? w.wq : kind == 1 ? w.wk : w.wv;
    const float *bias = kind == 0 ? w.bq : kind == 1 ? w.bk : w.bv;
    float acc[NT][4];
    gemv_tile<NT>(W + (size_t)rlo * H, W + (size_t)rhi * H, xhat, B, H, red, acc);
    if ((threadIdx.x >> 5) != 0) return;
    const float blo = bias[rlo], bhi = bias[rhi];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const int b = nt * 8 + 2 * t4 + c;
            if (b >= B) continue;
            float lo = acc[nt][c] + blo, hi = acc[nt][2 + c] + bhi;
            const int p = pos[b];
            if (p < 0 || p >= d.max_ctx) continue;  // outside the cache: the sequence is skipped
            if (kind < 2) {
                // RoPE pair 8 sub + g of the head: l cos - r sin, l sin + r cos
                double sn, cs;
                sincos((double)p * d.freq[8 * sub + g], &sn, &cs);
                const float cf = (float)(cs * d.rope_af), sf = (float)(sn * d.rope_af);
                const float l = lo, r = hi;
                lo = l * cf - r * sf;
                hi = l * sf + r * cf;
            }
            if (kind == 0) {
                q[(size_t)b * d.QH * kHeadDim + rlo] = lo;
                q[(size_t)b * d.QH * kHeadDim + rhi] = hi;
            } else {
                __half *cache = kind == 1 ? kc : vc;
                const size_t base = ((size_t)b * d.max_ctx + p) * d.KVH * kHeadDim;
                cache[base + rlo] = __float2half_rn(lo);
                cache[base + rhi] = __float2half_rn(hi);
            }
        }
}

// Visible context of sequence b (its new token at position p is the last).
__device__ __forceinline__ void visible_range(const AttnDims &d, int p, int &first, int &count) {
    const int n = p + 1;
    first = (d.window > 0 && n > d.window) ? n - d.window : 0;
    count = n - first;
}

// fp16 pair (x, y) rounded from fp32, and the pair of what that rounding left
// (so hi + lo carries about 22 significant bits of each value).
__device__ __forceinline__ void split_half2(float x, float y, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x, y);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ void mma_f16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kVPad = kHeadDim + 8;  // value row in shared memory (halves): ldmatrix rows on distinct banks

// Partials per (sequence, query head, chunk): max score, sum of exp(s - max),
// and the exp-weighted value sums [64], on the tensor cores (up to 16 query
// heads per kv head as the MMA's 16 rows).  Scores: q (split into fp16 high
// and low parts, about 22 significant bits together) against the fp16 keys
// (exact), warp w taking tokens 32 w .. 32 w + 31, each thread reading 16
// contiguous bytes of a key row per 32 dims and the matching slice of q (the
// MMA sees both in the same permuted k order).  Weighted values: the
// probabilities (split the same way) against the value rows staged in shared
// memory (transposed by ldmatrix), warp w taking dims 8 w .. 8 w + 7.
__global__ void __launch_bounds__(256) moe_attn_chunk_kernel(AttnDims d, const float *q, const int32_t *pos,
                                                             const __half *kc, const __half *vc, float *pm, float *pl,
                                                             float *pacc, int n_chunks) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int c = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t4 = lane & 3;
    const int G = d.QH / d.KVH;
    float *ss = reinterpret_cast<float *>(smem);                 // [16][256] scores, then probabilities
    __half *sv = reinterpret_cast<__half *>(ss + 16 * kChunk);  // [256][kVPad] value rows
    const int p = pos[b];
    if (p < 0 || p >= d.max_ctx) return;
    int first, count;
    visible_range(d, p, first, count);
    const int t0 = first + c * kChunk;
    const int nt = min(kChunk, first + count - t0);
    if (nt <= 0) return;
    const size_t row0 = ((size_t)b * d.max_ctx) * d.KVH * kHeadDim + (size_t)j * kHeadDim;
    const size_t rstride = (size_t)d.KVH * kHeadDim;
    // value rows of the chunk into shared memory (rows past the chunk: zeros)
    {
        const int t = tid;  // one row per thread
        uint4 *dst = reinterpret_cast<uint4 *>(sv + (size_t)t * kVPad);
        if (t < nt) {
            const __half *vr = vc + row0 + (size_t)(t0 + t) * rstride;
#pragma unroll
            for (int v = 0; v < kHeadDim / 8; v++) {
                const uint32_t da = static_cast<uint32_t>(__cvta_generic_to_shared(dst + v));
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(da), "l"(vr + 8 * v) : "memory");
            }
        } else {
#pragma unroll
            for (int v = 0; v < kHeadDim / 8; v++) dst[v] = make_uint4(0, 0, 0, 0);
        }
    }
    // q slices of heads g and g + 8 (zero rows past G), split high / low
    const float *qb = q + (size_t)b * d.QH * kHeadDim + (size_t)(j * G) * kHeadDim;
    uint32_t qh[2][2][4], ql[2][2][4];  // [row g / g+8][32-dim block][pair]
#pragma unroll
    for (int r = 0; r < 2; r++)
#pragma unroll
        for (int db = 0; db < 2; db++) {
            const int h = g + 8 * r;
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; e++) v[e] = h < G ? qb[(size_t)h * kHeadDim + 32 * db + 8 * t4 + e] : 0.f;
#pragma unroll
            for (int e = 0; e < 4; e++) split_half2(v[2 * e], v[2 * e + 1], qh[r][db][e], ql[r][db][e]);
        }
    // scores of this warp's 32 tokens (4 column tiles of 8)
    const float scale = rsqrtf((float)kHeadDim);
#pragma unroll
    for (int ni = 0; ni < 4; ni++) {
        const int tt = 32 * warp + 8 * ni + g;  // this thread's key row
        uint4 kv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (tt < nt) {
            const uint4 *kr = reinterpret_cast<const uint4 *>(kc + row0 + (size_t)(t0 + tt) * rstride);
            kv[0] = kr[t4];
            kv[1] = kr[4 + t4];
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int db = 0; db < 2; db++) {
            mma_f16(acc, qh[0][db][0], qh[1][db][0], qh[0][db][1], qh[1][db][1], kv[db].x, kv[db].y);
            mma_f16(acc, qh[0][db][2], qh[1][db][2], qh[0][db][3], qh[1][db][3], kv[db].z, kv[db].w);
            mma_f16(acc, ql[0][db][0], ql[1][db][0], ql[0][db][1], ql[1][db][1], kv[db].x, kv[db].y);
            mma_f16(acc, ql[0][db][2], ql[1][db][2], ql[0][db][3], ql[1][db][3], kv[db].z, kv[db].w);
        }
        // acc[0..1]: head g, tokens 2 t4, 2 t4 + 1 of the tile; acc[2..3]: head g + 8
#pragma unroll
        for (int qd = 0; qd < 4; qd++) {
            const int h = g + 8 * (qd >> 1), t = 32 * warp + 8 * ni + 2 * t4 + (qd & 1);
            if (h < G) ss[h * kChunk + t] = t < nt ? acc[qd] * scale : -INFINITY;
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    // per head (a warp each): max, exponentials (0 past the chunk), their sum
    for (int h = warp; h < G; h += 8) {
        float m = -INFINITY;
        for (int t = lane; t < nt; t += 32) m = fmaxf(m, ss[h * kChunk + t]);
#pragma unroll
        for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        for (int t = lane; t < kChunk; t += 32) {
            const float e = t < nt ? __expf(ss[h * kChunk + t] - m) : 0.f;
            ss[h * kChunk + t] = e;
            l += e;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            const size_t idx = ((size_t)b * d.QH + j * G + h) * n_chunks + c;
            pm[idx] = m;
            pl[idx] = l;
        }
    }
    __syncthreads();
    // weighted values: this warp's 8 dims, the chunk's tokens 16 at a time
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    const int ksteps = (nt + 15) / 16;
    for (int ks = 0; ks < ksteps; ks++) {
        const int kt = 16 * ks;
        uint32_t ph[4], plo[4];
        {
            const float *r0 = ss + (size_t)g * kChunk + kt + 2 * t4;        // head g
            const float *r1 = ss + (size_t)(g + 8) * kChunk + kt + 2 * t4;  // head g + 8
            const bool h1 = g + 8 < G;
            const bool h0 = g < G;
            split_half2(h0 ? r0[0] : 0.f, h0 ? r0[1] : 0.f, ph[0], plo[0]);
            split_half2(h1 ? r1[0] : 0.f, h1 ? r1[1] : 0.f, ph[1], plo[1]);
            split_half2(h0 ? r0[8] : 0.f, h0 ? r0[9] : 0.f, ph[2], plo[2]);
            split_half2(h1 ? r1[8] : 0.f, h1 ? r1[9] : 0.f, ph[3], plo[3]);
        }
        uint32_t b0, b1;
        {
            const __half *rowp = sv + (size_t)(kt + (lane & 15)) * kVPad + 8 * warp;
            const uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(rowp));
            asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                         : "=r"(b0), "=r"(b1)
                         : "r"(addr));
        }
        mma_f16(o, ph[0], ph[1], ph[2], ph[3], b0, b1);
        mma_f16(o, plo[0], plo[1], plo[2], plo[3], b0, b1);
    }
    // o[0..1]: head g, dims 8 w + 2 t4, + 1; o[2..3]: head g + 8
#pragma unroll
    for (int qd = 0; qd < 4; qd++) {
        const int h = g + 8 * (qd >> 1);
        if (h >= G) continue;
        const size_t idx = ((size_t)b * d.QH + j * G + h) * n_chunks + c;
        pacc[idx * kHeadDim + 8 * warp + 2 * t4 + (qd & 1)] = o[qd];
    }
}

size_t chunk_smem_bytes(const AttnDims &) {
    return (size_t)16 * kChunk * 4 + (size_t)kChunk * kVPad * 2;
}

// o[b][h][:] = (sum over chunks of acc e^(m_c - m)) / (sum of l e^(m_c - m) +
// e^(sink - m)), m the largest of the chunk maxima and the sink; rounded to bf16.
__global__ void moe_attn_merge_kernel(AttnDims d, const float *sinks, const int32_t *pos, const float *pm,
                                      const float *pl, const float *pacc, int n_chunks, uint16_t *o) {
    const int h = blockIdx.x, b = blockIdx.y, e = threadIdx.x;  // 64 threads
    const int p = pos[b];
    int first = 0, count = 0;
    if (p >= 0 && p < d.max_ctx) visible_range(d, p, first, count);
    const int nc = (count + kChunk - 1) / kChunk;
    const size_t base = ((size_t)b * d.QH + h) * n_chunks;
    const float sink = sinks[h];
    float m = sink;
    for (int c = 0; c < nc; c++) m = fmaxf(m, pm[base + c]);
    float den = __expf(sink - m), num = 0.f;
    for (int c = 0; c < nc; c++) {
        const float f = __expf(pm[base + c] - m);
        den = fmaf(pl[base + c], f, den);
        num = fmaf(pacc[(base + c) * kHeadDim + e], f, num);
    }
    const __nv_bfloat16 r = __float2bfloat16_rn(num / den);
    o[((size_t)b * d.QH + h) * kHeadDim + e] = *reinterpret_cast<const uint16_t *>(&r);
}

// out[b][r] = x[b][r] + (Wo o[b])[r] + bo[r], 16 consecutive rows per CTA.
template <int NT>
__global__ void __launch_bounds__(kGemvThreads) moe_attn_out_kernel(AttnDims d, AttnWeights w, const uint16_t *o,
                                                                    int B, const uint16_t *x, void *out, int out_bf16) {
    __shared__ float red[(kGemvWarps - 1) * NT * 32][4];
    const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
    const int K = d.QH * kHeadDim, H = d.H;
    const int rlo = blockIdx.x * 16 + g, rhi = rlo + 8;
    float acc[NT][4];
    gemv_tile<NT>(w.wo + (size_t)rlo * K, w.wo + (size_t)rhi * K, o, B, K, red, acc);
    if ((threadIdx.x >> 5) != 0) return;
    const float blo = w.bo[rlo], bhi = w.bo[rhi];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const int b = nt * 8 + 2 * t4 + c;
            if (b >= B) continue;
            const float lo = bf16_to_f32(x[(size_t)b * H + rlo]) + (acc[nt][c] + blo);
            const float hi = bf16_to_f32(x[(size_t)b * H + rhi]) + (acc[nt][2 + c] + bhi);
            if (out_bf16) {
                const __nv_bfloat16 l = __float2bfloat16_rn(lo), h = __float2bfloat16_rn(hi);
                static_cast<uint16_t *>(out)[(size_t)b * H + rlo] = *reinterpret_cast<const uint16_t *>(&l);
                static_cast<uint16_t *>(out)[(size_t)b * H + rhi] = *reinterpret_cast<const uint16_t *>(&h);
            } else {
                static_cast<float *>(out)[(size_t)b * H + rlo] = lo;
                static_cast<float *>(out)[(size_t)b * H + rhi] = hi;
            }
        }
}

template <template <int> class F, typename... A>
cudaError_t by_nt(int B, A... args) {
    if (B <= 8) return F<1>::run(args...);
    if (B <= 16) return F<2>::run(args...);
    if (B <= 24) return F<3>::run(args...);
    return F<4>::run(args...);
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

struct moe_attn {
    AttnDims d;
    AttnWeights w{};
    bool have_w = false;
    __half *kc = nullptr, *vc = nullptr;
    unsigned char *ws = nullptr;
    size_t ws_bytes = 0;
    bool out_bf16 = false;
    double rope_base = 150000.0, rope_factor = 32.0, rope_orig = 4096.0, beta_fast = 32.0, beta_slow = 1.0;
};

namespace {

void attn_rope(moe_attn *p) {
    // goosedump gpt_oss.rs Rope::new: frequencies blended by the YaRN ramp
    // between the correction dimensions of beta_fast and beta_slow
    const double D = kHeadDim;
    auto corr = [&](double rot) { return D * std::log(p->rope_orig / (rot * 2.0 * M_PI)) / (2.0 * std::log(p->rope_base)); };
    const double low = std::max(corr(p->beta_fast), 0.0), high = std::min(corr(p->beta_slow), D - 1.0);
    for (int i = 0; i < kHeadDim / 2; i++) {
        const double base_f = std::pow(p->rope_base, -(2.0 * i / D));
        const double ramp = std::min(std::max((i - low) / (high - low), 0.0), 1.0);
        p->d.freq[i] = base_f * (1.0 - ramp + ramp / p->rope_factor);
    }
    p->d.rope_af = 0.1 * std::log(p->rope_factor) + 1.0;
}

struct Carve {
    uint16_t *xhat;
    float *xnorm;
    int32_t *count;
    float *q;
    float *pm, *pl, *pacc;
    uint16_t *o;
};
size_t attn_carve(const AttnDims &d, unsigned char *base, Carve *c) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        unsigned char *q = base ? base + off : nullptr;
        off = (off + bytes + 255) & ~(size_t)255;
        return q;
    };
    const size_t S = d.max_seq, nch = (d.max_ctx + kChunk - 1) / kChunk, QD = (size_t)d.QH * kHeadDim;
    Carve t;
    t.xhat = reinterpret_cast<uint16_t *>(take(S * d.H * 2));
    t.xnorm = reinterpret_cast<float *>(take(S * 4));
    t.count = reinterpret_cast<int32_t *>(take(4));
    t.q = reinterpret_cast<float *>(take(S * QD * 4));
    t.pm = reinterpret_cast<float *>(take(S * d.QH * nch * 4));
    t.pl = reinterpret_cast<float *>(take(S * d.QH * nch * 4));
    t.pacc = reinterpret_cast<float *>(take(S * d.QH * nch * kHeadDim * 4));
    t.o = reinterpret_cast<uint16_t *>(take(S * QD * 2));
    if (c) *c = t;
    return off;
}

template <int NT>
struct QkvRun {
    static cudaError_t run(const AttnDims &d, const AttnWeights &w, const uint16_t *xh, int B, const int32_t *pos,
                           float *q, __half *kc, __half *vc, cudaStream_t st) {
        const int tiles = d.QH * 4 + 2 * d.KVH * 4;
        moe_attn_qkv_kernel<NT><<<tiles, kGemvThreads, 0, st>>>(d, w, xh, B, pos, q, kc, vc);
        return cudaGetLastError();
    }
};
template <int NT>
struct OutRun {
    static cudaError_t run(const AttnDims &d, const AttnWeights &w, const uint16_t *o, int B, const uint16_t *x,
                           void *out, int out_bf16, cudaStream_t st) {
        moe_attn_out_kernel<NT><<<d.H / 16, kGemvThreads, 0, st>>>(d, w, o, B, x, out, out_bf16);
        return cudaGetLastError();
    }
};

}  // namespace

extern "C" {

moe_attn *moe_attn_create(int hidden, int q_heads, int kv_heads, int head_dim, int max_seqs, int max_ctx) {
    if (hidden <= 0 || hidden % 32 != 0 || hidden / 8 > 512 || head_dim != kHeadDim || q_heads < 1 ||
        kv_heads < 1 || q_heads % kv_heads != 0 || q_heads / kv_heads > kMaxQPerKV || q_heads > 256 ||
        max_seqs < 1 || max_seqs > kMaxSeqs || max_ctx < 1 || max_ctx > 65536) {
        moe_set_error("moe_attn_create: bad arguments (hidden a multiple of 32 up to 4096, head_dim 64, "
                      "q_heads a multiple of kv_heads with at most %d per kv head, 1..%d sequences, "
                      "1..65536 context tokens)", kMaxQPerKV, kMaxSeqs);
        return nullptr;
    }
    moe_attn *p = new moe_attn;
    p->d.H = hidden;
    p->d.QH = q_heads;
    p->d.KVH = kv_heads;
    p->d.window = 0;
    p->d.max_seq = max_seqs;
    p->d.max_ctx = max_ctx;
    p->d.eps = 1e-5;
    attn_rope(p);
    return p;
}

void moe_attn_destroy(moe_attn *p) { delete p; }

int moe_attn_set_i(moe_attn *p, const char *key, long long v) {
    if (!p || !key) return moe_fail_status(MOE_EINVAL, "NULL argument");
    if (!strcmp(key, "sliding_window")) {
        if (v < 0 || v > 65536) return moe_fail_status(MOE_EINVAL, "sliding_window must be 0..65536");
        p->d.window = (int)v;
    } else if (!strcmp(key, "out_bf16")) {
        p->out_bf16 = v != 0;
    } else {
        return moe_fail_status(MOE_EINVAL, "unknown integer option '%s'", key);
    }
    return MOE_OK;
}

int moe_attn_set_f(moe_attn *p, const char *key, double v) {
    if (!p || !key) return moe_fail_status(MOE_EINVAL, "NULL argument");
    if (!(v > 0.0) || !std::isfinite(v)) return moe_fail_status(MOE_EINVAL, "'%s' must be positive and finite", key);
    if (!strcmp(key, "rms_eps")) p->d.eps = v;
    else if (!strcmp(key, "rope_base")) p->rope_base = v;
    else if (!strcmp(key, "rope_factor")) p->rope_factor = v;
    else if (!strcmp(key, "rope_original_context")) p->rope_orig = v;
    else if (!strcmp(key, "rope_beta_fast")) p->beta_fast = v;
    else if (!strcmp(key, "rope_beta_slow")) p->beta_slow = v;
    else return moe_fail_status(MOE_EINVAL, "unknown floating option '%s'", key);
    attn_rope(p);
    return MOE_OK;
}

size_t moe_attn_workspace_bytes(const moe_attn *p) { return p ? attn_carve(p->d, nullptr, nullptr) : 0; }

int moe_attn_set_workspace(moe_attn *p, void *dev, size_t bytes) {
    if (!p || !dev) return moe_fail_status(MOE_EINVAL, "NULL argument");
    if (((uintptr_t)dev & 255u) != 0) return moe_fail_status(MOE_EINVAL, "the workspace must be 256-byte aligned");
    if (bytes < attn_carve(p->d, nullptr, nullptr))
        return moe_fail_status(MOE_ENOMEM, "workspace of %zu bytes, %zu needed", bytes, attn_carve(p->d, nullptr, nullptr));
    p->ws = static_cast<unsigned char *>(dev);
    p->ws_bytes = bytes;
    return MOE_OK;
}

int moe_attn_set_cache(moe_attn *p, void *k_cache, void *v_cache) {
    if (!p || !k_cache || !v_cache) return moe_fail_status(MOE_EINVAL, "NULL argument");
    if (!aligned16(k_cache) || !aligned16(v_cache)) return moe_fail_status(MOE_EINVAL, "caches must be 16-byte aligned");
    p->kc = static_cast<__half *>(k_cache);
    p->vc = static_cast<__half *>(v_cache);
    return MOE_OK;
}

int moe_attn_load_weights(moe_attn *p, const moe_attn_weights *w) {
    if (!p || !w) return moe_fail_status(MOE_EINVAL, "NULL argument");
    const void *all[] = {w->gamma, w->wq, w->wk, w->wv, w->wo, w->bq, w->bk, w->bv, w->bo, w->sinks};
    for (const void *q : all) {
        if (!q) return moe_fail_status(MOE_EINVAL, "NULL weight pointer");
        if (!aligned16(q)) return moe_fail_status(MOE_EINVAL, "weight pointers must be 16-byte aligned");
    }
    p->w = AttnWeights{w->gamma, w->wq, w->wk, w->wv, w->wo, w->bq, w->bk, w->bv, w->bo, w->sinks};
    p->have_w = true;
    return MOE_OK;
}

int moe_attn_decode(moe_attn *p, const uint16_t *x, int n_seqs, const int32_t *positions, void *out, void *stream) {
    if (!p) return moe_fail_status(MOE_EINVAL, "NULL plan");
    if (!p->have_w) return moe_fail_status(MOE_ENOTREADY, "moe_attn_load_weights has not been called");
    if (!p->ws) return moe_fail_status(MOE_ENOTREADY, "moe_attn_set_workspace has not been called");
    if (!p->kc) return moe_fail_status(MOE_ENOTREADY, "moe_attn_set_cache has not been called");
    if (n_seqs < 0 || n_seqs > p->d.max_seq) return moe_fail_status(MOE_EINVAL, "n_seqs must be 0..%d", p->d.max_seq);
    if (n_seqs == 0) return MOE_OK;
    if (!x || !positions || !out) return moe_fail_status(MOE_EINVAL, "NULL x, positions or out");
    if (!aligned16(x) || !aligned16(out) || ((uintptr_t)positions & 3u))
        return moe_fail_status(MOE_EINVAL, "x and out must be 16-byte aligned, positions 4-byte aligned");
    const size_t xb = (size_t)n_seqs * p->d.H * 2, ob = (size_t)n_seqs * p->d.H * (p->out_bf16 ? 2 : 4);
    const char *xc = reinterpret_cast<const char *>(x), *oc = static_cast<const char *>(out);
    if (xc < oc + ob && oc < xc + xb) return moe_fail_status(MOE_EINVAL, "x and out must not overlap");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Carve c;
    attn_carve(p->d, p->ws, &c);
    const int nch = (p->d.max_ctx + kChunk - 1) / kChunk;
    cudaError_t e = launch_rms_norm_rows(x, p->w.gamma, n_seqs, p->d.H, p->d.eps, c.xhat, c.xnorm, c.count, st);
    if (e == cudaSuccess) e = by_nt<QkvRun>(n_seqs, p->d, p->w, (const uint16_t *)c.xhat, n_seqs, positions, c.q, p->kc, p->vc, st);
    if (e == cudaSuccess) {
        const size_t sm = chunk_smem_bytes(p->d);
        static bool opted = false;
        if (!opted) {
            e = cudaFuncSetAttribute(moe_attn_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
            opted = e == cudaSuccess;
        }
        if (e == cudaSuccess) {
            moe_attn_chunk_kernel<<<dim3(nch, p->d.KVH, n_seqs), 256, sm, st>>>(p->d, c.q, positions, p->kc, p->vc,
                                                                                c.pm, c.pl, c.pacc, nch);
            e = cudaGetLastError();
        }
    }
    if (e == cudaSuccess) {
        moe_attn_merge_kernel<<<dim3(p->d.QH, n_seqs), kHeadDim, 0, st>>>(p->d, p->w.sinks, positions, c.pm, c.pl,
                                                                          c.pacc, nch, c.o);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess)
        e = by_nt<OutRun>(n_seqs, p->d, p->w, (const uint16_t *)c.o, n_seqs, x, out, p->out_bf16 ? 1 : 0, st);
    return e == cudaSuccess ? MOE_OK : moe_fail_status(MOE_ECUDA, "moe_attn_decode: %s", cudaGetErrorString(e));
}

}  // extern "C"
