// moe_attn.cu -- the attention half of the gpt-oss layer: one decode step for
// a batch of sequences, or the prefill of a prompt (goosedump gpt_oss.rs
// `forward` and `prefill_attention_layer`: attention norm, the query/key/value
// projections with biases, `apply_rope` with `Rope::new`'s YaRN tables,
// `LayerCache::append` (fp16), `causal_gqa` / `causal_gqa_batch` /
// `attention_head` with the per-head sink logit and `attention_window`, the
// output projection with bias and the residual add; turbospark-runtime
// gptoss/mod.rs module doc comment).
//
// Kernels, in stream order (each after the first launched as a programmatic
// dependent of the one before):
//  * the routing's norm kernel: x_hat = bf16(rms_norm(x) * gamma), exact;
//  * moe_attn_proj_kernel<., 0>: q, k, v = W x_hat + b as one GEMV over
//    16-row tiles of the concatenated weights (mma.sync m16n8k16, bf16
//    weights and x_hat, fp32 accumulation; eight warps split K and add their
//    partials in a fixed order), fp32 to the workspace, and the RoPE table of
//    each row's position (cos and sin per pair, from the angle reduced in
//    double); a prefill block of more than 32 rows uses the tensor-core GEMM
//    (moe_attn_gemm.cu) and moe_attn_rope_kernel instead;
//  * moe_attn_append_kernel: every row's rotated key and its value into the
//    caller's fp16 cache;
//  * decode: moe_attn_stream_kernel, one CTA per (split of the visible
//    context, kv head, sequence), the split's 64-key chunks through a TMA
//    ring; the kv head's query heads are the MMA's rows (mma.sync m16n8k16
//    f16; fp32 q and probabilities split into fp16 high and low parts, keys
//    and values fp16 as cached; the probabilities stay in registers); then
//    moe_attn_merge_kernel: the splits and the head's sink logit combined
//    into o, rounded to bf16;
//  * prefill: moe_attn_flash_kernel, one CTA per (16 rows, kv head), o
//    directly;
//  * moe_attn_proj_kernel<., 1> (or the GEMM): out = x + Wo o + bo.
#include "moe_common.cuh"
#include "../../include/moe.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>

namespace {

constexpr int kHeadDim = 64;
constexpr int kMaxSeqs = 32;      // tokens per decode step (4 MMA column tiles of 8)
constexpr int kChunk = 256;       // context tokens per attention CTA
constexpr int kMaxQPerKV = 16;    // query heads sharing one kv head (the attention MMA's 16 rows)
constexpr int kMaxPrefillRows = 4096;  // prefill rows per block (workspace rows)

struct AttnDims {
    int H, QH, KVH;
    int window;       // 0: full causal attention; else the last `window` tokens
    int max_seq, max_ctx;
    int rows;         // rows a step holds in the workspace: max(max_seq, prefill rows)
    double eps;
    double rope_af;   // attention factor 0.1 ln(factor) + 1
    double freq[kHeadDim / 2];
};

struct AttnWeights {
    const float *gamma;
    const uint16_t *wq, *wk, *wv, *wo;
    const float *bq, *bk, *bv, *bo, *sinks;
};

// Row b of a step: decode, one new token per cache sequence (sequence b, its
// position pos[b]); prefill, consecutive new tokens of one sequence (sequence
// seq, position pos0 + b).
struct RowMap {
    const int32_t *pos;  // decode: [rows] on the device; prefill: null
    int pos0, seq;       // prefill: first position, cache sequence (seq < 0: decode)
};
__device__ __forceinline__ int row_pos(const RowMap &m, int b) { return m.pos ? m.pos[b] : m.pos0 + b; }
__device__ __forceinline__ int row_seq(const RowMap &m, int b) { return m.seq >= 0 ? m.seq : b; }

__device__ __forceinline__ void mma_bf16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- the projections ----
// One CTA per 16 weight rows (8 warps split K).  Each thread reads 16
// contiguous bytes of a weight row and of an activation row per 32-element
// block and hands them to two MMAs (mma.sync m16n8k16, bf16, fp32
// accumulate) as if their k order were permuted: the dot product does not
// depend on the order of k, and A and B see the same permutation.
constexpr double kTwoPi = 6.283185307179586476925;
constexpr double kInvTwoPi = 0.159154943091895335769;

struct ProjArgs {
    AttnDims d;
    int rows, K;           // weight rows, reduction length
    const uint16_t *w[3];  // Q/K/V: wq, wk, wv (rows in that order); output: Wo
    const float *bias[3];
    int r1, r2;            // first row of the second and the third matrix
    const uint16_t *x;     // activations [B][K]
    int B;
    // Q/K/V: q, k, v with biases, fp32 [B][rows]; the RoPE table (cos, sin)
    // x attention factor [B][32]
    float *raw;
    float2 *rope;
    RowMap rows_of;
    // output: out = res + Wo o + bo
    const uint16_t *res;
    void *out;
    int out_bf16;
};

__device__ __forceinline__ int proj_mat(const ProjArgs &a, int row) { return row < a.r1 ? 0 : row < a.r2 ? 1 : 2; }

// acc[nt][0..1]: row lo, tokens 8 nt + 2 t4, + 1; acc[nt][2..3]: row hi.
// Rows lo and hi (16-byte aligned row pointers, K elements each) against
// activation rows X[b] (K elements, 16-byte aligned rows, b < B), over the
// warp's share of the 32-element blocks; then the eight warps' partials are
// added in warp order (result valid in warp 0).
template <int NT>
__device__ void gemv_tile(const uint16_t *wlo, const uint16_t *whi, const uint16_t *X, int B, int K, float (*red)[4],
                          float (&acc)[NT][4]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const int nblk = K / 32, per = (nblk + 8 - 1) / 8;
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
        for (int w = 1; w < 8; w++)
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
#pragma unroll
                for (int q = 0; q < 4; q++) acc[nt][q] += red[((w - 1) * NT + nt) * 32 + lane][q];
}


// 16 rows per CTA: Q/K/V (raw: biases added, RoPE later) or the output
// (with the residual, fp32 or bf16).  The Q/K/V kernel also writes the RoPE
// table: per sequence and pair, the angle pos f in double less the nearest
// whole number of turns (exact to about 1e-11 at any position), then its
// cosine and sine in float, times the attention factor.
template <int NT, int KIND>
__global__ void __launch_bounds__(256) moe_attn_proj_kernel(const __grid_constant__ ProjArgs a) {
    __shared__ float red[7 * NT * 32][4];
    const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
    const int rlo = blockIdx.x * 16 + g, rhi = rlo + 8;
    const int m = proj_mat(a, rlo), base = m == 0 ? 0 : m == 1 ? a.r1 : a.r2;
    if (threadIdx.x == 0 && blockIdx.y == 0) {
        // the tile's 16 weight rows (contiguous) into L2 while the previous
        // kernel finishes: they do not depend on it
        const uint16_t *w0 = a.w[m] + (size_t)(blockIdx.x * 16 - base) * a.K;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(w0), "r"((uint32_t)(16 * a.K * 2)) : "memory");
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the activations come from the previous kernel
    asm volatile("griddepcontrol.launch_dependents;");
    const int tb = blockIdx.y * 8 * NT, B = min(8 * NT, a.B - tb);  // this CTA's tokens: tb .. tb + B - 1
    float acc[NT][4];
    gemv_tile<NT>(a.w[m] + (size_t)(rlo - base) * a.K, a.w[m] + (size_t)(rhi - base) * a.K, a.x + (size_t)tb * a.K, B,
                  a.K, red, acc);
    if ((threadIdx.x >> 5) != 0) return;
    const float blo = a.bias[m][rlo - base], bhi = a.bias[m][rhi - base];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const int b = tb + nt * 8 + 2 * t4 + c;
            if (b >= a.B) continue;
            const size_t ol = (size_t)b * a.rows + rlo, oh = (size_t)b * a.rows + rhi;
            const float lo = acc[nt][c] + blo, hi = acc[nt][2 + c] + bhi;
            if (KIND == 0) {
                a.raw[ol] = lo;
                a.raw[oh] = hi;
            } else {
                const float yl = bf16_to_f32(a.res[ol]) + lo, yh = bf16_to_f32(a.res[oh]) + hi;
                if (a.out_bf16) {
                    const __nv_bfloat16 l = __float2bfloat16_rn(yl), h = __float2bfloat16_rn(yh);
                    static_cast<uint16_t *>(a.out)[ol] = *reinterpret_cast<const uint16_t *>(&l);
                    static_cast<uint16_t *>(a.out)[oh] = *reinterpret_cast<const uint16_t *>(&h);
                } else {
                    static_cast<float *>(a.out)[ol] = yl;
                    static_cast<float *>(a.out)[oh] = yh;
                }
            }
        }
    if (KIND == 0 && blockIdx.y == 0)
        for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
            const double ang = (double)row_pos(a.rows_of, b) * a.d.freq[lane];
            const float r = (float)fma(-rint(ang * kInvTwoPi), kTwoPi, ang);
            float sn, cs;
            sincosf(r, &sn, &cs);
            a.rope[(size_t)b * 32 + lane] = make_float2(cs * (float)a.d.rope_af, sn * (float)a.d.rope_af);
        }
}

template <int KIND>
cudaError_t proj_launch(const ProjArgs &a, cudaStream_t st) {
    const dim3 grid(a.rows / 16, (a.B + 31) / 32), block(256);  // above 32 tokens: blocks of 32 on grid.y
    const int nt = a.B > 32 ? 4 : (a.B + 7) / 8;
    if (nt == 1) return launch_pdl(moe_attn_proj_kernel<1, KIND>, grid, block, 0, st, a);
    if (nt == 2) return launch_pdl(moe_attn_proj_kernel<2, KIND>, grid, block, 0, st, a);
    if (nt == 3) return launch_pdl(moe_attn_proj_kernel<3, KIND>, grid, block, 0, st, a);
    return launch_pdl(moe_attn_proj_kernel<4, KIND>, grid, block, 0, st, a);
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

constexpr int kOPad = kHeadDim + 8;  // a warp's weighted sums per head (floats): 64-bit stores on distinct banks

// The RoPE table of rows 0 .. n - 1 (as the Q/K/V GEMV writes it): per row
// and pair, the angle pos f in double less the nearest whole number of turns,
// then its cosine and sine in float, times the attention factor.  One warp
// per row.
__global__ void moe_attn_rope_kernel(AttnDims d, RowMap rm, int n, float2 *rope) {
    const int b = blockIdx.x, lane = threadIdx.x;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    if (b >= n) return;
    const double ang = (double)row_pos(rm, b) * d.freq[lane];
    const float r = (float)fma(-rint(ang * kInvTwoPi), kTwoPi, ang);
    float sn, cs;
    sincosf(r, &sn, &cs);
    rope[(size_t)b * 32 + lane] = make_float2(cs * (float)d.rope_af, sn * (float)d.rope_af);
}

// Prefill: every new row's key (rotated with its row of the RoPE table) and
// value into the cache of sequence seq at position pos0 + b, as fp16 (goosedump
// gpt_oss.rs prefill_attention_layer: the batch is appended before its
// attention).  One CTA per (row, kv head), 64 threads.
__global__ void moe_attn_append_kernel(AttnDims d, const float *raw, const float2 *rope, RowMap rm, __half *kc,
                                       __half *vc) {
    const int b = blockIdx.x, j = blockIdx.y, e = threadIdx.x;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // k, v and the RoPE table
    asm volatile("griddepcontrol.launch_dependents;");
    const int p = row_pos(rm, b);
    if (p < 0 || p >= d.max_ctx) return;
    const int RW = (d.QH + 2 * d.KVH) * kHeadDim;
    const float *rq = raw + (size_t)b * RW;
    const size_t at = (((size_t)row_seq(rm, b) * d.max_ctx + p) * d.KVH + j) * kHeadDim;
    if (e < 32) {
        const float l = rq[(d.QH + j) * kHeadDim + e], r = rq[(d.QH + j) * kHeadDim + e + 32];
        const float2 cs = rope[(size_t)b * 32 + e];
        kc[at + e] = __float2half_rn(l * cs.x - r * cs.y);
        kc[at + e + 32] = __float2half_rn(l * cs.y + r * cs.x);
    }
    vc[at + e] = __float2half_rn(rq[(d.QH + d.KVH + j) * kHeadDim + e]);
}

// Decode attention, streamed (goosedump gpt_oss.rs causal_gqa /
// attention_head): one CTA per (split of the visible context, kv head,
// sequence).  A producer warp copies the split's 64-key chunks of keys and
// values by TMA (2-D maps over the caches, 128-byte swizzle) into a 4-stage
// ring; four consumer warps take 16 keys of each chunk apiece, with the kv
// head's query heads as the MMA's 16 rows: scores (q rotated as it is read,
// fp32 split into fp16 high and low parts, keys by ldmatrix), a running
// maximum and sum per head, the value sums rescaled and the chunk's
// exponentials (split the same way) times the values (ldmatrix.trans).  The
// four warps' results are combined in warp order into the split's partials
// (max, sum, value sums), which the merge kernel combines with the sink.  The
// new token's key and value are in the cache already (the append kernel).
constexpr int kSKeys = 64;                        // keys per stage
constexpr int kSStages = 4;
constexpr int kSWarps = 4;                        // consumers; warp kSWarps is the producer
constexpr int kSStage = 2 * kSKeys * 128;         // bytes: keys then values, 128-byte rows
constexpr int kSSmem = 1024 + kSStages * kSStage;
constexpr uint64_t kSWaitNs = 2000000000ull;

struct KvMaps {
    CUtensorMap k, v;  // [max_seq * max_ctx rows][KVH * 64] fp16, box 64 x 64, 128-byte swizzle
};

__device__ __forceinline__ uint32_t s_smem(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ bool s_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(s_smem(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: false (and the status word set) after about 2 s, or when a
// failure was reported elsewhere first; drain: only the time limit ends it.
__device__ bool s_wait(uint64_t *b, uint32_t parity, int32_t *status, int where, bool drain = false) {
    if (s_try(b, parity)) return true;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (uint32_t i = 0;; i++) {
        if (s_try(b, parity)) return true;
        if ((i & 63) == 63) {
            if (!drain && *(volatile int32_t *)status != 0) return false;
            uint64_t t1;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
            if (t1 - t0 > kSWaitNs) {
                set_device_error(status, MOE_DEV_WAIT_TIMEOUT, where);
                return false;
            }
        }
    }
}

// Keys per split of a visible context of `count` tokens cut into `splits`:
// whole 64-key chunks (the merge kernel uses the same cut).
__device__ __forceinline__ int split_len(int count, int splits) {
    return ((count + splits - 1) / splits + kSKeys - 1) / kSKeys * kSKeys;
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__global__ void __launch_bounds__((kSWarps + 1) * 32) moe_attn_stream_kernel(
    AttnDims d, const float *raw, const float2 *rope, RowMap rm, float *pm, float *pl, float *pacc, int n_splits,
    int32_t *status, const __grid_constant__ KvMaps maps) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) uint64_t full[kSStages], empty[kSStages];
    __shared__ float sml[kSWarps][kMaxQPerKV][2];
    const int c = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t4 = lane & 3;
    const int G = d.QH / d.KVH;
    if (tid == 0) {
        for (int s = 0; s < kSStages; s++) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_smem(&full[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s_smem(&empty[s])), "r"(kSWarps));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");  // q, the RoPE table and the appended rows
    asm volatile("griddepcontrol.launch_dependents;");
    const int p = row_pos(rm, b);
    if (p < 0 || p >= d.max_ctx) return;
    int first, count;
    visible_range(d, p, first, count);
    const int per = split_len(count, n_splits);
    const int k_beg = first + c * per, k_end = min(first + count, k_beg + per);  // keys [k_beg, k_end)
    if (k_beg >= k_end) return;
    const int nst = (k_end - k_beg + kSKeys - 1) / kSKeys;  // chunks of this split
    const int seqrow = row_seq(rm, b) * d.max_ctx;
    if (warp == kSWarps) {
        // producer: one lane issues the two copies of each chunk
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nst; i++) {
                const int s = i % kSStages;
                if (i >= kSStages && !s_wait(&empty[s], ((i / kSStages) - 1) & 1, status, 80)) break;
                unsigned char *dst = smem + s * kSStage;
                asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
                                 s_smem(&full[s])),
                             "r"(kSStage)
                             : "memory");
#pragma unroll
                for (int kv = 0; kv < 2; kv++)
                    asm volatile(
                        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
                        "{%3, %4}], [%2];" ::"r"(s_smem(dst + kv * kSKeys * 128)),
                        "l"(reinterpret_cast<uint64_t>(kv ? &maps.v : &maps.k)), "r"(s_smem(&full[s])),
                        "r"(j * kHeadDim), "r"(seqrow + k_beg + i * kSKeys)
                        : "memory");
                issued++;
            }
            // copies still in flight land before the CTA's shared memory goes
            uint64_t t0;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
            for (int i = max(0, issued - kSStages); i < issued; i++)
                while (!s_try(&full[i % kSStages], (i / kSStages) & 1)) {
                    uint64_t t1;
                    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
                    if (t1 - t0 > kSWaitNs) {
                        set_device_error(status, MOE_DEV_WAIT_TIMEOUT, 81);
                        i = issued;
                        break;
                    }
                }
        }
    }
    float o[8][4];  // [dim tile][fragment]: heads g, g + 8; dims 8 dt + 2 t4, + 1
#pragma unroll
    for (int dt = 0; dt < 8; dt++) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
    if (warp < kSWarps) {
        // q of heads g and g + 8 (zero rows past G), rotated: A fragments of
        // the four 16-dim steps (dims 16 s + 2 t4 + {0, 1, 8, 9})
        const int RW = (d.QH + 2 * d.KVH) * kHeadDim;
        const float *qb = raw + (size_t)b * RW + (size_t)(j * G) * kHeadDim;
        const float2 *rt = rope + (size_t)b * 32;
        uint32_t qh[4][4], ql[4][4];
        {
            float q[2][16];
#pragma unroll
            for (int r = 0; r < 2; r++) {
                const int h = g + 8 * r;
#pragma unroll
                for (int sp = 0; sp < 2; sp++)
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int dd = 16 * sp + 2 * t4 + (e & 1) + 8 * (e >> 1);
                        float l = 0.f, rr = 0.f;
                        float2 cs = make_float2(0.f, 0.f);
                        if (h < G) {
                            l = qb[(size_t)h * kHeadDim + dd];
                            rr = qb[(size_t)h * kHeadDim + dd + 32];
                            cs = rt[dd];
                        }
                        q[r][4 * sp + e] = l * cs.x - rr * cs.y;
                        q[r][4 * (sp + 2) + e] = l * cs.y + rr * cs.x;
                    }
            }
#pragma unroll
            for (int s4 = 0; s4 < 4; s4++) {
                split_half2(q[0][4 * s4], q[0][4 * s4 + 1], qh[s4][0], ql[s4][0]);
                split_half2(q[1][4 * s4], q[1][4 * s4 + 1], qh[s4][1], ql[s4][1]);
                split_half2(q[0][4 * s4 + 2], q[0][4 * s4 + 3], qh[s4][2], ql[s4][2]);
                split_half2(q[1][4 * s4 + 2], q[1][4 * s4 + 3], qh[s4][3], ql[s4][3]);
            }
        }
        for (int i = 0; i < nst; i++) {
            const int s = i % kSStages, k0 = k_beg + i * kSKeys;
            if (!s_wait(&full[s], (i / kSStages) & 1, status, 82)) break;
            unsigned char *sk = smem + s * kSStage, *sv = sk + kSKeys * 128;
            const int r0 = 16 * warp;  // this warp's rows of the chunk
            if (k0 + r0 + 16 > k_end) {
                // rows past the split: zero values (their weights are zero, but
                // what the copy brought there need not be finite)
                for (int r = r0 + (lane >> 3); r < r0 + 16; r += 4)
                    if (k0 + r >= k_end) *reinterpret_cast<uint4 *>(sv + r * 128 + (lane & 7) * 16) = make_uint4(0, 0, 0, 0);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before a copy refills the stage
                __syncwarp();
            }
            // scores of keys r0 .. r0 + 15: two key tiles of 8
            float sc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; nt++) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                for (int s2 = 0; s2 < 4; s2 += 2) {
                    const int row = r0 + 8 * nt + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                                 : "r"(s_smem(sk) + sw128(row, 2 * s2 + (lane >> 3))));
                    mma_f16(sc[nt], qh[s2][0], qh[s2][1], qh[s2][2], qh[s2][3], b0, b1);
                    mma_f16(sc[nt], ql[s2][0], ql[s2][1], ql[s2][2], ql[s2][3], b0, b1);
                    mma_f16(sc[nt], qh[s2 + 1][0], qh[s2 + 1][1], qh[s2 + 1][2], qh[s2 + 1][3], b2, b3);
                    mma_f16(sc[nt], ql[s2 + 1][0], ql[s2 + 1][1], ql[s2 + 1][2], ql[s2 + 1][3], b2, b3);
                }
            }
            float cm[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < 2; nt++)
#pragma unroll
                for (int qd = 0; qd < 4; qd++) {
                    const int t = k0 + r0 + 8 * nt + 2 * t4 + (qd & 1);
                    sc[nt][qd] = t < k_end ? sc[nt][qd] * 0.125f : -INFINITY;  // 1 / sqrt(64)
                    cm[qd >> 1] = fmaxf(cm[qd >> 1], sc[nt][qd]);
                }
            float scale[2];
#pragma unroll
            for (int r = 0; r < 2; r++) {
                cm[r] = fmaxf(cm[r], __shfl_xor_sync(0xffffffffu, cm[r], 1));
                cm[r] = fmaxf(cm[r], __shfl_xor_sync(0xffffffffu, cm[r], 2));
                const float mn = fmaxf(mrun[r], cm[r]);
                scale[r] = mrun[r] == -INFINITY ? 0.f : __expf(mrun[r] - mn);
                mrun[r] = mn;
                lrun[r] *= scale[r];
            }
#pragma unroll
            for (int dt = 0; dt < 8; dt++) {
                o[dt][0] *= scale[0], o[dt][1] *= scale[0];
                o[dt][2] *= scale[1], o[dt][3] *= scale[1];
            }
            float e[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; nt++)
#pragma unroll
                for (int qd = 0; qd < 4; qd++) {
                    const float v = sc[nt][qd];
                    e[nt][qd] = v == -INFINITY ? 0.f : __expf(v - mrun[qd >> 1]);
                    lrun[qd >> 1] += e[nt][qd];
                }
            uint32_t ph[4], plo[4];
            split_half2(e[0][0], e[0][1], ph[0], plo[0]);
            split_half2(e[0][2], e[0][3], ph[1], plo[1]);
            split_half2(e[1][0], e[1][1], ph[2], plo[2]);
            split_half2(e[1][2], e[1][3], ph[3], plo[3]);
#pragma unroll
            for (int dt = 0; dt < 8; dt += 2) {
                const int row = r0 + (lane & 15);
                uint32_t v0, v1, v2, v3;
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                             : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                             : "r"(s_smem(sv) + sw128(row, dt + (lane >> 4))));
                mma_f16(o[dt], ph[0], ph[1], ph[2], ph[3], v0, v1);
                mma_f16(o[dt + 1], ph[0], ph[1], ph[2], ph[3], v2, v3);
                mma_f16(o[dt], plo[0], plo[1], plo[2], plo[3], v0, v1);
                mma_f16(o[dt + 1], plo[0], plo[1], plo[2], plo[3], v2, v3);
            }
            __syncwarp();
            if (lane == 0) asm volatile("{ .reg .b64 t; mbarrier.arrive.shared::cta.b64 t, [%0]; }" ::"r"(
                                            s_smem(&empty[s]))
                                        : "memory");
        }
#pragma unroll
        for (int r = 0; r < 2; r++) {
            lrun[r] += __shfl_xor_sync(0xffffffffu, lrun[r], 1);
            lrun[r] += __shfl_xor_sync(0xffffffffu, lrun[r], 2);
        }
        if (t4 == 0) {
            sml[warp][g][0] = mrun[0];
            sml[warp][g][1] = lrun[0];
            sml[warp][g + 8][0] = mrun[1];
            sml[warp][g + 8][1] = lrun[1];
        }
    }
    __syncthreads();  // every stage is consumed and every copy has landed (the producer drained)
    // the split's maximum per head and each warp's sums rescaled to it, then
    // added in warp order
    float *so = reinterpret_cast<float *>(smem);  // [4][16][kOPad]
    if (warp < kSWarps) {
#pragma unroll
        for (int r = 0; r < 2; r++) {
            const int h = g + 8 * r;
            float M = -INFINITY;
            for (int w = 0; w < kSWarps; w++) M = fmaxf(M, sml[w][h][0]);
            const float f = mrun[r] == -INFINITY ? 0.f : __expf(mrun[r] - M);
#pragma unroll
            for (int dt = 0; dt < 8; dt++)
                *reinterpret_cast<float2 *>(so + ((size_t)warp * kMaxQPerKV + h) * kOPad + 8 * dt + 2 * t4) =
                    make_float2(o[dt][2 * r] * f, o[dt][2 * r + 1] * f);
        }
    }
    __syncthreads();
    for (int i = tid; i < G * kHeadDim; i += blockDim.x) {
        const int h = i / kHeadDim, dd = i % kHeadDim;
        float acc = 0.f;
        for (int w = 0; w < kSWarps; w++) acc += so[((size_t)w * kMaxQPerKV + h) * kOPad + dd];
        const size_t idx = ((size_t)b * d.QH + j * G + h) * n_splits + c;
        pacc[idx * kHeadDim + dd] = acc;
    }
    if (tid < G) {
        const int h = tid;
        float M = -INFINITY;
        for (int w = 0; w < kSWarps; w++) M = fmaxf(M, sml[w][h][0]);
        float l = 0.f;
        for (int w = 0; w < kSWarps; w++)
            if (sml[w][h][0] != -INFINITY) l += __expf(sml[w][h][0] - M) * sml[w][h][1];
        const size_t idx = ((size_t)b * d.QH + j * G + h) * n_splits + c;
        pm[idx] = M;
        pl[idx] = l;
    }
}

// Prefill attention, flash style (goosedump gpt_oss.rs causal_gqa_batch): one
// CTA per (16 consecutive new tokens, kv head), warp w the kv head's query
// head w, the 16 tokens the MMA's rows.  The keys and values the block can
// see stream once through a two-stage shared-memory ring of 64-key chunks
// (asynchronous copies) shared by all the warps; per chunk each warp forms
// its 16 x 64 scores (q rotated as it is read, fp32 split into fp16 high and
// low parts, against the fp16 keys transposed by ldmatrix), masks them
// causally (and to the window), keeps a running maximum and sum per token,
// rescales its running value sums, and adds the chunk's exponentials (split
// the same way) times the values.  At the end the sink logit joins the
// maximum and the denominator, and o is written (bf16).  Requires the block's
// keys and values already in the cache (the append kernel).
constexpr int kFChunk = 64;                  // keys per stage
constexpr int kFPitch = kHeadDim + 8;        // shared row pitch (halves): ldmatrix rows on distinct banks
constexpr int kFStage = 2 * kFChunk * kFPitch;  // halves per stage: keys then values

__global__ void __launch_bounds__(256) moe_attn_flash_kernel(AttnDims d, const float *raw, const float2 *rope,
                                                             RowMap rm, int n, const __half *kc, const __half *vc,
                                                             const float *sinks, uint16_t *o) {
    __shared__ __align__(16) __half sm[2 * kFStage];
    const int T0 = blockIdx.x * 16, j = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, g = lane >> 2, t4 = lane & 3;
    // warp w: query head 8 blockIdx.z + w of the kv head (more than 8 heads
    // per kv head take further CTAs on grid.z)
    const int G = d.QH / d.KVH, hw = 8 * blockIdx.z + w, h = j * G + hw, nthr = blockDim.x;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the appended rows, q and the RoPE table
    asm volatile("griddepcontrol.launch_dependents;");
    const int nb = min(16, n - T0);  // tokens of this block
    const int P0 = row_pos(rm, T0), P1 = row_pos(rm, T0 + nb - 1);  // first and last position
    // keys the block can see: from the first token's window start to the last token
    const int kstart = (d.window > 0 && P0 + 1 > d.window) ? P0 + 1 - d.window : 0, kend = P1;
    const size_t seqbase = (size_t)row_seq(rm, T0) * d.max_ctx * d.KVH * kHeadDim + (size_t)j * kHeadDim;
    const size_t rstride = (size_t)d.KVH * kHeadDim;
    auto load_chunk = [&](int k0, int st) {
        __half *dst = sm + st * kFStage;
        for (int i = tid; i < 2 * kFChunk * 8; i += nthr) {
            const int v = i >= kFChunk * 8, r = (i >> 3) & (kFChunk - 1), pc = i & 7;
            __half *dp = dst + (v * kFChunk + r) * kFPitch + 8 * pc;
            const int t = k0 + r;
            if (t <= kend) {
                const __half *src = (v ? vc : kc) + seqbase + (size_t)t * rstride + 8 * pc;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                                 __cvta_generic_to_shared(dp))),
                             "l"(src)
                             : "memory");
            } else {
                *reinterpret_cast<uint4 *>(dp) = make_uint4(0, 0, 0, 0);  // past the block: zeros
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    load_chunk(kstart, 0);
    // q of tokens g and g + 8 (rows past the block: zeros), rotated; A
    // fragments of the four 16-dim steps, high and low parts
    uint32_t qh[4][4], ql[4][4];
    {
        float q[2][16];  // [token g / g+8][dims 16 s + 2 t4 + {0, 1, 8, 9}, s = 0..3]
#pragma unroll
        for (int r = 0; r < 2; r++) {
            const int tb = T0 + g + 8 * r;
            const bool ok = g + 8 * r < nb && hw < G;
            const float *qr = raw + (size_t)tb * (d.QH + 2 * d.KVH) * kHeadDim + (size_t)h * kHeadDim;
            const float2 *rt = rope + (size_t)tb * 32;
#pragma unroll
            for (int sp = 0; sp < 2; sp++)  // dims 16 sp + .. and their partners 32 + 16 sp + ..
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int dd = 16 * sp + 2 * t4 + (e & 1) + 8 * (e >> 1);
                    float l = 0.f, rr = 0.f;
                    float2 cs = make_float2(0.f, 0.f);
                    if (ok) {
                        l = qr[dd];
                        rr = qr[dd + 32];
                        cs = rt[dd];
                    }
                    q[r][4 * sp + e] = l * cs.x - rr * cs.y;
                    q[r][4 * (sp + 2) + e] = l * cs.y + rr * cs.x;
                }
        }
#pragma unroll
        for (int s4 = 0; s4 < 4; s4++) {
            split_half2(q[0][4 * s4], q[0][4 * s4 + 1], qh[s4][0], ql[s4][0]);      // token g, 2 t4 .. + 1
            split_half2(q[1][4 * s4], q[1][4 * s4 + 1], qh[s4][1], ql[s4][1]);      // token g + 8
            split_half2(q[0][4 * s4 + 2], q[0][4 * s4 + 3], qh[s4][2], ql[s4][2]);  // token g, 2 t4 + 8 .. + 9
            split_half2(q[1][4 * s4 + 2], q[1][4 * s4 + 3], qh[s4][3], ql[s4][3]);
        }
    }
    float oacc[8][4];
#pragma unroll
    for (int dt = 0; dt < 8; dt++) oacc[dt][0] = oacc[dt][1] = oacc[dt][2] = oacc[dt][3] = 0.f;
    float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
    const int tok[2] = {P0 + g, P0 + g + 8};  // positions of tokens g and g + 8
    int first[2];
#pragma unroll
    for (int r = 0; r < 2; r++) first[r] = (d.window > 0 && tok[r] + 1 > d.window) ? tok[r] + 1 - d.window : 0;
    int st = 0;
    for (int k0 = kstart; k0 <= kend; k0 += kFChunk, st ^= 1) {
        if (k0 + kFChunk <= kend) {
            load_chunk(k0 + kFChunk, st ^ 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
        const __half *sk = sm + st * kFStage, *sv = sk + kFChunk * kFPitch;
        if (hw < G) {
            // scores: 8 key tiles of 8
            float sc[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; nt++) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                for (int s2 = 0; s2 < 4; s2 += 2) {  // two 16-dim steps per ldmatrix.x4
                    const __half *rowp = sk + (size_t)(8 * nt + (lane & 7)) * kFPitch + 16 * s2 + 8 * (lane >> 3);
                    uint32_t b0, b1, b2, b3;
                    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(rowp))));
                    mma_f16(sc[nt], qh[s2][0], qh[s2][1], qh[s2][2], qh[s2][3], b0, b1);
                    mma_f16(sc[nt], ql[s2][0], ql[s2][1], ql[s2][2], ql[s2][3], b0, b1);
                    mma_f16(sc[nt], qh[s2 + 1][0], qh[s2 + 1][1], qh[s2 + 1][2], qh[s2 + 1][3], b2, b3);
                    mma_f16(sc[nt], ql[s2 + 1][0], ql[s2 + 1][1], ql[s2 + 1][2], ql[s2 + 1][3], b2, b3);
                }
            }
            // mask (causal, window, past the block's last key), chunk maximum per token
            float cm[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < 8; nt++)
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const int r = c >> 1, t = k0 + 8 * nt + 2 * t4 + (c & 1);
                    const bool ok = t >= first[r] && t <= tok[r] && t <= kend;
                    sc[nt][c] = ok ? sc[nt][c] * 0.125f : -INFINITY;  // 1 / sqrt(64)
                    cm[r] = fmaxf(cm[r], sc[nt][c]);
                }
            float scale[2];
#pragma unroll
            for (int r = 0; r < 2; r++) {
                cm[r] = fmaxf(cm[r], __shfl_xor_sync(0xffffffffu, cm[r], 1));
                cm[r] = fmaxf(cm[r], __shfl_xor_sync(0xffffffffu, cm[r], 2));
                const float mn = fmaxf(mrun[r], cm[r]);
                scale[r] = mrun[r] == -INFINITY ? 0.f : __expf(mrun[r] - mn);
                mrun[r] = mn;
                lrun[r] *= scale[r];
            }
#pragma unroll
            for (int dt = 0; dt < 8; dt++) {
                oacc[dt][0] *= scale[0], oacc[dt][1] *= scale[0];
                oacc[dt][2] *= scale[1], oacc[dt][3] *= scale[1];
            }
            // exponentials into the A fragments of the value products; sums
#pragma unroll
            for (int ks = 0; ks < 4; ks++) {  // keys 16 ks .. + 15 = key tiles 2 ks, 2 ks + 1
                float e[2][4];
#pragma unroll
                for (int hh = 0; hh < 2; hh++)
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const float v = sc[2 * ks + hh][c];
                        e[hh][c] = v == -INFINITY ? 0.f : __expf(v - mrun[c >> 1]);
                        lrun[c >> 1] += e[hh][c];
                    }
                uint32_t ph[4], pl[4];
                split_half2(e[0][0], e[0][1], ph[0], pl[0]);
                split_half2(e[0][2], e[0][3], ph[1], pl[1]);
                split_half2(e[1][0], e[1][1], ph[2], pl[2]);
                split_half2(e[1][2], e[1][3], ph[3], pl[3]);
#pragma unroll
                for (int dt = 0; dt < 8; dt += 2) {
                    const __half *rowp = sv + (size_t)(16 * ks + (lane & 15)) * kFPitch + 8 * dt + 8 * (lane >> 4);
                    uint32_t v0, v1, v2, v3;
                    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(rowp))));
                    mma_f16(oacc[dt], ph[0], ph[1], ph[2], ph[3], v0, v1);
                    mma_f16(oacc[dt + 1], ph[0], ph[1], ph[2], ph[3], v2, v3);
                    mma_f16(oacc[dt], pl[0], pl[1], pl[2], pl[3], v0, v1);
                    mma_f16(oacc[dt + 1], pl[0], pl[1], pl[2], pl[3], v2, v3);
                }
            }
        }
        __syncthreads();  // every warp is done with this stage before it is refilled
    }
    if (hw >= G) return;
    // the sink, and o
    const float sink = sinks[h];
#pragma unroll
    for (int r = 0; r < 2; r++) {
        lrun[r] += __shfl_xor_sync(0xffffffffu, lrun[r], 1);
        lrun[r] += __shfl_xor_sync(0xffffffffu, lrun[r], 2);
        const int b = T0 + g + 8 * r;
        const float mf = fmaxf(mrun[r], sink);
        const float f = mrun[r] == -INFINITY ? 0.f : __expf(mrun[r] - mf);
        const float inv = f / (lrun[r] * f + __expf(sink - mf));
        if (g + 8 * r >= nb) continue;
        uint16_t *orow = o + ((size_t)b * d.QH + h) * kHeadDim;
#pragma unroll
        for (int dt = 0; dt < 8; dt++) {
            const __nv_bfloat16 a0 = __float2bfloat16_rn(oacc[dt][2 * r] * inv);
            const __nv_bfloat16 a1 = __float2bfloat16_rn(oacc[dt][2 * r + 1] * inv);
            const uint32_t pr = (uint32_t)*reinterpret_cast<const uint16_t *>(&a0) |
                                ((uint32_t)*reinterpret_cast<const uint16_t *>(&a1) << 16);
            *reinterpret_cast<uint32_t *>(orow + 8 * dt + 2 * t4) = pr;
        }
    }
}

// o[b][h][:] = (sum over chunks of acc e^(m_c - m)) / (sum of l e^(m_c - m) +
// e^(sink - m)), m the largest of the chunk maxima and the sink; rounded to bf16.
constexpr int kMergeHeads = 4;  // query heads per merge CTA (64 threads each)
__global__ void moe_attn_merge_kernel(AttnDims d, const float *sinks, RowMap rm, const float *pm,
                                      const float *pl, const float *pacc, int n_chunks, uint16_t *o) {
    const int h = blockIdx.x * kMergeHeads + (threadIdx.x >> 6), b = blockIdx.y, e = threadIdx.x & 63;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the chunks' partials
    asm volatile("griddepcontrol.launch_dependents;");
    if (h >= d.QH) return;
    const int p = row_pos(rm, b);
    int first = 0, count = 0;
    if (p >= 0 && p < d.max_ctx) visible_range(d, p, first, count);
    const int per = split_len(count, n_chunks);
    const int nc = count > 0 ? (count + per - 1) / per : 0;  // the splits that hold keys
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
    KvMaps kv{};  // the caches as TMA maps (set with the caches)
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
    int32_t *status;  // the device status word and its detail (the prefill GEMM's bounded waits)
    uint16_t *xhat;
    float *xnorm;
    int32_t *count;
    float *raw;       // q, k, v with biases (before RoPE), fp32 [seq][(QH + 2 KVH) 64]
    float2 *rope;     // [seq][32] (cos, sin) x attention factor
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
    const size_t S = d.rows, nch = (d.max_ctx + kChunk - 1) / kChunk, QD = (size_t)d.QH * kHeadDim;
    Carve t;
    t.status = reinterpret_cast<int32_t *>(take(16));
    t.xhat = reinterpret_cast<uint16_t *>(take(S * d.H * 2));
    t.xnorm = reinterpret_cast<float *>(take(S * 4));
    t.count = reinterpret_cast<int32_t *>(take(4));
    t.raw = reinterpret_cast<float *>(take(S * (QD + 2 * (size_t)d.KVH * kHeadDim) * 4));
    t.rope = reinterpret_cast<float2 *>(take(S * 32 * 8));
    t.pm = reinterpret_cast<float *>(take(S * d.QH * nch * 4));
    t.pl = reinterpret_cast<float *>(take(S * d.QH * nch * 4));
    t.pacc = reinterpret_cast<float *>(take(S * d.QH * nch * kHeadDim * 4));
    t.o = reinterpret_cast<uint16_t *>(take(S * QD * 2));
    if (c) *c = t;
    return off;
}

PFN_cuTensorMapEncodeTiled_v12000 g_kv_encode = nullptr;

cudaError_t kv_encoder() {
    if (g_kv_encode) return cudaSuccess;
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_kv_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

// Splits of each row's context for the streamed decode attention: about
// three CTAs per SM over the (kv head, row) pairs, whole 64-key chunks, no
// more than the workspace's partials hold.
cudaError_t stream_splits(const AttnDims &d, int n, int most, int *splits) {
    static PerDevice<int> sms;
    int dev = 0;
    cudaError_t e = current_device_slot(&dev);
    if (e != cudaSuccess) return e;
    int &n_sm = sms.v[dev];
    if (!n_sm) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int pairs = d.KVH * n, cap = (d.max_ctx + kChunk - 1) / kChunk, chunks = (most + kSKeys - 1) / kSKeys;
    *splits = std::max(1, std::min({3 * n_sm / pairs, cap, chunks}));  // one wave: no partial second one
    return cudaSuccess;
}

// One step over n rows: norm, Q/K/V + RoPE table, (prefill: the append), the
// chunked attention, merge, output projection + residual.
cudaError_t attn_step(moe_attn *p, const uint16_t *x, int n, RowMap rm, void *out, cudaStream_t st) {
    Carve c;
    attn_carve(p->d, p->ws, &c);
    // chunks a row can need: a sliding layer's window, a prefill block's last
    // row's context, else the whole cache (launched CTAs past a row's
    // context exit at once, but each still costs a launch slot)
    int most = p->d.max_ctx;
    if (p->d.window > 0) most = std::min(most, p->d.window);
    if (rm.seq >= 0) most = std::min(most, rm.pos0 + n);
    cudaError_t e = launch_rms_norm_rows(x, p->w.gamma, n, p->d.H, p->d.eps, c.xhat, c.xnorm, c.count, st);
    const int RW = (p->d.QH + 2 * p->d.KVH) * kHeadDim, QD = p->d.QH * kHeadDim;
    ProjArgs a{};
    a.d = p->d;
    a.B = n;
    // above 32 rows (a prefill block) the projections run as tensor-core GEMMs
    const bool gemm = n > 32 && attn_gemm_supported(p->d.H, RW) && attn_gemm_supported(QD, p->d.H);
    if (e == cudaSuccess && gemm) {
        AttnGemm gq{};
        gq.n = n, gq.K = p->d.H, gq.rows = RW, gq.r1 = QD, gq.r2 = QD + p->d.KVH * kHeadDim;
        gq.x = c.xhat;
        gq.w[0] = p->w.wq, gq.w[1] = p->w.wk, gq.w[2] = p->w.wv;
        gq.bias[0] = p->w.bq, gq.bias[1] = p->w.bk, gq.bias[2] = p->w.bv;
        gq.kind = 0;
        gq.raw = c.raw;
        gq.status = c.status;
        e = launch_attn_gemm(gq, st);
        if (e == cudaSuccess) e = launch_pdl(moe_attn_rope_kernel, dim3(n), dim3(32), 0, st, p->d, rm, n, c.rope);
    } else if (e == cudaSuccess) {
        a.rows = RW;
        a.K = p->d.H;
        a.w[0] = p->w.wq, a.w[1] = p->w.wk, a.w[2] = p->w.wv;
        a.bias[0] = p->w.bq, a.bias[1] = p->w.bk, a.bias[2] = p->w.bv;
        a.r1 = QD;
        a.r2 = QD + p->d.KVH * kHeadDim;
        a.x = c.xhat;
        a.raw = c.raw;
        a.rope = c.rope;
        a.rows_of = rm;
        e = proj_launch<0>(a, st);
    }
    if (e == cudaSuccess && rm.seq >= 0)
        e = launch_pdl(moe_attn_append_kernel, dim3(n, p->d.KVH), dim3(kHeadDim), 0, st, p->d, (const float *)c.raw,
                       (const float2 *)c.rope, rm, p->kc, p->vc);
    if (e == cudaSuccess && rm.seq >= 0) {
        // prefill: the flash kernel over blocks of 16 tokens (a warp per query head)
        const int G = p->d.QH / p->d.KVH;
        e = launch_pdl(moe_attn_flash_kernel, dim3((n + 15) / 16, p->d.KVH, (G + 7) / 8), dim3(256), 0, st, p->d,
                       (const float *)c.raw, (const float2 *)c.rope, rm, n, (const __half *)p->kc,
                       (const __half *)p->vc, (const float *)p->w.sinks, c.o);
    } else {
        // decode: the new rows into the cache, the streamed attention over
        // splits of each row's context, the merge
        int splits = 1;
        if (e == cudaSuccess)
            e = launch_pdl(moe_attn_append_kernel, dim3(n, p->d.KVH), dim3(kHeadDim), 0, st, p->d,
                           (const float *)c.raw, (const float2 *)c.rope, rm, p->kc, p->vc);
        if (e == cudaSuccess) e = stream_splits(p->d, n, most, &splits);
        if (e == cudaSuccess) {
            static PerDevice<bool> opted;
            int dev = 0;
            e = current_device_slot(&dev);
            if (e == cudaSuccess && !opted.v[dev]) {
                e = cudaFuncSetAttribute(moe_attn_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSSmem);
                if (e == cudaSuccess) opted.v[dev] = true;
            }
        }
        if (e == cudaSuccess)
            e = launch_pdl(moe_attn_stream_kernel, dim3(splits, p->d.KVH, n), dim3((kSWarps + 1) * 32),
                           (size_t)kSSmem, st, p->d, (const float *)c.raw, (const float2 *)c.rope, rm, c.pm, c.pl,
                           c.pacc, splits, c.status, p->kv);
        if (e == cudaSuccess)
            e = launch_pdl(moe_attn_merge_kernel, dim3((p->d.QH + kMergeHeads - 1) / kMergeHeads, n),
                           dim3(kMergeHeads * kHeadDim), 0, st, p->d, (const float *)p->w.sinks,
                           rm, (const float *)c.pm, (const float *)c.pl, (const float *)c.pacc, splits, c.o);
    }
    if (e == cudaSuccess && gemm) {
        AttnGemm go{};
        go.n = n, go.K = QD, go.rows = p->d.H, go.r1 = go.r2 = p->d.H;
        go.x = c.o;
        go.w[0] = go.w[1] = go.w[2] = p->w.wo;
        go.bias[0] = go.bias[1] = go.bias[2] = p->w.bo;
        go.kind = 1;
        go.res = x;
        go.out = out;
        go.out_bf16 = p->out_bf16 ? 1 : 0;
        go.status = c.status;
        e = launch_attn_gemm(go, st);
    } else if (e == cudaSuccess) {
        a.rows = p->d.H;
        a.K = QD;
        a.w[0] = a.w[1] = a.w[2] = p->w.wo;
        a.bias[0] = a.bias[1] = a.bias[2] = p->w.bo;
        a.r1 = a.r2 = p->d.H;
        a.x = c.o;
        a.res = x;
        a.out = out;
        a.out_bf16 = p->out_bf16 ? 1 : 0;
        e = proj_launch<1>(a, st);
    }
    return e;
}

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
    p->d.rows = max_seqs;
    p->d.eps = 1e-5;
    attn_rope(p);
    return p;
}

void moe_attn_destroy(moe_attn *p) { delete p; }

int moe_attn_get_device_status(moe_attn *p, int *status, void *stream) {
    if (!p || !status) return moe_fail_status(MOE_EINVAL, "NULL argument");
    if (!p->ws) return moe_fail_status(MOE_ENOTREADY, "moe_attn_set_workspace has not been called");
    Carve c;
    attn_carve(p->d, p->ws, &c);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t h[4] = {0, 0, 0, 0};
    cudaError_t e = cudaMemcpyAsync(h, c.status, 16, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(c.status, 0, 16, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return moe_fail_status(MOE_ECUDA, "moe_attn_get_device_status: %s", cudaGetErrorString(e));
    *status = h[0];
    if (h[0]) return moe_fail_status(MOE_EDEVICE, "device status %d (detail %d)", h[0], h[1]);
    return MOE_OK;
}


int moe_attn_set_i(moe_attn *p, const char *key, long long v) {
    if (!p || !key) return moe_fail_status(MOE_EINVAL, "NULL argument");
    if (!strcmp(key, "sliding_window")) {
        if (v < 0 || v > 65536) return moe_fail_status(MOE_EINVAL, "sliding_window must be 0..65536");
        p->d.window = (int)v;
    } else if (!strcmp(key, "out_bf16")) {
        p->out_bf16 = v != 0;
    } else if (!strcmp(key, "prefill_rows")) {
        if (v < 1 || v > kMaxPrefillRows)
            return moe_fail_status(MOE_EINVAL, "prefill_rows must be 1..%d", kMaxPrefillRows);
        const int rows = std::max(p->d.max_seq, (int)v);
        if (rows != p->d.rows) {
            p->d.rows = rows;
            p->ws = nullptr;  // the workspace is sized by the rows: set it again
            p->ws_bytes = 0;
        }
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
    Carve c;
    attn_carve(p->d, static_cast<unsigned char *>(dev), &c);
    const cudaError_t e = cudaMemset(c.status, 0, 16);
    if (e != cudaSuccess) return moe_fail_status(MOE_ECUDA, "moe_attn_set_workspace: %s", cudaGetErrorString(e));
    p->ws = static_cast<unsigned char *>(dev);
    p->ws_bytes = bytes;
    return MOE_OK;
}

int moe_attn_set_cache(moe_attn *p, void *k_cache, void *v_cache) {
    if (!p || !k_cache || !v_cache) return moe_fail_status(MOE_EINVAL, "NULL argument");
    if (!aligned16(k_cache) || !aligned16(v_cache)) return moe_fail_status(MOE_EINVAL, "caches must be 16-byte aligned");
    cudaError_t e = kv_encoder();
    for (int i = 0; i < 2 && e == cudaSuccess; i++) {
        cuuint64_t dims[2] = {(cuuint64_t)p->d.KVH * kHeadDim, (cuuint64_t)p->d.max_seq * p->d.max_ctx};
        cuuint64_t strides[1] = {(cuuint64_t)p->d.KVH * kHeadDim * 2};
        cuuint32_t box[2] = {(cuuint32_t)kHeadDim, (cuuint32_t)kSKeys};
        cuuint32_t estr[2] = {1, 1};
        const CUresult r = g_kv_encode(i ? &p->kv.v : &p->kv.k, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, i ? v_cache : k_cache,
                                       dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) e = cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return moe_fail_status(MOE_ECUDA, "moe_attn_set_cache: tensor maps: %s", cudaGetErrorString(e));
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
    const cudaError_t e = attn_step(p, x, n_seqs, RowMap{positions, 0, -1}, out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : moe_fail_status(MOE_ECUDA, "moe_attn_decode: %s", cudaGetErrorString(e));
}

int moe_attn_prefill(moe_attn *p, const uint16_t *x, int n_tokens, int seq, int pos0, void *out, void *stream) {
    if (!p) return moe_fail_status(MOE_EINVAL, "NULL plan");
    if (!p->have_w) return moe_fail_status(MOE_ENOTREADY, "moe_attn_load_weights has not been called");
    if (!p->ws) return moe_fail_status(MOE_ENOTREADY, "moe_attn_set_workspace has not been called");
    if (!p->kc) return moe_fail_status(MOE_ENOTREADY, "moe_attn_set_cache has not been called");
    if (n_tokens < 0) return moe_fail_status(MOE_EINVAL, "n_tokens must be >= 0");
    if (n_tokens == 0) return MOE_OK;
    if (seq < 0 || seq >= p->d.max_seq) return moe_fail_status(MOE_EINVAL, "seq must be 0..%d", p->d.max_seq - 1);
    if (pos0 < 0 || (long long)pos0 + n_tokens > p->d.max_ctx)
        return moe_fail_status(MOE_EINVAL, "positions %d .. %lld outside the cache's %d rows", pos0,
                               (long long)pos0 + n_tokens - 1, p->d.max_ctx);
    if (!x || !out) return moe_fail_status(MOE_EINVAL, "NULL x or out");
    if (!aligned16(x) || !aligned16(out)) return moe_fail_status(MOE_EINVAL, "x and out must be 16-byte aligned");
    const size_t xb = (size_t)n_tokens * p->d.H * 2, ob = (size_t)n_tokens * p->d.H * (p->out_bf16 ? 2 : 4);
    const char *xc = reinterpret_cast<const char *>(x), *oc = static_cast<const char *>(out);
    if (xc < oc + ob && oc < xc + xb) return moe_fail_status(MOE_EINVAL, "x and out must not overlap");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // blocks of up to max(max_seqs, prefill_rows) rows (goosedump gpt_oss.rs
    // prefill_attention_layer: batches of PREFILL_BATCH_SIZE rows, each
    // appended, then attended)
    const size_t osz = p->out_bf16 ? 2 : 4;
    cudaError_t e = cudaSuccess;
    for (int r0 = 0; r0 < n_tokens && e == cudaSuccess; r0 += p->d.rows) {
        const int nb = std::min(p->d.rows, n_tokens - r0);
        e = attn_step(p, x + (size_t)r0 * p->d.H, nb, RowMap{nullptr, pos0 + r0, seq},
                      static_cast<char *>(out) + (size_t)r0 * p->d.H * osz, st);
    }
    return e == cudaSuccess ? MOE_OK : moe_fail_status(MOE_ECUDA, "moe_attn_prefill: %s", cudaGetErrorString(e));
}

}  // extern "C"
