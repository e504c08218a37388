// moe_decode.cu -- decode path: MXFP4 dequant-in-register GEMVs over the
// selected experts, the weighted combine with the residual, and the debug
// dequantiser that shares the GEMV's dequantisation routine.
//
// goosedump gpt_oss.rs `mixture_of_experts` (decode) evaluates, per selected
// expert, `matrix_vector_pair(gate, up)` + bias, `swiglu_inplace`,
// `matrix_vector(down)` + bias and scales by the route weight; the weighted
// outputs are summed in slot order and added to the residual in `forward`.
//
// Design (sm_103a):
//  * work item = (tile of <= 8*NT routes of one expert, 16 weight rows);
//    4 warps split the K dimension; each thread streams its rows' packed
//    codes with 128-bit loads straight from HBM into registers;
//  * dequantisation in registers: one 32-bit word of codes (8 nibbles) gives
//    four bf16x2 pairs (nibble i, nibble i+4) by two shifts and two masks,
//    scaled exactly by the E8M0 exponent with one bf16x2 multiply;
//  * the multiply-accumulate runs on the tensor cores (m16n8k16 bf16, fp32
//    accumulate) with the routed activations as the N=8 operand, staged in
//    shared memory in the matching pair order;
//  * gate/up kernel: bias + clamped SwiGLU epilogue writes h (bf16);
//    down kernel: bias, times the route weight, into a per-route fp32 buffer;
//    the combine kernel sums the slots of each token in slot order and adds x.
#include "moe_common.cuh"

namespace {

constexpr int kDecThreads = 128;  // 4 warps

struct DecodeArgs {
    BlockParams bp;
    Workspace ws;
    MatPtrs A0, A1;   // gate, up (GATEUP) or down, unused
    int Kdim;         // reduction length: H for gate/up, F for down
};

// 8 nibbles of one 32-bit word -> four bf16x2 (value * 2^-126, exact):
// pair i holds nibble i in the low half and nibble i+4 in the high half.
__device__ __forceinline__ void nibbles_to_bf16x2(uint32_t w, uint32_t p[4]) {
    p[0] = ((w << 6) & 0x01C001C0u) | ((w << 12) & 0x80008000u);
    p[1] = ((w << 2) & 0x01C001C0u) | ((w << 8) & 0x80008000u);
    p[2] = ((w >> 2) & 0x01C001C0u) | ((w << 4) & 0x80008000u);
    p[3] = ((w >> 6) & 0x01C001C0u) | (w & 0x80008000u);
}

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// E8M0 exponent -> bf16x2 multiplier(s) turning value*2^-126 into value*2^(s-127).
// For s <= 128 one factor 2^(s-1) suffices; above that two factors are used.
__device__ __forceinline__ uint32_t scale_lo(uint32_t s) {
    uint32_t b = (s <= 128u) ? ((s + 126u) << 7) : (253u << 7);  // 2^(s-1) or 2^126
    return b | (b << 16);
}
__device__ __forceinline__ uint32_t scale_hi(uint32_t s) {
    uint32_t b = (s <= 128u) ? 0x3F80u : (s << 7);                // 1 or 2^(s-127)
    return b | (b << 16);
}

template <bool BIG>
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t s1, uint32_t s2, uint32_t p[4]) {
    nibbles_to_bf16x2(w, p);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        p[i] = bmul2(p[i], s1);
        if (BIG) p[i] = bmul2(p[i], s2);
    }
}

__device__ __forceinline__ void mma_bf16_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Byte offset inside a staged activation row of 16-byte chunk k of 32-block b
// (chunk rotation by b/2 keeps the fragment loads bank-conflict free).
__device__ __forceinline__ int bstage_off(int b, int k) { return b * 64 + (((k + (b >> 1)) & 3) << 4); }

template <bool GATEUP, int NT, bool BIG>
__device__ __forceinline__ void decode_mainloop(const DecodeArgs &a, const uint8_t *c0, const uint8_t *c1,
                                                const uint8_t *sc, const unsigned char *bst, int Sb,
                                                float acc[2][NT][4]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int K = a.Kdim, nb = K / 32, nq = (nb + 3) / 4;
    const size_t rowb = (size_t)K / 2;
    constexpr int NM = GATEUP ? 2 : 1;
    for (int q = warp; q < nq; q += 4) {
        const int b = 4 * q + t4;
        const bool valid = b < nb;
        uint4 A[NM][2];
        uint32_t s1[NM][2], s2[NM][2];
#pragma unroll
        for (int m = 0; m < NM; m++) {
            const uint8_t *cb = (m == 0 ? c0 : c1);
#pragma unroll
            for (int h = 0; h < 2; h++) {
                if (valid) {
                    A[m][h] = ldg_stream(cb + (size_t)(g + 8 * h) * rowb + 16 * b);
                    uint32_t s = sc[(m * 16 + g + 8 * h) * nb + b];
                    s1[m][h] = scale_lo(s);
                    s2[m][h] = scale_hi(s);
                } else {
                    A[m][h] = make_uint4(0, 0, 0, 0);
                    s1[m][h] = s2[m][h] = 0x3F803F80u;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 4; k++) {
            uint4 B[NT];
#pragma unroll
            for (int n = 0; n < NT; n++) {
                B[n] = valid ? *reinterpret_cast<const uint4 *>(bst + (size_t)(n * 8 + g) * Sb + bstage_off(b, k))
                             : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int m = 0; m < NM; m++) {
                uint32_t w0 = (&A[m][0].x)[k], w1 = (&A[m][1].x)[k];
                uint32_t p0[4], p1[4];
                dequant_word<BIG>(w0, s1[m][0], s2[m][0], p0);
                dequant_word<BIG>(w1, s1[m][1], s2[m][1], p1);
#pragma unroll
                for (int n = 0; n < NT; n++) {
                    mma_bf16_16816(acc[m][n], p0[0], p1[0], p0[1], p1[1], B[n].x, B[n].y);
                    mma_bf16_16816(acc[m][n], p0[2], p1[2], p0[3], p1[3], B[n].z, B[n].w);
                }
            }
        }
    }
}

template <bool GATEUP, int NT>
__global__ void __launch_bounds__(kDecThreads) moe_decode_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int tile_idx = blockIdx.y;
    if (tile_idx >= *a.ws.n_tiles) return;
    const int4 tile = a.ws.tiles[tile_idx];
    const int e = tile.x, rstart = tile.y, rcount = tile.z;
    const int j0 = blockIdx.x * 16;
    const int K = a.Kdim, nb = K / 32;
    const int Sb = 2 * K + 32;                       // staged row stride (bytes)
    const int tid = threadIdx.x;
    const int E = a.bp.E;
    constexpr int NM = GATEUP ? 2 : 1;

    unsigned char *bst = smem;                                     // [8*NT][Sb]
    uint8_t *sc = smem + (size_t)8 * NT * Sb;                      // [NM][16][nb]
    float *red = reinterpret_cast<float *>(sc + ((NM * 16 * nb + 15) & ~15));  // [4][NM][NT][16][8]

    // stage the routed activations (already in MMA pair order) with the chunk rotation
    const int nchunk = K / 8;
    for (int i = tid; i < rcount * nchunk; i += kDecThreads) {
        int n = i / nchunk, c = i - n * nchunk;
        const uint16_t *src = GATEUP ? a.ws.xhat_mma + (size_t)a.ws.perm_token[rstart + n] * K
                                     : a.ws.h + (size_t)(rstart + n) * K;
        uint4 v = *reinterpret_cast<const uint4 *>(src + c * 8);
        *reinterpret_cast<uint4 *>(bst + (size_t)n * Sb + bstage_off(c >> 2, c & 3)) = v;
    }
    // stage the E8M0 scales of the 16 rows (contiguous in the canonical layout)
    const uint8_t *c0 = mat_codes(a.A0, e, E) + (size_t)j0 * (K / 2);
    const uint8_t *c1 = GATEUP ? mat_codes(a.A1, e, E) + (size_t)j0 * (K / 2) : nullptr;
    int big = 0;
    for (int m = 0; m < NM; m++) {
        const uint8_t *s = mat_scales(m == 0 ? a.A0 : a.A1, e, E) + (size_t)j0 * nb;
        for (int i = tid; i < 16 * nb; i += kDecThreads) {
            uint8_t v = s[i];
            sc[m * 16 * nb + i] = v;
            big |= (v > 128);
        }
    }
    big = __syncthreads_or(big);

    float acc[2][NT][4];
#pragma unroll
    for (int m = 0; m < 2; m++)
#pragma unroll
        for (int n = 0; n < NT; n++)
#pragma unroll
            for (int r = 0; r < 4; r++) acc[m][n][r] = 0.f;
    if (big)
        decode_mainloop<GATEUP, NT, true>(a, c0, c1, sc, bst, Sb, acc);
    else
        decode_mainloop<GATEUP, NT, false>(a, c0, c1, sc, bst, Sb, acc);

    // cross-warp reduction of the split-K partials (fixed order)
    const int lane = tid & 31, warp = tid >> 5, g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int m = 0; m < NM; m++)
#pragma unroll
        for (int n = 0; n < NT; n++) {
            float *r = red + (((warp * NM + m) * NT + n) * 16) * 8;
            r[g * 8 + 2 * t4] = acc[m][n][0];
            r[g * 8 + 2 * t4 + 1] = acc[m][n][1];
            r[(g + 8) * 8 + 2 * t4] = acc[m][n][2];
            r[(g + 8) * 8 + 2 * t4 + 1] = acc[m][n][3];
        }
    __syncthreads();
    for (int idx = tid; idx < 16 * 8 * NT; idx += kDecThreads) {
        const int row = idx & 15, col = idx >> 4;  // col = route within the tile
        if (col >= rcount) continue;
        const int n = col >> 3, c = col & 7;
        float s[NM];
#pragma unroll
        for (int m = 0; m < NM; m++) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < 4; w++) v += red[(((w * NM + m) * NT + n) * 16 + row) * 8 + c];
            s[m] = v;
        }
        const int j = j0 + row;
        const int route = rstart + col;
        if (GATEUP) {
            float gg = s[0] + mat_bias(a.A0, e, E)[j];
            float uu = s[1] + mat_bias(a.A1, e, E)[j];
            float hv = swiglu_clamped(gg, uu, a.bp.alpha, a.bp.limit);
            __nv_bfloat16 hb = __float2bfloat16_rn(hv);
            a.ws.h[(size_t)route * a.bp.F + mma_perm_pos(j)] = *reinterpret_cast<uint16_t *>(&hb);
        } else {
            float yv = s[0] + mat_bias(a.A0, e, E)[j];
            a.ws.y[(size_t)route * a.bp.H + j] = a.ws.perm_w[route] * yv;
        }
    }
}

// out[t] = x[t] + Σ_slot y[loc[t][slot]] (slot order; the shared expert last)
__global__ void __launch_bounds__(256) moe_combine_kernel(BlockParams bp, Workspace ws, const uint16_t *x,
                                                          float *out, int T) {
    const int t = blockIdx.y;
    const int KK = bp.K + bp.n_shared;
    const int H = bp.H;
    const int i4 = blockIdx.x * blockDim.x + threadIdx.x;  // float4 index
    if (i4 * 4 >= H) return;
    float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < KK; s++) {
        int p = ws.loc[t * KK + s];
        float4 v = *reinterpret_cast<const float4 *>(ws.y + (size_t)p * H + i4 * 4);
        m.x += v.x;
        m.y += v.y;
        m.z += v.z;
        m.w += v.w;
    }
    uint2 xv = *reinterpret_cast<const uint2 *>(x + (size_t)t * H + i4 * 4);
    float4 o;
    o.x = __uint_as_float(xv.x << 16) + m.x;
    o.y = __uint_as_float(xv.x & 0xFFFF0000u) + m.y;
    o.z = __uint_as_float(xv.y << 16) + m.z;
    o.w = __uint_as_float(xv.y & 0xFFFF0000u) + m.w;
    *reinterpret_cast<float4 *>(out + (size_t)t * H + i4 * 4) = o;
}

// One thread per 32-element block: the GEMV's dequantisation, un-permuted.
__global__ void moe_dequant_kernel(MatPtrs m, int expert, int n_experts, float *out) {
    const int nb = m.cols / 32;
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)m.rows * nb) return;
    const size_t row = i / nb, b = i - row * nb;
    const uint8_t *codes = mat_codes(m, expert, n_experts);
    const uint8_t *scales = mat_scales(m, expert, n_experts);
    uint4 v = *reinterpret_cast<const uint4 *>(codes + row * (m.cols / 2) + 16 * b);
    uint32_t s = scales[row * nb + b];
    uint32_t s1 = scale_lo(s), s2 = scale_hi(s);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float *o = out + row * m.cols + 32 * b;
    for (int k = 0; k < 4; k++) {
        uint32_t p[4];
        if (s > 128u)
            dequant_word<true>(w[k], s1, s2, p);
        else
            dequant_word<false>(w[k], s1, s2, p);
        for (int ii = 0; ii < 4; ii++) {
            o[8 * k + ii] = __uint_as_float(p[ii] << 16);
            o[8 * k + ii + 4] = __uint_as_float(p[ii] & 0xFFFF0000u);
        }
    }
}

__global__ void moe_scan_scales_kernel(const uint8_t *s, size_t n, int32_t *flag) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    size_t stride = (size_t)gridDim.x * blockDim.x;
    int bad = 0;
    for (; i < n; i += stride) bad |= (s[i] == 0xFF);
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(flag, 1);
}

}  // namespace

size_t decode_smem_bytes(bool gateup, int nt, int K) {
    int NM = gateup ? 2 : 1;
    size_t Sb = 2 * (size_t)K + 32;
    size_t sc = ((size_t)NM * 16 * (K / 32) + 15) & ~(size_t)15;
    return 8 * nt * Sb + sc + (size_t)4 * NM * nt * 16 * 8 * 4;
}

template <bool GATEUP, int NT>
static cudaError_t launch_one(const DecodeArgs &a, int rows, int max_tiles, cudaStream_t st) {
    size_t sm = decode_smem_bytes(GATEUP, NT, a.Kdim);
    static bool done = false;
    MOE_CUDA_TRY(smem_optin_once(moe_decode_kernel<GATEUP, NT>, done));
    dim3 grid(rows / 16, max_tiles);
    moe_decode_kernel<GATEUP, NT><<<grid, kDecThreads, sm, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_decode_stage(const BlockParams &bp, const Workspace &ws, const MatPtrs &a0, const MatPtrs &a1,
                                bool gateup, int T, int nt, cudaStream_t st) {
    const int R = T * (bp.K + bp.n_shared);
    // upper bound on the tile count: each expert's last tile may be partial
    int tiles = (R + 8 * nt - 1) / (8 * nt) + bp.E + bp.n_shared;
    if (tiles > ws.max_tiles) tiles = ws.max_tiles;
    if (gateup) {
        DecodeArgs gu{bp, ws, a0, a1, bp.H};
        return nt == 1 ? launch_one<true, 1>(gu, bp.F, tiles, st) : launch_one<true, 2>(gu, bp.F, tiles, st);
    }
    DecodeArgs dn{bp, ws, a0, a0, bp.F};
    return nt == 1 ? launch_one<false, 1>(dn, bp.H, tiles, st) : launch_one<false, 2>(dn, bp.H, tiles, st);
}

cudaError_t launch_combine(const BlockParams &bp, const Workspace &ws, const uint16_t *x, int T, float *out,
                           cudaStream_t st) {
    dim3 grid((bp.H / 4 + 255) / 256, T);
    moe_combine_kernel<<<grid, 256, 0, st>>>(bp, ws, x, out, T);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const MatPtrs &m, int expert, int n_experts, float *out, cudaStream_t st) {
    size_t n = (size_t)m.rows * (m.cols / 32);
    moe_dequant_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(m, expert, n_experts, out);
    return cudaGetLastError();
}

cudaError_t launch_scan_scales(const uint8_t *scales, size_t n, int32_t *flag, cudaStream_t st) {
    moe_scan_scales_kernel<<<1024, 256, 0, st>>>(scales, n, flag);
    return cudaGetLastError();
}
