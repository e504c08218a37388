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
//  * work item = (tile of <= 8*NT routes of one expert, 16 weight rows),
//    walked by persistent CTAs; 8 warps split the K dimension; each thread
//    streams its rows' packed codes with 128-bit loads straight from HBM into
//    registers, one iteration ahead;
//  * dequantisation in registers: one 32-bit word of codes (8 nibbles) gives
//    four bf16x2 pairs (nibble i, nibble i+4) by two shifts and two masks,
//    scaled exactly by the E8M0 exponent with one bf16x2 multiply;
//  * the multiply-accumulate runs on the tensor cores (m16n8k16 bf16, fp32
//    accumulate) with the routed activations as the N=8 operand, read in the
//    matching pair order from L1/L2;
//  * gate/up kernel: bias + clamped SwiGLU epilogue writes h (bf16);
//    down kernel: bias, times the route weight, into a per-route fp32 buffer;
//    the combine kernel sums the slots of each token in slot order and adds x.
#include "moe_common.cuh"

namespace {


struct DecodeArgs {
    BlockParams bp;
    Workspace ws;
    MatPtrs A0, A1;   // gate, up (GATEUP) or down, unused
    int Kdim;         // reduction length: H for gate/up, F for down
    int rows;         // output rows: F for gate/up, H for down
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

// Two exact dequantisers feed the tensor cores:
//  * fp16 (used when every E8M0 exponent of the work item lies in [104, 140],
//    where e2m1 * 2^(s-127) is exactly representable in fp16): the hardware
//    e2m1x2 -> f16x2 conversion turns one byte (two nibbles, low nibble =
//    even element) into a natural-order pair, then one f16x2 multiply applies
//    the power-of-two scale; MMA kind f16 against the fp16 activations;
//  * bf16 (any exponent): the shift/mask construction above, re-paired into
//    natural order with byte permutes, scaled by one or two bf16x2
//    multiplies; MMA kind bf16 against the bf16 activations.
// Both keep K in natural order, so the activations need no reordering.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t h[4]) {
    asm("{ .reg .b8 a, b, c, d;\n"
        "  mov.b32 {a, b, c, d}, %4;\n"
        "  cvt.rn.f16x2.e2m1x2 %0, a;\n"
        "  cvt.rn.f16x2.e2m1x2 %1, b;\n"
        "  cvt.rn.f16x2.e2m1x2 %2, c;\n"
        "  cvt.rn.f16x2.e2m1x2 %3, d; }"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}
// fp16 bits of 2^(s-127) in both halves, s in [104, 140]
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t s) {
    const uint32_t b = (s >= 113u) ? ((s - 112u) << 10) : (1u << (s - 103u));
    return b | (b << 16);
}
__device__ __forceinline__ bool f16_exact_scale(uint32_t s) { return s >= 104u && s <= 140u; }

// natural-order bf16 pairs (n0,n1),(n2,n3),(n4,n5),(n6,n7), exact, any exponent
template <bool BIG>
__device__ __forceinline__ void dequant_word_nat(uint32_t w, uint32_t s1, uint32_t s2, uint32_t o[4]) {
    uint32_t p[4];
    dequant_word<BIG>(w, s1, s2, p);
    o[0] = __byte_perm(p[0], p[1], 0x5410);
    o[1] = __byte_perm(p[2], p[3], 0x5410);
    o[2] = __byte_perm(p[0], p[1], 0x7632);
    o[3] = __byte_perm(p[2], p[3], 0x7632);
}

__device__ __forceinline__ void mma_f16_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Persistent CTAs of 8 warps, each owning a contiguous range of work items
// (tile, 16-row block).  The packed codes and E8M0 scales of an item (16 rows
// of one or two matrices, contiguous rows in the canonical layout) are
// streamed into a two-stage shared-memory ring by bulk asynchronous copies
// (one per row) while the
// previous item is computed.  The 8 warps split K (32-element blocks in groups
// of four per warp-iteration) and reduce through shared memory; each thread
// prefetches the next iteration's activation fragments into registers.
constexpr int kDecWarps = 8;
constexpr uint64_t kDecWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ bool dec_mbar_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait (about 2 s, or until another CTA reported a failure).
__device__ __forceinline__ bool dec_mbar_wait(uint64_t *b, uint32_t parity, int32_t *status, int where) {
    if (dec_mbar_try(b, parity)) return true;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (uint32_t i = 0;; i++) {
        if (dec_mbar_try(b, parity)) return true;
        if ((i & 63) == 63) {
            if (*(volatile int32_t *)status != 0) return false;
            uint64_t t1;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
            if (t1 - t0 > kDecWaitNs) {
                set_device_error(status, MOE_DEV_WAIT_TIMEOUT, where);
                return false;
            }
        }
    }
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Shared-memory geometry of one stage for reduction length K.
struct DecGeom {
    int rs;        // row stride of packed codes (bytes)
    int scb;       // bytes of one matrix's 16 rows of scales, rounded to 16
    int bias;      // offset of the [NM][16] fp32 biases in a stage
    int stage;     // bytes of one stage (NM matrices)
    __host__ __device__ DecGeom(int K, int NM) {
        const int rb = K / 2;
        rs = rb;  // unpadded: two stages + the reductions of two CTAs fit one SM
        scb = (16 * (K / 32) + 15) & ~15;
        bias = NM * (16 * rs + scb);
        stage = (bias + NM * 64 + 127) & ~127;
    }
};

// One warp-iteration covers 16 rows x 4 blocks of 32 (per thread: block 4q+t4
// of rows g and g+8).  If every exponent of the iteration admits the exact
// fp16 conversion (warp vote) the fp16 path runs on the prefetched fp16
// activations; otherwise the bf16 path runs on bf16 activations loaded for
// this iteration.
template <bool GATEUP, int NT>
__device__ __forceinline__ void decode_mainloop(int K, const unsigned char *st, const DecGeom &geo,
                                                const uint16_t *const (&brow16)[NT],
                                                const uint16_t *const (&browbf)[NT], float acc[2][NT][4]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int nb = K / 32, nq = (nb + 3) / 4;
    constexpr int NM = GATEUP ? 2 : 1;
    const unsigned char *codes = st;                    // [NM][16][rs]
    const uint8_t *sc = st + NM * 16 * geo.rs;          // [NM][scb]
    auto load_b = [&](uint4 (&B)[NT][4], const uint16_t *const (&brow)[NT], int q) {
        const int b = 4 * q + t4;
        const bool valid = q < nq && b < nb;
#pragma unroll
        for (int n = 0; n < NT; n++)
#pragma unroll
            for (int k = 0; k < 4; k++)
                B[n][k] = (valid && brow[n]) ? __ldg(reinterpret_cast<const uint4 *>(brow[n] + 32 * b) + k)
                                            : make_uint4(0, 0, 0, 0);
    };
    uint4 B[NT][4];
    load_b(B, brow16, warp);
    for (int q = warp; q < nq; q += kDecWarps) {
        const int b = 4 * q + t4;
        const bool valid = b < nb;
        uint4 Bn[NT][4];
        load_b(Bn, brow16, q + kDecWarps);
        uint4 A[2][2];
        uint32_t sv[2][2];
        bool f16ok = true;
#pragma unroll
        for (int m = 0; m < NM; m++)
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int r = g + 8 * h;
                A[m][h] = valid ? *reinterpret_cast<const uint4 *>(codes + (m * 16 + r) * geo.rs + 16 * b)
                                : make_uint4(0, 0, 0, 0);
                sv[m][h] = valid ? sc[m * geo.scb + r * nb + b] : 127u;
                f16ok = f16ok && f16_exact_scale(sv[m][h]);
            }
        if (__all_sync(0xffffffffu, f16ok)) {
#pragma unroll
            for (int k = 0; k < 4; k++) {
#pragma unroll
                for (int m = 0; m < NM; m++) {
                    uint32_t p0[4], p1[4];
                    e2m1x8_to_f16((&A[m][0].x)[k], p0);
                    e2m1x8_to_f16((&A[m][1].x)[k], p1);
                    const uint32_t s0 = scale_f16x2(sv[m][0]), s1 = scale_f16x2(sv[m][1]);
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        p0[i] = hmul2_f16(p0[i], s0);
                        p1[i] = hmul2_f16(p1[i], s1);
                    }
#pragma unroll
                    for (int n = 0; n < NT; n++) {
                        mma_f16_16816(acc[m][n], p0[0], p1[0], p0[1], p1[1], B[n][k].x, B[n][k].y);
                        mma_f16_16816(acc[m][n], p0[2], p1[2], p0[3], p1[3], B[n][k].z, B[n][k].w);
                    }
                }
            }
        } else {
            uint4 Bb[NT][4];
            load_b(Bb, browbf, q);
#pragma unroll
            for (int k = 0; k < 4; k++) {
#pragma unroll
                for (int m = 0; m < NM; m++) {
                    uint32_t p0[4], p1[4];
                    dequant_word_nat<true>((&A[m][0].x)[k], scale_lo(sv[m][0]), scale_hi(sv[m][0]), p0);
                    dequant_word_nat<true>((&A[m][1].x)[k], scale_lo(sv[m][1]), scale_hi(sv[m][1]), p1);
#pragma unroll
                    for (int n = 0; n < NT; n++) {
                        mma_bf16_16816(acc[m][n], p0[0], p1[0], p0[1], p1[1], Bb[n][k].x, Bb[n][k].y);
                        mma_bf16_16816(acc[m][n], p0[2], p1[2], p0[3], p1[3], Bb[n][k].z, Bb[n][k].w);
                    }
                }
            }
        }
#pragma unroll
        for (int n = 0; n < NT; n++)
#pragma unroll
            for (int k = 0; k < 4; k++) B[n][k] = Bn[n][k];
    }
}

__device__ __forceinline__ void dec_arrive(uint64_t *b) {
    asm volatile("{ .reg .b64 t; mbarrier.arrive.shared::cta.b64 t, [%0]; }" ::"r"(smem_addr(b)) : "memory");
}

// Warp roles: warps 0..7 consume (split-K over the item's 16 rows), warp 8
// produces (bulk copies).  mbarriers: full[s] (codes landed), empty[s] (8
// consumer warps done with stage s), redfull[r] (8 partials written),
// redempty[r] (epilogue done with reduction buffer r).  The epilogue of item
// k runs on consumer warp k % 8; no CTA-wide barrier is used in the loop.
template <bool GATEUP, int NT>
__global__ void __launch_bounds__((kDecWarps + 1) * 32, 2) moe_decode_kernel(DecodeArgs a) {
    constexpr int NM = GATEUP ? 2 : 1;
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(16) float red[2][kDecWarps][NM][NT][16][8];  // split-K partials, double-buffered
    __shared__ __align__(8) uint64_t bars[8];
    uint64_t *full = bars, *empty = bars + 2, *redfull = bars + 4, *redempty = bars + 6;
    const int K = a.Kdim, nb = K / 32;
    const DecGeom geo(K, NM);
    const int RB = a.rows / 16;
    asm volatile("griddepcontrol.launch_dependents;");
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&empty[i])), "r"(kDecWarps));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&redfull[i])), "r"(kDecWarps));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&redempty[i])));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // the tile table, activations and (for down) h come from the previous kernels
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_items = *a.ws.n_tiles * RB;
    const int per = (n_items + gridDim.x - 1) / gridDim.x;
    const int begin = blockIdx.x * per, end = min(n_items, begin + per);
    const int n = end - begin;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t4 = lane & 3;
    const int E = a.bp.E;
    int32_t *status = a.ws.status;

    if (warp == kDecWarps) {
        // ---------------------------------------------------------- producer
        int issued = 0;
        for (int k = 0; k < n; k++) {
            const int s = k & 1, item = begin + k;
            if (k >= 2 && !dec_mbar_wait(&empty[s], ((k >> 1) - 1) & 1, status, 51)) break;
            const int4 tile = a.ws.tiles[item / RB];
            const int e = tile.x, j0 = (item % RB) * 16;
            unsigned char *st = dsm + s * geo.stage;
            if (lane == 0) {
                const uint32_t bytes = NM * (16 * (K / 2) + 16 * nb + 64);
                asm volatile("{ .reg .b64 t; mbarrier.arrive.expect_tx.shared::cta.b64 t, [%0], %1; }" ::"r"(
                                 smem_addr(&full[s])),
                             "r"(bytes)
                             : "memory");
            }
            __syncwarp();
#pragma unroll
            for (int m = 0; m < NM; m++) {
                const MatPtrs &M = m == 0 ? a.A0 : a.A1;
                if (lane < 16)
                    bulk_g2s(st + (m * 16 + lane) * geo.rs, mat_codes(M, e, E) + (size_t)(j0 + lane) * (K / 2), K / 2,
                             &full[s]);
                if (lane == 16 + m) {
                    bulk_g2s(st + NM * 16 * geo.rs + m * geo.scb, mat_scales(M, e, E) + (size_t)j0 * nb, 16 * nb,
                             &full[s]);
                    bulk_g2s(st + geo.bias + m * 64, mat_bias(M, e, E) + j0, 64, &full[s]);
                }
            }
            issued = k + 1;
        }
        // the copies of the last two stages must have landed before this warp exits
        for (int k = max(0, issued - 2); k < issued; k++) dec_mbar_wait(&full[k & 1], (k >> 1) & 1, status, 52);
        return;
    }

    // -------------------------------------------------------------- consumers
    int cur_tile = -1;
    int4 tile = make_int4(0, 0, 0, 0);
    for (int k = 0; k < n; k++) {
        const int item = begin + k, s = k & 1, r = k & 1;
        if (item / RB != cur_tile) {
            cur_tile = item / RB;
            tile = a.ws.tiles[cur_tile];
        }
        const int rstart = tile.y, rcount = tile.z;
        const int j0 = (item % RB) * 16;
        if (!dec_mbar_wait(&full[s], (k >> 1) & 1, status, 50)) break;
        const unsigned char *st = dsm + s * geo.stage;
        const uint16_t *brow16[NT], *browbf[NT];
#pragma unroll
        for (int nn = 0; nn < NT; nn++) {
            const int col = nn * 8 + g;
            brow16[nn] = browbf[nn] = nullptr;
            if (col < rcount) {
                if (GATEUP) {
                    const size_t tok = (size_t)a.ws.perm_token[rstart + col];
                    brow16[nn] = a.ws.xhat16 + tok * K;
                    browbf[nn] = a.ws.xhat + tok * K;
                } else {
                    brow16[nn] = a.ws.h16 + (size_t)(rstart + col) * K;
                    browbf[nn] = a.ws.h + (size_t)(rstart + col) * K;
                }
            }
        }
        const bool epi = warp == (k % kDecWarps);
        float b0 = 0.f, b1 = 0.f;  // biases of row lane & 15 (epilogue warp only), read before the stage is released
        if (epi) {
            const float *sb = reinterpret_cast<const float *>(st + geo.bias);
            b0 = sb[lane & 15];
            if (GATEUP) b1 = sb[16 + (lane & 15)];
        }
        float acc[2][NT][4];
#pragma unroll
        for (int m = 0; m < 2; m++)
#pragma unroll
            for (int nn = 0; nn < NT; nn++)
#pragma unroll
                for (int q = 0; q < 4; q++) acc[m][nn][q] = 0.f;
        decode_mainloop<GATEUP, NT>(K, st, geo, brow16, browbf, acc);
        __syncwarp();
        if (lane == 0) dec_arrive(&empty[s]);  // this warp no longer reads stage s
        if (k >= 2 && !dec_mbar_wait(&redempty[r], ((k >> 1) - 1) & 1, status, 53)) break;
#pragma unroll
        for (int m = 0; m < NM; m++)
#pragma unroll
            for (int nn = 0; nn < NT; nn++) {
                float(*rp)[8] = red[r][warp][m][nn];
                rp[g][2 * t4] = acc[m][nn][0];
                rp[g][2 * t4 + 1] = acc[m][nn][1];
                rp[g + 8][2 * t4] = acc[m][nn][2];
                rp[g + 8][2 * t4 + 1] = acc[m][nn][3];
            }
        __syncwarp();
        if (lane == 0) dec_arrive(&redfull[r]);
        if (epi) {
            if (!dec_mbar_wait(&redfull[r], (k >> 1) & 1, status, 54)) break;
            for (int idx = lane; idx < 16 * 8 * NT; idx += 32) {
                const int row = idx & 15, col = idx >> 4;  // col = route within the tile
                const float bb0 = __shfl_sync(0xffffffffu, b0, row);
                const float bb1 = __shfl_sync(0xffffffffu, b1, row);
                if (col >= rcount) continue;
                const int nn = col >> 3, c = col & 7;
                float sm[NM];
#pragma unroll
                for (int m = 0; m < NM; m++) {
                    float v = 0.f;
#pragma unroll
                    for (int w = 0; w < kDecWarps; w++) v += red[r][w][m][nn][row][c];
                    sm[m] = v;
                }
                const int j = j0 + row;
                const int route = rstart + col;
                if (GATEUP) {
                    const float hv = swiglu_clamped(sm[0] + bb0, sm[1] + bb1, a.bp.alpha, a.bp.limit);
                    const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                    const __half h16 = __float2half_rn(__bfloat162float(hb));  // exact for |h| >= 2^-14
                    a.ws.h[(size_t)route * a.bp.F + j] = *reinterpret_cast<const uint16_t *>(&hb);
                    a.ws.h16[(size_t)route * a.bp.F + j] = *reinterpret_cast<const uint16_t *>(&h16);
                } else {
                    a.ws.y[(size_t)route * a.bp.H + j] = a.ws.perm_w[route] * (sm[0] + bb0);
                }
            }
            __syncwarp();
            if (lane == 0) dec_arrive(&redempty[r]);
        }
    }
}

// out[t] = x[t] + Σ_slot y[loc[t][slot]] (slot order; the shared expert last)
__global__ void __launch_bounds__(256) moe_combine_kernel(BlockParams bp, Workspace ws, const uint16_t *x,
                                                          float *out, int T) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
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

// One thread per 32-element block: the GEMV's element converters (fp16 where
// the exponent allows it exactly, bf16 otherwise), written out in natural order.
__global__ void moe_dequant_kernel(MatPtrs m, int expert, int n_experts, float *out) {
    const int nb = m.cols / 32;
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)m.rows * nb) return;
    const size_t row = i / nb, b = i - row * nb;
    const uint8_t *codes = mat_codes(m, expert, n_experts);
    const uint8_t *scales = mat_scales(m, expert, n_experts);
    const uint4 v = *reinterpret_cast<const uint4 *>(codes + row * (m.cols / 2) + 16 * b);
    const uint32_t s = scales[row * nb + b];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float *o = out + row * m.cols + 32 * b;
    for (int k = 0; k < 4; k++) {
        uint32_t p[4];
        if (f16_exact_scale(s)) {
            e2m1x8_to_f16(w[k], p);
            for (int ii = 0; ii < 4; ii++) p[ii] = hmul2_f16(p[ii], scale_f16x2(s));
            for (int ii = 0; ii < 4; ii++) {
                o[8 * k + 2 * ii] = __half2float(__ushort_as_half((unsigned short)(p[ii] & 0xFFFFu)));
                o[8 * k + 2 * ii + 1] = __half2float(__ushort_as_half((unsigned short)(p[ii] >> 16)));
            }
        } else {
            if (s > 128u)
                dequant_word_nat<true>(w[k], scale_lo(s), scale_hi(s), p);
            else
                dequant_word_nat<false>(w[k], scale_lo(s), scale_hi(s), p);
            for (int ii = 0; ii < 4; ii++) {
                o[8 * k + 2 * ii] = __uint_as_float(p[ii] << 16);
                o[8 * k + 2 * ii + 1] = __uint_as_float(p[ii] & 0xFFFF0000u);
            }
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

size_t decode_smem_bytes(bool gateup, int, int K) { return 2 * (size_t)DecGeom(K, gateup ? 2 : 1).stage; }

template <bool GATEUP, int NT>
static cudaError_t launch_one(const DecodeArgs &a, int n_items_max, cudaStream_t st) {
    static int per_sm = 0, n_sm = 0;
    static bool done = false;
    const size_t smem = decode_smem_bytes(GATEUP, NT, a.Kdim);
    MOE_CUDA_TRY(smem_optin_once(moe_decode_kernel<GATEUP, NT>, done));
    if (!per_sm) {
        int dev = 0;
        MOE_CUDA_TRY(cudaGetDevice(&dev));
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
        MOE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, moe_decode_kernel<GATEUP, NT>,
                                                                   (kDecWarps + 1) * 32, smem));
        if (per_sm < 1) per_sm = 1;
    }
    int grid = n_sm * per_sm;
    if (grid > n_items_max) grid = n_items_max;
    if (grid < 1) grid = 1;
    return launch_pdl(moe_decode_kernel<GATEUP, NT>, dim3(grid), dim3((kDecWarps + 1) * 32), smem, st, a);
}

cudaError_t launch_decode_stage(const BlockParams &bp, const Workspace &ws, const MatPtrs &a0, const MatPtrs &a1,
                                bool gateup, int T, int nt, cudaStream_t st) {
    const int R = T * (bp.K + bp.n_shared);
    // upper bound on the tile count: each expert's last tile may be partial
    int tiles = (R + 8 * nt - 1) / (8 * nt) + bp.E + bp.n_shared;
    if (tiles > ws.max_tiles) tiles = ws.max_tiles;
    if (gateup) {
        DecodeArgs gu{bp, ws, a0, a1, bp.H, bp.F};
        const int items = tiles * (bp.F / 16);
        return nt == 1 ? launch_one<true, 1>(gu, items, st) : launch_one<true, 2>(gu, items, st);
    }
    DecodeArgs dn{bp, ws, a0, a0, bp.F, bp.H};
    const int items = tiles * (bp.H / 16);
    return nt == 1 ? launch_one<false, 1>(dn, items, st) : launch_one<false, 2>(dn, items, st);
}

cudaError_t launch_combine(const BlockParams &bp, const Workspace &ws, const uint16_t *x, int T, float *out,
                           cudaStream_t st) {
    dim3 grid((bp.H / 4 + 255) / 256, T);
    return launch_pdl(moe_combine_kernel, grid, dim3(256), 0, st, bp, ws, x, out, T);
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
