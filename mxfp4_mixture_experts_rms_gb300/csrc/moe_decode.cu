// moe_decode.cu -- decode path: MXFP4 dequant-in-register GEMVs over the
// selected experts, the weighted combine with the residual, and the debug
// dequantiser that shares the GEMV's element converter.
//
// goosedump gpt_oss.rs `mixture_of_experts` (decode) evaluates, per selected
// expert, `matrix_vector_pair(gate, up)` + bias, `swiglu_inplace`,
// `matrix_vector(down)` + bias and scales by the route weight; the weighted
// outputs are summed in slot order and added to the residual in `forward`.
//
// Design (sm_103a), for each of the two projections:
//  * one persistent CTA per SM: 14 consumer warps, 1 producer warp and 1
//    epilogue warp (16 warps: 4 per SM sub-partition, up to 128 registers a
//    thread);
//  * work item = (tile of <= 8*NT routes of one expert, 16 weight rows of gate
//    and of up, or 32 rows of down -- about 46 KB of codes either way); each
//    CTA walks a contiguous range of items;
//  * the producer streams every item into a ring of S shared-memory stages
//    (S = 2..8, as deep as shared memory allows), so that several items are in
//    flight from HBM while one is computed.  The item's 16 rows of packed codes
//    are contiguous: one bulk asynchronous copy per matrix (the copy engine's
//    cost is per copy, so it only gets large ranges); the E8M0 scales and the
//    biases go by 16-byte asynchronous copies of the producer's 32 lanes;
//  * the consumer warps split K in pairs of 32-element blocks; for tiles of up
//    to 8 routes each keeps the routed activations of its K range in registers
//    for the whole tile (16-route tiles load them per block pair, one ahead);
//  * ldmatrix hands each thread one 32-bit word (8 codes) of two rows of a
//    block; the hardware e2m1x2 -> f16x2 conversion yields the E2M1 values
//    exactly; two m16n8k16 MMAs (fp32 accumulate) form the unscaled block dot
//    product, which one FFMA per output multiplies by 2^(e-127) (exact) into
//    the accumulator;
//  * the 14 split-K partials meet in shared memory; the epilogue warp sums
//    them and applies bias + clamped SwiGLU (gate/up) or bias x route weight
//    (down), off the consumers' critical path, while the producer warp does
//    nothing but keep the copy engine busy (a bulk-copy issue blocks while the
//    engine is saturated, so any other work there idles HBM).
//
// Activations are fp16 (x_hat and h are bf16 values; fp16 holds them exactly
// for 2^-17 <= |v| < 65504) unless the plan found at load time that they can
// leave the fp16 range (huge gamma or SwiGLU limit); then the bf16 variant
// (template BF) converts the E2M1 values to bf16 and multiplies in bf16.
#include "moe_common.cuh"

// Timeline marker (no-op unless an instrumented build defines it).
#ifndef MOE_DEC_MARK
#define MOE_DEC_MARK(slot, k)
#endif

namespace {

constexpr int kCW = 14;                      // consumer warps
constexpr int kProd = kCW, kEpi = kCW + 1;   // producer warp, epilogue warp
constexpr int kDecThreads = (kCW + 2) * 32;
constexpr int kMaxPairs = 5;                 // block pairs per consumer warp: K <= 14 * 5 * 64 = 4480
constexpr int kMaxStages = 8;
constexpr uint64_t kDecWaitNs = 2000000000ull;

struct DecodeArgs {
    BlockParams bp;
    Workspace ws;
    MatPtrs A0, A1;  // gate, up (GATEUP) or down, unused
    int Kdim;        // reduction length: H for gate/up, F for down
    int rows;        // output rows: F for gate/up, H for down
    int stages;      // shared-memory ring depth
    int h_bf16;      // gate/up: write h as bf16 (else fp16)
    int stall;       // test hook: consumers first wait on a barrier nothing completes
    int slot_index;  // expert cache: the matrices are slot-major and a tile's slot is its fourth field
};

// f16x2 holding two E2M1 values (0, +-0.5 .. +-6) -> the same values as bf16x2.
// Non-zero E2M1 magnitudes in fp16 are 0x3800..0x4600 (bit 13 or 14 set, low
// byte zero); the bf16 pattern is (fp16 magnitude >> 3) + 0x3800.
__device__ __forceinline__ uint32_t e2m1_f16x2_to_bf16x2(uint32_t h) {
    const uint32_t mag = h & 0x7FFF7FFFu;
    const uint32_t t = ((mag >> 3) & 0x0FFF0FFFu) + 0x38003800u;
    const uint32_t nz = ((mag >> 13) | (mag >> 14)) & 0x00010001u;  // 1 per non-zero half
    return (t & (nz * 0xFFFFu)) | (h & 0x80008000u);
}

// 2^(e-127) as fp32 (e = 0 gives the subnormal 2^-127); e = 255 is rejected at load.
__device__ __forceinline__ float e8m0_f32(uint32_t e) { return __uint_as_float(max(e << 23, 0x00400000u)); }

__device__ __forceinline__ void mma_16816(bool bf, float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    if (bf)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A*B (C = 0)
__device__ __forceinline__ void mma_16816_z(bool bf, float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
    if (bf)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%10,%10,%10};\n"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%10,%10,%10};\n"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

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
// Wait for copies already issued to land before the CTA's shared memory goes:
// only the time limit ends it (a failure reported elsewhere does not).
__device__ __forceinline__ void dec_mbar_drain(uint64_t *b, uint32_t parity, int32_t *status) {
    if (dec_mbar_try(b, parity)) return;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
        if (dec_mbar_try(b, parity)) return;
        uint64_t t1;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
        if (t1 - t0 > kDecWaitNs) {
            set_device_error(status, MOE_DEV_WAIT_TIMEOUT, 58);
            return;
        }
    }
}
__device__ __forceinline__ void dec_arrive(uint64_t *b) {
    asm volatile("{ .reg .b64 t; mbarrier.arrive.shared::cta.b64 t, [%0]; }" ::"r"(smem_addr(b)) : "memory");
}
// L2 policy for the weight stream: each weight byte is read once per
// forward, so its lines go first when L2 needs room.  Everything else of a
// forward (its activations and tables, and the kernels' own code) then stays
// in L2 while gigabytes of weights pass through it; measured on a GB300 this
// shortened the routing kernel's serial tail from 7.6 to 2.9 us at 16 tokens.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t r[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}

// Shared-memory geometry of one stage for reduction length K.
struct DecGeom {
    int rs;     // row stride of packed codes (bytes)
    int scb;    // bytes of one matrix's 16 rows of scales, rounded to 16
    int bias;   // offset of the [NM][16] fp32 biases in a stage
    int stage;  // bytes of one stage (NM matrices)
    __host__ __device__ DecGeom(int K, int NM) {
        rs = K / 2;
        scb = (16 * (K / 32) + 15) & ~15;
        bias = NM * (16 * rs + scb);
        stage = (bias + NM * 64 + 127) & ~127;
    }
};
// split-K partials: [2][kCW][NM][NT][16 rows][8 columns] fp32
__host__ __device__ constexpr size_t dec_red_bytes(int NM, int NT) { return (size_t)2 * kCW * NM * NT * 128 * 4; }

// NM: matrices per item -- gate and up (gate/up), or for down 1 or 2 groups of
// 16 consecutive rows (an item of 32 rows carries as many bytes as a gate/up item)
template <bool GATEUP, int NT, bool BF, int MP, int NM>
__global__ void __launch_bounds__(kDecThreads, 1) moe_decode_kernel(DecodeArgs a) {
    static_assert(!GATEUP || NM == 2, "gate/up items hold both matrices");
    constexpr int IR = GATEUP ? 16 : 16 * NM;  // output rows per item
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t bars[2 * kMaxStages + 5];
    uint64_t *full = bars, *empty = bars + kMaxStages, *redfull = bars + 2 * kMaxStages, *redempty = redfull + 2;
    uint64_t *never = redempty + 2;  // completed by nobody (the stall test hook waits on it)
    const int K = a.Kdim, nb = K / 32, S = a.stages;
    const DecGeom geo(K, NM);
    float *red = reinterpret_cast<float *>(dsm + (size_t)S * geo.stage);
    const int RB = a.rows / IR;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; i++) {
            // one arrival with the codes' byte count + one per producer lane (its small copies)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 33;" ::"r"(smem_addr(&full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&empty[i])), "r"(kCW + 1));
        }
        for (int i = 0; i < 2; i++) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&redfull[i])), "r"(kCW));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&redempty[i])));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(never)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Gate/up needs the routing kernel's results everywhere.  The down kernel
    // is let in only once every gate/up CTA has passed its own wait, so the
    // tile table is complete: its producer starts streaming weights at once
    // (into the SMs gate/up has left) and only its consumers and epilogue wait
    // for gate/up's results.
    if (GATEUP || threadIdx.x < kCW * 32 || threadIdx.x >= kEpi * 32) asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    // the producer's lanes fetch the first 64 tile-table entries together with
    // the tile count, so that the first copy waits for one round trip, not two
    int4 tpre[2] = {make_int4(0, 0, 0, 0), make_int4(0, 0, 0, 0)};
    if ((threadIdx.x >> 5) == kProd) {
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int ti = (threadIdx.x & 31) + 32 * h;
            if (ti < a.ws.max_tiles) tpre[h] = __ldcg(a.ws.tiles + ti);
        }
    }
    const int n_items = *a.ws.n_tiles * RB;
    const int per = (n_items + gridDim.x - 1) / gridDim.x;
    const int begin = blockIdx.x * per, end = min(n_items, begin + per);
    const int n = end - begin;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t4 = lane & 3;
    const int E = a.bp.E;
    int32_t *status = a.ws.status;

    if (warp == kProd) {
        // ---------------------------------------------------------- producer
        const uint64_t pol = l2_evict_first();
        auto tile_of = [&](int ti) {  // warp-uniform ti
            if (ti >= 64) return a.ws.tiles[ti];
            const int4 v = ti < 32 ? tpre[0] : tpre[1];
            const int src = ti & 31;
            return make_int4(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src),
                             __shfl_sync(0xffffffffu, v.z, src), __shfl_sync(0xffffffffu, v.w, src));
        };
        auto issue = [&](int k) {
            const int s = k % S, item = begin + k;
            const int4 tile = tile_of(item / RB);
            // the matrix index: the expert, or with the expert cache its slot
            // (the shared expert, index E, is never cached)
            const int e = a.slot_index && tile.x < E ? tile.w : tile.x, j0 = (item % RB) * IR;
            unsigned char *st = dsm + (size_t)s * geo.stage;
            if (lane == 0) {
                const uint32_t bytes = NM * 16 * (K / 2);
                asm volatile("{ .reg .b64 t; mbarrier.arrive.expect_tx.shared::cta.b64 t, [%0], %1; }" ::"r"(
                                 smem_addr(&full[s])),
                             "r"(bytes)
                             : "memory");
#pragma unroll
                for (int m = 0; m < NM; m++) {
                    const MatPtrs &M = m == 0 ? a.A0 : a.A1;
                    const int jm = GATEUP ? j0 : j0 + 16 * m;
                    bulk_g2s(st + m * 16 * geo.rs, mat_codes(M, e, E) + (size_t)jm * (K / 2), 16 * (K / 2), &full[s], pol);
                }
            }
#pragma unroll
            for (int m = 0; m < NM; m++) {
                const MatPtrs &M = m == 0 ? a.A0 : a.A1;
                const int jm = GATEUP ? j0 : j0 + 16 * m;
                const uint8_t *scs = mat_scales(M, e, E) + (size_t)jm * nb;
                unsigned char *scd = st + NM * 16 * geo.rs + m * geo.scb;
                for (int c = lane; c < nb; c += 32) cp_async16(scd + 16 * c, scs + 16 * c, pol);
                if (lane < 4) cp_async16(st + geo.bias + m * 64 + 16 * lane, mat_bias(M, e, E) + jm + 4 * lane, pol);
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(&full[s])) : "memory");
            if (lane == 0) MOE_DEC_MARK(0, k);
        };
        int issued = 0;
        for (int k = 0; k < n; k++) {
            if (k >= S && !dec_mbar_wait(&empty[k % S], ((k / S) - 1) & 1, status, 51)) break;
            issue(k);
            issued++;
        }
        // the copies still in flight must land before this warp exits: the
        // last S issued (each earlier one was consumed before its stage was
        // refilled), waited for even when the kernel is failing
        for (int k = max(0, issued - S); k < issued; k++) dec_mbar_drain(&full[k % S], (k / S) & 1, status);
        return;
    }
    if (warp == kEpi) {
        // ---------------------------------------------------------- epilogue
        for (int k = 0; k < n; k++) {
            const int s = k % S, r = k & 1, item = begin + k;
            // this item's biases, read before the stage may be refilled
            if (!dec_mbar_wait(&full[s], (k / S) & 1, status, 55)) break;
            const float *sb = reinterpret_cast<const float *>(dsm + (size_t)s * geo.stage + geo.bias);
            const float b0 = sb[lane >> 1], b1 = NM == 2 ? sb[16 + (lane >> 1)] : 0.f;
            asm volatile("" ::"f"(b0), "f"(b1));
            __syncwarp();
            if (lane == 0) dec_arrive(&empty[s]);
            if (!dec_mbar_wait(&redfull[r], (k >> 1) & 1, status, 54)) break;
            if (lane == 0) MOE_DEC_MARK(3, k);
            const int4 tile = a.ws.tiles[item / RB];
            const int rstart = tile.y, rcount = tile.z, j0 = (item % RB) * IR;
            // lane: row lane/2, columns 4*(lane&1) .. +3 of every column group nn
            const int row = lane >> 1, c0 = 4 * (lane & 1);
            const float *rr = red + (size_t)r * kCW * NM * NT * 128;
#pragma unroll
            for (int nn = 0; nn < NT; nn++) {
                float4 sm[NM];
#pragma unroll
                for (int m = 0; m < NM; m++) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int w = 0; w < kCW; w++) {
                        const float4 q =
                            *reinterpret_cast<const float4 *>(rr + ((w * NM + m) * NT + nn) * 128 + row * 8 + c0);
                        v.x += q.x;
                        v.y += q.y;
                        v.z += q.z;
                        v.w += q.w;
                    }
                    sm[m] = v;
                }
                const float s0[4] = {sm[0].x, sm[0].y, sm[0].z, sm[0].w};
                const float s1[4] = {sm[NM - 1].x, sm[NM - 1].y, sm[NM - 1].z, sm[NM - 1].w};
                const int j = j0 + row;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const int col = nn * 8 + c0 + c;  // route within the tile
                    if (col >= rcount) continue;
                    const int route = rstart + col;
                    if (GATEUP) {
                        const float hv = swiglu_clamped(s0[c] + b0, s1[c] + b1, a.bp.alpha, a.bp.limit);
                        const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                        if (a.h_bf16) {
                            a.ws.h[(size_t)route * a.bp.F + j] = *reinterpret_cast<const uint16_t *>(&hb);
                        } else {
                            const __half h16 = __float2half_rn(__bfloat162float(hb));
                            a.ws.h16[(size_t)route * a.bp.F + j] = *reinterpret_cast<const uint16_t *>(&h16);
                        }
                    } else {
                        a.ws.y[(size_t)route * a.bp.H + j] = a.ws.perm_w[route] * (s0[c] + b0);
                    }
                }
                if (!GATEUP && NM == 2) {
                    // the second group of 16 rows (a separate pass keeps the live ranges short)
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const int col = nn * 8 + c0 + c;
                        if (col >= rcount) continue;
                        const int route = rstart + col;
                        a.ws.y[(size_t)route * a.bp.H + j + 16] = a.ws.perm_w[route] * (s1[c] + b1);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) MOE_DEC_MARK(4, k);
            if (lane == 0) dec_arrive(&redempty[r]);
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    // test hook: a bounded wait that runs out (nothing completes `never`); the
    // status word then stops the producer and the epilogue, which drain and exit
    if (GATEUP && a.stall && !dec_mbar_wait(never, 0, status, 59)) return;
    const int npairs = (nb + 1) >> 1;
    // activations of pair p = warp + kCW*i: block 2p+bb, token column nn*8 + g,
    // elements 8*t4 .. 8*t4+7 of the block (zero past the end of K or of the tile)
    const uint16_t *brow[NT];
    auto load_pair = [&](uint4(&dst)[2][NT], int i) {
        const int p = warp + kCW * i;
#pragma unroll
        for (int bb = 0; bb < 2; bb++) {
            const int b = 2 * p + bb;
#pragma unroll
            for (int nn = 0; nn < NT; nn++)
                dst[bb][nn] = (p < npairs && b < nb && brow[nn])
                                  ? __ldg(reinterpret_cast<const uint4 *>(brow[nn] + 32 * b + 8 * t4))
                                  : make_uint4(0, 0, 0, 0);
        }
    };
    constexpr bool kRegB = NT == 1;  // whole-tile activations in registers
    uint4 Bc[kRegB ? MP : 1][2][NT];
    int cur_tile = -1;
    int rstart = 0, rcount = 0;
    // ldmatrix row address pattern: matrices (rows 0-7, block 2p), (rows 8-15, 2p),
    // (rows 0-7, 2p+1), (rows 8-15, 2p+1); this lane supplies row lrow of matrix lane/8
    const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lblk = lane >> 4;
#pragma unroll 1
    for (int k = 0; k < n; k++) {
        const int item = begin + k, s = k % S, r = k & 1;
        if (item / RB != cur_tile) {
            cur_tile = item / RB;
            const int4 tile = a.ws.tiles[cur_tile];
            rstart = tile.y;
            rcount = tile.z;
#pragma unroll
            for (int nn = 0; nn < NT; nn++) {
                const int col = nn * 8 + g;
                brow[nn] = nullptr;
                if (col < rcount) {
                    if (GATEUP)
                        brow[nn] = (BF ? a.ws.xhat : a.ws.xhat16) + (size_t)a.ws.perm_token[rstart + col] * K;
                    else
                        brow[nn] = (BF ? a.ws.h : a.ws.h16) + (size_t)(rstart + col) * K;
                }
            }
            if (kRegB) {
#pragma unroll
                for (int i = 0; i < MP; i++) load_pair(Bc[kRegB ? i : 0], i);
            }
        }
        uint4 Bcur[2][NT], Bnext[2][NT];
        if (!kRegB) load_pair(Bcur, 0);
        if (!dec_mbar_wait(&full[s], (k / S) & 1, status, 50)) break;
        if (warp == 0 && lane == 0) MOE_DEC_MARK(1, k);
        const unsigned char *st = dsm + (size_t)s * geo.stage;
        float acc[NM][NT][4];
#pragma unroll
        for (int m = 0; m < NM; m++)
#pragma unroll
            for (int nn = 0; nn < NT; nn++)
#pragma unroll
                for (int q = 0; q < 4; q++) acc[m][nn][q] = 0.f;
#pragma unroll
        for (int i = 0; i < MP; i++) {
            const int p = warp + kCW * i;
            if (p < npairs) {
                if (!kRegB && i + 1 < MP) load_pair(Bnext, i + 1);
                const int bk0 = 2 * p, bk1 = min(2 * p + 1, nb - 1);  // a missing odd block has zero activations
#pragma unroll
                for (int m = 0; m < NM; m++) {
                    const unsigned char *codes = st + m * 16 * geo.rs;
                    const uint8_t *sc = st + NM * 16 * geo.rs + m * geo.scb;
                    uint32_t wv[4];
                    ldmatrix_x4(wv, codes + lrow * geo.rs + 16 * (lblk ? bk1 : bk0));
                    const float f[2][2] = {{e8m0_f32(sc[g * nb + bk0]), e8m0_f32(sc[(g + 8) * nb + bk0])},
                                           {e8m0_f32(sc[g * nb + bk1]), e8m0_f32(sc[(g + 8) * nb + bk1])}};
#pragma unroll
                    for (int bb = 0; bb < 2; bb++) {
                        uint32_t hg[4], hg8[4];
                        e2m1x8_to_f16(wv[2 * bb], hg);
                        e2m1x8_to_f16(wv[2 * bb + 1], hg8);
                        if (BF) {
#pragma unroll
                            for (int q = 0; q < 4; q++) {
                                hg[q] = e2m1_f16x2_to_bf16x2(hg[q]);
                                hg8[q] = e2m1_f16x2_to_bf16x2(hg8[q]);
                            }
                        }
#pragma unroll
                        for (int nn = 0; nn < NT; nn++) {
                            float t[4];
                            const uint4 bv = kRegB ? Bc[kRegB ? i : 0][bb][nn] : Bcur[bb][nn];
                            mma_16816_z(BF, t, hg[0], hg8[0], hg[1], hg8[1], bv.x, bv.y);
                            mma_16816(BF, t, hg[2], hg8[2], hg[3], hg8[3], bv.z, bv.w);
                            acc[m][nn][0] = fmaf(t[0], f[bb][0], acc[m][nn][0]);
                            acc[m][nn][1] = fmaf(t[1], f[bb][0], acc[m][nn][1]);
                            acc[m][nn][2] = fmaf(t[2], f[bb][1], acc[m][nn][2]);
                            acc[m][nn][3] = fmaf(t[3], f[bb][1], acc[m][nn][3]);
                        }
                    }
                }
                if (!kRegB) {
#pragma unroll
                    for (int bb = 0; bb < 2; bb++)
#pragma unroll
                        for (int nn = 0; nn < NT; nn++) Bcur[bb][nn] = Bnext[bb][nn];
                }
            }
            // keep the shared-memory reads of one pair from being hoisted into the
            // previous one (register pressure)
            asm volatile("" ::: "memory");
        }
        __syncwarp();
        if (warp == 0 && lane == 0) MOE_DEC_MARK(2, k);
        if (lane == 0) MOE_DEC_MARK(6 + warp, k);
        if (lane == 0) dec_arrive(&empty[s]);  // this warp no longer reads stage s
        if (k >= 2 && !dec_mbar_wait(&redempty[r], ((k >> 1) - 1) & 1, status, 53)) break;
        float *rw = red + (size_t)(r * kCW + warp) * NM * NT * 128;
#pragma unroll
        for (int m = 0; m < NM; m++)
#pragma unroll
            for (int nn = 0; nn < NT; nn++) {
                float *rp = rw + (m * NT + nn) * 128;
                *reinterpret_cast<float2 *>(rp + g * 8 + 2 * t4) = make_float2(acc[m][nn][0], acc[m][nn][1]);
                *reinterpret_cast<float2 *>(rp + (g + 8) * 8 + 2 * t4) = make_float2(acc[m][nn][2], acc[m][nn][3]);
            }
        __syncwarp();
        if (lane == 0) dec_arrive(&redfull[r]);
    }
}

// out[t] = x[t] + Σ_slot y[loc[t][slot]] (slot order; the shared expert last),
// as fp32, or (BF16OUT) rounded to bf16 (nearest, ties to even): the input of
// a next stacked block, written here instead of by a separate cast.
template <bool BF16OUT>
__global__ void __launch_bounds__(256) moe_combine_kernel(BlockParams bp, Workspace ws, const uint16_t *x, void *out,
                                                          int T) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");  // a following cast may set itself up
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
    if (BF16OUT) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
        reinterpret_cast<uint2 *>(out)[((size_t)t * H + i4 * 4) / 4] =
            make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
    } else {
        *reinterpret_cast<float4 *>(static_cast<float *>(out) + (size_t)t * H + i4 * 4) = o;
    }
}

// One thread per 32-element block: the GEMV's element converter (E2M1 -> fp16,
// exact) and its fp32 block scale, written out in natural order.
__global__ void moe_dequant_kernel(MatPtrs m, int expert, int n_experts, float *out) {
    const int nb = m.cols / 32;
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)m.rows * nb) return;
    const size_t row = i / nb, b = i - row * nb;
    const uint8_t *codes = mat_codes(m, expert, n_experts);
    const uint8_t *scales = mat_scales(m, expert, n_experts);
    const uint4 v = *reinterpret_cast<const uint4 *>(codes + row * (m.cols / 2) + 16 * b);
    const float f = e8m0_f32(scales[row * nb + b]);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float *o = out + row * m.cols + 32 * b;
    for (int k = 0; k < 4; k++) {
        uint32_t p[4];
        e2m1x8_to_f16(w[k], p);
        for (int ii = 0; ii < 4; ii++) {
            o[8 * k + 2 * ii] = __half2float(__ushort_as_half((unsigned short)(p[ii] & 0xFFFFu))) * f;
            o[8 * k + 2 * ii + 1] = __half2float(__ushort_as_half((unsigned short)(p[ii] >> 16))) * f;
        }
    }
}

// flag bit 0: an exponent holds the NaN code 0xFF; bit 1: an exponent lies
// outside [104, 140] (where e2m1 * 2^(e-127) stops being exact in fp16)
__global__ void moe_scan_scales_kernel(const uint8_t *s, size_t n, int32_t *flag) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    size_t stride = (size_t)gridDim.x * blockDim.x;
    int bad = 0, wide = 0;
    for (; i < n; i += stride) {
        bad |= (s[i] == 0xFF);
        wide |= (s[i] < 104 || s[i] > 140);
    }
    bad = __syncthreads_or(bad);
    wide = __syncthreads_or(wide);
    if (threadIdx.x == 0 && (bad || wide)) atomicOr(flag, (bad ? 1 : 0) | (wide ? 2 : 0));
}

// max |v| over n floats (NaN counts as +inf), as the bit pattern of a
// non-negative float: the integer order of such patterns is their value order.
__global__ void moe_absmax_kernel(const float *v, int n, uint32_t *out) {
    uint32_t m = 0;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float a = fabsf(v[i]);
        m = max(m, a != a ? 0x7F800000u : __float_as_uint(a));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(out, m);
}

struct KernelInfo {
    bool done = false;
    int n_sm = 0, avail = 0;
};

template <bool GATEUP, int NT, bool BF, int MP, int NM>
static cudaError_t launch_one(DecodeArgs a, int n_items_max, cudaStream_t st) {
    static PerDevice<KernelInfo> kis;
    static PerDevice<bool> opt;
    auto kern = moe_decode_kernel<GATEUP, NT, BF, MP, NM>;
    int dev = 0;
    MOE_CUDA_TRY(current_device_slot(&dev));
    KernelInfo &ki = kis.v[dev];
    if (!ki.done) {
        MOE_CUDA_TRY(smem_optin_once(kern, opt));
        int optin = 0;
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&ki.n_sm, cudaDevAttrMultiProcessorCount, dev));
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
        cudaFuncAttributes fa;
        MOE_CUDA_TRY(cudaFuncGetAttributes(&fa, kern));
        ki.avail = optin - (int)fa.sharedSizeBytes;
        ki.done = true;
    }
    const DecGeom geo(a.Kdim, NM);
    int S = (int)((ki.avail - (long long)dec_red_bytes(NM, NT)) / geo.stage);
    if (S > kMaxStages) S = kMaxStages;
    if (S < 2) return cudaErrorInvalidValue;
    a.stages = S;
    int grid = ki.n_sm;
    if (grid > n_items_max) grid = n_items_max;
    if (grid < 1) grid = 1;
    const size_t smem = (size_t)S * geo.stage + dec_red_bytes(NM, NT);
    return launch_pdl(kern, dim3(grid), dim3(kDecThreads), smem, st, a);
}

// variant choice: bf16 activations, and the number of block pairs a warp covers
// (fewer pairs, fewer registers for the activations of 8-route tiles)
template <bool GATEUP, int NT, bool BF, int NM>
static cudaError_t launch_mp(const DecodeArgs &a, int n_items_max, cudaStream_t st) {
    const int ppw = ((a.Kdim / 32 + 1) / 2 + kCW - 1) / kCW;
    if (ppw <= 3) return launch_one<GATEUP, NT, BF, 3, NM>(a, n_items_max, st);
    if (ppw <= 4) return launch_one<GATEUP, NT, BF, 4, NM>(a, n_items_max, st);
    return launch_one<GATEUP, NT, BF, kMaxPairs, NM>(a, n_items_max, st);
}
template <bool GATEUP, int NT, int NM>
static cudaError_t launch_bf(const DecodeArgs &a, bool bf, int n_items_max, cudaStream_t st) {
    return bf ? launch_mp<GATEUP, NT, true, NM>(a, n_items_max, st)
              : launch_mp<GATEUP, NT, false, NM>(a, n_items_max, st);
}
// down items of 32 rows when H allows it and two such stages fit beside the partials
bool down_rows32(const BlockParams &bp) {
    return bp.H % 32 == 0 && 2 * (size_t)DecGeom(bp.F, 2).stage + dec_red_bytes(2, 2) + 1024 <= 227 * 1024;
}

}  // namespace

bool decode_supported(const BlockParams &bp) {
    // K range of the register-resident activations, and two ring stages next to the partials
    const int kmax = kCW * kMaxPairs * 64;
    if (bp.H > kmax || bp.F > kmax) return false;
    const size_t optin = 227 * 1024;
    return 2 * (size_t)DecGeom(bp.H, 2).stage + dec_red_bytes(2, 2) + 1024 <= optin &&
           2 * (size_t)DecGeom(bp.F, 1).stage + dec_red_bytes(1, 2) + 1024 <= optin;
}

cudaError_t launch_decode_stage(const BlockParams &bp, const Workspace &ws, const MatPtrs &a0, const MatPtrs &a1,
                                bool gateup, int T, int nt, bool x_bf16, bool h_bf16, int stall, bool slot_index,
                                cudaStream_t st) {
    const int R = T * (bp.K + bp.n_shared);
    // upper bound on the tile count: each expert's last tile may be partial
    int tiles = (R + 8 * nt - 1) / (8 * nt) + bp.E + bp.n_shared;
    if (tiles > ws.max_tiles) tiles = ws.max_tiles;
    if (gateup) {
        DecodeArgs gu{bp, ws, a0, a1, bp.H, bp.F, 0, h_bf16 ? 1 : 0, stall, slot_index ? 1 : 0};
        const int items = tiles * (bp.F / 16);
        return nt == 1 ? launch_bf<true, 1, 2>(gu, x_bf16, items, st) : launch_bf<true, 2, 2>(gu, x_bf16, items, st);
    }
    DecodeArgs dn{bp, ws, a0, a0, bp.F, bp.H, 0, 0, 0, slot_index ? 1 : 0};
    if (down_rows32(bp)) {
        const int items = tiles * (bp.H / 32);
        return nt == 1 ? launch_bf<false, 1, 2>(dn, h_bf16, items, st) : launch_bf<false, 2, 2>(dn, h_bf16, items, st);
    }
    const int items = tiles * (bp.H / 16);
    return nt == 1 ? launch_bf<false, 1, 1>(dn, h_bf16, items, st) : launch_bf<false, 2, 1>(dn, h_bf16, items, st);
}

cudaError_t launch_combine(const BlockParams &bp, const Workspace &ws, const uint16_t *x, int T, void *out,
                           int out_bf16, cudaStream_t st) {
    dim3 grid((bp.H / 4 + 255) / 256, T);
    return out_bf16 ? launch_pdl(moe_combine_kernel<true>, grid, dim3(256), 0, st, bp, ws, x, out, T)
                    : launch_pdl(moe_combine_kernel<false>, grid, dim3(256), 0, st, bp, ws, x, out, T);
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

cudaError_t launch_absmax(const float *v, int n, uint32_t *out, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    const int blocks = (n + 255) / 256 < 64 ? (n + 255) / 256 : 64;
    moe_absmax_kernel<<<blocks, 256, 0, st>>>(v, n, out);
    return cudaGetLastError();
}
