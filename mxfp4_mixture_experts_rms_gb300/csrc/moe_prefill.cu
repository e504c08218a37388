// moe_prefill.cu -- prefill path: grouped per-expert GEMMs on the 5th-gen
// tensor cores (tcgen05.mma kind::f16, bf16 operands in shared memory, fp32
// accumulators in TMEM), with MXFP4 weight tiles staged by TMA and
// dequantised to bf16 in shared memory.
//
// goosedump gpt_oss.rs `expert_batch_output` gathers the routed rows of one
// expert and runs `matrix_matrix_pair(gate, up)` + bias, `swiglu_inplace`,
// `matrix_matrix(down)` + bias and the route weight; `mix_expert_outputs`
// then sums each token's slots.  Here one CTA computes one (expert tile of
// <= 128 routes) x (weight row tile) block:
//
//   gate/up kernel: A = [64 gate rows ; the same 64 up rows] (M = 128),
//                   B = the tile's x_hat rows, D = TMEM [128 lanes][N];
//                   epilogue: bias + clamped SwiGLU -> h (bf16)
//   down kernel:    A = 128 rows of Wd, B = the tile's h rows;
//                   epilogue: bias, times the route weight -> per-route fp32
//
// Warp roles (320 threads): warp 0 issues the TMA loads of the packed codes
// and of the B tile (128-byte swizzled, straight into the MMA layout; the
// x_hat rows are first gathered into route order by moe_gather_kernel);
// warp 1 owns TMEM and issues the MMAs (one elected lane); warps 2..9
// dequantise A (two threads per row) and warps 2..5 run the epilogue.  A 4-stage mbarrier ring connects them.
// Activations use a 32-block pair order (x_hat_mma / h), and A is written in
// that order straight from the nibble-pair dequantiser, so the K permutation
// cancels in every dot product.
//
// Every wait is bounded (about 2 s of %globaltimer); on a timeout the kernel
// records MOE_DEV_WAIT_TIMEOUT in the status word, drains what it issued,
// frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "moe_common.cuh"

namespace {

constexpr int kStages = 4;
constexpr int kBK = 64;            // K elements per stage (one 128-byte swizzle row of bf16)
constexpr int kBN = 128;           // max routes per tile
constexpr int kDqWarps = 8;                   // dequantising warps (2 threads per A row)
constexpr int kThreads = 64 + 32 * kDqWarps;
constexpr int kABytes = 128 * 128;     // A stage: 128 rows x 128 B
constexpr int kBBytes = kBN * 128;     // B stage
constexpr int kFp4Bytes = 128 * 32;    // packed codes of one stage
constexpr uint64_t kWaitNs = 2000000000ull;

struct PrefillArgs {
    BlockParams bp;
    Workspace ws;
    MatPtrs A0, A1;     // gate, up (GATEUP) or down
    int Kdim;           // H (gate/up) or F (down)
    int rows;           // F (gate/up) or H (down)
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(smem_u32(b)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: false (and the status word set) after ~2 s or when another
// thread of the grid already reported a failure.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, int32_t *status, int where) {
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 0;; i++) {
        if (mbar_try(b, parity)) return true;
        if ((i & 63) == 63) {
            if (*(volatile int32_t *)status != 0) return false;
            if (globaltimer() - t0 > kWaitNs) {
                set_device_error(status, MOE_DEV_WAIT_TIMEOUT, where);
                return false;
            }
        }
    }
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// UMMA shared-memory descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;              // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset
    d |= (uint64_t)1 << 46;              // descriptor version
    d |= (uint64_t)2 << 61;              // SWIZZLE_128B
    return d;
}
// Instruction descriptor, kind::f16: D f32, A/B bf16, both K-major, M x N.
__host__ __device__ __forceinline__ uint32_t umma_idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(dtmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float v[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------- dequantisation
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}
// 8 nibbles -> 4 bf16x2 in pair order (nibble i, nibble i+4), value*2^(s-127).
__device__ __forceinline__ uint4 dequant8(uint32_t w, uint32_t s1, uint32_t s2, bool big) {
    uint32_t p0 = ((w << 6) & 0x01C001C0u) | ((w << 12) & 0x80008000u);
    uint32_t p1 = ((w << 2) & 0x01C001C0u) | ((w << 8) & 0x80008000u);
    uint32_t p2 = ((w >> 2) & 0x01C001C0u) | ((w << 4) & 0x80008000u);
    uint32_t p3 = ((w >> 6) & 0x01C001C0u) | (w & 0x80008000u);
    p0 = bmul2(p0, s1);
    p1 = bmul2(p1, s1);
    p2 = bmul2(p2, s1);
    p3 = bmul2(p3, s1);
    if (big) {
        p0 = bmul2(p0, s2);
        p1 = bmul2(p1, s2);
        p2 = bmul2(p2, s2);
        p3 = bmul2(p3, s2);
    }
    return make_uint4(p0, p1, p2, p3);
}
__device__ __forceinline__ uint32_t scale_lo(uint32_t s) {
    uint32_t b = (s <= 128u) ? ((s + 126u) << 7) : (253u << 7);
    return b | (b << 16);
}
__device__ __forceinline__ uint32_t scale_hi(uint32_t s) {
    uint32_t b = (s <= 128u) ? 0x3F80u : (s << 7);
    return b | (b << 16);
}
// byte offset of 16-byte chunk c of row r in a 128B-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

template <bool GATEUP>
__global__ void __launch_bounds__(kThreads, 1) moe_prefill_kernel(const __grid_constant__ PrefillArgs a,
                                                                    const __grid_constant__ TmaMaps maps,
                                                                    const __grid_constant__ CUtensorMap bmap) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = smem;                                   // [kStages][128 rows][128 B] swizzled
    unsigned char *sB = sA + kStages * kABytes;                 // [kStages][kBN rows][128 B] swizzled
    unsigned char *sF = sB + kStages * kBBytes;                 // [kStages][128 rows][32 B] packed codes
    uint64_t *bars = reinterpret_cast<uint64_t *>(sF + kStages * kFp4Bytes);
    uint64_t *full_fp4 = bars, *full_ab = bars + kStages, *empty = bars + 2 * kStages, *full_b = bars + 3 * kStages;
    uint64_t *acc_full = bars + 4 * kStages, *drain = acc_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);

    const int tile_idx = blockIdx.x;
    if (tile_idx >= *a.ws.n_tiles) return;
    const int4 tile = a.ws.tiles[tile_idx];
    const int e = tile.x, rstart = tile.y, rcount = tile.z;
    const int E = a.bp.E, K = a.Kdim, nb = K / 32, nkb = K / kBK;
    const int mt = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_mma = max(16, (rcount + 15) & ~15);
    int32_t *status = a.ws.status;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&full_fp4[s], 1);
            mbar_init(&full_ab[s], kDqWarps);
            mbar_init(&full_b[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;" ::"r"(smem_u32(tmem_slot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (codes)
        if (lane == 0) {
            const bool shared_e = e >= E;
            const CUtensorMap *m0 = shared_e ? &maps.m[2] : &maps.m[0];
            const CUtensorMap *m1 = shared_e ? &maps.m[3] : &maps.m[1];
            const int ebase = shared_e ? 0 : e;
            int issued_upto = 0;
            bool ok = true;
            for (int kb = 0; kb < nkb && ok; kb++) {
                const int s = kb % kStages;
                if (kb >= kStages) ok = mbar_wait(&empty[s], ((kb / kStages) - 1) & 1, status, 10);
                if (!ok) break;
                // B: the tile's 128 activation rows (rows past the tile belong to other
                // tiles or lie outside the tensor, read as zeros: their columns are ignored)
                // (in boxes of 32 rows, as many as the tile's routes need: the MMA
                // reads only the first n_mma rows)
                const int nbox = (rcount + 31) / 32;
                mbar_expect_tx(&full_b[s], (uint32_t)nbox * 32 * 128);
                for (int bx = 0; bx < nbox; bx++)
                    tma_load_2d(sB + s * kBBytes + bx * 32 * 128, &bmap, &full_b[s], kb * kBK, rstart + 32 * bx);
                mbar_expect_tx(&full_fp4[s], kFp4Bytes);
                unsigned char *dst = sF + s * kFp4Bytes;
                if (GATEUP) {
                    const int y = ebase * a.rows + mt * 64;
                    tma_load_2d(dst, m0, &full_fp4[s], kb * 32, y);
                    tma_load_2d(dst + 64 * 32, m1, &full_fp4[s], kb * 32, y);
                } else {
                    tma_load_2d(dst, m0, &full_fp4[s], kb * 32, ebase * a.rows + mt * 128);
                }
                issued_upto = kb + 1;
            }
            // make sure every copy this thread issued has landed before exiting
            for (int kb = max(0, issued_upto - kStages); kb < issued_upto; kb++) {
                mbar_wait(&full_fp4[kb % kStages], (kb / kStages) & 1, status, 11);
                mbar_wait(&full_b[kb % kStages], (kb / kStages) & 1, status, 12);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16(128, n_mma);
            int done = 0;
            bool ok = true;
            for (int kb = 0; kb < nkb; kb++) {
                const int s = kb % kStages;
                ok = mbar_wait(&full_ab[s], (kb / kStages) & 1, status, 20) &&
                     mbar_wait(&full_b[s], (kb / kStages) & 1, status, 22);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a_addr = smem_u32(sA + s * kABytes), b_addr = smem_u32(sB + s * kBBytes);
#pragma unroll
                for (int k = 0; k < kBK / 16; k++) {
                    umma_bf16(tmem, umma_desc_sw128(a_addr + 32 * k), umma_desc_sw128(b_addr + 32 * k), idesc,
                              (kb | k) != 0);
                }
                umma_commit(&empty[s]);
                done = kb + 1;
            }
            if (ok && done == nkb) {
                umma_commit(acc_full);
            } else {
                // drain the MMAs already issued before TMEM is released
                umma_commit(drain);
                mbar_wait(drain, 0, status, 21);
            }
        }
    } else {
        // ----------------------------------------------- dequant (warps 2..9)
        const int t = threadIdx.x - 64;  // 0..255
        const int arow = t >> 1, half = t & 1;  // A row and which 32-element block of the stage
        const MatPtrs &M = (GATEUP && arow >= 64) ? a.A1 : a.A0;
        int wrow;                        // weight row of A row arow (may be >= rows for the last down tile)
        if (GATEUP)
            wrow = mt * 64 + (arow & 63);
        else
            wrow = mt * 128 + arow;
        const bool row_ok = wrow < a.rows;
        const uint8_t *srow = mat_scales(M, e, E) + (size_t)(row_ok ? wrow : 0) * nb + half;
        // this thread's scale byte per k-block, loaded four k-blocks ahead
        auto ldsc = [&](int k) -> uint32_t { return (k < nkb && row_ok) ? (uint32_t)__ldg(srow + 2 * k) : 127u; };
        uint32_t q0 = ldsc(0), q1 = ldsc(1), q2 = ldsc(2), q3 = ldsc(3);
        bool ok = true;
        for (int kb = 0; kb < nkb; kb++) {
            const int s = kb % kStages;
            if (kb >= kStages) {
                ok = mbar_wait(&empty[s], ((kb / kStages) - 1) & 1, status, 30);
                if (!ok) break;
            }
            const uint32_t sc = q0;
            q0 = q1;
            q1 = q2;
            q2 = q3;
            q3 = ldsc(kb + 4);
            // A: wait for the packed codes, dequantise half a row
            ok = mbar_wait(&full_fp4[s], (kb / kStages) & 1, status, 31);
            if (!ok) break;
            const uint4 c = *reinterpret_cast<const uint4 *>(sF + s * kFp4Bytes + arow * 32 + half * 16);
            const bool big = sc > 128u;
            const uint32_t l = scale_lo(sc), h = scale_hi(sc);
            unsigned char *adst = sA + s * kABytes;
            *reinterpret_cast<uint4 *>(adst + sw128(arow, half * 4 + 0)) = dequant8(c.x, l, h, big);
            *reinterpret_cast<uint4 *>(adst + sw128(arow, half * 4 + 1)) = dequant8(c.y, l, h, big);
            *reinterpret_cast<uint4 *>(adst + sw128(arow, half * 4 + 2)) = dequant8(c.z, l, h, big);
            *reinterpret_cast<uint4 *>(adst + sw128(arow, half * 4 + 3)) = dequant8(c.w, l, h, big);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full_ab[s]);
        }
        if (warp < 6) {
        // ------------------------------------------------------------ epilogue
        if (ok) ok = mbar_wait(acc_full, 0, status, 40);
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld below is warp-collective
        tc_fence_after();
        const int q = warp & 3;                  // TMEM lane quarter of this warp
        const int lrow = q * 32 + lane;          // accumulator row (= A row)
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
        float *xch = reinterpret_cast<float *>(sA);  // [64][33] exchange buffer (stages are idle now)
        for (int c0 = 0; c0 < n_mma; c0 += 32) {
            float v[32];
            if (ok) tmem_ld32(taddr + c0, v);
            if (GATEUP) {
                if (q >= 2) {
#pragma unroll
                    for (int c = 0; c < 32; c++) xch[(lrow - 64) * 33 + c] = v[c];
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (q < 2 && ok) {
                    const int j = mt * 64 + lrow;
                    const float bg = mat_bias(a.A0, e, E)[j], bu = mat_bias(a.A1, e, E)[j];
                    const int pj = mma_perm_pos(j);
#pragma unroll
                    for (int c = 0; c < 32; c++) {
                        if (c0 + c >= rcount) continue;
                        const float hv = swiglu_clamped(v[c] + bg, xch[lrow * 33 + c] + bu, a.bp.alpha, a.bp.limit);
                        __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                        a.ws.h[(size_t)(rstart + c0 + c) * a.bp.F + pj] = *reinterpret_cast<uint16_t *>(&hb);
                    }
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
            } else if (ok) {
                const int i = mt * 128 + lrow;
                if (i < a.rows) {
                    const float bd = mat_bias(a.A0, e, E)[i];
#pragma unroll
                    for (int c = 0; c < 32; c++) {
                        if (c0 + c >= rcount) continue;
                        const int route = rstart + c0 + c;
                        a.ws.y[(size_t)route * a.bp.H + i] = a.ws.perm_w[route] * (v[c] + bd);
                    }
                }
            }
        }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;" ::"r"(tmem));
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder() {
    if (g_encode) return cudaSuccess;
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

// 2D map over packed codes: [n_rows][cols/2] bytes, box 32 bytes x box_rows.
cudaError_t make_codes_map(CUtensorMap *m, const uint8_t *codes, size_t n_rows, int cols, int box_rows) {
    if (!codes) {
        memset(m, 0, sizeof *m);
        return cudaSuccess;
    }
    cuuint64_t dims[2] = {(cuuint64_t)(cols / 2), (cuuint64_t)n_rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols / 2)};
    cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

size_t prefill_smem_bytes() { return 1024 + kStages * (kABytes + kBBytes + kFp4Bytes) + 256; }

// 2D map over a bf16 activation matrix [rows][K]: box 64 elements (128 B) x 32
// rows, 128-byte swizzle (the K-major layout the MMA descriptors expect; a
// 32-row box is four whole 8-row swizzle atoms).
cudaError_t make_act_map(CUtensorMap *m, const uint16_t *base, int rows, int K) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// xs[pos] = x_hat_mma[perm_token[pos]] (16-byte chunks), pos < R.
__global__ void __launch_bounds__(256) moe_gather_kernel(Workspace ws, int H, int R) {
    const int cpr = H / 8;  // 16-byte chunks per row
    const size_t n = (size_t)R * cpr;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int pos = (int)(i / cpr), c = (int)(i - (size_t)pos * cpr);
        const int tok = ws.perm_token[pos];
        reinterpret_cast<uint4 *>(ws.xs + (size_t)pos * H)[c] =
            reinterpret_cast<const uint4 *>(ws.xhat_mma + (size_t)tok * H)[c];
    }
}

}  // namespace

int prefill_tile_rows() { return kBN; }

cudaError_t prefill_make_maps(const BlockParams &bp, const MatPtrs &gate, const MatPtrs &up, const MatPtrs &down,
                              PrefillMaps *out) {
    MOE_CUDA_TRY(get_encoder());
    const int E = bp.E;
    TmaMaps &g = out->gateup, &d = out->down;
    MOE_CUDA_TRY(make_codes_map(&g.m[0], gate.codes, (size_t)E * gate.rows, gate.cols, 64));
    MOE_CUDA_TRY(make_codes_map(&g.m[1], up.codes, (size_t)E * up.rows, up.cols, 64));
    MOE_CUDA_TRY(make_codes_map(&g.m[2], bp.n_shared ? gate.sh_codes : nullptr, gate.rows, gate.cols, 64));
    MOE_CUDA_TRY(make_codes_map(&g.m[3], bp.n_shared ? up.sh_codes : nullptr, up.rows, up.cols, 64));
    MOE_CUDA_TRY(make_codes_map(&d.m[0], down.codes, (size_t)E * down.rows, down.cols, 128));
    d.m[1] = d.m[0];
    MOE_CUDA_TRY(make_codes_map(&d.m[2], bp.n_shared ? down.sh_codes : nullptr, down.rows, down.cols, 128));
    d.m[3] = d.m[2];
    return cudaSuccess;
}

cudaError_t launch_gather(const BlockParams &bp, const Workspace &ws, int T, cudaStream_t st) {
    const int R = T * (bp.K + bp.n_shared);
    const size_t n = (size_t)R * (bp.H / 8);
    const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    moe_gather_kernel<<<blocks, 256, 0, st>>>(ws, bp.H, R);
    return cudaGetLastError();
}

cudaError_t launch_prefill_stage(const BlockParams &bp, const Workspace &ws, const MatPtrs &a0, const MatPtrs &a1,
                                 bool gateup, int T, const TmaMaps &maps, cudaStream_t st) {
    PrefillArgs args{bp, ws, a0, a1, gateup ? bp.H : bp.F, gateup ? bp.F : bp.H};
    const int R = T * (bp.K + bp.n_shared);
    CUtensorMap bmap;
    MOE_CUDA_TRY(get_encoder());
    MOE_CUDA_TRY(make_act_map(&bmap, gateup ? ws.xs : ws.h, R, args.Kdim));
    int tiles = (R + kBN - 1) / kBN + bp.E + bp.n_shared;
    if (tiles > ws.max_tiles) tiles = ws.max_tiles;
    const int mtiles = gateup ? bp.F / 64 : (bp.H + 127) / 128;
    const size_t sm = prefill_smem_bytes();
    static bool done_gu = false, done_dn = false;
    if (gateup) {
        MOE_CUDA_TRY(smem_optin_once(moe_prefill_kernel<true>, done_gu));
        moe_prefill_kernel<true><<<dim3(tiles, mtiles), kThreads, sm, st>>>(args, maps, bmap);
    } else {
        MOE_CUDA_TRY(smem_optin_once(moe_prefill_kernel<false>, done_dn));
        moe_prefill_kernel<false><<<dim3(tiles, mtiles), kThreads, sm, st>>>(args, maps, bmap);
    }
    return cudaGetLastError();
}
