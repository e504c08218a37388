// moe_prefill.cu -- prefill path: grouped per-expert GEMMs on the 5th-gen
// tensor cores (tcgen05.mma kind::f16, fp32 accumulators in TMEM), with MXFP4
// weight tiles staged by TMA and dequantised by the SM into TMEM.
//
// goosedump gpt_oss.rs `expert_batch_output` gathers the routed rows of one
// expert and runs `matrix_matrix_pair(gate, up)` + bias, `swiglu_inplace`,
// `matrix_matrix(down)` + bias and the route weight; `mix_expert_outputs`
// then sums each token's slots.  Here a work item is one (expert tile of
// <= 128 routes) x (weight row block) block:
//
//   gate/up kernel: A = the tile's x_hat rows (M = 128 routes), B = [128 gate
//                   rows ; the same 128 up rows] (N = 256), D = TMEM
//                   [128 lanes = routes][256 columns];
//                   epilogue: bias + clamped SwiGLU -> h
//   down kernel:    A = the tile's h rows, B = 256 rows of Wd;
//                   epilogue: bias, times the route weight -> per-route fp32
//
// The kernel is persistent (one CTA per SM walking a static list of items)
// with warp roles: a TMA warp for the packed codes and their scales, a TMA
// warp for the activation tile, A (128-byte swizzled, straight into the MMA layout; the
// x_hat rows are first gathered into route order by moe_gather_kernel), an
// MMA warp that owns all 512 TMEM columns, eight dequantising warps that
// write B into 128-byte-swizzled shared memory, and four epilogue warps that
// drain one of two TMEM accumulators while the MMA fills the other.  mbarrier
// rings connect them.  The bf16 variant keeps activations in a 32-block pair
// order (x_hat_mma / h) and produces B in that order straight from the
// nibble-pair dequantiser, so the K permutation cancels in every dot product.
//
// Every wait is bounded (about 2 s of %globaltimer); on a timeout the kernel
// records MOE_DEV_WAIT_TIMEOUT in the status word, drains what it issued,
// frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "moe_common.cuh"

// Timeline markers (no-ops unless an instrumented build defines them).
#ifndef MOE_PF_MARK
#define MOE_PF_MARK(slot)
#endif
#ifndef MOE_PF_KMARK
#define MOE_PF_KMARK(kind, kb)
#endif

namespace {

constexpr int kStages = 3;          // A (activations, by TMA) + B (dequantised weights) stages, consumed by the MMA
constexpr int kCK = 2;              // k-blocks per packed-code stage
constexpr int kCStages = 4;         // packed-code stages (8 k-blocks ahead)
constexpr int kBK = 64;             // K elements per stage (one 128-byte swizzle row of 16-bit values)
constexpr int kTM = 128;            // routes per tile (the MMA's M)
constexpr int kWN = 256;            // weight rows per item (the MMA's N): 128 gate + 128 up rows, or 256 down rows
constexpr int kWarpCodes = 0, kWarpMma = 1, kWarpA = 2, kWarpDq0 = 3;
constexpr int kDqWarps = 8;                   // dequantising warps
constexpr int kDqGroups = 2;                  // k-blocks are dealt round-robin to this many warp groups
constexpr int kDqGroupWarps = kDqWarps / kDqGroups;
constexpr int kWarpEpi0 = kWarpDq0 + kDqWarps, kEpiWarps = 4;
constexpr int kThreads = 32 * (kWarpEpi0 + kEpiWarps);
constexpr int kAccCols = kWN;                 // one fp32 accumulator: 128 lanes (routes) x 256 columns (rows)
constexpr int kTmemCols = 2 * kAccCols;       // two accumulators (MMA fills one, the epilogue drains the other)
static_assert(kTmemCols == 512, "TMEM budget");
constexpr int kSmTiles = 256;                 // route tiles cached in shared memory
constexpr int kBiasFloats = kWN;              // an epilogue warp's copy of the item's 256 biases
constexpr int kABytes = kTM * 128;            // A stage: 128 route rows x 128 B
constexpr int kBBytes = kWN * 128;            // B stage: 256 weight rows x 128 B
constexpr int kFp4Bytes = kWN * 32 * kCK;     // packed codes of one code stage: 256 rows x 64 B, 64-byte swizzle
constexpr int kScBytes = (kWN / 64) * 128 * kCK;  // its scale bytes: per 64-row block, kCK chunks of 128 B
constexpr int kCStageBytes = kFp4Bytes + kScBytes;  // a multiple of 512 B (the 64-byte swizzle period)
constexpr uint64_t kWaitNs = 2000000000ull;

// TMA descriptors of the activation operand (A) with boxes of 32, 64 and 128
// rows: one copy per k-block, the smallest box that covers the tile's routes
// (the MMA reads all 128 rows; rows past the box are stale and only feed
// accumulator lanes the epilogue skips).
struct AMaps {
    CUtensorMap m[3];
};

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
__device__ __forceinline__ void mbar_arrive_n(uint64_t *b, uint32_t n) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0], %1; }" ::"r"(smem_u32(b)), "r"(n)
                 : "memory");
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
// Wait that ignores the status word (only the time limit ends it): used to let
// copies or MMAs already issued land before the CTA's shared memory or TMEM goes.
__device__ __forceinline__ void mbar_wait_drain(uint64_t *b, uint32_t parity, int32_t *status) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try(b, parity))
        if (globaltimer() - t0 > kWaitNs) {
            set_device_error(status, MOE_DEV_WAIT_TIMEOUT, 90);
            return;
        }
}
// The last min(issued, n) copies of an n-stage ring have landed (one ~2 s
// limit for all of them: a full barrier that also counts other arrivals may
// never complete once the kernel is failing).
__device__ __forceinline__ void drain_ring(uint64_t *full, int n, int issued, int32_t *status) {
    const uint64_t t0 = globaltimer();
    for (int g = max(0, issued - n); g < issued; g++)
        while (!mbar_try(&full[g % n], (g / n) & 1))
            if (globaltimer() - t0 > kWaitNs) {
                set_device_error(status, MOE_DEV_WAIT_TIMEOUT, 91);
                return;
            }
}
// Stage index and phase bit of a ring walked in order.  Consumers wait on a
// full barrier with parity ph; producers wait on an empty barrier with parity
// ph ^ 1, which a fresh barrier already satisfies (every stage starts free).
struct Ring {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next(int n) {
        if (++s == n) {
            s = 0;
            ph ^= 1;
        }
    }
};

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// The same for the weight stream, with an L2 evict-first policy (each weight
// byte is read once per forward: its lines go first, the activation tiles
// that every weight-row block re-reads stay).
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_2d_ef(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y,
                                               uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void bulk_load_ef(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
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
// Instruction descriptor, kind::f16: D f32, A/B both bf16 (bf = true) or both
// f16, both K-major, M x N.
__host__ __device__ __forceinline__ uint32_t umma_idesc(int M, int N, bool bf) {
    const uint32_t ab = bf ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D (TMEM, fp32) (+)= A x B, both from shared memory (K-major, 128-byte swizzle)
__device__ __forceinline__ void umma_ss(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(dtmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
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
__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}
// fp16 2^(s-127) in both halves for s in [104, 140] (subnormal below 113): the
// product with an E2M1 value is then exact in fp16
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t s) {
    const uint32_t b = (s >= 113u) ? ((s - 112u) << 10) : (1u << (s - 103u));
    return b | (b << 16);
}
// 8 codes -> 8 fp16 values, natural order, times 2^(s-127) (fp16 variant)
__device__ __forceinline__ uint4 dequant8_f16(uint32_t w, uint32_t sc2) {
    uint32_t h[4];
    e2m1x8_to_f16(w, h);
    return make_uint4(hmul2_f16(h[0], sc2), hmul2_f16(h[1], sc2), hmul2_f16(h[2], sc2), hmul2_f16(h[3], sc2));
}

// Clamped SwiGLU with the hardware exponential and a fast divide: within a few
// fp32 ulps of the correctly rounded form, far inside the bf16 rounding of h.
// For α·g below about -87 the divide returns 0 where the exact value is a
// normal below 1e-36 in magnitude.
__device__ __forceinline__ float swiglu_fast(float g, float u, float alpha, float limit) {
    const float gc = (g > limit) ? limit : g;
    const float uc = (u > limit) ? limit : ((u < -limit) ? -limit : u);
    return __fdividef(gc, 1.0f + __expf(-alpha * gc)) * (uc + 1.0f);
}

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Persistent grouped GEMM.  A launch covers n_tiles x mtiles work items, item
// i = (route tile i / mtiles, weight-row block i % mtiles); CTA b takes items
// b, b + gridDim.x, ...  Every role walks that same sequence with its own ring
// counters, so the producers run ahead into the next item while the epilogue
// drains the previous one from the other of two TMEM accumulators.
//
// Operands: A = the tile's activation rows (M = 128 routes, by TMA), B = 256
// dequantised weight rows (N = 256): a tcgen05.mma of M = 128, K = 16 costs
// the same issue slot whatever N is, so N is the weight dimension, always 256,
// and the routes (often fewer than 128 per expert) take M.  D = TMEM [128
// lanes = routes][256 columns = weight rows]; for gate/up the 256 rows are 128
// gate rows then the same 128 up rows, so one thread holds both halves of its
// route's SwiGLU inputs.
//
// Warps: 0 TMA for the packed codes and their scales, 1 MMA issue (and TMEM
// owner), 2 TMA for the activation tile, 3..10 dequantisation into the
// 128-byte-swizzled B stage (two groups of four warps, k-blocks dealt
// round-robin, two weight rows per thread), 11..14 epilogue (one TMEM lane
// quarter each).  Each producer has a warp of its own: a lane blocked in
// mbarrier.try_wait holds up every other lane of its warp.
//
// F16: the fp16 variant (every E8M0 exponent in [104, 140], activations in the
// fp16 range): hardware e2m1 -> f16 conversion, natural K order, fp16 MMA
// operands (x_hat16 / h16); otherwise the bf16 variant (any exponent,
// nibble-pair order, bf16 operands x_hat_mma / h).
template <bool GATEUP, bool F16>
__global__ void __launch_bounds__(kThreads, 1) moe_prefill_kernel(const __grid_constant__ PrefillArgs a,
                                                                    const __grid_constant__ TmaMaps maps,
                                                                    const __grid_constant__ AMaps amaps) {
    constexpr int RPI = GATEUP ? kWN / 2 : kWN;  // output rows per item
    const int mtiles = (a.rows + RPI - 1) / RPI;
    const int n_tiles = *a.ws.n_tiles;
    const int n_items = n_tiles * mtiles;
    if ((int)blockIdx.x >= n_items) return;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = smem;                                   // [kStages][128 route rows][128 B] swizzled
    unsigned char *sB = sA + kStages * kABytes;                 // [kStages][256 weight rows][128 B] swizzled
    unsigned char *sF = sB + kStages * kBBytes;                 // [kCStages][codes 256 x 64 B, scales 4 x 256 B]
    int4 *s_tiles = reinterpret_cast<int4 *>(sF + kCStages * kCStageBytes);  // [kSmTiles]
    float *s_bias = reinterpret_cast<float *>(s_tiles + kSmTiles);           // [kEpiWarps][kBiasFloats]
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_bias + kEpiWarps * kBiasFloats);
    uint64_t *full_c = bars, *empty_c = bars + kCStages;    // code ring
    uint64_t *full_ab = empty_c + kCStages;                  // A/B ring: A by TMA, B from the dequantisers
    uint64_t *empty = full_ab + kStages;
    uint64_t *acc_full = empty + kStages, *acc_empty = acc_full + 2, *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);

    MOE_PF_MARK(0);
    const int E = a.bp.E, K = a.Kdim, nkb = K / kBK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *status = a.ws.status;

    for (int i = threadIdx.x; i < min(n_tiles, kSmTiles); i += blockDim.x) s_tiles[i] = a.ws.tiles[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < kCStages; s++) {
            mbar_init(&full_c[s], 1);
            mbar_init(&empty_c[s], kCK * kDqGroupWarps);
        }
        for (int s = 0; s < kStages; s++) {
            mbar_init(&full_ab[s], kDqGroupWarps + 1);  // + the A copy's expect_tx arrival
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kEpiWarps);
        }
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "n"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto tile_at = [&](int t) -> int4 { return t < kSmTiles ? s_tiles[t] : a.ws.tiles[t]; };

    if (warp == kWarpCodes) {
        // ------------------------------------------- packed codes + scales (TMA)
        if (lane == 0) {
            const uint64_t pol = l2_evict_first();
            Ring r;
            int issued = 0, g = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const int tile = it / mtiles, mt = it - tile * mtiles;
                const int e = tile_at(tile).x;
                const bool shared_e = e >= E;
                const CUtensorMap *m0 = shared_e ? &maps.m[2] : &maps.m[0];
                const CUtensorMap *m1 = shared_e ? &maps.m[3] : &maps.m[1];
                const int ebase = shared_e ? 0 : e;
                // the item's four 64-row scale blocks, kCK chunks per code stage
                const size_t cb = (size_t)nkb * 128;
                const uint8_t *scp[4];
                if (GATEUP) {
                    const uint8_t *g0 = maps.sc[shared_e ? 2 : 0] + (size_t)(ebase * maps.row_blocks + 2 * mt) * cb;
                    const uint8_t *u0 = maps.sc[shared_e ? 3 : 1] + (size_t)(ebase * maps.row_blocks + 2 * mt) * cb;
                    scp[0] = g0;
                    scp[1] = g0 + cb;
                    scp[2] = u0;
                    scp[3] = u0 + cb;
                } else {
                    const uint8_t *d0 = maps.sc[shared_e ? 2 : 0] + (size_t)(ebase * maps.row_blocks + 4 * mt) * cb;
                    for (int j = 0; j < 4; j++) scp[j] = d0 + j * cb;
                }
                // past the end of K (or of the matrix) the boxes read zeros; the scale
                // chunks there belong to the next block or the pad, and are never used
                for (int kb = 0; kb < nkb; kb += kCK, g++) {
                    if (!mbar_wait(&empty_c[r.s], r.ph ^ 1, status, 10)) {
                        ok = false;
                        break;
                    }
                    MOE_PF_KMARK(5, g);
                    mbar_expect_tx(&full_c[r.s], kCStageBytes);
                    unsigned char *dst = sF + r.s * kCStageBytes;
                    if (GATEUP) {
                        const int y = ebase * a.rows + mt * RPI;
                        tma_load_2d_ef(dst, m0, &full_c[r.s], kb * 32, y, pol);
                        tma_load_2d_ef(dst + kFp4Bytes / 2, m1, &full_c[r.s], kb * 32, y, pol);
                    } else {
                        tma_load_2d_ef(dst, m0, &full_c[r.s], kb * 32, ebase * a.rows + mt * RPI, pol);
                    }
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        bulk_load_ef(dst + kFp4Bytes + j * 128 * kCK, scp[j] + (size_t)kb * 128, 128 * kCK, &full_c[r.s],
                                     pol);
                    issued++;
                    r.next(kCStages);
                }
            }
            drain_ring(full_c, kCStages, issued, status);
        }
    } else if (warp == kWarpA) {
        // ------------------------------------- activation tile (TMA, A operand)
        if (lane == 0) {
            Ring r;
            int issued = 0, g = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const int4 tl = tile_at(it / mtiles);
                const int rstart = tl.y, mi = tl.z <= 32 ? 0 : (tl.z <= 64 ? 1 : 2);
                const CUtensorMap *am = &amaps.m[mi];
                const uint32_t abytes = (uint32_t)(32 << mi) * 128;
                for (int kb = 0; kb < nkb; kb++, g++) {
                    if (!mbar_wait(&empty[r.s], r.ph ^ 1, status, 13)) {
                        ok = false;
                        break;
                    }
                    MOE_PF_KMARK(4, g);
                    mbar_expect_tx(&full_ab[r.s], abytes);
                    tma_load_2d(sA + r.s * kABytes, am, &full_ab[r.s], kb * kBK, rstart);
                    issued++;
                    r.next(kStages);
                }
            }
            drain_ring(full_ab, kStages, issued, status);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = umma_idesc(kTM, kWN, !F16);
            Ring r;
            bool ok = true;
            int li = 0, g = 0;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, li++) {
                const int ab = li & 1;
                // the epilogue has read this accumulator out (free on its first use)
                ok = mbar_wait(&acc_empty[ab], ((li >> 1) & 1) ^ 1, status, 23);
                if (!ok) break;
                tc_fence_after();
                const uint32_t dt = tmem + (uint32_t)(ab * kAccCols);
                for (int kb = 0; kb < nkb; kb++, g++) {
                    ok = mbar_wait(&full_ab[r.s], r.ph, status, 20);
                    MOE_PF_KMARK(0, g);
                    if (!ok) break;
                    tc_fence_after();
                    MOE_PF_KMARK(3, g);
                    const uint32_t a_addr = smem_u32(sA + r.s * kABytes), b_addr = smem_u32(sB + r.s * kBBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; k++)
                        umma_ss(dt, umma_desc_sw128(a_addr + 32 * k), umma_desc_sw128(b_addr + 32 * k), idesc,
                                (kb | k) != 0);
                    umma_commit(&empty[r.s]);
                    MOE_PF_KMARK(1, g);
                    r.next(kStages);
                }
                if (ok) umma_commit(&acc_full[ab]);
            }
            if (!ok) {
                // the MMAs already issued finish before TMEM is released
                umma_commit(drain);
                mbar_wait_drain(drain, 0, status);
            }
        }
    } else if (warp < kWarpEpi0) {
        // ------------------------------------------ dequant (warps 3..10)
        // Two groups of four warps; group grp dequantises k-blocks g = grp,
        // grp + 2, ... of the CTA's sequence into the whole 256 x 64 B stage:
        // thread t of the group handles weight rows t and t + 128.
        const int grp = (warp - kWarpDq0) / kDqGroupWarps;
        const int t = threadIdx.x - 32 * (kWarpDq0 + grp * kDqGroupWarps);  // 0..127
        const int my_items = (n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
        const int total = my_items * nkb, ncs = (nkb + kCK - 1) / kCK;
        for (int g = grp; g < total; g += kDqGroups) {
            const int li = g / nkb, kb = g - li * nkb;
            const int qq = li * ncs + kb / kCK;  // this CTA's code stage holding k-block kb
            const int s = g % kStages, cs = qq % kCStages, kh = kb % kCK;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&empty[s], ((g / kStages) & 1) ^ 1, status, 30) &&
                                                        mbar_wait(&full_c[cs], (qq / kCStages) & 1, status, 31));
            if (!ok) break;
            if (warp == kWarpDq0 && lane == 0) MOE_PF_KMARK(2, g);
            const unsigned char *cst = sF + cs * kCStageBytes;
            unsigned char *bdst = sB + s * kBBytes;
#pragma unroll
            for (int rr = 0; rr < 2; rr++) {
                const int row = t + 128 * rr;
                const int swz = (row >> 1) & 3;  // the code box's 64-byte swizzle for this row
                const uint4 c0 = *reinterpret_cast<const uint4 *>(cst + row * 64 + (((2 * kh) ^ swz) << 4));
                const uint4 c1 = *reinterpret_cast<const uint4 *>(cst + row * 64 + (((2 * kh + 1) ^ swz) << 4));
                const uint32_t sc2 = *reinterpret_cast<const uint16_t *>(cst + kFp4Bytes + (row >> 6) * 128 * kCK +
                                                                          kh * 128 + (row & 63) * 2);
                const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                for (int hf = 0; hf < 2; hf++) {
                    const uint32_t sc = (sc2 >> (8 * hf)) & 0xFFu;
                    if (F16) {
                        const uint32_t sx = scale_f16x2(sc);
#pragma unroll
                        for (int j = 0; j < 4; j++)
                            *reinterpret_cast<uint4 *>(bdst + sw128(row, 4 * hf + j)) = dequant8_f16(w[4 * hf + j], sx);
                    } else {
                        const bool big = sc > 128u;
                        const uint32_t l = scale_lo(sc), h = scale_hi(sc);
#pragma unroll
                        for (int j = 0; j < 4; j++)
                            *reinterpret_cast<uint4 *>(bdst + sw128(row, 4 * hf + j)) = dequant8(w[4 * hf + j], l, h, big);
                    }
                }
            }
            if (warp == kWarpDq0 && lane == 0) MOE_PF_KMARK(9, g);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&full_ab[s]);
                // the last stage of an item may hold fewer than kCK k-blocks: arrive for the missing ones too
                mbar_arrive_n(&empty_c[cs], kb + 1 == nkb ? (uint32_t)(kCK - kh) : 1u);
            }
            if (warp == kWarpDq0 && lane == 0) MOE_PF_KMARK(6, g);
        }
    } else {
        // ------------------------------------------ epilogue (warps 11..14)
        // lane quarter q: routes 32 q .. 32 q + 31 of the tile, one per thread;
        // a thread writes its route's row of h (or y) with 16-byte stores
        const int q = warp & 3, lrow = q * 32 + lane;
        int li = 0;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x, li++) {
            const int tile = it / mtiles, mt = it - tile * mtiles;
            const int4 tl = tile_at(tile);
            const int e = tl.x, rstart = tl.y, rcount = tl.z;
            const int ab = li & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[ab], (li >> 1) & 1, status, 40))) break;
            if (it == (int)blockIdx.x && warp == kWarpEpi0 && lane == 0) MOE_PF_MARK(1);
            if (warp == kWarpEpi0 && lane == 0) MOE_PF_KMARK(7, li);
            tc_fence_after();
            const uint32_t taddr = tmem + (uint32_t)(ab * kAccCols) + ((uint32_t)(q * 32) << 16);
            const bool mine = lrow < rcount;
            if (q * 32 < rcount) {  // warp-uniform: the quarter holds routes of the tile
                // the item's 256 biases (gate then up, or down), staged once per warp
                float *bias = s_bias + (warp - kWarpEpi0) * kBiasFloats;
#pragma unroll
                for (int i = lane; i < kWN; i += 32) {
                    const int half = GATEUP ? i / RPI : 0, row = mt * RPI + (GATEUP ? i % RPI : i);
                    bias[i] = row < a.rows ? __ldg(mat_bias(half ? a.A1 : a.A0, e, E) + row) : 0.0f;
                }
                __syncwarp();
                if (GATEUP) {
                    uint16_t *hrow = (F16 ? a.ws.h16 : a.ws.h) + (size_t)(rstart + lrow) * a.bp.F;
#pragma unroll 1
                    for (int c0 = 0; c0 < RPI; c0 += 32) {
                        const int j0 = mt * RPI + c0;
                        if (j0 >= a.rows) break;  // F is a multiple of 64: whole 32-column chunks
                        float gv[32], uv[32];
                        tmem_ld32(taddr + c0, gv);
                        tmem_ld32(taddr + RPI + c0, uv);
                        if (!mine) continue;
                        uint32_t bits[32];
#pragma unroll
                        for (int c = 0; c < 32; c++) {
                            const float hv = swiglu_fast(gv[c] + bias[c0 + c], uv[c] + bias[RPI + c0 + c],
                                                         a.bp.alpha, a.bp.limit);
                            const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                            bits[c] = *reinterpret_cast<const uint16_t *>(&hb);
                            if (F16) {
                                const __half hh = __float2half_rn(__bfloat162float(hb));  // exact in the fp16 range
                                bits[c] = *reinterpret_cast<const uint16_t *>(&hh);
                            }
                        }
                        // fp16: natural order; bf16: the 32-block pair order (elements i and
                        // i + 4 of every 8 share a word), as the next GEMM's B-side expects
                        uint32_t wd[16];
#pragma unroll
                        for (int k = 0; k < 16; k++) {
                            const int lo = F16 ? 2 * k : 8 * (k >> 2) + (k & 3), hi = F16 ? 2 * k + 1 : lo + 4;
                            wd[k] = bits[lo] | (bits[hi] << 16);
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(hrow + j0);
#pragma unroll
                        for (int k = 0; k < 4; k++)
                            dst[k] = make_uint4(wd[4 * k], wd[4 * k + 1], wd[4 * k + 2], wd[4 * k + 3]);
                    }
                } else {
                    const float w = mine ? a.ws.perm_w[rstart + lrow] : 0.0f;
                    float *yrow = a.ws.y + (size_t)(rstart + lrow) * a.bp.H;
#pragma unroll 1
                    for (int c0 = 0; c0 < RPI; c0 += 32) {
                        const int i0 = mt * RPI + c0;
                        if (i0 >= a.rows) break;  // H is a multiple of 64: whole 32-column chunks
                        float v[32];
                        tmem_ld32(taddr + c0, v);
                        if (!mine) continue;
                        float4 *dst = reinterpret_cast<float4 *>(yrow + i0);
#pragma unroll
                        for (int k = 0; k < 8; k++)
                            dst[k] = make_float4(w * (v[4 * k] + bias[c0 + 4 * k]), w * (v[4 * k + 1] + bias[c0 + 4 * k + 1]),
                                                 w * (v[4 * k + 2] + bias[c0 + 4 * k + 2]),
                                                 w * (v[4 * k + 3] + bias[c0 + 4 * k + 3]));
                    }
                }
            }
            // the accumulator may be overwritten once every lane's TMEM reads are done
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ab]);
            if (warp == kWarpEpi0 && lane == 0) MOE_PF_KMARK(8, li);
        }
        if (warp == kWarpEpi0 && lane == 0) MOE_PF_MARK(2);
    }
    tc_fence_before();
    __syncthreads();
    MOE_PF_MARK(3);
    if (warp == kWarpMma)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols));
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

// 2D map over packed codes: [n_rows][cols/2] bytes, box 32 kCK bytes x box_rows, 64-byte swizzle.
cudaError_t make_codes_map(CUtensorMap *m, const uint8_t *codes, size_t n_rows, int cols, int box_rows) {
    if (!codes) {
        memset(m, 0, sizeof *m);
        return cudaSuccess;
    }
    cuuint64_t dims[2] = {(cuuint64_t)(cols / 2), (cuuint64_t)n_rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols / 2)};
    cuuint32_t box[2] = {32 * kCK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

size_t prefill_smem_bytes() {
    return 1024 + kStages * (kABytes + kBBytes) + kCStages * kCStageBytes + kSmTiles * 16 +
           kEpiWarps * kBiasFloats * 4 + 512;
}

// 2D map over a 16-bit activation matrix [rows][K] (the MMA's A operand): box
// 64 elements (128 B) x box_rows (32, 64, 128), 128-byte swizzle (the K-major
// layout the MMA descriptors expect; the box is whole 8-row swizzle atoms).
cudaError_t make_act_map(CUtensorMap *m, const uint16_t *base, int rows, int K, bool f16, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<uint16_t *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// xs[pos] = src[perm_token[pos]] (16-byte chunks), pos < R; src is x_hat16
// (fp16 variant) or x_hat_mma (bf16 variant).
__global__ void __launch_bounds__(256) moe_gather_kernel(Workspace ws, const uint16_t *src, int H, int R) {
    const int cpr = H / 8;  // 16-byte chunks per row
    const size_t n = (size_t)R * cpr;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int pos = (int)(i / cpr), c = (int)(i - (size_t)pos * cpr);
        const int tok = ws.perm_token[pos];
        reinterpret_cast<uint4 *>(ws.xs + (size_t)pos * H)[c] =
            reinterpret_cast<const uint4 *>(src + (size_t)tok * H)[c];
    }
}

// Scale repack: out chunk (block b, k-block kb) byte 2 r + h = scale of row
// 64 (b % row_blocks) + r of expert b / row_blocks, 32-element block 2 kb + h;
// rows past the matrix (and the trailing pad block) read 127, a scale of 1.
__global__ void __launch_bounds__(256) moe_pack_scales_kernel(const uint8_t *in, uint8_t *out, int n_exp, int rows,
                                                               int cols, size_t n_out) {
    const int nb = cols / 32, nkb = cols / kBK, rb = (rows + 63) / 64;
    const size_t per_block = (size_t)nkb * 128;
    for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < n_out; o += (size_t)gridDim.x * blockDim.x) {
        const size_t blk = o / per_block;
        const int rem = (int)(o - blk * per_block);
        const int kb = rem >> 7, r = (rem & 127) >> 1, h = rem & 1;
        const int e = (int)(blk / rb), row = (int)(blk % rb) * 64 + r;
        out[o] = (e < n_exp && row < rows) ? in[((size_t)e * rows + row) * nb + 2 * kb + h] : (uint8_t)127;
    }
}

// blocks of one repacked matrix set: n_exp experts plus four pad blocks (a
// down item's four blocks may run three past the last real one, and a code
// stage's chunk pair one chunk further)
size_t packed_blocks(int n_exp, int rows) { return (size_t)n_exp * ((rows + 63) / 64) + 4; }
size_t packed_bytes(int n_exp, int rows, int cols) {
    return (packed_blocks(n_exp, rows) * (size_t)(cols / kBK) * 128 + 255) & ~(size_t)255;
}

}  // namespace

int prefill_tile_rows() { return kTM; }

cudaError_t prefill_make_maps(const BlockParams &bp, const MatPtrs &gate, const MatPtrs &up, const MatPtrs &down,
                              PrefillMaps *out) {
    MOE_CUDA_TRY(get_encoder());
    const int E = bp.E;
    TmaMaps &g = out->gateup, &d = out->down;
    // gate/up items: 128 gate rows + the same 128 up rows; down items: 256 rows
    MOE_CUDA_TRY(make_codes_map(&g.m[0], gate.codes, (size_t)E * gate.rows, gate.cols, kWN / 2));
    MOE_CUDA_TRY(make_codes_map(&g.m[1], up.codes, (size_t)E * up.rows, up.cols, kWN / 2));
    MOE_CUDA_TRY(make_codes_map(&g.m[2], bp.n_shared ? gate.sh_codes : nullptr, gate.rows, gate.cols, kWN / 2));
    MOE_CUDA_TRY(make_codes_map(&g.m[3], bp.n_shared ? up.sh_codes : nullptr, up.rows, up.cols, kWN / 2));
    MOE_CUDA_TRY(make_codes_map(&d.m[0], down.codes, (size_t)E * down.rows, down.cols, kWN));
    d.m[1] = d.m[0];
    MOE_CUDA_TRY(make_codes_map(&d.m[2], bp.n_shared ? down.sh_codes : nullptr, down.rows, down.cols, kWN));
    d.m[3] = d.m[2];
    return cudaSuccess;
}

size_t prefill_scales_bytes(const BlockParams &bp) {
    const int ns = bp.n_shared ? 1 : 0;
    return 2 * (packed_bytes(bp.E, bp.F, bp.H) + packed_bytes(ns, bp.F, bp.H)) + packed_bytes(bp.E, bp.H, bp.F) +
           packed_bytes(ns, bp.H, bp.F);
}

cudaError_t prefill_pack_scales(const BlockParams &bp, const MatPtrs &gate, const MatPtrs &up, const MatPtrs &down,
                                uint8_t *buf, PrefillMaps *out, cudaStream_t st) {
    const MatPtrs *ms[3] = {&gate, &up, &down};
    TmaMaps *tm[3] = {&out->gateup, &out->gateup, &out->down};
    const int slot[3] = {0, 1, 0};
    for (int i = 0; i < 3; i++) {
        const MatPtrs &m = *ms[i];
        for (int sh = 0; sh < 2; sh++) {
            const int n_exp = sh ? (bp.n_shared ? 1 : 0) : bp.E;
            const uint8_t *src = sh ? m.sh_scales : m.scales;
            const size_t n = packed_bytes(n_exp, m.rows, m.cols);
            const uint8_t *dst = nullptr;
            if (n_exp) {
                const size_t nout = packed_blocks(n_exp, m.rows) * (size_t)(m.cols / kBK) * 128;
                const int blocks = (int)((nout + 255) / 256 < 8192 ? (nout + 255) / 256 : 8192);
                moe_pack_scales_kernel<<<blocks, 256, 0, st>>>(src, buf, n_exp, m.rows, m.cols, nout);
                MOE_CUDA_TRY(cudaGetLastError());
                dst = buf;
                buf += n;
            }
            tm[i]->sc[slot[i] + 2 * sh] = dst;
        }
        tm[i]->row_blocks = (m.rows + 63) / 64;
    }
    out->down.sc[1] = out->down.sc[0];
    out->down.sc[3] = out->down.sc[2];
    return cudaSuccess;
}

cudaError_t launch_gather(const BlockParams &bp, const Workspace &ws, int T, bool f16, cudaStream_t st) {
    const int R = T * (bp.K + bp.n_shared);
    const size_t n = (size_t)R * (bp.H / 8);
    const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    moe_gather_kernel<<<blocks, 256, 0, st>>>(ws, f16 ? ws.xhat16 : ws.xhat_mma, bp.H, R);
    return cudaGetLastError();
}

template <bool GATEUP, bool F16>
cudaError_t launch_pf(const PrefillArgs &args, const TmaMaps &maps, const AMaps &amaps, dim3 grid,
                      cudaStream_t st) {
    static PerDevice<bool> done;
    MOE_CUDA_TRY(smem_optin_once(moe_prefill_kernel<GATEUP, F16>, done));
    moe_prefill_kernel<GATEUP, F16><<<grid, kThreads, prefill_smem_bytes(), st>>>(args, maps, amaps);
    return cudaGetLastError();
}

cudaError_t launch_prefill_stage(const BlockParams &bp, const Workspace &ws, const MatPtrs &a0, const MatPtrs &a1,
                                 bool gateup, int T, const TmaMaps &maps, bool f16, cudaStream_t st) {
    PrefillArgs args{bp, ws, a0, a1, gateup ? bp.H : bp.F, gateup ? bp.F : bp.H};
    const int R = T * (bp.K + bp.n_shared);
    AMaps amaps;
    MOE_CUDA_TRY(get_encoder());
    const uint16_t *bsrc = gateup ? ws.xs : (f16 ? ws.h16 : ws.h);
    for (int i = 0; i < 3; i++) MOE_CUDA_TRY(make_act_map(&amaps.m[i], bsrc, R, args.Kdim, f16, 32 << i));
    int tiles = (R + kTM - 1) / kTM + bp.E + bp.n_shared;
    if (tiles > ws.max_tiles) tiles = ws.max_tiles;
    const int mtiles = gateup ? (bp.F + kWN / 2 - 1) / (kWN / 2) : (bp.H + kWN - 1) / kWN;
    // persistent: one CTA per SM, or fewer when there are fewer work items
    static PerDevice<int> sms;
    int dev = 0;
    MOE_CUDA_TRY(current_device_slot(&dev));
    int &n_sm = sms.v[dev];
    if (!n_sm) MOE_CUDA_TRY(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
    const long items = (long)tiles * mtiles;
    const dim3 grid((unsigned)(items < n_sm ? items : n_sm));
    if (gateup)
        return f16 ? launch_pf<true, true>(args, maps, amaps, grid, st) : launch_pf<true, false>(args, maps, amaps, grid, st);
    return f16 ? launch_pf<false, true>(args, maps, amaps, grid, st) : launch_pf<false, false>(args, maps, amaps, grid, st);
}
