// moe_mxf4.cu -- the grouped per-expert GEMMs on the block-scaled FP4 tensor
// cores: tcgen05.mma kind::mxf4 with both operands MXFP4 (E2M1 codes in
// 32-element blocks with one E8M0 scale each), the scales in tensor memory,
// no dequantisation anywhere.
//
// The activations take the FP4 activation encoding of ds4.c (FP4 activation
// quantisation `dsv4_fp4_act_quantize_row_inplace_cpu`, nearest value as in
// `dsv4_e2m1fn_dequant_cpu`) along the contracted dimension: x_hat before
// gate/up, h (after its bf16 rounding) before down.  The weights already have
// that format.  Everything else is the block of goosedump gpt_oss.rs
// `expert_batch_output`: per expert, gate/up + bias, clamped SwiGLU, down +
// bias, times the route weight.
//
// Work item = (route tile of <= 128 routes of one expert, block of weight
// rows): M = 128 routes, N = 192 weight rows (96 gate rows then the same 96
// up rows, or 192 down rows), K in stages of 256 (128 bytes of codes per row,
// four MMAs of K = 64).  Per stage two producer threads bring in by TMA the
// tile's A codes and the item's B codes (both 128-byte swizzled; a weight box
// covers 96 or 192 rows of one expert, rows past its end read as zeros), and
// by bulk copies the 512-byte scale atoms of A and B; the MMA thread copies
// the atoms into tensor memory (tcgen05.cp .32x128b.warpx4: atom byte
// 16 (r % 32) + 4 (r / 32) + j holds row r's scale for the j-th 32-element
// block of the 128-element group, and lands in the row's lane, column r / 32,
// byte j), then issues the MMAs with scale ID = byte 0 or 2 of that column.
// Two 192-column fp32 accumulators (with the scale slots, 480 of the 512 TMEM
// columns) let four epilogue warps drain one item while the next accumulates:
// measured on GB300, a single accumulator left the MMA waiting for the
// epilogue ~45 % of the time.  The gate/up epilogue applies bias and SwiGLU,
// rounds h to bf16 and encodes it straight into the down GEMM's A operand
// (codes by route row, scales into the tile's atoms); the down epilogue
// writes bias-added, route-weighted rows of y for the combine.
//
// Every mbarrier wait is bounded (about 2 s of %globaltimer): on a timeout
// the kernel records MOE_DEV_WAIT_TIMEOUT, lets issued copies and MMAs land,
// frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "moe_common.cuh"

// Timeline marker (no-op unless an instrumented build defines it).
#ifndef MOE_Q_MARK
#define MOE_Q_MARK(slot, idx)
#endif

namespace {

constexpr int kQStages = 4;                 // operand stages
constexpr int kQK = 256;                    // K elements per stage (128 bytes of codes per row)
constexpr int kQM = 128;                    // routes per tile (MMA M)
constexpr int kQN = 192;                    // weight rows per item (MMA N)
constexpr int kQABytes = kQM * 128;         // A codes of a stage
constexpr int kQBBytes = kQN * 128;         // B codes of a stage
constexpr int kQSfABytes = 1024;            // A scale atoms of a stage: 2 groups of 128 K elements x 128 rows
constexpr int kQSfBBytes = 2048;            // B scale atoms of a stage: 2 groups x 2 row halves (rows 0-127, 128-191)
constexpr int kQStageBytes = kQABytes + kQBBytes + kQSfABytes + kQSfBBytes;
static_assert(kQStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
// warps: 0 weight producer (B codes + B scale atoms), 1 MMA issuer, 2
// activation producer (A codes + A scale atoms), 3..6 epilogue.  A copy
// instruction holds its issuing thread for ~0.1 us (measured on GB300 with
// 4 KB bulk copies), so the two operand streams get a thread each.
constexpr int kQWarpProd = 0, kQWarpMma = 1, kQWarpProdA = 2, kQWarpEpi0 = 3, kQEpiWarps = 4;
constexpr int kQThreads = 32 * (kQWarpEpi0 + kQEpiWarps);
constexpr int kQAcc = kQN;                  // an fp32 accumulator: 128 lanes x 192 columns; two of them
constexpr int kQSfCol0 = 2 * kQAcc;         // scale slots: stage s -> A at kQSfCol0 + 24 s (8 columns), B at + 8 (16)
constexpr int kQTmemCols = 512;
static_assert(kQSfCol0 + 24 * kQStages <= kQTmemCols, "TMEM budget");
constexpr int kQSmTiles = 256;
constexpr uint64_t kQWaitNs = 2000000000ull;

struct Mxf4Maps {
    CUtensorMap b[4];      // B codes: [0] routed gate (or down), [1] routed up, [2] shared gate (or down), [3] shared up
    CUtensorMap a[3];      // A codes (route-ordered activations): boxes of 32, 64, 128 rows
    const uint8_t *bsf;    // routed B scale atoms [E][row blocks][nqe][2 row halves][512]
    const uint8_t *bsf_sh; // the shared expert's
    const uint8_t *asf;    // A scale atoms [tile][nqe][512]
    int row_blocks;        // item row blocks per expert matrix
    int nqe;               // 128-element scale groups per row, rounded up to even
};

struct Mxf4Args {
    BlockParams bp;
    Workspace ws;
    MatPtrs A0, A1;    // gate, up (GATEUP) or down
    int Kdim, rows;    // K = H (gate/up) or F (down); output rows F or H
    uint8_t *hq;       // gate/up: h codes out [R][F/2] (route rows)
    uint8_t *hsf;      // gate/up: h scale atoms out [tile][nqe(F)][512]
    int hnqe;          // nqe(F)
};

__device__ __forceinline__ uint32_t q_smem(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ uint64_t q_time() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void q_init(uint64_t *b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(q_smem(b)), "r"(n));
}
__device__ __forceinline__ void q_arrive(uint64_t *b) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(q_smem(b)) : "memory");
}
__device__ __forceinline__ void q_expect(uint64_t *b, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(q_smem(b)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool q_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(q_smem(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: false (status set) after ~2 s or once another thread reported a failure.
__device__ __forceinline__ bool q_wait(uint64_t *b, uint32_t parity, int32_t *status, int where) {
    if (q_try(b, parity)) return true;
    const uint64_t t0 = q_time();
    for (uint32_t i = 0;; i++) {
        if (q_try(b, parity)) return true;
        if ((i & 63) == 63) {
            if (*(volatile int32_t *)status != 0) return false;
            if (q_time() - t0 > kQWaitNs) {
                set_device_error(status, MOE_DEV_WAIT_TIMEOUT, where);
                return false;
            }
        }
    }
}
// The last min(issued, n) phases of an n-stage ring have completed (only the
// time limit ends it): issued copies land before the CTA's shared memory goes.
__device__ __forceinline__ void q_drain(uint64_t *full, int n, int issued, int32_t *status) {
    const uint64_t t0 = q_time();
    for (int g = max(0, issued - n); g < issued; g++)
        while (!q_try(&full[g % n], (g / n) & 1))
            if (q_time() - t0 > kQWaitNs) {
                set_device_error(status, MOE_DEV_WAIT_TIMEOUT, 191);
                return;
            }
}
__device__ __forceinline__ uint64_t q_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void q_tma(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(q_smem(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(q_smem(bar)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void q_tma3_ef(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y, int z,
                                          uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%3, %4, %5}], [%2], %6;" ::"r"(q_smem(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(q_smem(bar)), "r"(x), "r"(y), "r"(z), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void q_bulk(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     q_smem(dst)),
                 "l"(src), "r"(bytes), "r"(q_smem(bar))
                 : "memory");
}
__device__ __forceinline__ void q_bulk_ef(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            q_smem(dst)),
        "l"(src), "r"(bytes), "r"(q_smem(bar)), "l"(pol)
        : "memory");
}
// Shared-memory matrix descriptors: K-major 128-byte swizzle (8-row groups
// 1024 B apart), and the plain layout of a scale atom (32 rows of 16 bytes;
// both offsets 128 B, so either reading of the two fields is the same).
__device__ __forceinline__ uint64_t q_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ uint64_t q_desc_atom(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) |
           ((uint64_t)1 << 46);
}
// Instruction descriptor, kind::mxf4: A and B E2M1 (format 1), K-major, E8M0
// scales (bit 23), N = 128, M = 128, scale IDs (byte within the scale column)
// for A (bits 29-30) and B (bits 4-5).
__device__ __forceinline__ uint32_t q_idesc(uint32_t sf_id) {
    return (sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kQN >> 3) << 17) | (1u << 23) |
           ((uint32_t)(kQM >> 4) << 24) | (sf_id << 29);
}
__device__ __forceinline__ void q_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                      uint32_t acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %6, 0; tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, "
        "%2, %3, [%4], [%5], p; }" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc));
}
__device__ __forceinline__ void q_cp_atom(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc));
}
__device__ __forceinline__ void q_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(q_smem(bar))
                 : "memory");
}
__device__ __forceinline__ void q_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void q_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void q_ld32(uint32_t taddr, float v[32]) {
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
// Two 32-column loads, one wait.
__device__ __forceinline__ void q_ld32x2(uint32_t t0, float v0[32], uint32_t t1, float v1[32]) {
    uint32_t r[32], u[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(t0));
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]), "=r"(u[8]),
          "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]),
          "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]),
          "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
        : "r"(t1));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) {
        v0[i] = __uint_as_float(r[i]);
        v1[i] = __uint_as_float(u[i]);
    }
}
// Byte of row r (< 128) and 32-element block j (< 4) inside a 512-byte scale atom.
__device__ __forceinline__ int q_atom_byte(int r, int j) { return 16 * (r & 31) + 4 * (r >> 5) + j; }

// Clamped SwiGLU with the hardware exponential and a fast divide (a few fp32
// ulps, far inside the bf16 rounding of h that follows).
__device__ __forceinline__ float q_swiglu(float g, float u, float alpha, float limit) {
    const float gc = (g > limit) ? limit : g;
    const float uc = (u > limit) ? limit : ((u < -limit) ? -limit : u);
    return __fdividef(gc, 1.0f + __expf(-alpha * gc)) * (uc + 1.0f);
}

// Persistent grouped GEMM.  Items it = (route tile it / mtiles, weight-row
// block it % mtiles); CTA b takes items b, b + gridDim.x, ...; every role
// walks the same sequence with its own ring counters.
template <bool GATEUP>
__global__ void __launch_bounds__(kQThreads, 1) moe_mxf4_kernel(const __grid_constant__ Mxf4Args a,
                                                                 const __grid_constant__ Mxf4Maps maps) {
    constexpr int RPI = GATEUP ? kQN / 2 : kQN;  // output rows per item
    const int mtiles = (a.rows + RPI - 1) / RPI;
    const int n_tiles = *a.ws.n_tiles;
    const int n_items = n_tiles * mtiles;
    if ((int)blockIdx.x >= n_items) return;
    extern __shared__ unsigned char q_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(((uintptr_t)q_raw + 1023) & ~(uintptr_t)1023);
    int4 *s_tiles = reinterpret_cast<int4 *>(smem + kQStages * kQStageBytes);   // [kQSmTiles]
    float *s_bias = reinterpret_cast<float *>(s_tiles + kQSmTiles);              // [kQEpiWarps][kQN]
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_bias + kQEpiWarps * kQN);
    uint64_t *full = bars, *empty = bars + kQStages, *acc_full = empty + kQStages, *acc_empty = acc_full + 2,
             *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    const int E = a.bp.E, K = a.Kdim, nks = (K + kQK - 1) / kQK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *status = a.ws.status;
    for (int i = threadIdx.x; i < min(n_tiles, kQSmTiles); i += blockDim.x) s_tiles[i] = a.ws.tiles[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; s++) {
            q_init(&full[s], 2);  // the two producers' expect_tx arrivals
            q_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            q_init(&acc_full[b], 1);
            q_init(&acc_empty[b], kQEpiWarps);
        }
        q_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kQWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(q_smem(tmem_slot)),
                     "n"(kQTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    q_fence_before();
    __syncthreads();
    q_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto tile_at = [&](int t) -> int4 { return t < kQSmTiles ? s_tiles[t] : a.ws.tiles[t]; };

    if (warp == kQWarpProd || warp == kQWarpProdA) {
        // ------------------------------------------- TMA producers (B and A)
        if (lane == 0) {
            const bool wB = warp == kQWarpProd;
            const uint64_t pol = q_evict_first();
            int s = 0, issued = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const int tile = it / mtiles, mt = it - tile * mtiles;
                const int4 tl = tile_at(tile);
                const int e = tl.x, rstart = tl.y, rcount = tl.z;
                const bool sh = e >= E;
                const int ebase = sh ? 0 : e;
                const int mi = rcount <= 32 ? 0 : (rcount <= 64 ? 1 : 2);
                const uint32_t abytes = (uint32_t)(32 << mi) * 128;
                const uint8_t *bsf = (sh ? maps.bsf_sh : maps.bsf) +
                                     ((size_t)(ebase * maps.row_blocks + mt) * maps.nqe) * 1024;
                const uint8_t *asf = maps.asf + (size_t)tile * maps.nqe * 512;
                for (int ks = 0; ks < nks; ks++) {
                    if (!q_wait(&empty[s], ph ^ 1, status, wB ? 110 : 111)) {
                        ok = false;
                        break;
                    }
                    MOE_Q_MARK(wB ? 7 : 8, issued);
                    unsigned char *st = smem + s * kQStageBytes;
                    if (wB) {
                        q_expect(&full[s], kQBBytes + kQSfBBytes);
                        if (GATEUP) {
                            q_tma3_ef(st + kQABytes, &maps.b[sh ? 2 : 0], &full[s], ks * 128, mt * RPI, ebase, pol);
                            q_tma3_ef(st + kQABytes + kQBBytes / 2, &maps.b[sh ? 3 : 1], &full[s], ks * 128, mt * RPI,
                                      ebase, pol);
                        } else {
                            q_tma3_ef(st + kQABytes, &maps.b[sh ? 2 : 0], &full[s], ks * 128, mt * RPI, ebase, pol);
                        }
                        q_bulk_ef(st + kQABytes + kQBBytes + kQSfABytes, bsf + (size_t)ks * kQSfBBytes, kQSfBBytes,
                                  &full[s], pol);
                    } else {
                        q_expect(&full[s], abytes + kQSfABytes);
                        q_tma(st, &maps.a[mi], &full[s], ks * 128, rstart);
                        q_bulk(st + kQABytes + kQBBytes, asf + (size_t)ks * kQSfABytes, kQSfABytes, &full[s]);
                    }
                    MOE_Q_MARK(wB ? 0 : 1, issued);
                    issued++;
                    if (++s == kQStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            q_drain(full, kQStages, issued, status);
        }
    } else if (warp == kQWarpMma) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int s = 0, li = 0, g = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, li++) {
                // the epilogue has read this accumulator out (free on its first use)
                const int ab = li & 1;
                if (!(ok = q_wait(&acc_empty[ab], ((li >> 1) & 1) ^ 1, status, 120))) break;
                MOE_Q_MARK(4, li);
                q_fence_after();
                const uint32_t d = tmem + (uint32_t)(ab * kQAcc);
                for (int ks = 0; ks < nks; ks++, g++) {
                    if (!(ok = q_wait(&full[s], ph, status, 121))) break;
                    MOE_Q_MARK(2, g);
                    q_fence_after();
                    const uint32_t sa = q_smem(smem + s * kQStageBytes), sb = sa + kQABytes;
                    const uint32_t sfa = sb + kQBBytes, sfb = sfa + kQSfABytes;
                    const uint32_t ta = tmem + (uint32_t)(kQSfCol0 + 24 * s), tb = ta + 8;
                    // A: group g -> columns ta + 4 g; B: group g, row half h -> columns tb + 8 g + 4 h
                    q_cp_atom(ta, q_desc_atom(sfa));
                    q_cp_atom(ta + 4, q_desc_atom(sfa + 512));
#pragma unroll
                    for (int j = 0; j < 4; j++) q_cp_atom(tb + 4 * j, q_desc_atom(sfb + 512 * j));
                    const int nk = min(4, (K - ks * kQK) / 64);
                    for (int i = 0; i < nk; i++)
                        q_mma(d, q_desc_sw128(sa + 32 * i), q_desc_sw128(sb + 32 * i),
                              q_idesc((uint32_t)(i & 1) * 2), ta + 4 * (i >> 1), tb + 8 * (i >> 1),
                              (uint32_t)((ks | i) != 0));
                    q_commit(&empty[s]);
                    MOE_Q_MARK(3, g);
                    if (++s == kQStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (ok) q_commit(&acc_full[ab]);
            }
            if (!ok) {
                // the copies and MMAs already issued finish before TMEM is released
                q_commit(drain);
                const uint64_t t0 = q_time();
                while (!q_try(drain, 0))
                    if (q_time() - t0 > kQWaitNs) {
                        set_device_error(status, MOE_DEV_WAIT_TIMEOUT, 192);
                        break;
                    }
            }
        }
    } else {
        // ------------------------------------------------- epilogue (4 warps)
        // lane quarter q: routes 32 q .. 32 q + 31 of the tile, one per thread
        const int q = warp & 3, lrow = q * 32 + lane;
        float *bias = s_bias + (warp - kQWarpEpi0) * kQN;
        int li = 0;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x, li++) {
            const int tile = it / mtiles, mt = it - tile * mtiles;
            const int4 tl = tile_at(tile);
            const int e = tl.x, rstart = tl.y, rcount = tl.z;
            const int ab = li & 1;
            if (!__all_sync(0xffffffffu, q_wait(&acc_full[ab], (li >> 1) & 1, status, 130))) break;
            if (warp == kQWarpEpi0 && lane == 0) MOE_Q_MARK(5, li);
            q_fence_after();
            const uint32_t taddr = tmem + (uint32_t)(ab * kQAcc) + ((uint32_t)(q * 32) << 16);
            const bool mine = lrow < rcount;
            const int pos = rstart + lrow;
            if (q * 32 < rcount) {  // warp-uniform: the quarter holds routes of the tile
                for (int i = lane; i < kQN; i += 32) {
                    const int half = GATEUP ? i / RPI : 0, row = mt * RPI + (GATEUP ? i % RPI : i);
                    bias[i] = row < a.rows ? __ldg(mat_bias(half ? a.A1 : a.A0, e, E) + row) : 0.0f;
                }
                __syncwarp();
                if (GATEUP) {
                    // h rows j0 .. j0 + 95: three 32-element blocks of the down GEMM's K
                    const int j0 = mt * RPI;
#pragma unroll 1
                    for (int c0 = 0; c0 < RPI; c0 += 32) {
                        if (j0 + c0 >= a.rows) break;  // F is a multiple of 64: whole 32-column chunks
                        float gv[32], uv[32];
                        q_ld32x2(taddr + c0, gv, taddr + RPI + c0, uv);
                        if (!mine) continue;
                        float hv[32];
#pragma unroll
                        for (int c = 0; c < 32; c++) {
                            const float h = q_swiglu(gv[c] + bias[c0 + c], uv[c] + bias[RPI + c0 + c], a.bp.alpha,
                                                     a.bp.limit);
                            hv[c] = __bfloat162float(__float2bfloat16_rn(h));  // h's contractual bf16 rounding
                        }
                        uint32_t sb;
                        const uint4 codes = mxq_encode_block(hv, sb);
                        const int blk = (j0 + c0) / 32;
                        *reinterpret_cast<uint4 *>(a.hq + (size_t)pos * (a.bp.F / 2) + (j0 + c0) / 2) = codes;
                        a.hsf[((size_t)tile * a.hnqe + blk / 4) * 512 + q_atom_byte(lrow, blk & 3)] = (uint8_t)sb;
                    }
                } else {
                    const float w = mine ? a.ws.perm_w[pos] : 0.0f;
                    float *yrow = a.ws.y + (size_t)pos * a.bp.H;
#pragma unroll 1
                    for (int c0 = 0; c0 < RPI; c0 += 32) {
                        const int i0 = mt * RPI + c0;
                        if (i0 >= a.rows) break;  // H is a multiple of 64: whole 32-column chunks
                        float v[32];
                        q_ld32(taddr + c0, v);
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
            q_fence_before();
            __syncwarp();
            if (lane == 0) q_arrive(&acc_empty[ab]);
            if (warp == kQWarpEpi0 && lane == 0) MOE_Q_MARK(6, li);
        }
    }
    q_fence_before();
    __syncthreads();
    if (warp == kQWarpMma)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kQTmemCols));
}

// x_hat rows of each route tile, FP4-encoded into route order (the gate/up
// GEMM's A codes, [R][H/2]) with the tile's scale atoms ([tile][nqe][512]).
// Grid (tiles, 128 / 8): one warp per route row of the tile, lane l encoding
// 32-element blocks l, l + 32, ...; all of a row's loads are issued before
// any is used (the row index itself is one load, the row another: two L2
// round trips in all).
constexpr int kGatherRowsPerCta = 8;
constexpr int kGatherMaxBlocks = 4;  // blocks per lane: H <= 4 * 32 * 32 = 4096
__global__ void __launch_bounds__(32 * kGatherRowsPerCta) moe_mxf4_gather_kernel(Workspace ws, int H, uint8_t *xq,
                                                                                  uint8_t *xsf, int nqe) {
    const int tile = blockIdx.x;
    if (tile >= *ws.n_tiles) return;
    const int4 tl = ws.tiles[tile];
    const int r = blockIdx.y * kGatherRowsPerCta + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (r >= tl.z) return;
    const int pos = tl.y + r, nb = H / 32;
    const uint4 *src = reinterpret_cast<const uint4 *>(ws.xhat + (size_t)ws.perm_token[pos] * H);
    uint4 v[kGatherMaxBlocks][4];
#pragma unroll
    for (int j = 0; j < kGatherMaxBlocks; j++) {
        const int b = lane + 32 * j;
#pragma unroll
        for (int c = 0; c < 4; c++) v[j][c] = b < nb ? __ldg(src + 4 * b + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kGatherMaxBlocks; j++) {
        const int b = lane + 32 * j;
        if (b >= nb) break;
        float x[32];
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const uint32_t w[4] = {v[j][c].x, v[j][c].y, v[j][c].z, v[j][c].w};
#pragma unroll
            for (int k = 0; k < 4; k++) {
                x[8 * c + 2 * k] = __uint_as_float(w[k] << 16);
                x[8 * c + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            }
        }
        uint32_t sb;
        const uint4 codes = mxq_encode_block(x, sb);
        *reinterpret_cast<uint4 *>(xq + (size_t)pos * (H / 2) + 16 * b) = codes;
        xsf[((size_t)tile * nqe + b / 4) * 512 + q_atom_byte(r, b & 3)] = (uint8_t)sb;
    }
}

// Weight scales repacked into the atoms the kernel copies: item block b of
// expert e, 128-element group g, row half h: atom (((e * blocks + b) * nqe + g)
// * 2 + h) holds, for atom row r, the scales of the weight row behind item row
// n = 128 h + r (gate/up: gate row 96 b + n for n < 96, up row 96 b + n - 96
// for n < 192; down: row 192 b + n for n < 192) for the four 32-element
// blocks 4 g .. 4 g + 3.  Item rows past 192 or past the matrix and blocks
// past K read 127 (a scale of 1; their codes are zeros or unused).
__global__ void __launch_bounds__(256) moe_mxf4_pack_kernel(const uint8_t *s0, const uint8_t *s1, int n_exp, int rows,
                                                            int cols, int gateup, int nqe, uint8_t *out, size_t n_out) {
    const int nb = cols / 32, rpb = gateup ? kQN / 2 : kQN, blocks = (rows + rpb - 1) / rpb;
    for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < n_out; o += (size_t)gridDim.x * blockDim.x) {
        const size_t atom = o / 512;
        const int byte = (int)(o - atom * 512);
        const int h = (int)(atom & 1);
        const size_t ag = atom >> 1;
        const int g = (int)(ag % nqe);
        const size_t eb = ag / nqe;
        const int b = (int)(eb % blocks), e = (int)(eb / blocks);
        const int lo = byte >> 4, rem = byte & 15;  // lo = row % 32, rem = 4 * (row / 32) + j
        const int n = 128 * h + lo + 32 * (rem >> 2), j = rem & 3;
        const int kb = 4 * g + j;
        const bool up_half = gateup && n >= rpb;
        const uint8_t *src = up_half ? s1 : s0;
        const int wr = rpb * b + (up_half ? n - rpb : n);
        const bool valid = e < n_exp && n < kQN && wr < rows && kb < nb;
        out[o] = valid ? src[((size_t)e * rows + wr) * nb + kb] : (uint8_t)127;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 q_encode = nullptr;

cudaError_t q_get_encoder() {
    if (q_encode) return cudaSuccess;
    cudaDriverEntryPointQueryResult qr;
    void *fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr);
    if (e != cudaSuccess) return e;
    if (qr != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    q_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

// 2D map over packed FP4 codes [n_rows][cols/2] bytes: box 128 bytes x box_rows,
// 128-byte swizzle (the K-major layout of the MMA descriptors).
cudaError_t q_codes_map(CUtensorMap *m, const uint8_t *codes, size_t n_rows, int cols, int box_rows, bool promote) {
    if (!codes || n_rows == 0) {
        memset(m, 0, sizeof *m);
        return cudaSuccess;
    }
    cuuint64_t dims[2] = {(cuuint64_t)(cols / 2), (cuuint64_t)n_rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols / 2)};
    cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = q_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          promote ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3D map over the weight codes of n_exp experts, [n_exp][rows][cols/2] bytes:
// box 128 bytes x box_rows x 1 expert, 128-byte swizzle; rows past an
// expert's end are outside the box's expert and read as zeros.
cudaError_t q_weight_map(CUtensorMap *m, const uint8_t *codes, int n_exp, int rows, int cols, int box_rows) {
    if (!codes || n_exp == 0) {
        memset(m, 0, sizeof *m);
        return cudaSuccess;
    }
    cuuint64_t dims[3] = {(cuuint64_t)(cols / 2), (cuuint64_t)rows, (cuuint64_t)n_exp};
    cuuint64_t strides[2] = {(cuuint64_t)(cols / 2), (cuuint64_t)rows * (cuuint64_t)(cols / 2)};
    cuuint32_t box[3] = {128, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = q_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(codes), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

size_t q_smem_bytes() {
    return 1024 + (size_t)kQStages * kQStageBytes + kQSmTiles * 16 + kQEpiWarps * kQN * 4 + 256;
}

}  // namespace

int mxf4_nqe(int K) { return 2 * ((K + kQK - 1) / kQK); }

size_t mxf4_scales_bytes(const BlockParams &bp) {
    const int ns = bp.n_shared ? 1 : 0;
    auto one = [](int n_exp, int rows, int cols, bool gu) {
        const int rpb = gu ? kQN / 2 : kQN;
        return ((size_t)n_exp * ((rows + rpb - 1) / rpb) * mxf4_nqe(cols) * 1024 + 255) & ~(size_t)255;
    };
    return one(bp.E, bp.F, bp.H, true) + one(ns, bp.F, bp.H, true) + one(bp.E, bp.H, bp.F, false) +
           one(ns, bp.H, bp.F, false);
}

cudaError_t mxf4_prepare(const BlockParams &bp, const MatPtrs &gate, const MatPtrs &up, const MatPtrs &down,
                         uint8_t *buf, Mxf4Weights *out, cudaStream_t st) {
    MOE_CUDA_TRY(q_get_encoder());
    const int E = bp.E, ns = bp.n_shared ? 1 : 0;
    Mxf4Weights &w = *out;
    MOE_CUDA_TRY(q_weight_map(&w.gu.b[0], gate.codes, E, bp.F, bp.H, kQN / 2));
    MOE_CUDA_TRY(q_weight_map(&w.gu.b[1], up.codes, E, bp.F, bp.H, kQN / 2));
    MOE_CUDA_TRY(q_weight_map(&w.gu.b[2], ns ? gate.sh_codes : nullptr, ns, bp.F, bp.H, kQN / 2));
    MOE_CUDA_TRY(q_weight_map(&w.gu.b[3], ns ? up.sh_codes : nullptr, ns, bp.F, bp.H, kQN / 2));
    MOE_CUDA_TRY(q_weight_map(&w.dn.b[0], down.codes, E, bp.H, bp.F, kQN));
    w.dn.b[1] = w.dn.b[0];
    MOE_CUDA_TRY(q_weight_map(&w.dn.b[2], ns ? down.sh_codes : nullptr, ns, bp.H, bp.F, kQN));
    w.dn.b[3] = w.dn.b[2];
    auto pack = [&](const uint8_t *s0, const uint8_t *s1, int n_exp, int rows, int cols, bool gu) -> const uint8_t * {
        if (!n_exp) return nullptr;
        const int rpb = gu ? kQN / 2 : kQN;
        const size_t n = (size_t)n_exp * ((rows + rpb - 1) / rpb) * mxf4_nqe(cols) * 1024;
        const int blocks = (int)((n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192);
        moe_mxf4_pack_kernel<<<blocks, 256, 0, st>>>(s0, s1, n_exp, rows, cols, gu ? 1 : 0, mxf4_nqe(cols), buf, n);
        const uint8_t *r = buf;
        buf += (n + 255) & ~(size_t)255;
        return r;
    };
    w.gu.bsf = pack(gate.scales, up.scales, E, bp.F, bp.H, true);
    w.gu.bsf_sh = pack(gate.sh_scales, up.sh_scales, ns, bp.F, bp.H, true);
    w.dn.bsf = pack(down.scales, down.scales, E, bp.H, bp.F, false);
    w.dn.bsf_sh = pack(down.sh_scales, down.sh_scales, ns, bp.H, bp.F, false);
    w.gu.row_blocks = (bp.F + kQN / 2 - 1) / (kQN / 2);
    w.dn.row_blocks = (bp.H + kQN - 1) / kQN;
    w.gu.nqe = mxf4_nqe(bp.H);
    w.dn.nqe = mxf4_nqe(bp.F);
    return cudaGetLastError();
}

cudaError_t launch_mxf4_stage(const BlockParams &bp, const Workspace &ws, const MatPtrs &gate, const MatPtrs &up,
                              const MatPtrs &down, const Mxf4Weights &w, int T, bool gateup, cudaStream_t st) {
    MOE_CUDA_TRY(q_get_encoder());
    static PerDevice<int> sms;
    static PerDevice<bool> done_g, done_d;
    int dev = 0;
    MOE_CUDA_TRY(current_device_slot(&dev));
    int &n_sm = sms.v[dev];
    if (!n_sm) MOE_CUDA_TRY(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
    bool &done = (gateup ? done_g : done_d).v[dev];
    if (!done) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(gateup ? moe_mxf4_kernel<true> : moe_mxf4_kernel<false>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)q_smem_bytes()));
        done = true;
    }
    const int R = T * (bp.K + bp.n_shared);
    int tiles = (R + kQM - 1) / kQM + bp.E + bp.n_shared;
    if (tiles > ws.max_tiles) tiles = ws.max_tiles;
    const Mxf4Side &side = gateup ? w.gu : w.dn;
    Mxf4Maps m;
    for (int i = 0; i < 4; i++) m.b[i] = side.b[i];
    const int K = gateup ? bp.H : bp.F;
    const uint8_t *acodes = gateup ? ws.xq : ws.hq;
    for (int i = 0; i < 3; i++) MOE_CUDA_TRY(q_codes_map(&m.a[i], acodes, (size_t)R, K, 32 << i, true));
    m.bsf = side.bsf;
    m.bsf_sh = side.bsf_sh;
    m.asf = gateup ? ws.xsf : ws.hsf;
    m.row_blocks = side.row_blocks;
    m.nqe = side.nqe;
    if (gateup) {
        // x_hat -> route-ordered FP4 codes and the tiles' scale atoms
        if (bp.H > 32 * 32 * kGatherMaxBlocks) return cudaErrorInvalidValue;
        moe_mxf4_gather_kernel<<<dim3(tiles, kQM / kGatherRowsPerCta), 32 * kGatherRowsPerCta, 0, st>>>(
            ws, bp.H, ws.xq, ws.xsf, w.gu.nqe);
        MOE_CUDA_TRY(cudaGetLastError());
        Mxf4Args ag{bp, ws, gate, up, bp.H, bp.F, ws.hq, ws.hsf, w.dn.nqe};
        const long items = (long)tiles * w.gu.row_blocks;
        moe_mxf4_kernel<true><<<(unsigned)(items < n_sm ? items : n_sm), kQThreads, q_smem_bytes(), st>>>(ag, m);
    } else {
        Mxf4Args ad{bp, ws, down, down, bp.F, bp.H, nullptr, nullptr, 0};
        const long items = (long)tiles * w.dn.row_blocks;
        moe_mxf4_kernel<false><<<(unsigned)(items < n_sm ? items : n_sm), kQThreads, q_smem_bytes(), st>>>(ad, m);
    }
    return cudaGetLastError();
}
