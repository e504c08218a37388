// moe_attn_gemm.cu -- the attention projections of a prefill block as a dense
// bf16 GEMM on the tensor cores (goosedump gpt_oss.rs prefill_attention_layer:
// `matrix_matrix_triple` for the query, key and value projections of a batch
// of rows, `matrix_matrix` for the output projection).
//
// y[t][r] = sum_k x[t][k] W[r][k] + b[r] for the block's tokens t and the rows
// r of up to three matrices laid end to end (Wq, Wk, Wv; or Wo alone).  One
// CTA per (TN weight rows, 128 tokens) tile, TN = 256, or 128 when twice the
// tiles still make one wave:
//  * warp 0 (one lane): per 64-element k-block, one TMA copy of the tokens'
//    activations (128 rows x 128 B) and one of the weight rows (TN rows x
//    128 B), both 128-byte swizzled, into a 4-stage ring;
//  * warp 1 (one lane; it owns the TN TMEM columns): four
//    tcgen05.mma.cta_group::1.kind::f16 (M = 128 tokens, N = TN rows,
//    K = 16, bf16 operands, fp32 accumulator in TMEM) per k-block, each
//    stage released by tcgen05.commit;
//  * warps 2..5: the epilogue, one TMEM lane quarter (32 tokens) each:
//    tcgen05.ld of 32 columns at a time, + bias (+ residual), stores.
// Every wait is bounded (about 2 s) and reports through the plan's status
// word; on a failure the MMAs already issued complete before TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "moe_common.cuh"

namespace {

constexpr int kGM = 128;                 // tokens per tile (TMEM lanes)
constexpr int kGN = 256;                 // weight rows per tile (TMEM columns): 256, or 128 when that fills more SMs
constexpr int kGK = 64;                  // elements per k-block: one 128-byte swizzle row
constexpr int kGStages = 4;
constexpr int kGABytes = kGM * kGK * 2;  // 16 KB
constexpr int kGBBytes = kGN * kGK * 2;  // 32 KB (the stage's room; an N = 128 tile uses half)
constexpr int kGThreads = 6 * 32;
constexpr uint64_t kGWaitNs = 2000000000ull;

struct GemmMaps {
    CUtensorMap a;     // activations [n][K]
    CUtensorMap b[3];  // the matrices [rows_i][K]
};

__device__ __forceinline__ uint32_t g_smem(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ uint64_t g_time() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void g_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(g_smem(b)), "r"(count));
}
__device__ __forceinline__ void g_expect(uint64_t *b, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(g_smem(b)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool g_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(g_smem(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: false (and the status word set) after about 2 s, or when a
// failure was reported elsewhere first; drain: only the time limit ends it.
__device__ bool g_wait(uint64_t *b, uint32_t parity, int32_t *status, int where, bool drain = false) {
    if (g_try(b, parity)) return true;
    const uint64_t t0 = g_time();
    for (uint32_t i = 0;; i++) {
        if (g_try(b, parity)) return true;
        if ((i & 63) == 63) {
            if (!drain && *(volatile int32_t *)status != 0) return false;
            if (g_time() - t0 > kGWaitNs) {
                set_device_error(status, MOE_DEV_WAIT_TIMEOUT, where);
                return false;
            }
        }
    }
}
__device__ __forceinline__ void g_tma(void *dst, const CUtensorMap *m, uint64_t *bar, int x, int y, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%3, %4}], [%2], %5;" ::"r"(g_smem(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(g_smem(bar)), "r"(x), "r"(y), "l"(pol)
        : "memory");
}
// UMMA shared-memory descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t g_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)2 << 61;            // SWIZZLE_128B
    return d;
}
// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major, M x N.
constexpr uint32_t g_idesc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void g_mma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(dtmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void g_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(g_smem(bar))
                 : "memory");
}
__device__ __forceinline__ void g_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void g_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
// 32 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void g_ld32(uint32_t taddr, float v[32]) {
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

// Tile blockIdx.x over the matrices' TN-row tiles (a tile never spans two
// matrices), tokens 128 blockIdx.y .. + 127.
template <int TN>
__global__ void __launch_bounds__(kGThreads, 1) moe_attn_gemm_kernel(const __grid_constant__ AttnGemm g,
                                                                      const __grid_constant__ GemmMaps maps) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = smem, *sB = smem + kGStages * kGABytes;
    __shared__ __align__(8) uint64_t full[kGStages], empty[kGStages], acc_full, drain;
    __shared__ uint32_t tmem_slot;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this tile's matrix and rows
    const int starts[3] = {0, g.r1, g.r2}, ends[3] = {g.r1, g.r2, g.rows};
    int m = 0, t = blockIdx.x;
    for (; m < 2; m++) {
        const int nt = (ends[m] - starts[m] + TN - 1) / TN;
        if (t < nt) break;
        t -= nt;
    }
    const int n0 = t * TN, mrows = ends[m] - starts[m], m0 = blockIdx.y * kGM;
    const int nkb = (g.K + kGK - 1) / kGK;
    int32_t *status = g.status;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGStages; s++) {
            g_init(&full[s], 1);
            g_init(&empty[s], 1);
        }
        g_init(&acc_full, 1);
        g_init(&drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(g_smem(&tmem_slot)),
                     "n"(TN));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    g_fence_before();
    __syncthreads();
    g_fence_after();
    const uint32_t tmem = tmem_slot;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the activations come from the previous kernel
    asm volatile("griddepcontrol.launch_dependents;");

    if (warp == 0) {
        if (lane == 0) {
            uint64_t pol;  // the weight tiles are read once per token tile: theirs go first
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
            int issued = 0;
            for (int kb = 0; kb < nkb; kb++) {
                const int s = kb % kGStages;
                if (kb >= kGStages && !g_wait(&empty[s], ((kb / kGStages) - 1) & 1, status, 70)) break;
                g_expect(&full[s], kGABytes + TN * kGK * 2);
                g_tma(sA + s * kGABytes, &maps.a, &full[s], kb * kGK, m0, 0ull);
                g_tma(sB + s * kGBBytes, &maps.b[m], &full[s], kb * kGK, n0, pol);
                issued++;
            }
            // copies still in flight land before the CTA's shared memory goes
            const uint64_t t0 = g_time();
            for (int kb = max(0, issued - kGStages); kb < issued; kb++)
                while (!g_try(&full[kb % kGStages], (kb / kGStages) & 1))
                    if (g_time() - t0 > kGWaitNs) {
                        set_device_error(status, MOE_DEV_WAIT_TIMEOUT, 71);
                        kb = issued;
                        break;
                    }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = g_idesc(kGM, TN);
            bool ok = true;
            for (int kb = 0; kb < nkb; kb++) {
                const int s = kb % kGStages;
                if (!g_wait(&full[s], (kb / kGStages) & 1, status, 72)) {
                    ok = false;
                    break;
                }
                g_fence_after();
                const uint32_t a_addr = g_smem(sA + s * kGABytes), b_addr = g_smem(sB + s * kGBBytes);
#pragma unroll
                for (int k = 0; k < kGK / 16; k++)
                    g_mma(tmem, g_desc(a_addr + 32 * k), g_desc(b_addr + 32 * k), idesc, (kb | k) != 0);
                g_commit(&empty[s]);
            }
            if (ok) {
                g_commit(&acc_full);
            } else {
                // the MMAs already issued finish before TMEM is released
                g_commit(&drain);
                g_wait(&drain, 0, status, 73, true);
            }
        }
    } else {
        // epilogue: warp w - 2 reads TMEM lanes 32 (w - 2) .. + 31 (the warp's
        // lane quarter is fixed by its index modulo 4)
        const int q = warp & 3, tok = m0 + 32 * q + lane;
        if (g_wait(&acc_full, 0, status, 74)) {
            g_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16);
            const float *bias = g.bias[m];
#pragma unroll 1
            for (int c0 = 0; c0 < TN; c0 += 32) {
                if (n0 + c0 >= mrows) break;  // past the matrix (whole 32-row chunks: rows are multiples of 32)
                float v[32];
                g_ld32(taddr + c0, v);
                if (tok >= g.n) continue;
                const int row = starts[m] + n0 + c0;  // row of the concatenated outputs
#pragma unroll
                for (int c = 0; c < 32; c++) v[c] += __ldg(bias + n0 + c0 + c);
                if (g.kind == 0) {
                    float4 *dst = reinterpret_cast<float4 *>(g.raw + (size_t)tok * g.rows + row);
#pragma unroll
                    for (int k = 0; k < 8; k++) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                } else {
                    const uint4 *rp = reinterpret_cast<const uint4 *>(g.res + (size_t)tok * g.rows + row);
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        const uint4 rv = rp[k];
                        const uint32_t w[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            v[8 * k + 2 * e] += bf16_to_f32((uint16_t)(w[e] & 0xFFFFu));
                            v[8 * k + 2 * e + 1] += bf16_to_f32((uint16_t)(w[e] >> 16));
                        }
                    }
                    if (g.out_bf16) {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(g.out) + (size_t)tok * g.rows + row);
#pragma unroll
                        for (int k = 0; k < 4; k++) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; e++) {
                                const __nv_bfloat16 lo = __float2bfloat16_rn(v[8 * k + 2 * e]);
                                const __nv_bfloat16 hi = __float2bfloat16_rn(v[8 * k + 2 * e + 1]);
                                w[e] = (uint32_t)*reinterpret_cast<const uint16_t *>(&lo) |
                                       ((uint32_t)*reinterpret_cast<const uint16_t *>(&hi) << 16);
                            }
                            dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(g.out) + (size_t)tok * g.rows + row);
#pragma unroll
                        for (int k = 0; k < 8; k++)
                            dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                    }
                }
            }
        }
    }
    g_fence_before();
    __syncthreads();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(TN));
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t gemm_encoder() {
    if (g_encode) return cudaSuccess;
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

// bf16 [rows][K], box 64 elements (128 B) x box_rows, 128-byte swizzle.
cudaError_t gemm_map(CUtensorMap *m, const uint16_t *base, int rows, int K, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kGK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool attn_gemm_supported(int K, int rows) {
    // TMA: 16-byte row strides; the epilogue's 32-row chunks and 16-byte stores
    return K % 8 == 0 && rows % 32 == 0;
}

cudaError_t launch_attn_gemm(const AttnGemm &g, cudaStream_t st) {
    static PerDevice<bool> opted;
    static PerDevice<int> sms;
    int dev = 0;
    MOE_CUDA_TRY(current_device_slot(&dev));
    const int smem = 1024 + kGStages * (kGABytes + kGBBytes);
    if (!opted.v[dev]) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(moe_attn_gemm_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        MOE_CUDA_TRY(cudaFuncSetAttribute(moe_attn_gemm_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms.v[dev], cudaDevAttrMultiProcessorCount, dev));
        opted.v[dev] = true;
    }
    MOE_CUDA_TRY(gemm_encoder());
    const int starts[3] = {0, g.r1, g.r2}, ends[3] = {g.r1, g.r2, g.rows};
    const int mt = (g.n + kGM - 1) / kGM;
    // 256-row tiles, or 128-row ones when twice as many tiles still make one wave
    int tiles256 = 0, tiles128 = 0;
    for (int i = 0; i < 3; i++) {
        const int rows = ends[i] - starts[i];
        if (rows <= 0) continue;
        tiles256 += (rows + 255) / 256;
        tiles128 += (rows + 127) / 128;
    }
    const int tn = tiles128 * mt <= sms.v[dev] ? 128 : 256;
    GemmMaps maps;
    memset(&maps, 0, sizeof maps);
    MOE_CUDA_TRY(gemm_map(&maps.a, g.x, g.n, g.K, kGM));
    for (int i = 0; i < 3; i++) {
        const int rows = ends[i] - starts[i];
        if (rows > 0) MOE_CUDA_TRY(gemm_map(&maps.b[i], g.w[i], rows, g.K, tn));
    }
    const dim3 grid(tn == 128 ? tiles128 : tiles256, mt);
    if (tn == 128) return launch_pdl(moe_attn_gemm_kernel<128>, grid, dim3(kGThreads), (size_t)smem, st, g, maps);
    return launch_pdl(moe_attn_gemm_kernel<256>, grid, dim3(kGThreads), (size_t)smem, st, g, maps);
}
