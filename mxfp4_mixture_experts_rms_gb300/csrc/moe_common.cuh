// moe_common.cuh -- shared device helpers and the plan's kernel parameters.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#define MOE_MAX_TOPK 8
#define MOE_MAX_EXPERTS 256

// Device status codes written into MoeWorkspace::status[0]
#define MOE_DEV_OK 0
#define MOE_DEV_WAIT_TIMEOUT 1
#define MOE_DEV_BAD_ROUTE 2

// Pointers to one expert matrix of all experts plus the shared expert.
struct MatPtrs {
    const uint8_t *codes;     // [E][rows][cols/2]
    const uint8_t *scales;    // [E][rows][cols/32]
    const float *bias;        // [E][rows]
    const uint8_t *sh_codes;  // shared expert (index E), may be null
    const uint8_t *sh_scales;
    const float *sh_bias;
    int rows, cols;
};

__device__ __forceinline__ const uint8_t *mat_codes(const MatPtrs &m, int e, int n_experts) {
    return e < n_experts ? m.codes + (size_t)e * m.rows * (m.cols / 2) : m.sh_codes;
}
__device__ __forceinline__ const uint8_t *mat_scales(const MatPtrs &m, int e, int n_experts) {
    return e < n_experts ? m.scales + (size_t)e * m.rows * (m.cols / 32) : m.sh_scales;
}
__device__ __forceinline__ const float *mat_bias(const MatPtrs &m, int e, int n_experts) {
    return e < n_experts ? m.bias + (size_t)e * m.rows : m.sh_bias;
}

// Device-side view of the workspace carved by the host plan.
struct Workspace {
    uint16_t *xhat;        // [T][H] bf16
    uint16_t *xhat_mma;    // [T][H] bf16, pair order of the prefill dequantiser inside each 8-element chunk
    uint16_t *xhat16;      // [T][H] fp16 copy of x_hat (decode GEMV operand)
    int32_t *ids;          // [T][K]
    float *route_w;        // [T][K]
    int32_t *counts;       // [E + 1] (index E: shared expert)
    int32_t *offsets;      // [E + 2]
    int32_t *perm_token;   // [R]
    int32_t *perm_slot;    // [R]
    float *perm_w;         // [R]
    int32_t *loc;          // [T][K + n_shared]
    int4 *tiles;           // [max_tiles]: (expert, route start, route count, cache slot or 0)
    int32_t *n_tiles;      // [1]
    uint16_t *h;           // [R][F] bf16 (decode: natural order, bf16-activation plans only; prefill: pair order)
    uint16_t *h16;         // [R][F] fp16 h of the decode GEMVs (natural order)
    float *y;              // [R][H] weighted expert outputs
    uint16_t *xs;          // [R][H] x_hat rows in route order (grouped GEMM operand, fp16 or bf16; aliases y,
                           //         which is written only after the gate/up GEMM has read these)
    float *logits;         // [T][E] router logits (fp32) of the routing kernel
    float *lbound;         // [T][E] their rounding-error bounds
    float *xnorm;          // [T] upper bounds of |x_hat| (large-batch routing)
    float *wnorm;          // [E] upper bounds of the router rows' |w| (large-batch routing)
    int32_t *status;       // [4] device error flag + detail
    uint32_t *tickets;     // [T + 1] last-CTA counters of the routing kernel (grid, token groups)
    // FP4-activation grouped GEMM (plans with act_fp4 only)
    uint8_t *xq;           // [R][H/2] FP4 codes of the routes' x_hat rows (aliases y, like xs)
    uint8_t *hq;           // [R][F/2] FP4 codes of h (aliases h16)
    uint8_t *xsf;          // [tiles][nqe(H)][512] scale atoms of xq, per route tile
    uint8_t *hsf;          // [tiles][nqe(F)][512] scale atoms of hq
    int max_tiles;
};

struct BlockParams {
    int H, F, E, K, n_shared;
    float alpha, limit, wscale;
    double eps;
};

// bf16 bits <-> float
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Round a double to bf16 with one rounding (nearest, ties to even), working on
// the IEEE-754 bit pattern: keep 7 fraction bits in the normal range, quantum
// 2^-133 below 2^-126.
__device__ __forceinline__ uint16_t bf16_from_double_rne(double v) {
    unsigned long long b = (unsigned long long)__double_as_longlong(v);
    uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
    unsigned long long a = b & 0x7FFFFFFFFFFFFFFFull;
    if (a > 0x7FF0000000000000ull) return 0x7FC0;            // NaN
    if (a >= (897ull << 52)) {                                 // |v| >= 2^-126
        unsigned long long lsb = (a >> 45) & 1ull;
        a += 0x00000FFFFFFFFFFFull + lsb;                      // 2^44 - 1 + lsb
        a &= ~0x00001FFFFFFFFFFFull;                           // clear 45 bits
        long long ex = (long long)(a >> 52) - 1023;
        if (ex > 127) return sign | 0x7F80;                    // overflow / inf
        return sign | (uint16_t)(((ex + 127) << 7) | ((a >> 45) & 0x7F));
    }
    double m = rint(__longlong_as_double((long long)a) * 0x1p133);  // exact scaling
    return sign | (uint16_t)m;                                 // m in [0, 128]
}

__device__ __forceinline__ void set_device_error(int32_t *status, int code, int detail) {
    if (atomicCAS(status, 0, code) == 0) status[1] = detail;
}

// 8 E2M1 codes of one 32-bit word -> four f16x2 in natural order (hardware conversion)
// (element 2i in the low half of h[i]), exact: byte i holds elements 2i, 2i+1.
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

// FP4 activation encoding of one 32-element block (ds4.c, FP4 activation
// quantisation `dsv4_fp4_act_quantize_row_inplace_cpu`, nearest value as in
// `dsv4_e2m1fn_dequant_cpu`): scale 2^k with k = ceil(log2(amax / 6)), amax at
// least 6 * 2^-126.  For a bf16-valued amax = m * 2^e (m in [1, 2)), k = e - 2
// + (m > 1.5), exactly the ceiling of the float quotient (no division).
// mxq_exponent takes amax (a bf16 value held in a float; NaN elements never
// raise it) and returns k in [-126, 127] (127 for an infinite amax).
__device__ __forceinline__ int mxq_exponent(float amax) {
    const uint32_t ab = max(__float_as_uint(amax) >> 16, 0x01C0u);
    return ab >= 0x7F80u ? 127 : (int)(ab >> 7) - 129 + ((ab & 0x7Fu) > 0x40u ? 1 : 0);
}
// 2^-k as float for k in [-126, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float mxq_inv_scale(int k) {
    return k <= 126 ? __uint_as_float((uint32_t)(127 - k) << 23) : __uint_as_float(0x00400000u);
}
// Four floats -> four E2M1 codes in bits 0..15 (x0 in bits 0..3, x1 in 4..7,
// x2 in 8..11, x3 in 12..15): round to nearest even, magnitudes above 6 (and
// infinities) saturated to 6.  The conversion puts its first source operand
// in the high nibble of its byte.
__device__ __forceinline__ uint32_t e2m1x4(float x0, float x1, float x2, float x3) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "mov.b32 %0, {b0, b1, 0, 0};\n\t}"
        : "=r"(r)
        : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
    return r;
}
// One whole 32-element block held by one thread -> 16 bytes of codes (element
// 2i in the low nibble of byte i) and the E8M0 scale byte k + 127.  Each
// element goes in as fmin(x * 2^-k + 0, 6): exact scaling; +0 turns -0 into +0
// and fmin turns NaN into 6, as the page's sign test and clamp do.
__device__ __forceinline__ uint4 mxq_encode_block(const float (&x)[32], uint32_t &scale_byte) {
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; i++) am = fmaxf(am, fabsf(x[i]));
    const int k = mxq_exponent(am);
    const float inv = mxq_inv_scale(k);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        float f[8];
#pragma unroll
        for (int i = 0; i < 8; i++) f[i] = fminf(fmaf(x[8 * q + i], inv, 0.0f), 6.0f);
        w[q] = e2m1x4(f[0], f[1], f[2], f[3]) | (e2m1x4(f[4], f[5], f[6], f[7]) << 16);
    }
    scale_byte = (uint32_t)(k + 127);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Clamped SwiGLU (gate clamped from above, up to [-L, L]); NaN propagates.
__device__ __forceinline__ float swiglu_clamped(float g, float u, float alpha, float limit) {
    float gc = (g > limit) ? limit : g;
    float uc = (u > limit) ? limit : ((u < -limit) ? -limit : u);
    float glu = gc / (1.0f + expf(-alpha * gc));
    return glu * (uc + 1.0f);
}

// Position of element j inside its 32-element block in the decode-MMA order:
// element 8q + i + 4hh (q, i in 0..3, hh in 0..1) goes to 8q + 2i + hh, so that
// elements (8q+i, 8q+i+4) form one bf16x2 pair, matching the nibble pairs the
// dequantiser extracts from one 32-bit word of codes.
__device__ __forceinline__ int mma_perm_pos(int j) {
    int b = j & ~31, e = j & 31;
    int q = e >> 3, r = e & 7, i = r & 3, hh = r >> 2;
    return b + (q << 3) + (i << 1) + hh;
}

// Host-side setup done once per device (kernel attributes and device
// properties belong to a device, not to the process): the current device's
// slot in a PerDevice table.
constexpr int kMaxDevices = 64;
template <class T>
struct PerDevice {
    T v[kMaxDevices]{};
};
inline cudaError_t current_device_slot(int *dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e == cudaSuccess && (*dev < 0 || *dev >= kMaxDevices)) e = cudaErrorInvalidDevice;
    return e;
}

// Raise a kernel's dynamic shared memory limit to the device maximum, once per
// device (host-side setup; kept out of the per-forward launch sequence).
template <class F>
inline cudaError_t smem_optin_once(F *kernel, PerDevice<bool> &flag) {
    int dev = 0, optin = 0;
    cudaError_t e = current_device_slot(&dev);
    if (e != cudaSuccess || flag.v[dev]) return e;
    bool &done = flag.v[dev];
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
    if (e == cudaSuccess) done = true;
    return e;
}

// Launch with programmatic dependent launch: the kernel may be scheduled while
// its predecessor on the stream drains; it must execute griddepcontrol.wait
// before touching the predecessor's results.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Host+device-visible launch helpers
#define MOE_CUDA_TRY(expr)                                  \
    do {                                                    \
        cudaError_t _e = (expr);                            \
        if (_e != cudaSuccess) return _e;                   \
    } while (0)

// x_hat copies the routing kernels write besides the natural bf16 one, as
// the expert kernels of the chosen path read them.
constexpr int kFormF16 = 1;  // fp16 (the GEMVs, the fp16 grouped GEMM)
constexpr int kFormMma = 2;  // bf16 in the grouped GEMM's pair order (its bf16 variant)

// The thread's last-error message (moe_last_error), set from any translation unit.
int moe_fail_status(int code, const char *fmt, ...);
void moe_set_error(const char *fmt, ...);
// Enqueue the recording of T tokens' routes of one layer into a locality profiler.
// Dense bf16 GEMM on the tensor cores for the attention projections of a
// prefill block (csrc/moe_attn_gemm.cu): for each token t < n and row r of up
// to three matrices laid end to end (w[0] rows [0, r1), w[1] [r1, r2), w[2]
// [r2, rows)), y = sum_k x[t][k] w[r][k] + bias[r]; kind 0 writes y to
// raw[t][r] (fp32), kind 1 writes res[t][r] + y to out[t][r] (fp32, or bf16).
struct AttnGemm {
    int n, K, rows, r1, r2;
    const uint16_t *x;  // [n][K] bf16, 16-byte aligned rows
    const uint16_t *w[3];
    const float *bias[3];
    int kind;
    float *raw;
    const uint16_t *res;
    void *out;
    int out_bf16;
    int32_t *status;  // bounded waits that gave up
};
bool attn_gemm_supported(int K, int rows);
cudaError_t launch_attn_gemm(const AttnGemm &g, cudaStream_t st);

struct moe_locality;
cudaError_t locality_enqueue(moe_locality *p, int layer, const int32_t *ids, const float *w, int T,
                             long long first_pos, cudaStream_t st);

// Launchers implemented in the .cu files (host side).
int route_ticket_count(int T);
cudaError_t launch_rms_norm_rows(const uint16_t *x, const float *gamma, int T, int H, double eps, uint16_t *xhat,
                                 float *xnorm_scratch, int32_t *count_scratch, cudaStream_t st);
cudaError_t launch_route(const BlockParams &bp, const Workspace &ws, const uint16_t *x,
                         const float *gamma, const uint16_t *router_w, const float *router_b,
                         int T, int32_t *ids_out, float *rw_out, uint16_t *xhat_out, int tile_rows,
                         int router_exact, int forms, cudaStream_t st);
// x_bf16 / h_bf16: the gate/up (down) GEMV reads bf16 activations instead of fp16.
// stall (test hook, gate/up only): the consumers first wait on a barrier that
// nothing completes, so the bounded wait runs out and the kernel reports
// MOE_DEV_WAIT_TIMEOUT (detail 59) and drains.
cudaError_t launch_decode_stage(const BlockParams &bp, const Workspace &ws, const MatPtrs &a0,
                                const MatPtrs &a1, bool gateup, int T, int nt, bool x_bf16, bool h_bf16,
                                int stall, bool slot_index, cudaStream_t st);
// dst = bf16_rne(src), n elements (any n; 16-byte aligned pointers)
cudaError_t launch_cast_bf16(const float *src, uint16_t *dst, size_t n, cudaStream_t st);
cudaError_t launch_mx_fp4_quantize(const uint16_t *x, size_t n_blocks, uint8_t *codes, uint8_t *scales,
                                   cudaStream_t st);
// Expert cache (plans with expert_cache_slots): device tables owned by the plan.
struct CacheTables {
    int32_t *slot_of;    // [E]: slot of each expert, -1 when not resident
    int32_t *expert_of;  // [slots]: expert in each slot, -1 when empty
    long long *stamp;    // [slots]: index of the last forward that used the slot, -1 when empty
    int2 *miss;          // [E]: (expert, slot) of this forward's misses
    int32_t *n_miss;     // [1]
    long long *stats;    // [3]: hits, misses, forwards (cumulative)
    long long *fwd;      // [1]: index of the last forward
    int slots;
};
// The arrays a slot holds: codes, scales and biases of gate, up and down.
constexpr int kCacheArrays = 9;
struct CacheArrays {
    const uint4 *src[kCacheArrays];  // the store's arrays (expert-major), device-accessible
    uint4 *dst[kCacheArrays];        // the slots' arrays (slot-major)
    long long words[kCacheArrays];   // 16-byte words per expert
};
cudaError_t launch_cache_assign(const CacheTables &c, const BlockParams &bp, const Workspace &ws, cudaStream_t st);
cudaError_t launch_cache_copy(const CacheTables &c, const CacheArrays &arr, cudaStream_t st);

cudaError_t launch_combine(const BlockParams &bp, const Workspace &ws, const uint16_t *x, int T,
                           void *out, int out_bf16, cudaStream_t st);
// What the grouped GEMM reads its weights through: TMA descriptors of the
// packed codes and the scales repacked into 128-byte chunks (the two E8M0
// bytes of one 64-element k-block for 64 consecutive rows, chunk (block b,
// k-block kb) at byte ((b * nkb) + kb) * 128, b = expert * row_blocks + row / 64).
// Index [0] routed A0, [1] routed A1, [2] shared A0, [3] shared A1.
struct TmaMaps {
    CUtensorMap m[4];
    const uint8_t *sc[4];
    int row_blocks;     // 64-row blocks per expert matrix
};
struct PrefillMaps {
    TmaMaps gateup, down;
};
cudaError_t prefill_make_maps(const BlockParams &bp, const MatPtrs &gate, const MatPtrs &up, const MatPtrs &down,
                              PrefillMaps *out);
// Bytes of the repacked scale buffer, and the repack itself (enqueued on st;
// fills the sc / row_blocks fields of *out).
size_t prefill_scales_bytes(const BlockParams &bp);
cudaError_t prefill_pack_scales(const BlockParams &bp, const MatPtrs &gate, const MatPtrs &up, const MatPtrs &down,
                                uint8_t *buf, PrefillMaps *out, cudaStream_t st);
// f16: the fp16-operand variant (E8M0 exponents in [104, 140], fp16-range activations).
cudaError_t launch_prefill_stage(const BlockParams &bp, const Workspace &ws, const MatPtrs &a0,
                                 const MatPtrs &a1, bool gateup, int T, const TmaMaps &maps, bool f16,
                                 cudaStream_t st);
// x_hat rows gathered into route order (ws.xs) for the grouped GEMM.
cudaError_t launch_gather(const BlockParams &bp, const Workspace &ws, int T, bool f16, cudaStream_t st);
int prefill_tile_rows();
cudaError_t launch_dequant(const MatPtrs &m, int expert, int n_experts, float *out, cudaStream_t st);

// Block-scaled FP4 grouped GEMM (tcgen05.mma kind::mxf4).  Per matrix side
// (gate/up, down): TMA maps of the weight codes with 128-byte boxes and the
// weight scales repacked into the 512-byte atoms the kernel copies into
// tensor memory.
struct Mxf4Side {
    CUtensorMap b[4];       // [0] routed gate (or down), [1] routed up, [2] shared gate (or down), [3] shared up
    const uint8_t *bsf;     // routed scale atoms [E][row blocks][nqe][512]
    const uint8_t *bsf_sh;  // the shared expert's
    int row_blocks;         // item row blocks per expert matrix (64 gate/up rows, or 128 down rows)
    int nqe;                // 128-element scale groups per row, rounded up to even
};
struct Mxf4Weights {
    Mxf4Side gu, dn;
};
int mxf4_nqe(int K);
size_t mxf4_scales_bytes(const BlockParams &bp);
// Builds the maps and repacks the scales into buf (mxf4_scales_bytes bytes), enqueued on st.
cudaError_t mxf4_prepare(const BlockParams &bp, const MatPtrs &gate, const MatPtrs &up, const MatPtrs &down,
                         uint8_t *buf, Mxf4Weights *out, cudaStream_t st);
// gateup: x_hat FP4 encoding into route order + the gate/up GEMM (bias, SwiGLU, h's bf16 rounding and FP4
// encoding in the epilogue); otherwise the down GEMM (bias x route weight -> y).
cudaError_t launch_mxf4_stage(const BlockParams &bp, const Workspace &ws, const MatPtrs &gate, const MatPtrs &up,
                              const MatPtrs &down, const Mxf4Weights &w, int T, bool gateup, cudaStream_t st);
cudaError_t launch_scan_scales(const uint8_t *scales, size_t n, int32_t *flag, cudaStream_t st);
