// moe_mxq.cu -- FP4 activation encoding: bf16 rows -> MXFP4 codes and E8M0
// block scales in the layout the expert weights use, the operand format of a
// block-scaled FP4 tensor-core product.
//
// ds4.c, FP4 activation quantisation (`dsv4_fp4_act_quantize_row_inplace_cpu`
// with its nearest-value step `dsv4_e2m1fn_dequant_cpu`): per 32-element block
// the scale is 2^k, k = ceil(log2(amax / 6)) with amax at least 6 * 2^-126,
// and each element becomes the E2M1 value nearest to x / 2^k clamped to +-6,
// ties to the even code.  Here k comes from amax's bits: amax = m * 2^e with
// m in [1, 2) makes amax / 6 = (m / 1.5) * 2^(e-2), so k = e - 2 + (m > 1.5);
// a bf16 amax (8 significant bits) is never within a float rounding of
// 6 * 2^j without being equal to it, so this is also the ceiling of the
// quotient rounded to float, without a division.  The nearest
// value from the hardware conversion to E2M1 (round to nearest even,
// saturating at +-6).  The scaled value goes in as fmin(x * 2^-k + 0, 6): the
// +0 turns -0 into +0 and fmin turns NaN into 6, the page's answers for both
// (its sign test x < 0 is false for them, and its clamp takes NaN to 6).
#include "moe_common.cuh"

namespace {

// Encode 16-byte chunk u of x (elements 8u..8u+7 of block u / 4: rows are
// contiguous, so blocks are numbered straight through the matrix) into the
// 32-bit code word u; the four lanes of a block meet by shuffles, so the whole
// warp calls this, `active` or not.
__device__ __forceinline__ void encode_chunk(const uint4 v, size_t u, bool active, int lane, uint32_t *codes,
                                             uint8_t *scales) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float xf[8];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        xf[2 * q] = __uint_as_float(w[q] << 16);
        xf[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
    // largest |x| of the block (fmax passes over NaN)
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) am = fmaxf(am, fabsf(xf[i]));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    const int k = mxq_exponent(am);
    const float inv = mxq_inv_scale(k);
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; i++) f[i] = fminf(fmaf(xf[i], inv, 0.0f), 6.0f);  // exact scaling
    const uint32_t out = e2m1x4(f[0], f[1], f[2], f[3]) | (e2m1x4(f[4], f[5], f[6], f[7]) << 16);
    if (active) {
        codes[u] = out;
        if ((lane & 3) == 0) scales[u >> 2] = (uint8_t)(k + 127);
    }
}

// Four lanes per 32-element block, eight elements (one 16-byte load) each; a
// warp reads 512 contiguous bytes per chunk set and writes 128.  Each thread
// issues kU loads before encoding any of them.  Measured on GB300: two loads a
// thread at eight CTAs per SM (all 2048 threads resident) beat four at four,
// eight at three and sixteen at two.
constexpr int kU = 2;           // chunks in flight per thread
constexpr int kCtasPerSm = 8;
__global__ void __launch_bounds__(256, kCtasPerSm) moe_mx_fp4_quantize_kernel(const uint16_t *x, size_t n_chunks,
                                                                      uint32_t *codes, uint8_t *scales) {
    const int lane = threadIdx.x & 31;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    // whole warps walk the loop together, so the group shuffles see all four lanes
    for (size_t u0 = (size_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31u); u0 < n_chunks; u0 += kU * stride) {
        uint4 v[kU];
#pragma unroll
        for (int j = 0; j < kU; j++) {
            const size_t u = u0 + j * stride + lane;
            v[j] = u < n_chunks ? __ldg(reinterpret_cast<const uint4 *>(x) + u) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kU; j++) {
            const size_t u = u0 + j * stride + lane;
            encode_chunk(v[j], u, u < n_chunks, lane, codes, scales);
        }
    }
}

}  // namespace

cudaError_t launch_mx_fp4_quantize(const uint16_t *x, size_t n_blocks, uint8_t *codes, uint8_t *scales,
                                   cudaStream_t st) {
    const size_t n_chunks = 4 * n_blocks;
    // enough CTAs for kU chunks a thread, at most kCtasPerSm per SM of a 152-SM GPU
    size_t grid = (n_chunks + 256 * kU - 1) / (256 * kU);
    if (grid < 1) grid = 1;
    if (grid > 152 * kCtasPerSm) grid = 152 * kCtasPerSm;
    moe_mx_fp4_quantize_kernel<<<(unsigned)grid, 256, 0, st>>>(x, n_chunks, reinterpret_cast<uint32_t *>(codes),
                                                               scales);
    return cudaGetLastError();
}
