// moe_cast.cu -- the residual stream between stacked blocks: a block's fp32
// output rounded (nearest, ties to even) to the bf16 input of the next block.
#include "moe_common.cuh"

namespace {
// Four elements per thread (one 16-byte load, one 8-byte store), the tail
// element-wise.  Launched as a programmatic dependent of whatever precedes it
// on the stream: it waits for that grid (complete, its writes visible) before
// reading src.
__global__ void __launch_bounds__(256) moe_cast_bf16_kernel(const float *src, uint16_t *dst, size_t n) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t n4 = n / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = reinterpret_cast<const float4 *>(src)[i];
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        reinterpret_cast<uint2 *>(dst)[i] =
            make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
    }
    const size_t t = 4 * n4 + (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t < n) {
        const __nv_bfloat16 b = __float2bfloat16_rn(src[t]);
        dst[t] = *reinterpret_cast<const uint16_t *>(&b);
    }
}
}  // namespace

cudaError_t launch_cast_bf16(const float *src, uint16_t *dst, size_t n, cudaStream_t st) {
    const size_t n4 = n / 4;
    size_t blocks = (n4 + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > 4096) blocks = 4096;
    return launch_pdl(moe_cast_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0, st, src, dst, n);
}
