// nvfp4.cu -- NVFP4 quantisation: FP4 E2M1 values, 16-element blocks with
// E4M3 block scales, one fp32 scale per tensor.
//
// The FP4 variant that "RL at 1T Scale: prime-rl Performance Deep Dive"
// lists as future work for training and inference (closing section); the
// format is NVIDIA's NVFP4.  Two passes over the tensor:
//   nvfp4_amax_kernel   amax over the whole tensor (the tensor scale needs
//                       it before any block can be encoded);
//   nvfp4_quant_kernel  one thread per 16-element block: s_enc = 2688 /
//                       amax, block scale byte = e4m3((amax_b / 6) * s_enc),
//                       codes = e2m1(x * (s_enc / scale)), every step one
//                       binary32 operation in that order, so the codes and
//                       scales are exactly determined.
// Both passes are HBM-bound: the input is read twice (2 bytes per element
// each), 0.5 + 1/16 bytes per element are written.
#include <cuda_fp4.h>

#include "common.cuh"
#include "nvfp4_internal.cuh"

namespace moe {

// non-negative binary32 values order as their bit patterns
__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const uint16_t *__restrict__ x, int64_t n8,
                                                         float *__restrict__ amax)
{
    float m = 0.0f;
    const uint4 *x4 = reinterpret_cast<const uint4 *>(x);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        float f[8];
        unpack_bf16x8(__ldg(x4 + i), f);
#pragma unroll
        for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(f[j]));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if ((threadIdx.x & 31) == 0 && m > 0.0f) atomicMax(reinterpret_cast<int *>(amax), __float_as_int(m));
}

__device__ __forceinline__ float e4m3_value(uint8_t b)
{
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(b, __NV_E4M3)));
}

__global__ void __launch_bounds__(256) nvfp4_quant_kernel(const uint16_t *__restrict__ x, int64_t rows, int64_t cols,
                                                          float *__restrict__ tensor_scale, uint8_t *__restrict__ q,
                                                          uint8_t *__restrict__ sc)
{
    const float amax_t = tensor_scale[1];
    const float s_enc = amax_t == 0.0f ? 1.0f : __fdiv_rn(6.0f * 448.0f, amax_t);
    if (blockIdx.x == 0 && threadIdx.x == 0) tensor_scale[0] = s_enc;
    const int64_t nb = cols / 16;
    const int64_t nblocks = rows * nb;
    for (int64_t blk = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; blk < nblocks;
         blk += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = blk / nb, b = blk - r * nb;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + r * cols + b * 16);
        float f[16];
        unpack_bf16x8(__ldg(src), f);
        unpack_bf16x8(__ldg(src + 1), f + 8);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(f[i]));
        const float bd = __fdiv_rn(amax, 6.0f);
        const uint8_t sb = (uint8_t)__nv_cvt_float_to_fp8(__fmul_rn(bd, s_enc), __NV_SATFINITE, __NV_E4M3);
        const float sbv = e4m3_value(sb);
        const float s_elem = sbv == 0.0f ? 0.0f : __fdiv_rn(s_enc, sbv);
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; i++) {
            // element 2i in the low nibble, 2i+1 in the high nibble
            const uint32_t byte = (uint32_t)__nv_cvt_float2_to_fp4x2(
                make_float2(__fmul_rn(f[2 * i], s_elem), __fmul_rn(f[2 * i + 1], s_elem)), __NV_E2M1,
                cudaRoundNearest);
            w[i >> 2] |= (byte & 0xFFu) << (8 * (i & 3));
        }
        *reinterpret_cast<uint2 *>(q + r * (cols / 2) + b * 8) = make_uint2(w[0], w[1]);
        sc[blk] = sb;
    }
}

moe_status nvfp4_quant_blocks(const uint16_t *src, int64_t rows, int64_t cols, float *tensor_scale, uint8_t *q,
                              uint8_t *scales, cudaStream_t st)
{
    const int64_t cap = (int64_t)sm_count() * 8;
    // launched even for rows == 0: it writes the tensor scale (1 for an
    // empty or all-zero tensor)
    int64_t g2 = (rows * (cols / 16) + 255) / 256;
    if (g2 < 1) g2 = 1;
    if (g2 > cap) g2 = cap;
    nvfp4_quant_kernel<<<(unsigned)g2, 256, 0, st>>>(src, rows, cols, tensor_scale, q, scales);
    return launch_status();
}

} // namespace moe

using namespace moe;

MOE_API moe_status fp8_quant_nvfp4(const uint16_t *src, int64_t rows, int64_t cols, uint8_t *q, uint8_t *scales,
                                   float *tensor_scale, void *stream)
{
    if (rows < 0 || cols <= 0 || cols % 16 != 0) return MOE_ERR_SHAPE;
    if (!tensor_scale || (rows > 0 && (!src || !q || !scales))) return MOE_ERR_NULL;
    if (rows > 0 && (!aligned16(src) || !aligned16(q))) return MOE_ERR_ALIGN;
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(tensor_scale, 0, 2 * sizeof(float), st) != cudaSuccess) return MOE_ERR_CUDA;
    const int64_t n8 = rows * cols / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (n8 > 0) {
        int64_t g1 = (n8 + 255) / 256;
        if (g1 > cap) g1 = cap;
        nvfp4_amax_kernel<<<(unsigned)g1, 256, 0, st>>>(src, n8, tensor_scale + 1);
    }
    return nvfp4_quant_blocks(src, rows, cols, tensor_scale, q, scales, st);
}
