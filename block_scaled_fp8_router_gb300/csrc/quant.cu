// quant.cu -- fused amax / scale / E4M3 block quantiser.
//
// Block-scaled FP8 as in the DeepSeek-V3 recipe that the prime-rl post
// ("RL at 1T Scale", section "FP8 training") trains with: one fp32 scale per
// 1x128 activation tile or 128x128 weight block, s = amax / 448, codes =
// E4M3(v / s) rounded to nearest even and saturated.
//
// HBM-bound: 2 bytes read and 1 + 4/128 (1x128) or 1 + 4/16384 (128x128)
// bytes written per element.  Each 16-byte load carries 8 bf16; a 1x128 block
// is 16 lanes of one half-warp (amax by 4 shuffles), a 128x128 block is one
// 256-thread CTA holding its 64 values per thread in registers between the
// amax pass and the encode pass (the block is read from HBM once).
//
// MX = true is the power-of-two variant (the scale format of the hardware
// block-scaled MMA, UE8M0): the block scale is the smallest power of two
// 2^p with amax <= 448 * 2^p, stored as the biased exponent byte p + 127;
// codes are v / 2^p (an exact division), so none saturates.
#include "common.cuh"

namespace moe {

// biased exponent of the UE8M0 block scale, read off amax's bits:
// amax = 1.m * 2^E needs p = E - 8 (448 = 1.75 * 2^8), one more when
// 1.m > 1.75; subnormal amax clamps to p = -127 (exponent byte 0)
__device__ __forceinline__ uint32_t ue8m0_exp(float amax)
{
    const uint32_t bits = __float_as_uint(amax);
    const int32_t ef = (int32_t)(bits >> 23);
    if (amax == 0.0f) return 127u;
    if (ef == 0) return 0u;
    int32_t e = ef - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return (uint32_t)(e < 0 ? 0 : (e > 254 ? 254 : e));
}

__device__ __forceinline__ float ue8m0_value(uint32_t e)
{
    return e == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);   // 2^(e-127)
}

// the block's scale value; *stored is the fp32 scale or the exponent byte
template <bool MX>
__device__ __forceinline__ float rule_scale(float amax, uint32_t &e8)
{
    if (MX) {
        e8 = ue8m0_exp(amax);
        return ue8m0_value(e8);
    }
    e8 = 0;
    return block_scale(amax);
}

template <bool MX>
__device__ __forceinline__ void store_scale(void *scales, int64_t i, float s, uint32_t e8)
{
    if (MX) reinterpret_cast<uint8_t *>(scales)[i] = (uint8_t)e8;
    else reinterpret_cast<float *>(scales)[i] = s;
}

// One half-warp per 1x128 block, each lane's 16 bytes of the next QD - 1
// blocks in flight: every lane copies its piece of a block into its own
// slot of a QD-deep shared-memory ring with cp.async (no registers held,
// and no barrier: a lane reads back only its own slots).  A half-warp's
// blocks are hw, hw + nhw, ...; their (row, column block) advance by the
// fixed quotient and remainder of nhw / nbc.
constexpr int QD = 8;

template <bool MX>
__global__ void __launch_bounds__(256) quant_1x128_kernel(const uint16_t *__restrict__ src, int64_t rows,
                                                          int64_t cols, int64_t ld, uint8_t *__restrict__ q,
                                                          void *__restrict__ scales)
{
    __shared__ __align__(16) uint4 ring[QD][256];
    const int nbc = (int)(cols >> 7);
    const int tid = threadIdx.x, lane = tid & 31;
    const int sub = lane & 15;
    const unsigned half_mask = 0xFFFFu << (lane & 16);
    const int64_t hw = (blockIdx.x * (int64_t)blockDim.x + tid) >> 4;
    const int64_t nhw = ((int64_t)gridDim.x * blockDim.x) >> 4;
    const int64_t dr = nhw / nbc;
    const int dc = (int)(nhw - dr * nbc);
    auto advance = [&](int64_t &r, int &cb) {
        cb += dc;
        r += dr;
        if (cb >= nbc) {
            cb -= nbc;
            r++;
        }
    };
    int64_t ir = hw / nbc;                       // the next block to copy
    int icb = (int)(hw - ir * nbc);
    int64_t pr = ir;                             // the next block to encode
    int pcb = icb;
    auto issue = [&](int slot) {
        if (ir < rows) cp_async16_zfill(&ring[slot][tid], src + ir * ld + icb * 128 + sub * 8, true);
        cp_async_commit();
        advance(ir, icb);
    };
#pragma unroll
    for (int i = 0; i < QD - 1; i++) issue(i);
    for (int i = 0; pr < rows; i++) {
        issue((i + QD - 1) % QD);
        cp_async_wait<QD - 1>();                 // this lane's piece of block i
        float v[8];
        unpack_bf16x8(ring[i % QD][tid], v);
        float amax = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                           fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(half_mask, amax, o, 16));
        uint32_t e8;
        const float s = rule_scale<MX>(amax, e8);
        *reinterpret_cast<uint2 *>(q + pr * cols + pcb * 128 + sub * 8) = e4m3x8_scaled<1>(v, s);
        if (sub == 0) store_scale<MX>(scales, pr * nbc + pcb, s, e8);
        advance(pr, pcb);
    }
    cp_async_wait<0>();
}

template <bool MX>
__global__ void __launch_bounds__(256) quant_128x128_kernel(const uint16_t *__restrict__ src, int64_t cols,
                                                            int64_t ld, uint8_t *__restrict__ q,
                                                            void *__restrict__ scales)
{
    __shared__ float warp_amax[8];
    const int64_t nbc = cols >> 7;
    const int64_t b = blockIdx.x;
    const int64_t br = b / nbc, bc = b - br * nbc;
    const int tid = threadIdx.x, tr = tid >> 4, tc = tid & 15;
    uint4 raw[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int64_t r = br * 128 + tr + 16 * i;
        raw[i] = __ldcs(reinterpret_cast<const uint4 *>(src + r * ld + bc * 128 + tc * 8));
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        float v[8];
        unpack_bf16x8(raw[i], v);
#pragma unroll
        for (int j = 0; j < 8; j++) amax = fmaxf(amax, fabsf(v[j]));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((tid & 31) == 0) warp_amax[tid >> 5] = amax;
    __syncthreads();
    amax = warp_amax[0];
#pragma unroll
    for (int w = 1; w < 8; w++) amax = fmaxf(amax, warp_amax[w]);
    uint32_t e8;
    const float s = rule_scale<MX>(amax, e8);
#pragma unroll
    for (int i = 0; i < 8; i++) {
        float v[8];
        unpack_bf16x8(raw[i], v);
        const uint2 out = e4m3x8_scaled<1>(v, s);
        const int64_t r = br * 128 + tr + 16 * i;
        *reinterpret_cast<uint2 *>(q + r * cols + bc * 128 + tc * 8) = out;
    }
    if (tid == 0) store_scale<MX>(scales, b, s, e8);
}

} // namespace moe

using namespace moe;

namespace moe {

template <bool MX>
static moe_status quant_launch(const uint16_t *src, int64_t rows, int64_t cols, int64_t ld_src, int block_rows,
                               uint8_t *q, void *scales, void *stream)
{
    if (rows < 0 || cols <= 0 || cols % 128 != 0 || ld_src < cols) return MOE_ERR_SHAPE;
    if (block_rows != 1 && block_rows != 128) return MOE_ERR_SHAPE;
    if (block_rows == 128 && rows % 128 != 0) return MOE_ERR_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!src || !q || !scales) return MOE_ERR_NULL;
    if (!aligned16(src) || !aligned16(q) || (ld_src * 2) % 16 != 0) return MOE_ERR_ALIGN;
    cudaStream_t st = as_stream(stream);
    if (block_rows == 1) {
        const int64_t nblocks = rows * (cols / 128);
        // one resident wave (six CTAs per SM: 6 x 32 KB of rings, 40
        // registers), each half-warp streaming many blocks through its ring
        int64_t grid = (nblocks + 15) / 16;
        const int64_t cap = (int64_t)sm_count() * 6;
        if (grid > cap) grid = cap;
        quant_1x128_kernel<MX><<<(unsigned)grid, 256, 0, st>>>(src, rows, cols, ld_src, q, scales);
    } else {
        const int64_t nblocks = (rows / 128) * (cols / 128);
        if (nblocks > 0x7FFFFFFFLL) return MOE_ERR_SHAPE;
        quant_128x128_kernel<MX><<<(unsigned)nblocks, 256, 0, st>>>(src, cols, ld_src, q, scales);
    }
    return launch_status();
}

} // namespace moe

MOE_API moe_status fp8_block_quant(const uint16_t *src, int64_t rows, int64_t cols, int64_t ld_src,
                                   int block_rows, uint8_t *q, float *scales, void *stream)
{
    return quant_launch<false>(src, rows, cols, ld_src, block_rows, q, scales, stream);
}

MOE_API moe_status fp8_block_quant_ue8m0(const uint16_t *src, int64_t rows, int64_t cols, int64_t ld_src,
                                         int block_rows, uint8_t *q, uint8_t *scale_exp, void *stream)
{
    return quant_launch<true>(src, rows, cols, ld_src, block_rows, q, scale_exp, stream);
}
