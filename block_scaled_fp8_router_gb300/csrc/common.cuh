// common.cuh -- small device/host helpers shared by the libmoe_r3 kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "moe_r3.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

static inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

static inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static inline int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

static inline moe_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// 8 packed bf16 (one 16-byte vector) -> 8 floats, exact
__device__ __forceinline__ void unpack_bf16x8(const uint4 &v, float *f)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// two floats -> packed bf16x2 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

// two floats -> two E4M3 codes (round to nearest even, saturate to +-448),
// `lo` in the low byte
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi)
{
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// block scale of the DeepSeek-V3 recipe: amax / 448 (IEEE division), 1 when
// 0.  For 2^-100 <= amax <= 2^127 the quotient comes from the constant
// RN(1/448) and one fused correction step q + RN(amax - 448 q) / 448 (the
// step Markstein's theorem describes), which equals the IEEE quotient for
// every such binary32 amax (checked exhaustively against IEEE division; see
// the division test); other values take __fdiv_rn.
__device__ __forceinline__ float block_scale(float amax)
{
    if (!(amax >= 0x1p-100f && amax <= 0x1p127f)) {
        const float s = __fdiv_rn(amax, 448.0f);
        return s == 0.0f ? 1.0f : s;
    }
    constexpr float y = 1.0f / 448.0f;
    const float q = __fmul_rn(amax, y);          // never contracted into an FMA
    return fmaf(fmaf(q, -448.0f, amax), y, q);
}

// Division by a block scale with the scale's reciprocal shared by the block,
// giving the correctly rounded v / s (the value of __fdiv_rn(v, s)) on the
// fast path.  y = RN(1/s), q0 = RN(v*y), and each step replaces q by
// q - RN(q*s - v) * y with fused multiply-adds, i.e. q + RN(v - q*s) * y.
// Markstein's theorem (J.-M. Muller et al., Handbook of Floating-Point
// Arithmetic, on division with an FMA): when q is a faithful rounding of v/s
// the residual is exact and one step returns RN(v/s).  q0 can be 1.5 ulp off,
// but one step from it lands within 2^-22 ulp of v/s before rounding, so it
// is faithful: STEPS = 2 is correct for every input.  STEPS = 1 returns
// RN(v/s) for every bf16 v and every scale of the 1 x 128 rule on the fast
// path (checked exhaustively against IEEE division; see the division test).
// The fast path needs 2^-90 <= s <= 2^126 (residuals above the underflow
// threshold for |v / s| >= 2^-12, and a normal reciprocal); other scales,
// inf and NaN take __fdiv_rn.  A quotient below 2^-12 can differ from
// RN(v/s) in its last bits, which does not change its E4M3 code (zero of the
// same sign).  The residual is taken negated, q*s - v, so that a zero
// dividend keeps its sign: -0 gives q0 = -0, residual +0, and
// -0 + (-(+0) * y) = -0.
__device__ __forceinline__ bool fast_scale(float s) { return s >= 0x1p-90f && s <= 0x1p126f; }

template <int STEPS>
__device__ __forceinline__ float div_fast(float v, float s, float y)
{
    float q = __fmul_rn(v, y);                   // never contracted into an FMA
#pragma unroll
    for (int i = 0; i < STEPS; i++) q = fmaf(-fmaf(q, s, -v), y, q);
    return q;
}

// eight values divided by one scale -> eight E4M3 codes (round to nearest
// even, saturated), value 0 in the low byte; one branch per block
template <int STEPS>
__device__ __forceinline__ uint2 e4m3x8_scaled(const float (&v)[8], float s)
{
    float q[8];
    if (fast_scale(s)) {
        const float y = __frcp_rn(s);
#pragma unroll
        for (int i = 0; i < 8; i++) q[i] = div_fast<STEPS>(v[i], s, y);
    } else {
#pragma unroll
        for (int i = 0; i < 8; i++) q[i] = __fdiv_rn(v[i], s);
    }
    uint2 out;
    out.x = (uint32_t)pack_e4m3x2(q[0], q[1]) | ((uint32_t)pack_e4m3x2(q[2], q[3]) << 16);
    out.y = (uint32_t)pack_e4m3x2(q[4], q[5]) | ((uint32_t)pack_e4m3x2(q[6], q[7]) << 16);
    return out;
}

// The reciprocal a block's divisions share: RN(1/s) on the fast path, else 0
// (a fast-path reciprocal is never 0), which sends e4m3x4_div and
// e4m3x2_div to IEEE division.  Computed once per block scale, by the
// thread that forms the scale, when many threads encode with it.
__device__ __forceinline__ float scale_recip(float s) { return fast_scale(s) ? __frcp_rn(s) : 0.0f; }

// four values (v0..v3) divided by one scale s -> four codes (value 0 in the
// low byte), the scale's reciprocal y = scale_recip(s) given
template <int STEPS>
__device__ __forceinline__ uint32_t e4m3x4_div(float v0, float v1, float v2, float v3, float s, float y)
{
    float q[4] = {v0, v1, v2, v3};
    if (y != 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; i++) q[i] = div_fast<STEPS>(q[i], s, y);
    } else {
#pragma unroll
        for (int i = 0; i < 4; i++) q[i] = __fdiv_rn(q[i], s);
    }
    return (uint32_t)pack_e4m3x2(q[0], q[1]) | ((uint32_t)pack_e4m3x2(q[2], q[3]) << 16);
}

// two values (v0 in the low byte) with the reciprocal given
template <int STEPS>
__device__ __forceinline__ uint16_t e4m3x2_div(float v0, float v1, float s, float y)
{
    if (y != 0.0f) return pack_e4m3x2(div_fast<STEPS>(v0, s, y), div_fast<STEPS>(v1, s, y));
    return pack_e4m3x2(__fdiv_rn(v0, s), __fdiv_rn(v1, s));
}

__device__ __forceinline__ void dev_flag(int32_t *status, int32_t bits)
{
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- cp.async (16 bytes, global -> shared; zero fill when !valid) ----
__device__ __forceinline__ uint32_t smem_u32(const void *p);
__device__ __forceinline__ void cp_async16_zfill(void *dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---- mbarrier helpers (shared::cta) ----
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// `timeout_ns` of wall time.  Returns false on expiry.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t timeout_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 64; i++)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

} // namespace moe
