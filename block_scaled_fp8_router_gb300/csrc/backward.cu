// backward.cu -- the HBM-bound steps of the expert path's backward pass.
//
// The trainer replays the captured routing ("RL at 1T Scale: prime-rl
// Performance Deep Dive", section "Router replay") and trains through the
// layer with block-scaled FP8 GEMMs (section "FP8 training").  With the ids
// fixed, the backward of the expert path is:
//   combine backward   d_out[r] = g[t,j] * dy[t] (quantised 1x128 for the
//                      dgrad GEMM), d_g[t,j] = <dy[t], out[r]>;
//   GEMM2 dgrad        d_act = d_out W2   (grouped GEMM, grouped_ffn.cu);
//   SwiGLU backward    d_g = d_act * u * silu'(g), d_u = d_act * silu(g),
//                      quantised 1x128 along 2F;
//   GEMM1 dgrad        dx_sorted = dh W13 (grouped GEMM);
//   dispatch backward  dx[t] = sum of its rows' gradients (combine with unit
//                      gates, dispatch.cu).
// The dgrad GEMMs take the weights transposed; fp8_weight_transpose makes
// that copy once per weight update (block quantisation commutes with
// transposition, so it is the quantisation of the transposed weights).
#include "common.cuh"

namespace moe {

// One warp per token: the token's dy row is read once (16 bytes per lane per
// step) and multiplied by each slot's gate; every 128-column block of the
// product is one half-warp (amax by four shuffles) and is written with its
// scale to the slot's sorted row.  The gate gradient is the warp-reduced dot
// of dy with the slot's expert output row.
__global__ void __launch_bounds__(256) combine_backward_kernel(const uint16_t *__restrict__ dy,
                                                               const float *__restrict__ gates,
                                                               const uint16_t *__restrict__ out_sorted,
                                                               const int32_t *__restrict__ slot_to_sorted, int T,
                                                               int k, int d, int64_t A, uint8_t *__restrict__ d_out_q,
                                                               float *__restrict__ d_out_s,
                                                               float *__restrict__ d_gates)
{
    const int lane = threadIdx.x & 31;
    const int sub = lane & 15;
    const unsigned half_mask = 0xFFFFu << (lane & 16);
    const int nvec = d >> 3;
    const int nb = d >> 7;
    const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t t = gw; t < T; t += nw) {
        for (int j = 0; j < k; j++) {
            const int32_t r = __ldg(slot_to_sorted + t * k + j);
            if (r < 0 || r >= A) {
                if (lane == 0) d_gates[t * k + j] = 0.0f;
                continue;
            }
            const float g = __ldg(gates + t * k + j);
            float dot = 0.0f;
            // 32 lanes x 8 columns = two 128-column blocks per step (the
            // second half-warp idles on the last step when d / 128 is odd)
            for (int v0 = 0; v0 < nvec; v0 += 32) {
                const int v = v0 + lane;
                const bool on = v < nvec;
                float f[8], o[8];
                unpack_bf16x8(on ? __ldg(reinterpret_cast<const uint4 *>(dy + t * d) + v) : make_uint4(0, 0, 0, 0), f);
                unpack_bf16x8(on ? __ldcs(reinterpret_cast<const uint4 *>(out_sorted + (int64_t)r * d) + v)
                                 : make_uint4(0, 0, 0, 0),
                              o);
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    dot = fmaf(f[i], o[i], dot);
                    f[i] = g * f[i];
                    amax = fmaxf(amax, fabsf(f[i]));
                }
#pragma unroll
                for (int off = 8; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(half_mask, amax, off, 16));
                const float s = block_scale(amax);
                uint2 q;
                q.x = (uint32_t)pack_e4m3x2(__fdiv_rn(f[0], s), __fdiv_rn(f[1], s)) |
                      ((uint32_t)pack_e4m3x2(__fdiv_rn(f[2], s), __fdiv_rn(f[3], s)) << 16);
                q.y = (uint32_t)pack_e4m3x2(__fdiv_rn(f[4], s), __fdiv_rn(f[5], s)) |
                      ((uint32_t)pack_e4m3x2(__fdiv_rn(f[6], s), __fdiv_rn(f[7], s)) << 16);
                if (on) {
                    __stcs(reinterpret_cast<uint2 *>(d_out_q + (int64_t)r * d + (int64_t)v * 8), q);
                    if (sub == 0) d_out_s[(int64_t)r * nb + (v >> 4)] = s;
                }
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
            if (lane == 0) d_gates[t * k + j] = dot;
        }
    }
}

// One half-warp per (row, 128-column block of F): 8 columns per lane of
// d_act (bf16), gate and up (fp32); the two dh blocks (gate part at column
// 128b, up part at F + 128b) are quantised separately.
__global__ void __launch_bounds__(256) swiglu_backward_kernel(const uint16_t *__restrict__ d_act,
                                                              const float *__restrict__ h, int64_t rows, int F,
                                                              uint8_t *__restrict__ dh_q, float *__restrict__ dh_s)
{
    const int lane = threadIdx.x & 31;
    const int sub = lane & 15;
    const unsigned half_mask = 0xFFFFu << (lane & 16);
    const int nbf = F >> 7;
    const int64_t nblocks = rows * nbf;
    int64_t b = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 4;
    const int64_t step = ((int64_t)gridDim.x * blockDim.x) >> 4;
    for (; b < nblocks; b += step) {
        const int64_t r = b / nbf, cb = b - r * nbf;
        const int64_t c0 = cb * 128 + sub * 8;
        float da[8], gt[8], up[8];
        unpack_bf16x8(__ldcs(reinterpret_cast<const uint4 *>(d_act + r * F + c0)), da);
        const float4 *hg = reinterpret_cast<const float4 *>(h + r * 2 * F + c0);
        const float4 *hu = reinterpret_cast<const float4 *>(h + r * 2 * F + F + c0);
        const float4 g0 = __ldcs(hg), g1 = __ldcs(hg + 1), u0 = __ldcs(hu), u1 = __ldcs(hu + 1);
        gt[0] = g0.x; gt[1] = g0.y; gt[2] = g0.z; gt[3] = g0.w; gt[4] = g1.x; gt[5] = g1.y; gt[6] = g1.z; gt[7] = g1.w;
        up[0] = u0.x; up[1] = u0.y; up[2] = u0.z; up[3] = u0.w; up[4] = u1.x; up[5] = u1.y; up[6] = u1.z; up[7] = u1.w;
        float dg[8], du[8], ag = 0.0f, au = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float sg = __fdiv_rn(1.0f, 1.0f + expf(-gt[i]));
            dg[i] = da[i] * up[i] * sg * (1.0f + gt[i] * (1.0f - sg));
            du[i] = da[i] * (gt[i] * sg);
            ag = fmaxf(ag, fabsf(dg[i]));
            au = fmaxf(au, fabsf(du[i]));
        }
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) {
            ag = fmaxf(ag, __shfl_xor_sync(half_mask, ag, off, 16));
            au = fmaxf(au, __shfl_xor_sync(half_mask, au, off, 16));
        }
        const float sg_ = block_scale(ag), su = block_scale(au);
        uint2 qg, qu;
        qg.x = (uint32_t)pack_e4m3x2(__fdiv_rn(dg[0], sg_), __fdiv_rn(dg[1], sg_)) |
               ((uint32_t)pack_e4m3x2(__fdiv_rn(dg[2], sg_), __fdiv_rn(dg[3], sg_)) << 16);
        qg.y = (uint32_t)pack_e4m3x2(__fdiv_rn(dg[4], sg_), __fdiv_rn(dg[5], sg_)) |
               ((uint32_t)pack_e4m3x2(__fdiv_rn(dg[6], sg_), __fdiv_rn(dg[7], sg_)) << 16);
        qu.x = (uint32_t)pack_e4m3x2(__fdiv_rn(du[0], su), __fdiv_rn(du[1], su)) |
               ((uint32_t)pack_e4m3x2(__fdiv_rn(du[2], su), __fdiv_rn(du[3], su)) << 16);
        qu.y = (uint32_t)pack_e4m3x2(__fdiv_rn(du[4], su), __fdiv_rn(du[5], su)) |
               ((uint32_t)pack_e4m3x2(__fdiv_rn(du[6], su), __fdiv_rn(du[7], su)) << 16);
        *reinterpret_cast<uint2 *>(dh_q + r * 2 * F + c0) = qg;
        *reinterpret_cast<uint2 *>(dh_q + r * 2 * F + F + c0) = qu;
        if (sub == 0) {
            dh_s[r * 2 * nbf + cb] = sg_;
            dh_s[r * 2 * nbf + nbf + cb] = su;
        }
    }
}

// Codes [R, C] -> [C, R] per expert through a 64 x 64 shared tile (16-byte
// loads along C, 4-byte stores along R); scales [R/128, C/128] transposed by
// the first CTA row of each expert.
__global__ void __launch_bounds__(256) transpose_codes_kernel(const uint8_t *__restrict__ q, int64_t R, int64_t C,
                                                              uint8_t *__restrict__ qt)
{
    __shared__ uint8_t tile[64][64 + 4];
    const int64_t e = blockIdx.z;
    const int64_t r0 = (int64_t)blockIdx.y * 64, c0 = (int64_t)blockIdx.x * 64;
    const uint8_t *src = q + e * R * C;
    uint8_t *dst = qt + e * R * C;
    const int tid = threadIdx.x;
    {
        const int rr = tid >> 2, cc = (tid & 3) * 16;      // 64 rows x 4 x 16 bytes
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src + (r0 + rr) * C + c0 + cc));
        const uint8_t *b = reinterpret_cast<const uint8_t *>(&v);
#pragma unroll
        for (int i = 0; i < 16; i++) tile[rr][cc + i] = b[i];
    }
    __syncthreads();
    {
        const int cc = tid >> 2, rr = (tid & 3) * 16;      // 64 output rows (= input cols) x 4 x 16 bytes
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; i++)
            w[i] = (uint32_t)tile[rr + 4 * i][cc] | ((uint32_t)tile[rr + 4 * i + 1][cc] << 8) |
                   ((uint32_t)tile[rr + 4 * i + 2][cc] << 16) | ((uint32_t)tile[rr + 4 * i + 3][cc] << 24);
        *reinterpret_cast<uint4 *>(dst + (c0 + cc) * R + r0 + rr) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__global__ void transpose_scales_kernel(const float *__restrict__ s, int64_t E, int64_t br, int64_t bc,
                                        float *__restrict__ st)
{
    const int64_t n = E * br * bc;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = i / (br * bc), rem = i - e * br * bc, r = rem / bc, c = rem - r * bc;
        st[e * br * bc + c * br + r] = s[i];
    }
}

// ---------------------------------------------------------------------------
// Weight gradients.  dW2[e] = d_out^T act and dW13[e] = dh^T x over expert
// e's rows: the contraction runs over tokens, so both operands are
// re-quantised 128 x 1 (one scale per channel per 128-row block of the
// expert) and stored channel-major with each expert's rows padded to a
// multiple of 128: q [C, ld], s [C, ld/128] with the rows of expert e at
// columns pad[e] .. (ld is a host-known bound of pad[E], so that tensor
// maps can be built without reading pad back).

// pad[e] = sum of the 128-rounded row counts of experts before e (one CTA)
__global__ void pad_offsets_kernel(const int32_t *__restrict__ offsets, int E, int32_t *__restrict__ pad)
{
    if (threadIdx.x != 0) return;
    int32_t acc = 0;
    for (int e = 0; e < E; e++) {
        pad[e] = acc;
        acc += ((offsets[e + 1] - offsets[e] + 127) / 128) * 128;
    }
    pad[E] = acc;
}

// the operand's value at sorted row r, channel c (fp32)
enum { SRC_GDY = 0, SRC_ACT = 1, SRC_DH = 2, SRC_X = 3 };
struct WgSrc {
    const uint16_t *dy;          // SRC_GDY: [T, C] bf16, with gates [T*k] and the slot map
    const float *gates;
    const uint16_t *x;           // SRC_X: [T, C] bf16
    const int32_t *sorted_to_slot;
    const float *h;              // SRC_ACT, SRC_DH: [A, 2F] fp32 pre-activations (C = F or 2F)
    const uint16_t *d_act;       // SRC_DH: [A, F] bf16
    int k, F;
};

// 32 consecutive channels c0 .. c0+31 of sorted row r (16-byte loads)
template <int SRC>
__device__ __forceinline__ void wg_row32(const WgSrc &w, int64_t r, int64_t c0, int64_t C, float *v)
{
    if (SRC == SRC_GDY || SRC == SRC_X) {
        const int32_t slot = __ldg(w.sorted_to_slot + r);
        const float g = SRC == SRC_GDY ? __ldg(w.gates + slot) : 1.0f;
        const uint4 *src = reinterpret_cast<const uint4 *>((SRC == SRC_GDY ? w.dy : w.x) + (int64_t)(slot / w.k) * C + c0);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            unpack_bf16x8(__ldg(src + i), v + 8 * i);
            if (SRC == SRC_GDY) {
#pragma unroll
                for (int j = 0; j < 8; j++) v[8 * i + j] = g * v[8 * i + j];
            }
        }
    } else if (SRC == SRC_ACT) {
        const float4 *hg = reinterpret_cast<const float4 *>(w.h + r * 2 * w.F + c0);
        const float4 *hu = reinterpret_cast<const float4 *>(w.h + r * 2 * w.F + w.F + c0);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float4 g4 = __ldg(hg + i), u4 = __ldg(hu + i);
            v[4 * i + 0] = __fdiv_rn(g4.x, 1.0f + expf(-g4.x)) * u4.x;
            v[4 * i + 1] = __fdiv_rn(g4.y, 1.0f + expf(-g4.y)) * u4.y;
            v[4 * i + 2] = __fdiv_rn(g4.z, 1.0f + expf(-g4.z)) * u4.z;
            v[4 * i + 3] = __fdiv_rn(g4.w, 1.0f + expf(-g4.w)) * u4.w;
        }
    } else {
        const bool up_half = c0 >= w.F;
        const int64_t f0 = up_half ? c0 - w.F : c0;
        float da[32];
        const uint4 *a4 = reinterpret_cast<const uint4 *>(w.d_act + r * w.F + f0);
#pragma unroll
        for (int i = 0; i < 4; i++) unpack_bf16x8(__ldg(a4 + i), da + 8 * i);
        const float4 *hg = reinterpret_cast<const float4 *>(w.h + r * 2 * w.F + f0);
        const float4 *hu = reinterpret_cast<const float4 *>(w.h + r * 2 * w.F + w.F + f0);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float4 g4 = __ldg(hg + i), u4 = __ldg(hu + i);
            const float gg[4] = {g4.x, g4.y, g4.z, g4.w}, uu[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const float g = gg[j], sg = __fdiv_rn(1.0f, 1.0f + expf(-g));
                const float a = da[4 * i + j];
                v[4 * i + j] = up_half ? a * (g * sg) : a * uu[j] * sg * (1.0f + g * (1.0f - sg));
            }
        }
    }
}

// the transpose tile: row stride 65 words, and each 32-row group shifted by 8
// more words, so that the column reads (8 channels x 4 row groups per warp)
// and the row writes (32 rows per warp) hit 32 distinct banks
__device__ __forceinline__ int q1_idx(int r, int c) { return r * 65 + c + (r >> 5) * 8; }
constexpr int Q1_TILE = 127 * 65 + 64 + 3 * 8;

// One CTA per (64 channels, padded 128-row block): the block's values are
// staged in shared memory, each channel's amax over the expert's rows is a
// 4-thread reduction, and each thread writes 32 codes of one channel (the
// 128 codes of a channel are one contiguous 128-byte run of q).
// Scales channel-major sc[c * ld/128 + kb] or block-major sc[kb * C + c] (the
// layout the weight-gradient GEMM takes for both operands: a tile's 128
// scales of one K block are one contiguous 512-byte run).
template <int SRC>
__global__ void __launch_bounds__(256) quant_128x1_kernel(WgSrc w, const int32_t *__restrict__ offsets,
                                                          const int32_t *__restrict__ pad, int E, int64_t C,
                                                          int64_t ld, bool kb_major, uint8_t *__restrict__ q,
                                                          float *__restrict__ sc)
{
    __shared__ float tile[Q1_TILE];
    __shared__ int64_t s_r0, s_rend;
    const int64_t P = __ldg(pad + E);
    const int64_t kb = blockIdx.y;
    if (kb * 128 >= P || kb * 128 >= ld) return;
    // the expert with pad[e] <= 128 kb < pad[e+1] (E <= 1024: each thread
    // checks up to four experts with independent loads; with offsets from
    // moe_wgrad_pad_offsets exactly one matches, otherwise the block is empty)
    if (threadIdx.x == 0) s_r0 = s_rend = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t p0 = __ldg(pad + e), p1 = __ldg(pad + e + 1);
        if (p0 <= kb * 128 && kb * 128 < p1) {
            s_r0 = __ldg(offsets + e) + (kb * 128 - p0);     // first sorted row of the block
            s_rend = __ldg(offsets + e + 1);
        }
    }
    __syncthreads();
    const int64_t r0 = s_r0, rend = s_rend;
    const int64_t c0 = (int64_t)blockIdx.x * 64;
    const int tid = threadIdx.x;
    {
        const int rr = tid & 127, ch = (tid >> 7) * 32;
        const int64_t r = r0 + rr;
        float v[32];
        if (r < rend) {
            wg_row32<SRC>(w, r, c0 + ch, C, v);
        } else {
#pragma unroll
            for (int i = 0; i < 32; i++) v[i] = 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 32; i++) tile[q1_idx(rr, ch + i)] = v[i];
    }
    __syncthreads();
    const int cc = tid >> 2, part = tid & 3;
    float amax = 0.0f;
#pragma unroll 8
    for (int i = 0; i < 32; i++) amax = fmaxf(amax, fabsf(tile[q1_idx(part * 32 + i, cc)]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    const float s = block_scale(amax);
    const int64_t c = c0 + cc;
    if (c < C) {
        uint32_t wds[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float *t4 = &tile[q1_idx(part * 32 + 4 * i, cc)];   // rows +1..+3 are +65 words each
            wds[i] = (uint32_t)pack_e4m3x2(__fdiv_rn(t4[0], s), __fdiv_rn(t4[65], s)) |
                     ((uint32_t)pack_e4m3x2(__fdiv_rn(t4[130], s), __fdiv_rn(t4[195], s)) << 16);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(q + c * ld + kb * 128 + part * 32);
        dst[0] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
        dst[1] = make_uint4(wds[4], wds[5], wds[6], wds[7]);
        if (part == 0) sc[kb_major ? kb * C + c : c * (ld / 128) + kb] = s;
    }
}

} // namespace moe

using namespace moe;

MOE_API moe_status moe_combine_backward(const uint16_t *dy, const float *gates, const uint16_t *out_sorted,
                                        const int32_t *slot_to_sorted, int T, int k, int d, int64_t A,
                                        uint8_t *d_out_q, float *d_out_s, float *d_gates, void *stream)
{
    if (T < 0 || k < 1 || k > 32 || d <= 0 || d % 128 != 0 || A < 0) return MOE_ERR_SHAPE;
    if (T == 0) return MOE_OK;
    if (!dy || !gates || !out_sorted || !slot_to_sorted || !d_out_q || !d_out_s || !d_gates) return MOE_ERR_NULL;
    if (!aligned16(dy) || !aligned16(out_sorted) || !aligned16(d_out_q)) return MOE_ERR_ALIGN;
    int64_t grid = ((int64_t)T + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (grid > cap) grid = cap;
    combine_backward_kernel<<<(unsigned)grid, 256, 0, as_stream(stream)>>>(dy, gates, out_sorted, slot_to_sorted, T,
                                                                          k, d, A, d_out_q, d_out_s, d_gates);
    return launch_status();
}

MOE_API moe_status moe_swiglu_backward(const uint16_t *d_act, const float *h, int64_t rows, int F, uint8_t *dh_q,
                                       float *dh_s, void *stream)
{
    if (rows < 0 || F <= 0 || F % 128 != 0) return MOE_ERR_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!d_act || !h || !dh_q || !dh_s) return MOE_ERR_NULL;
    if (!aligned16(d_act) || !aligned16(h) || !aligned16(dh_q)) return MOE_ERR_ALIGN;
    const int64_t nblocks = rows * (F / 128);
    int64_t grid = (nblocks + 15) / 16;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (grid > cap) grid = cap;
    swiglu_backward_kernel<<<(unsigned)grid, 256, 0, as_stream(stream)>>>(d_act, h, rows, F, dh_q, dh_s);
    return launch_status();
}

MOE_API moe_status fp8_weight_transpose(const uint8_t *q, const float *s, int64_t E, int64_t R, int64_t C,
                                        uint8_t *qt, float *st, void *stream)
{
    if (E < 0 || R <= 0 || C <= 0 || R % 128 != 0 || C % 128 != 0 || E > 65535) return MOE_ERR_SHAPE;
    if (E == 0) return MOE_OK;
    if (!q || !s || !qt || !st) return MOE_ERR_NULL;
    if (!aligned16(q) || !aligned16(qt)) return MOE_ERR_ALIGN;
    if (R / 64 > 65535) return MOE_ERR_SHAPE;
    cudaStream_t stm = as_stream(stream);
    transpose_codes_kernel<<<dim3((unsigned)(C / 64), (unsigned)(R / 64), (unsigned)E), 256, 0, stm>>>(q, R, C, qt);
    const int64_t ns = E * (R / 128) * (C / 128);
    transpose_scales_kernel<<<(unsigned)((ns + 255) / 256 < 4096 ? (ns + 255) / 256 : 4096), 256, 0, stm>>>(
        s, E, R / 128, C / 128, st);
    return launch_status();
}

MOE_API moe_status moe_wgrad_pad_offsets(const int32_t *expert_offsets, int E, int32_t *pad, void *stream)
{
    if (E < 1 || E > 1024) return MOE_ERR_SHAPE;
    if (!expert_offsets || !pad) return MOE_ERR_NULL;
    pad_offsets_kernel<<<1, 32, 0, as_stream(stream)>>>(expert_offsets, E, pad);
    return launch_status();
}

MOE_API moe_status moe_wgrad_quant(int src, const uint16_t *dy, const float *gates, const uint16_t *x,
                                   const int32_t *sorted_to_slot, int k, const float *h, const uint16_t *d_act,
                                   int F, const int32_t *expert_offsets, const int32_t *pad, int E, int64_t C,
                                   int64_t max_pad, int scales_kb_major, uint8_t *q, float *scales, void *stream)
{
    if (E < 1 || E > 1024 || C <= 0 || C % 128 != 0 || max_pad < 0 || max_pad % 128 != 0 || k < 1 || k > 32)
        return MOE_ERR_SHAPE;
    if (!expert_offsets || !pad || !q || !scales) return MOE_ERR_NULL;
    WgSrc w{dy, gates, x, sorted_to_slot, h, d_act, k, F};
    if (src < 0 || src > 3 || (src == SRC_ACT && (F <= 0 || C != F)) || (src == SRC_DH && (F <= 0 || C != 2 * F)))
        return MOE_ERR_SHAPE;
    if ((src == SRC_GDY && (!dy || !gates || !sorted_to_slot)) || (src == SRC_X && (!x || !sorted_to_slot)) ||
        (src == SRC_ACT && !h) || (src == SRC_DH && (!h || !d_act)))
        return MOE_ERR_NULL;
    // rows are read 16 bytes at a time
    if (!aligned16(q) || (dy && !aligned16(dy)) || (x && !aligned16(x)) || (h && !aligned16(h)) ||
        (d_act && !aligned16(d_act)))
        return MOE_ERR_ALIGN;
    if (max_pad == 0) return MOE_OK;
    // one CTA per (64 channels, 128-row block) of the largest possible padded
    // extent; blocks past pad[E] (known on the device only) return at once
    const dim3 grid((unsigned)((C + 63) / 64), (unsigned)(max_pad / 128));
    cudaStream_t st = as_stream(stream);
    switch (src) {
    case SRC_GDY: quant_128x1_kernel<SRC_GDY><<<grid, 256, 0, st>>>(w, expert_offsets, pad, E, C, max_pad, scales_kb_major != 0, q, scales); break;
    case SRC_ACT: quant_128x1_kernel<SRC_ACT><<<grid, 256, 0, st>>>(w, expert_offsets, pad, E, C, max_pad, scales_kb_major != 0, q, scales); break;
    case SRC_DH: quant_128x1_kernel<SRC_DH><<<grid, 256, 0, st>>>(w, expert_offsets, pad, E, C, max_pad, scales_kb_major != 0, q, scales); break;
    case SRC_X: quant_128x1_kernel<SRC_X><<<grid, 256, 0, st>>>(w, expert_offsets, pad, E, C, max_pad, scales_kb_major != 0, q, scales); break;
    default: return MOE_ERR_SHAPE;
    }
    return launch_status();
}
