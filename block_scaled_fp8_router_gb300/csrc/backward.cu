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
#include "tcgen05.cuh"

namespace moe {

// SwiGLU backward of one element from the gate pre-activation g, the up
// value u and the incoming gradient a = d_act: d_gate = a * u * sg *
// (1 + g * (1 - sg)) and d_up = a * g * sg with sg = sigmoid(g) (fast
// exponential and reciprocal, as the GEMM1 epilogue forms silu; below
// g = -87 the reciprocal of a sum past 2^126 is 0, the limit).  The dgrad operand (swiglu_backward_kernel)
// and the weight-gradient operand (quant_128x1_dh_kernel) both take it from here.
__device__ __forceinline__ float dswiglu_gate(float a, float g, float u, float sg)
{
    return a * u * sg * (1.0f + g * (1.0f - sg));
}
__device__ __forceinline__ float dswiglu_up(float a, float g, float sg) { return a * (g * sg); }
__device__ __forceinline__ float sigmoid_fast(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }

// One warp per (token, slot): the slot's gate times the token's dy row,
// 32 lanes x 8 columns per step (two 128-column blocks; the second half-warp
// idles on the last step when d / 128 is odd), CB_U steps loaded before the
// first is encoded.  Every 128-column block is one half-warp (amax by four
// shuffles), written with its scale to the slot's sorted row.  The gate
// gradient is the warp-reduced dot of dy with the slot's expert output row
// (each lane accumulates its columns in order).
constexpr int CB_U = 4;

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
    const int64_t n = (int64_t)T * k;
    const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t p = gw; p < n; p += nw) {
        const int32_t r = __ldg(slot_to_sorted + p);
        if (r < 0 || r >= A) {
            if (lane == 0) d_gates[p] = 0.0f;
            continue;
        }
        const int64_t t = p / k;
        const float g = __ldg(gates + p);
        const uint4 *dyr = reinterpret_cast<const uint4 *>(dy + t * d);
        const uint4 *outr = reinterpret_cast<const uint4 *>(out_sorted + (int64_t)r * d);
        float dot = 0.0f;
        for (int v0 = 0; v0 < nvec; v0 += 32 * CB_U) {
            uint4 a[CB_U], b[CB_U];
#pragma unroll
            for (int u = 0; u < CB_U; u++) {
                const int v = v0 + 32 * u + lane;
                a[u] = make_uint4(0u, 0u, 0u, 0u);
                b[u] = make_uint4(0u, 0u, 0u, 0u);
                if (v < nvec) {
                    a[u] = __ldg(dyr + v);
                    b[u] = __ldcs(outr + v);
                }
            }
#pragma unroll
            for (int u = 0; u < CB_U; u++) {
                if (v0 + 32 * u >= nvec) break;                 // uniform over the warp
                const int v = v0 + 32 * u + lane;
                float f[8], o[8];
                unpack_bf16x8(a[u], f);
                unpack_bf16x8(b[u], o);
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
                const uint2 q = e4m3x8_scaled<2>(f, s);
                if (v < nvec) {
                    __stcs(reinterpret_cast<uint2 *>(d_out_q + (int64_t)r * d + (int64_t)v * 8), q);
                    if (sub == 0) d_out_s[(int64_t)r * nb + (v >> 4)] = s;
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
        if (lane == 0) d_gates[p] = dot;
    }
}

// The same combine backward with the rows staged in shared memory by bulk
// asynchronous copies (d <= CBT_MAX_D).  A producer lane copies each token's
// dy row (two buffers) and the expert output row of each routed slot (a
// CBT_STAGES ring) with 1-D bulk copies, so that whole rows stay in flight
// to HBM; 16 consumer warps (32 half-warps, each holding its 128-column
// blocks of the token's dy) form g * dy, its 1x128 codes and scales, and
// each warp's part of the dot with the output row.  A warp releases a stage with its part of the dot; the
// producer, before it refills the stage, sums the parts in warp order (a
// fixed order) into the slot's gate gradient.  Persistent: CTA c takes tokens c, c + grid, ...
// Every wait is bounded: one that runs out sets MOE_DEV_TIMEOUT and the
// abort flag, the consumers leave, and the producer waits (bounded) for its
// copies still in flight before the CTA exits.
constexpr int CBT_WARPS = 16;
constexpr int CBT_THREADS = (CBT_WARPS + 1) * 32;
constexpr int CBT_STAGES = 4;
constexpr int CBT_MAX_D = 8192;
constexpr int CBT_MAXB = CBT_MAX_D / 128 / (2 * CBT_WARPS);     // blocks per half-warp
constexpr int CBT_HDR = 512;

struct CbtHdr {
    uint64_t dy_full[2], dy_empty[2], out_full[CBT_STAGES], out_empty[CBT_STAGES];
    float partial[CBT_STAGES][CBT_WARPS];
    int abort_flag;
};
static_assert(sizeof(CbtHdr) <= CBT_HDR, "combine backward header");

// a bounded wait whose outcome is the same for the whole warp
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *dev_status)
{
    // one poll, then polls 32 ns apart with the time limit checked after
    // each (bounded like wait_or_abort; measured 3% faster than its 32 polls
    // per check for this kernel, whatever the sleep length)
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
        const uint64_t t0 = globaltimer_ns();
        while (true) {
            __nanosleep(32);
            if (mbar_try_wait(bar, parity)) {
                ok = true;
                break;
            }
            if (*abort_flag) break;
            if (globaltimer_ns() - t0 > ffn::TIMEOUT_NS) {
                *abort_flag = 1;
                dev_flag(dev_status, MOE_DEV_TIMEOUT);
                break;
            }
        }
    }
    return __all_sync(0xFFFFFFFFu, ok);
}

__global__ void __launch_bounds__(CBT_THREADS, 2)
    combine_backward_tma_kernel(const uint16_t *__restrict__ dy, const float *__restrict__ gates,
                                const uint16_t *__restrict__ out_sorted, const int32_t *__restrict__ slot_to_sorted,
                                int T, int k, int d, int64_t A, uint8_t *__restrict__ d_out_q,
                                float *__restrict__ d_out_s, float *__restrict__ d_gates, int32_t *dev_status)
{
    extern __shared__ __align__(128) uint8_t smem[];
    CbtHdr &hd = *reinterpret_cast<CbtHdr *>(smem);
    uint16_t *dyb = reinterpret_cast<uint16_t *>(smem + CBT_HDR);        // [2][d]
    uint16_t *outb = dyb + 2 * (int64_t)d;                                // [CBT_STAGES][d]
    volatile int *abort_flag = &hd.abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t row_bytes = (uint32_t)d * 2u;
    if (tid == 0) {
        for (int i = 0; i < 2; i++) {
            mbar_init(&hd.dy_full[i], 1);
            mbar_init(&hd.dy_empty[i], CBT_WARPS);
        }
        for (int i = 0; i < CBT_STAGES; i++) {
            mbar_init(&hd.out_full[i], 1);
            mbar_init(&hd.out_empty[i], CBT_WARPS);
        }
        hd.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == CBT_WARPS) {
        if (lane != 0) return;
        // producer; pend[st] is the slot whose gate gradient stage st holds
        int64_t pend[CBT_STAGES] = {};
        int64_t it = 0, sc = 0;
        bool ok = true;
        // the gate gradient of use u of a stage, once its eight parts are in
        auto finish = [&](int64_t u) -> bool {
            const int st = (int)(u % CBT_STAGES);
            if (!ffn::wait_or_abort(&hd.out_empty[st], (uint32_t)((u / CBT_STAGES) & 1), abort_flag, dev_status))
                return false;
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < CBT_WARPS; w++) sum += hd.partial[st][w];
            d_gates[pend[st]] = sum;
            return true;
        };
        for (int64_t t = blockIdx.x; t < T && ok; t += gridDim.x, it++) {
            const int db = (int)(it & 1);
            if (it >= 2 && !ffn::wait_or_abort(&hd.dy_empty[db], (uint32_t)(((it >> 1) - 1) & 1), abort_flag,
                                               dev_status)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&hd.dy_full[db], row_bytes);
            ffn::bulk_load_1d(dyb + (int64_t)db * d, dy + t * d, row_bytes, &hd.dy_full[db]);
            for (int j = 0; j < k; j++) {
                const int64_t p = t * k + j;
                const int32_t r = __ldg(slot_to_sorted + p);
                if (r < 0 || r >= A) {
                    d_gates[p] = 0.0f;
                    continue;
                }
                const int st = (int)(sc % CBT_STAGES);
                if (sc >= CBT_STAGES && !finish(sc - CBT_STAGES)) {
                    ok = false;
                    break;
                }
                pend[st] = p;
                mbar_arrive_expect_tx(&hd.out_full[st], row_bytes);
                ffn::bulk_load_1d(outb + (int64_t)st * d, out_sorted + (int64_t)r * d, row_bytes, &hd.out_full[st]);
                sc++;
            }
        }
        // the last uses of the stages
        for (int64_t u = sc - CBT_STAGES < 0 ? 0 : sc - CBT_STAGES; u < sc && ok; u++) ok = finish(u);
        // drain: every copy issued has landed before the CTA may exit
        for (int64_t u = it - 2 < 0 ? 0 : it - 2; u < it; u++)
            if (!mbar_wait_bounded(&hd.dy_full[u & 1], (uint32_t)((u >> 1) & 1), ffn::TIMEOUT_NS))
                dev_flag(dev_status, MOE_DEV_TIMEOUT);
        for (int64_t u = sc - CBT_STAGES < 0 ? 0 : sc - CBT_STAGES; u < sc; u++)
            if (!mbar_wait_bounded(&hd.out_full[u % CBT_STAGES], (uint32_t)((u / CBT_STAGES) & 1),
                                   ffn::TIMEOUT_NS))
                dev_flag(dev_status, MOE_DEV_TIMEOUT);
        return;
    }
    // consumers: half-warp h of a token holds its blocks h, h + 32, ... of dy
    // in registers for all the token's slots (the split rotated from token to
    // token), with each block's amax of |dy|: since rounding is monotonic,
    // the amax of a block of RN(g * dy) is exactly RN(|g| * amax |dy|), so a
    // slot's block scales need no reduction
    const int sub = lane & 15, hwid = tid >> 4;
    const unsigned half_mask = 0xFFFFu << (lane & 16);
    const int nb = d >> 7;
    int64_t it = 0, sc = 0;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x, it++) {
        const int db = (int)(it & 1);
        if (!warp_wait(&hd.dy_full[db], (uint32_t)((it >> 1) & 1), abort_flag, dev_status)) return;
        const uint16_t *dyr = dyb + (int64_t)db * d;
        const int h = (hwid + (int)(it & 1) * CBT_WARPS) & (2 * CBT_WARPS - 1);
        float dv[CBT_MAXB][8], am[CBT_MAXB];
#pragma unroll
        for (int u = 0; u < CBT_MAXB; u++) {
            const int blk = h + 2 * CBT_WARPS * u;
            unpack_bf16x8(blk < nb ? *reinterpret_cast<const uint4 *>(dyr + blk * 128 + sub * 8)
                                   : make_uint4(0u, 0u, 0u, 0u),
                          dv[u]);
            am[u] = fmaxf(fmaxf(fmaxf(fabsf(dv[u][0]), fabsf(dv[u][1])), fmaxf(fabsf(dv[u][2]), fabsf(dv[u][3]))),
                          fmaxf(fmaxf(fabsf(dv[u][4]), fabsf(dv[u][5])), fmaxf(fabsf(dv[u][6]), fabsf(dv[u][7]))));
        }
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) {
#pragma unroll
            for (int u = 0; u < CBT_MAXB; u++) am[u] = fmaxf(am[u], __shfl_xor_sync(half_mask, am[u], off, 16));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd.dy_empty[db]);            // dy now lives in registers
        for (int j = 0; j < k; j++) {
            const int64_t p = t * k + j;
            const int32_t r = __ldg(slot_to_sorted + p);
            if (r < 0 || r >= A) continue;
            const int st = (int)(sc % CBT_STAGES);
            if (!warp_wait(&hd.out_full[st], (uint32_t)((sc / CBT_STAGES) & 1), abort_flag, dev_status)) return;
            sc++;
            const float g = __ldg(gates + p), ag = fabsf(g);
            const uint16_t *outr = outb + (int64_t)st * d;
            float dot = 0.0f;
#pragma unroll
            for (int u = 0; u < CBT_MAXB; u++) {
                const int blk = h + 2 * CBT_WARPS * u;
                if (blk < nb) {
                    float o[8], f[8];
                    unpack_bf16x8(*reinterpret_cast<const uint4 *>(outr + blk * 128 + sub * 8), o);
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        dot = fmaf(dv[u][i], o[i], dot);
                        f[i] = g * dv[u][i];
                    }
                    const float s = block_scale(__fmul_rn(ag, am[u]));
                    __stcs(reinterpret_cast<uint2 *>(d_out_q + (int64_t)r * d + blk * 128 + sub * 8),
                           e4m3x8_scaled<2>(f, s));
                    if (sub == 0) d_out_s[(int64_t)r * nb + blk] = s;
                }
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
            if (lane == 0) {
                hd.partial[st][warp] = dot;
                mbar_arrive(&hd.out_empty[st]);
            }
        }
    }
}

// One half-warp per (row, 128-column block of F): 8 columns per lane of
// d_act (bf16), gate and up (fp32); the two dh blocks (gate part at column
// 128b, up part at F + 128b) are quantised separately.  SB blocks per pass
// with all their loads issued first (80 bytes per block per lane); the
// (row, block) pairs advance by the quotient and remainder of the stride.
constexpr int SB = 2;

__global__ void __launch_bounds__(256) swiglu_backward_kernel(const uint16_t *__restrict__ d_act,
                                                              const float *__restrict__ h, int64_t rows, int F,
                                                              uint8_t *__restrict__ dh_q, float *__restrict__ dh_s)
{
    const int lane = threadIdx.x & 31;
    const int sub = lane & 15;
    const unsigned half_mask = 0xFFFFu << (lane & 16);
    const int nbf = F >> 7;
    const int64_t hw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 4;
    const int64_t nhw = ((int64_t)gridDim.x * blockDim.x) >> 4;
    const int64_t dr = nhw / nbf;
    const int dc = (int)(nhw - dr * nbf);
    int64_t r = hw / nbf;
    int cb = (int)(hw - r * nbf);
    while (r < rows) {
        int64_t rr[SB];
        int cc[SB];
        uint4 ra[SB];
        float4 rg[SB][2], ru[SB][2];
#pragma unroll
        for (int u = 0; u < SB; u++) {
            rr[u] = r;
            cc[u] = cb;
            ra[u] = make_uint4(0u, 0u, 0u, 0u);
            rg[u][0] = rg[u][1] = ru[u][0] = ru[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < rows) {
                const int64_t c0 = (int64_t)cb * 128 + sub * 8;
                ra[u] = __ldcs(reinterpret_cast<const uint4 *>(d_act + r * F + c0));
                const float4 *hg = reinterpret_cast<const float4 *>(h + r * 2 * F + c0);
                const float4 *hu = reinterpret_cast<const float4 *>(h + r * 2 * F + F + c0);
                rg[u][0] = __ldcs(hg);
                rg[u][1] = __ldcs(hg + 1);
                ru[u][0] = __ldcs(hu);
                ru[u][1] = __ldcs(hu + 1);
            }
            cb += dc;
            r += dr;
            if (cb >= nbf) {
                cb -= nbf;
                r++;
            }
        }
#pragma unroll
        for (int u = 0; u < SB; u++) {
            if (rr[u] >= rows) break;                            // uniform over the half-warp
            const int64_t c0 = (int64_t)cc[u] * 128 + sub * 8;
            float da[8];
            unpack_bf16x8(ra[u], da);
            const float gt[8] = {rg[u][0].x, rg[u][0].y, rg[u][0].z, rg[u][0].w,
                                 rg[u][1].x, rg[u][1].y, rg[u][1].z, rg[u][1].w};
            const float up[8] = {ru[u][0].x, ru[u][0].y, ru[u][0].z, ru[u][0].w,
                                 ru[u][1].x, ru[u][1].y, ru[u][1].z, ru[u][1].w};
            float dg[8], du[8], ag = 0.0f, au = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const float sg = sigmoid_fast(gt[i]);
                dg[i] = dswiglu_gate(da[i], gt[i], up[i], sg);
                du[i] = dswiglu_up(da[i], gt[i], sg);
                ag = fmaxf(ag, fabsf(dg[i]));
                au = fmaxf(au, fabsf(du[i]));
            }
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) {
                ag = fmaxf(ag, __shfl_xor_sync(half_mask, ag, off, 16));
                au = fmaxf(au, __shfl_xor_sync(half_mask, au, off, 16));
            }
            const float sg_ = block_scale(ag), su = block_scale(au);
            const uint2 qg = e4m3x8_scaled<2>(dg, sg_), qu = e4m3x8_scaled<2>(du, su);
            *reinterpret_cast<uint2 *>(dh_q + rr[u] * 2 * F + c0) = qg;
            *reinterpret_cast<uint2 *>(dh_q + rr[u] * 2 * F + F + c0) = qu;
            if (sub == 0) {
                dh_s[rr[u] * 2 * nbf + cc[u]] = sg_;
                dh_s[rr[u] * 2 * nbf + nbf + cc[u]] = su;
            }
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

// The sorted rows [r0, rend) of padded 128-row block kb: the expert with
// pad[e] <= 128 kb < pad[e+1] (E <= 1024; the CTA's threads check the
// experts with independent loads; with offsets from moe_wgrad_pad_offsets
// exactly one matches, otherwise the block is empty).  Called by every
// thread of the CTA (two barriers).
__device__ __forceinline__ void padded_block_rows(const int32_t *__restrict__ pad,
                                                  const int32_t *__restrict__ offsets, int E, int64_t kb,
                                                  int64_t &s_r0, int64_t &s_rend)
{
    if (threadIdx.x == 0) s_r0 = s_rend = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t p0 = __ldg(pad + e), p1 = __ldg(pad + e + 1);
        if (p0 <= kb * 128 && kb * 128 < p1) {
            s_r0 = __ldg(offsets + e) + (kb * 128 - p0);
            s_rend = __ldg(offsets + e + 1);
        }
    }
    __syncthreads();
}

// The act operand (C = F): act = silu(gate) * up as the GEMM1 epilogue forms
// it, one CTA per (64 channels, padded 128-row block).  Thread (rg, cg) =
// (tid / 8, tid % 8) holds rows 4 rg .. 4 rg + 3 and channels 8 cg .. 8 cg + 7
// (every load of the four rows issued before the first value is formed).
// Channel amax: over the thread's four rows, the warp's four row groups (two
// shuffles) and the eight warps (shared memory).  The four codes of a
// channel form one 32-bit word, stored to a [channel][32 words] shared tile
// at word (rg + 4 cg) mod 32 (conflict-free); each channel's 128 codes then
// leave as eight 16-byte stores (one contiguous 128-byte run of q).
// Scales, in every 128 x 1 kernel here: channel-major sc[c * ld/128 + kb] or
// block-major sc[kb * C + c] (the layout the weight-gradient GEMM takes for
// both operands: a tile's 128 scales of one K block are one contiguous
// 512-byte run).
__global__ void __launch_bounds__(256) quant_128x1_act_kernel(WgSrc w, const int32_t *__restrict__ offsets,
                                                              const int32_t *__restrict__ pad, int E, int64_t C,
                                                              int64_t ld, bool kb_major, uint8_t *__restrict__ q,
                                                              float *__restrict__ sc)
{
    __shared__ __align__(16) uint32_t tq[64 * 32];
    __shared__ float red[8][64];
    __shared__ __align__(16) float ssc[64], ysc[64];
    __shared__ int64_t s_r0, s_rend;
    const int64_t P = __ldg(pad + E);
    const int64_t kb = blockIdx.y;
    if (kb * 128 >= P || kb * 128 >= ld) return;
    padded_block_rows(pad, offsets, E, kb, s_r0, s_rend);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid & 7, rg = tid >> 3;
    const int64_t cbase = (int64_t)blockIdx.x * 64, c0 = cbase + 8 * cg;
    const int64_t r0 = s_r0 + 4 * rg, rend = s_rend;
    const int F = w.F;
    float4 hg[4][2], hu[4][2];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        hg[i][0] = hg[i][1] = hu[i][0] = hu[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r0 + i < rend) {
            const float4 *pg = reinterpret_cast<const float4 *>(w.h + (r0 + i) * 2 * F + c0);
            const float4 *pu = reinterpret_cast<const float4 *>(w.h + (r0 + i) * 2 * F + F + c0);
            hg[i][0] = __ldg(pg);
            hg[i][1] = __ldg(pg + 1);
            hu[i][0] = __ldg(pu);
            hu[i][1] = __ldg(pu + 1);
        }
    }
    float v[4][8];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float gg[8] = {hg[i][0].x, hg[i][0].y, hg[i][0].z, hg[i][0].w,
                             hg[i][1].x, hg[i][1].y, hg[i][1].z, hg[i][1].w};
        const float uu[8] = {hu[i][0].x, hu[i][0].y, hu[i][0].z, hu[i][0].w,
                             hu[i][1].x, hu[i][1].y, hu[i][1].z, hu[i][1].w};
#pragma unroll
        for (int j = 0; j < 8; j++) v[i][j] = __fdividef(gg[j], 1.0f + __expf(-gg[j])) * uu[j];
    }
    float am[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
        am[j] = fmaxf(fmaxf(fabsf(v[0][j]), fabsf(v[1][j])), fmaxf(fabsf(v[2][j]), fabsf(v[3][j])));
        am[j] = fmaxf(am[j], __shfl_xor_sync(0xFFFFFFFFu, am[j], 8));
        am[j] = fmaxf(am[j], __shfl_xor_sync(0xFFFFFFFFu, am[j], 16));
    }
    if (lane < 8) {
#pragma unroll
        for (int j = 0; j < 8; j++) red[warp][8 * cg + j] = am[j];
    }
    __syncthreads();
    if (tid < 64) {
        float a = red[0][tid];
#pragma unroll
        for (int i = 1; i < 8; i++) a = fmaxf(a, red[i][tid]);
        const float s = block_scale(a);
        ssc[tid] = s;
        ysc[tid] = scale_recip(s);
        const int64_t c = cbase + tid;
        sc[kb_major ? kb * C + c : c * (ld / 128) + kb] = s;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; j++)
        tq[(8 * cg + j) * 32 + ((rg + 4 * cg) & 31)] =
            e4m3x4_div<2>(v[0][j], v[1][j], v[2][j], v[3][j], ssc[8 * cg + j], ysc[8 * cg + j]);
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 2; it++) {
        const int u = tid + 256 * it, ch = u >> 3, chunk = u & 7;
        const uint4 val = *reinterpret_cast<const uint4 *>(&tq[ch * 32 + ((4 * chunk + 4 * (ch >> 3)) & 31)]);
        *reinterpret_cast<uint4 *>(q + (cbase + ch) * ld + kb * 128 + 16 * chunk) = val;
    }
}

// The dh operand (C = 2F): one CTA per (32 columns f0 .. f0 + 31 of F,
// padded 128-row block), holding channels f (the gate part) and F + f (the
// up part) of those columns.  Thread (rg, cg) = (tid / 4, tid % 4) owns
// rows 2 rg, 2 rg + 1 and columns f0 + 8 cg .. + 7: it reads d_act, the gate
// and the up pre-activations there once and forms both d_gate and d_up with
// one sigmoid per element.  Channel amax: the thread's two rows, its warp
// (three shuffles) and the eight warps (shared memory).  The two codes of a
// channel's row pair are one halfword of the channel's row of the code
// tile, at halfword (rg + 8 cg) mod 64 (conflict-free; 16-byte runs stay
// whole), and each channel's 128 codes leave as eight 16-byte stores.
__global__ void __launch_bounds__(256) quant_128x1_dh_kernel(WgSrc w, const int32_t *__restrict__ offsets,
                                                             const int32_t *__restrict__ pad, int E, int64_t C,
                                                             int64_t ld, bool kb_major, uint8_t *__restrict__ q,
                                                             float *__restrict__ sc)
{
    __shared__ __align__(16) uint16_t tq[64 * 64];
    __shared__ float red[8][64];
    __shared__ float ssc[64], ysc[64];
    __shared__ int64_t s_r0, s_rend;
    const int64_t P = __ldg(pad + E);
    const int64_t kb = blockIdx.y;
    if (kb * 128 >= P || kb * 128 >= ld) return;
    padded_block_rows(pad, offsets, E, kb, s_r0, s_rend);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid & 3, rg = tid >> 2;
    const int F = w.F;
    const int64_t f0 = (int64_t)blockIdx.x * 32, fc = f0 + 8 * cg;
    const int64_t r0 = s_r0 + 2 * rg, rend = s_rend;
    uint4 ra[2];
    float4 hg[2][2], hu[2][2];
#pragma unroll
    for (int i = 0; i < 2; i++) {
        ra[i] = make_uint4(0u, 0u, 0u, 0u);
        hg[i][0] = hg[i][1] = hu[i][0] = hu[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r0 + i < rend) {
            const float4 *pg = reinterpret_cast<const float4 *>(w.h + (r0 + i) * 2 * F + fc);
            const float4 *pu = reinterpret_cast<const float4 *>(w.h + (r0 + i) * 2 * F + F + fc);
            hg[i][0] = __ldg(pg);
            hg[i][1] = __ldg(pg + 1);
            hu[i][0] = __ldg(pu);
            hu[i][1] = __ldg(pu + 1);
            ra[i] = __ldg(reinterpret_cast<const uint4 *>(w.d_act + (r0 + i) * F + fc));
        }
    }
    float vg[2][8], vu[2][8];
#pragma unroll
    for (int i = 0; i < 2; i++) {
        float da[8];
        unpack_bf16x8(ra[i], da);
        const float gg[8] = {hg[i][0].x, hg[i][0].y, hg[i][0].z, hg[i][0].w,
                             hg[i][1].x, hg[i][1].y, hg[i][1].z, hg[i][1].w};
        const float uu[8] = {hu[i][0].x, hu[i][0].y, hu[i][0].z, hu[i][0].w,
                             hu[i][1].x, hu[i][1].y, hu[i][1].z, hu[i][1].w};
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const float sg = sigmoid_fast(gg[j]);
            vg[i][j] = dswiglu_gate(da[j], gg[j], uu[j], sg);
            vu[i][j] = dswiglu_up(da[j], gg[j], sg);
        }
    }
    float ag[8], au[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
        ag[j] = fmaxf(fabsf(vg[0][j]), fabsf(vg[1][j]));
        au[j] = fmaxf(fabsf(vu[0][j]), fabsf(vu[1][j]));
    }
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
#pragma unroll
        for (int j = 0; j < 8; j++) {
            ag[j] = fmaxf(ag[j], __shfl_xor_sync(0xFFFFFFFFu, ag[j], off));
            au[j] = fmaxf(au[j], __shfl_xor_sync(0xFFFFFFFFu, au[j], off));
        }
    }
    if (lane < 4) {
#pragma unroll
        for (int j = 0; j < 8; j++) {
            red[warp][8 * cg + j] = ag[j];
            red[warp][32 + 8 * cg + j] = au[j];
        }
    }
    __syncthreads();
    auto gch = [&](int ch) -> int64_t { return ch < 32 ? f0 + ch : F + f0 + ch - 32; };
    if (tid < 64) {
        float a = red[0][tid];
#pragma unroll
        for (int i = 1; i < 8; i++) a = fmaxf(a, red[i][tid]);
        const float s = block_scale(a);
        ssc[tid] = s;
        ysc[tid] = scale_recip(s);
        const int64_t c = gch(tid);
        sc[kb_major ? kb * C + c : c * (ld / 128) + kb] = s;
    }
    __syncthreads();
    const int hp = (rg + 8 * cg) & 63;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const int chg = 8 * cg + j, chu = 32 + 8 * cg + j;
        tq[chg * 64 + hp] = e4m3x2_div<2>(vg[0][j], vg[1][j], ssc[chg], ysc[chg]);
        tq[chu * 64 + hp] = e4m3x2_div<2>(vu[0][j], vu[1][j], ssc[chu], ysc[chu]);
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 2; it++) {
        const int u = tid + 256 * it, ch = u >> 3, chunk = u & 7;
        const int pchunk = (chunk + ((ch & 31) >> 3)) & 7;
        const uint4 val = *reinterpret_cast<const uint4 *>(&tq[ch * 64 + 8 * pchunk]);
        *reinterpret_cast<uint4 *>(q + gch(ch) * ld + kb * 128 + 16 * chunk) = val;
    }
}

// The same quantiser for the bf16 operands (SRC_GDY: g * dy of each routed
// row's token, SRC_X: x of that token), persistent over channel tiles so
// that loads stay in flight across them: a CTA of 256 threads takes one
// padded 128-row block and Q1_TPC consecutive 64-channel tiles.
// Loads: thread (rg, cg) = (tid / 8, tid % 8) looks the tokens of rows
// 4 rg .. 4 rg + 3 up once and copies their 16-byte pieces cg (channels
// 8 cg .. 8 cg + 7) of each tile into a Q1_STAGES-deep shared-memory ring
// with cp.async (eight lanes read a row's 128 contiguous bytes); piece cg
// of row r lands at position cg ^ ((r / 4) % 8) of the row.
// Work: warp w owns channels 8 w .. 8 w + 7 of the tile for all 128 rows,
// lane l rows 4 l .. 4 l + 3 (the swizzle makes the warp's reads of one
// piece column conflict-free), so a channel's amax is a warp reduction: a
// reduce-scatter of nine shuffles leaves channel (l / 4) % 8's amax in
// lane l, which forms that channel's scale and reciprocal, and sixteen
// shuffles hand all eight to the warp.  The four codes of a channel's rows
// in lane l form one word of the warp's own 8 x 32-word code tile, and
// each channel's 128 codes leave as eight 16-byte stores.  One CTA barrier
// per tile publishes the stage to every warp and frees the stage that is
// refilled next.
constexpr int Q1_STAGES = 4;
constexpr int Q1_TPC = 28;  // 14, 56 and 112 measured slower
constexpr int Q1_STAGE_BYTES = 128 * 64 * 2;
constexpr int Q1_SMEM = Q1_STAGES * Q1_STAGE_BYTES;

template <int SRC>
__global__ void __launch_bounds__(256, 3) quant_128x1_bf16_kernel(WgSrc w, const int32_t *__restrict__ offsets,
                                                               const int32_t *__restrict__ pad, int E, int64_t C,
                                                               int64_t ld, bool kb_major, uint8_t *__restrict__ q,
                                                               float *__restrict__ sc)
{
    extern __shared__ __align__(128) uint8_t q1_ring[];
    __shared__ __align__(16) uint32_t tq[8][8 * 32];       // per warp: [channel][32 words]
    __shared__ int64_t s_r0, s_rend;
    const int64_t P = __ldg(pad + E);
    const int64_t kb = blockIdx.y;
    const int ntiles = (int)(C / 64);
    const int t0 = blockIdx.x * Q1_TPC;
    const int t1 = t0 + Q1_TPC < ntiles ? t0 + Q1_TPC : ntiles;
    if (kb * 128 >= P || kb * 128 >= ld || t0 >= ntiles) return;
    padded_block_rows(pad, offsets, E, kb, s_r0, s_rend);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid & 7, rg = tid >> 3;
    const int64_t rend = s_rend;
    const uint16_t *src = SRC == SRC_GDY ? w.dy : w.x;
    int64_t off[4];            // loader rows 4 rg + i: element offset of the token's piece, or -1
    float g[4];                // worker rows 4 lane + i: the gate (g * dy)
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int64_t r = s_r0 + 4 * rg + i;
        const int32_t slot = r < rend ? __ldg(w.sorted_to_slot + r) : -1;
        off[i] = slot >= 0 ? (int64_t)(slot / w.k) * C + 8 * cg : -1;
        g[i] = 1.0f;
        if (SRC == SRC_GDY) {
            const int64_t rw = s_r0 + 4 * lane + i;
            const int32_t sw = rw < rend ? __ldg(w.sorted_to_slot + rw) : -1;
            if (sw >= 0) g[i] = __ldg(w.gates + sw);
        }
    }
    uint4 *ring = reinterpret_cast<uint4 *>(q1_ring);      // [stage][row][position]
    auto issue = [&](int t) {
        uint4 *dst = ring + (t % Q1_STAGES) * (128 * 8) + (4 * rg) * 8 + (cg ^ (rg & 7));
#pragma unroll
        for (int i = 0; i < 4; i++)
            cp_async16_zfill(dst + 8 * i, off[i] >= 0 ? src + off[i] + (int64_t)t * 64 : src, off[i] >= 0);
    };
#pragma unroll
    for (int u = 0; u < Q1_STAGES - 1; u++) {
        if (t0 + u < t1) issue(t0 + u);
        cp_async_commit();
    }
    uint32_t *tqw = tq[warp];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    for (int t = t0; t < t1; t++) {
        cp_async_wait<Q1_STAGES - 2>();                   // this thread's pieces of tile t
        __syncthreads();                                  // every piece of tile t; stage t - 1 read by all
        if (t + Q1_STAGES - 1 < t1) issue(t + Q1_STAGES - 1);
        cp_async_commit();
        const uint4 *stg = ring + (t % Q1_STAGES) * (128 * 8);
        float v[4][8];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            unpack_bf16x8(stg[(4 * lane + i) * 8 + (warp ^ (lane & 7))], v[i]);
            if (SRC == SRC_GDY) {
#pragma unroll
                for (int j = 0; j < 8; j++) v[i][j] = g[i] * v[i][j];
            }
        }
        float am[8];
#pragma unroll
        for (int j = 0; j < 8; j++)
            am[j] = fmaxf(fmaxf(fabsf(v[0][j]), fabsf(v[1][j])), fmaxf(fabsf(v[2][j]), fabsf(v[3][j])));
        // reduce-scatter: the xor-16, -8 and -4 steps each keep half of the
        // channels (lane bit 4, 3, 2 chooses which), leaving channel
        // 4 b4 + 2 b3 + b2 = (lane / 4) % 8; xor 2 and 1 finish its max
        float a4[4], a2[2];
#pragma unroll
        for (int i = 0; i < 4; i++)
            a4[i] = fmaxf(b4 ? am[4 + i] : am[i], __shfl_xor_sync(0xFFFFFFFFu, b4 ? am[i] : am[4 + i], 16));
#pragma unroll
        for (int i = 0; i < 2; i++)
            a2[i] = fmaxf(b3 ? a4[2 + i] : a4[i], __shfl_xor_sync(0xFFFFFFFFu, b3 ? a4[i] : a4[2 + i], 8));
        float a1 = fmaxf(b2 ? a2[1] : a2[0], __shfl_xor_sync(0xFFFFFFFFu, b2 ? a2[0] : a2[1], 4));
        a1 = fmaxf(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, 2));
        a1 = fmaxf(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, 1));
        const float s = block_scale(a1), y = scale_recip(s);
        const int64_t cbase = (int64_t)t * 64 + 8 * warp;
        if ((lane & 3) == 0) {
            const int64_t c = cbase + (lane >> 2);
            sc[kb_major ? kb * C + c : c * (ld / 128) + kb] = s;
        }
        __syncwarp();                                     // the previous tile's code reads are done
#pragma unroll
        for (int j = 0; j < 8; j++) {
            // x is bf16 (one correction step suffices); g * dy is an fp32 product
            constexpr int ST = SRC == SRC_X ? 1 : 2;
            tqw[j * 32 + lane] = e4m3x4_div<ST>(v[0][j], v[1][j], v[2][j], v[3][j], __shfl_sync(0xFFFFFFFFu, s, 4 * j),
                                                __shfl_sync(0xFFFFFFFFu, y, 4 * j));
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 2; r++) {
            const int p = lane + 32 * r, ch = p >> 3, chunk = p & 7;
            const uint4 val = *reinterpret_cast<const uint4 *>(&tqw[ch * 32 + 4 * chunk]);
            *reinterpret_cast<uint4 *>(q + (cbase + ch) * ld + kb * 128 + 16 * chunk) = val;
        }
    }
    cp_async_wait<0>();
}

} // namespace moe

using namespace moe;

MOE_API moe_status moe_combine_backward(const uint16_t *dy, const float *gates, const uint16_t *out_sorted,
                                        const int32_t *slot_to_sorted, int T, int k, int d, int64_t A,
                                        uint8_t *d_out_q, float *d_out_s, float *d_gates, int32_t *dev_status,
                                        void *stream)
{
    if (T < 0 || k < 1 || k > 32 || d <= 0 || d % 128 != 0 || A < 0) return MOE_ERR_SHAPE;
    if (T == 0) return MOE_OK;
    if (!dy || !gates || !out_sorted || !slot_to_sorted || !d_out_q || !d_out_s || !d_gates) return MOE_ERR_NULL;
    if (!aligned16(dy) || !aligned16(out_sorted) || !aligned16(d_out_q)) return MOE_ERR_ALIGN;
    cudaStream_t st = as_stream(stream);
    if (d <= CBT_MAX_D) {
        const size_t smem = CBT_HDR + (size_t)(2 + CBT_STAGES) * d * 2;
        if (cudaFuncSetAttribute(combine_backward_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return MOE_ERR_CUDA;
        // two CTAs per SM (both fit in the SM's shared memory for every
        // d <= CBT_MAX_D), persistent over tokens
        const int per_sm = smem * 2 <= 227 * 1024 ? 2 : 1;
        int64_t grid = (int64_t)sm_count() * per_sm;
        if (grid > T) grid = T;
        combine_backward_tma_kernel<<<(unsigned)grid, CBT_THREADS, smem, st>>>(
            dy, gates, out_sorted, slot_to_sorted, T, k, d, A, d_out_q, d_out_s, d_gates, dev_status);
        return launch_status();
    }
    int64_t grid = ((int64_t)T * k + 7) / 8;                  // one warp per (token, slot)
    const int64_t cap = (int64_t)sm_count() * 8;
    if (grid > cap) grid = cap;
    combine_backward_kernel<<<(unsigned)grid, 256, 0, st>>>(dy, gates, out_sorted, slot_to_sorted, T, k, d, A,
                                                           d_out_q, d_out_s, d_gates);
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
    // extent (the bf16 operands: per (Q1_TPC 64-channel tiles, 128-row
    // block)); blocks past pad[E] (known on the device only) return at once
    const dim3 grid((unsigned)(src == SRC_DH ? F / 32 : (C + 63) / 64), (unsigned)(max_pad / 128));
    const dim3 grid_bf16((unsigned)((C / 64 + Q1_TPC - 1) / Q1_TPC), (unsigned)(max_pad / 128));
    cudaStream_t st = as_stream(stream);
    const bool kbm = scales_kb_major != 0;
    switch (src) {
    case SRC_GDY:
        if (cudaFuncSetAttribute(quant_128x1_bf16_kernel<SRC_GDY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Q1_SMEM) != cudaSuccess)
            return MOE_ERR_CUDA;
        quant_128x1_bf16_kernel<SRC_GDY><<<grid_bf16, 256, Q1_SMEM, st>>>(w, expert_offsets, pad, E, C, max_pad, kbm,
                                                                         q, scales);
        break;
    case SRC_ACT:
        quant_128x1_act_kernel<<<grid, 256, 0, st>>>(w, expert_offsets, pad, E, C, max_pad, kbm, q, scales);
        break;
    case SRC_DH:
        quant_128x1_dh_kernel<<<grid, 256, 0, st>>>(w, expert_offsets, pad, E, C, max_pad, kbm, q, scales);
        break;
    case SRC_X:
        if (cudaFuncSetAttribute(quant_128x1_bf16_kernel<SRC_X>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Q1_SMEM) != cudaSuccess)
            return MOE_ERR_CUDA;
        quant_128x1_bf16_kernel<SRC_X><<<grid_bf16, 256, Q1_SMEM, st>>>(w, expert_offsets, pad, E, C, max_pad, kbm, q,
                                                                       scales);
        break;
    default: return MOE_ERR_SHAPE;
    }
    return launch_status();
}
