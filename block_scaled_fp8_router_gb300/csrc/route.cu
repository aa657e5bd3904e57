// route.cu -- MoE router: fused fp32 logits + warp top-k + gates + capture,
// and replay of a captured routing payload.
//
// Router replay (R3) in "RL at 1T Scale: prime-rl Performance Deep Dive",
// section "Router replay": the routing decision made at inference is
// captured into a [num_layers, top_k, seq_len] payload and replayed on the
// trainer.  For the replay to be exact, the decision must be
// bit-reproducible: every logit is one binary32 fma chain in ascending hidden
// index, computed by one thread (a SIMT register-tiled GEMM, not the tensor
// cores, whose accumulation order is not specified).
//
// route_topk_kernel: CTA = 128 threads, 32 tokens x all experts (passes of
// 256); each thread owns 8 tokens x 8 experts of fp32 accumulators (6
// shared-memory wavefronts per 64 FMAs per warp); bf16 tiles of x and W_r (32
// deep) are widened to fp32 in shared memory with conflict-free stores, the
// next tile is loaded into registers while the current one is consumed.
// Logits never leave the SM: they go to shared memory, and each warp then
// selects top-k for 8 tokens with k rounds of a (value, index) arg-max.
#include "common.cuh"

namespace moe {

constexpr int RT_BT = 32;   // tokens per CTA
constexpr int RT_EP = 256;  // experts per pass
constexpr int RT_BK = 32;   // hidden indices per shared-memory tile
constexpr int RR_BK = 256;  // replay: hidden indices per staged x chunk

// Strict total order of the selection: larger value first, -0 == +0, NaN
// below every number, equal keys by lower index.
__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib)
{
    const bool na = isnan(a), nb = isnan(b);
    if (na != nb) return nb;
    if (!na && a != b) return a > b;
    return ia < ib;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Gate of the slot held by `lane` (lanes < k hold the chosen logits).  The
// same code serves routing and replay so that a replayed capture reproduces
// its gates bit for bit.  For softmax without renormalisation the caller
// passes the max and the exp-sum over all E (full_max, full_sum).
__device__ __forceinline__ float warp_gate(int lane, int k, float my_l, int score_fn, int renorm,
                                           float route_scale, float full_max, float full_sum)
{
    const bool mine = lane < k;
    float g;
    if (score_fn == MOE_SCORE_SOFTMAX) {
        if (renorm) {
            const float m = warp_max(mine ? my_l : -INFINITY);
            const float e = mine ? expf(my_l - m) : 0.0f;
            g = __fdiv_rn(e, warp_sum(e));
        } else {
            g = __fdiv_rn(expf(my_l - full_max), full_sum);
        }
    } else {
        const float s = mine ? __fdiv_rn(1.0f, 1.0f + expf(-my_l)) : 0.0f;
        g = renorm ? __fdiv_rn(s, warp_sum(s)) : s;
    }
    return g * route_scale;
}

__global__ void __launch_bounds__(128, 3) route_topk_kernel(const uint16_t *__restrict__ x,
                                                            const uint16_t *__restrict__ wr, int T, int d, int E,
                                                            int k, int score_fn, int renorm, float route_scale,
                                                            int32_t *__restrict__ ids, float *__restrict__ gates,
                                                            int32_t *__restrict__ capture,
                                                            float *__restrict__ logits_out)
{
    extern __shared__ float4 smem4[];
    float *xs = reinterpret_cast<float *>(smem4);   // [RT_BK][RT_BT]
    float *ws = xs + RT_BK * RT_BT;                  // [RT_BK][RT_EP]
    float *lg = ws + RT_BK * RT_EP;                  // [RT_BT][Epad]
    const int Epad = (E + 31) & ~31;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * RT_BT;
    const int tt = (lane >> 3) * 8;                // my 8 tokens in the tile
    const int ee = warp * 64 + (lane & 7) * 8;     // my 8 experts in the pass

    // tile loaders: x chunk (token = tid & 31, 8-wide part = tid >> 5) and
    // 8 W_r chunks (expert = tid + 128 (r & 1), part = r >> 1); consecutive
    // lanes write consecutive shared-memory words (no bank conflicts)
    const int xt = tid & 31, xp = tid >> 5;
    for (int e0 = 0; e0 < E; e0 += RT_EP) {
        float acc[8][8];
#pragma unroll
        for (int a = 0; a < 8; a++)
#pragma unroll
            for (int b = 0; b < 8; b++) acc[a][b] = 0.0f;

        uint4 rx, rw[8];
        auto load_tile = [&](int k0) {
            const int t = t0 + xt;
            rx = t < T ? __ldg(reinterpret_cast<const uint4 *>(x + (int64_t)t * d + k0 + xp * 8))
                       : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int r = 0; r < 8; r++) {
                const int e = e0 + tid + 128 * (r & 1), p = r >> 1;
                rw[r] = e < E ? __ldg(reinterpret_cast<const uint4 *>(wr + (int64_t)e * d + k0 + p * 8))
                              : make_uint4(0, 0, 0, 0);
            }
        };
        load_tile(0);
        for (int k0 = 0; k0 < d; k0 += RT_BK) {
            __syncthreads();
            {
                float f[8];
                unpack_bf16x8(rx, f);
#pragma unroll
                for (int j = 0; j < 8; j++) xs[(xp * 8 + j) * RT_BT + xt] = f[j];
#pragma unroll
                for (int r = 0; r < 8; r++) {
                    const int e = tid + 128 * (r & 1), p = r >> 1;
                    unpack_bf16x8(rw[r], f);
#pragma unroll
                    for (int j = 0; j < 8; j++) ws[(p * 8 + j) * RT_EP + e] = f[j];
                }
            }
            __syncthreads();
            if (k0 + RT_BK < d) load_tile(k0 + RT_BK);
#pragma unroll
            for (int i = 0; i < RT_BK; i++) {
                const float4 x0 = *reinterpret_cast<const float4 *>(&xs[i * RT_BT + tt]);
                const float4 x1 = *reinterpret_cast<const float4 *>(&xs[i * RT_BT + tt + 4]);
                const float4 w0 = *reinterpret_cast<const float4 *>(&ws[i * RT_EP + ee]);
                const float4 w1 = *reinterpret_cast<const float4 *>(&ws[i * RT_EP + ee + 4]);
                const float xa[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                const float wb[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int a = 0; a < 8; a++)
#pragma unroll
                    for (int b = 0; b < 8; b++) acc[a][b] = fmaf(xa[a], wb[b], acc[a][b]);
            }
        }
#pragma unroll
        for (int a = 0; a < 8; a++)
#pragma unroll
            for (int b = 0; b < 8; b++) {
                const int e = e0 + ee + b;
                if (e < E) lg[(tt + a) * Epad + e] = acc[a][b];
            }
    }
    __syncthreads();

    // ---- top-k + gates: warp w handles tokens 8w .. 8w+7 of the tile ----
    for (int tl = warp * 8; tl < warp * 8 + 8; tl++) {
        const int t = t0 + tl;
        if (t >= T) break;
        const float *row = lg + tl * Epad;
        if (logits_out)
            for (int e = lane; e < E; e += 32) logits_out[(int64_t)t * E + e] = row[e];
        uint32_t taken = 0;
        int my_id = -1;
        float my_l = 0.0f;
        for (int j = 0; j < k; j++) {
            float bv = 0.0f;
            int bi = -1;
            for (int m = 0; m * 32 + lane < E; m++) {
                if (taken & (1u << m)) continue;
                const int e = m * 32 + lane;
                const float v = row[e];
                if (bi < 0 || ranks_before(v, e, bv, bi)) {
                    bv = v;
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
                const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
                if (oi >= 0 && (bi < 0 || ranks_before(ov, oi, bv, bi))) {
                    bv = ov;
                    bi = oi;
                }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == j) {
                my_id = bi;
                my_l = bv;
            }
        }
        float full_max = 0.0f, full_sum = 0.0f;
        if (score_fn == MOE_SCORE_SOFTMAX && !renorm) {
            full_max = __shfl_sync(0xFFFFFFFFu, my_l, 0);
            float s = 0.0f;
            for (int e = lane; e < E; e += 32) s += expf(row[e] - full_max);
            full_sum = warp_sum(s);
        }
        const float g = warp_gate(lane, k, my_l, score_fn, renorm, route_scale, full_max, full_sum);
        if (lane < k) {
            ids[(int64_t)t * k + lane] = my_id;
            gates[(int64_t)t * k + lane] = g;
            if (capture) capture[(int64_t)lane * T + t] = my_id;
        }
    }
}

// Replay: CTA = 32 tokens.  Copies the layer slab [k, T] to [T, k], checks
// ids, and (if x is given) evaluates the router logits of the replayed
// experts -- one fma chain per (token, slot), as in route_topk_kernel -- for
// the gates.
__global__ void __launch_bounds__(256) route_replay_kernel(const int32_t *__restrict__ replay_kT,
                                                           const uint16_t *__restrict__ x,
                                                           const uint16_t *__restrict__ wr, int T, int d, int E,
                                                           int k, int score_fn, int renorm, float route_scale,
                                                           int32_t *__restrict__ ids,
                                                           float *__restrict__ gates,
                                                           int32_t *__restrict__ dev_status)
{
    __shared__ int32_t sid[RT_BT * 32];
    __shared__ float slg[RT_BT * 32];
    __shared__ int sbad[RT_BT];
    __shared__ float xs[RT_BT * (RR_BK + 1)];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * RT_BT;
    const int nt = min(RT_BT, T - t0);

    for (int idx = tid; idx < RT_BT * k; idx += blockDim.x) {
        const int j = idx / RT_BT, tl = idx % RT_BT;
        if (tl < nt) {
            const int32_t v = replay_kT[(int64_t)j * T + t0 + tl];
            sid[tl * k + j] = v;
            ids[(int64_t)(t0 + tl) * k + j] = v;
        }
    }
    __syncthreads();
    if (tid < nt) {
        int bad = 0;
        for (int j = 0; j < k; j++) {
            const int32_t v = sid[tid * k + j];
            if (v < 0 || v >= E) bad = 1;
            for (int i = 0; i < j; i++)
                if (sid[tid * k + i] == v) bad = 1;
        }
        sbad[tid] = bad;
        if (bad) dev_flag(dev_status, MOE_DEV_BAD_IDS);
    }
    if (x == nullptr) return;

    // logits of the replayed experts: pair p = (tl, j), p = tid + 256 r
    constexpr int MAXP = (RT_BT * 32) / 256;  // k <= 32
    float acc[MAXP];
#pragma unroll
    for (int r = 0; r < MAXP; r++) acc[r] = 0.0f;
    const int npairs = nt * k;
    for (int c0 = 0; c0 < d; c0 += RR_BK) {
        __syncthreads();
        for (int idx = tid; idx < RT_BT * (RR_BK / 8); idx += blockDim.x) {
            const int tl = idx / (RR_BK / 8), p = idx % (RR_BK / 8);
            float f[8];
            if (tl < nt) {
                unpack_bf16x8(__ldg(reinterpret_cast<const uint4 *>(x + (int64_t)(t0 + tl) * d + c0 + p * 8)), f);
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++) f[j] = 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 8; j++) xs[tl * (RR_BK + 1) + p * 8 + j] = f[j];
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < MAXP; r++) {
            const int p = tid + 256 * r;
            if (p < npairs) {
                const int tl = p / k;
                const int32_t e = sid[p];
                if (e >= 0 && e < E) {
                    const uint16_t *wrow = wr + (int64_t)e * d + c0;
                    const float *xrow = xs + tl * (RR_BK + 1);
                    float a = acc[r];
                    for (int i = 0; i < RR_BK; i += 8) {
                        float f[8];
                        unpack_bf16x8(__ldg(reinterpret_cast<const uint4 *>(wrow + i)), f);
#pragma unroll
                        for (int j = 0; j < 8; j++) a = fmaf(xrow[i + j], f[j], a);
                    }
                    acc[r] = a;
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < MAXP; r++) {
        const int p = tid + 256 * r;
        if (p < npairs) slg[p] = acc[r];
    }
    __syncthreads();
    for (int tl = warp; tl < nt; tl += 8) {
        const float my_l = lane < k ? slg[tl * k + lane] : 0.0f;
        float g = warp_gate(lane, k, my_l, score_fn, renorm, route_scale, 0.0f, 0.0f);
        if (sbad[tl]) g = 0.0f;
        if (lane < k) gates[(int64_t)(t0 + tl) * k + lane] = g;
    }
}

static moe_status check_route_args(int T, int d, int E, int k, int score_fn)
{
    if (T < 0 || d <= 0 || d % 128 != 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E)
        return MOE_ERR_SHAPE;
    if (score_fn != MOE_SCORE_SOFTMAX && score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_SHAPE;
    if ((int64_t)T * k >= (1LL << 31)) return MOE_ERR_SHAPE;
    return MOE_OK;
}

} // namespace moe

using namespace moe;

MOE_API moe_status moe_route_topk(const uint16_t *x, const uint16_t *w_router, int T, int d, int E, int k,
                                  int score_fn, int renorm, float route_scale, int32_t *topk_ids,
                                  float *topk_gates, int32_t *capture_kT, float *logits_out, void *stream)
{
    moe_status s = check_route_args(T, d, E, k, score_fn);
    if (s != MOE_OK) return s;
    if (T == 0) return MOE_OK;
    if (!x || !w_router || !topk_ids || !topk_gates) return MOE_ERR_NULL;
    if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_ALIGN;
    const int Epad = (E + 31) & ~31;
    const size_t smem = sizeof(float) * (RT_BK * RT_BT + RT_BK * RT_EP + (size_t)RT_BT * Epad);
    if (cudaFuncSetAttribute(route_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    const int grid = (T + RT_BT - 1) / RT_BT;
    route_topk_kernel<<<grid, 128, smem, as_stream(stream)>>>(x, w_router, T, d, E, k, score_fn, renorm,
                                                               route_scale, topk_ids, topk_gates, capture_kT,
                                                               logits_out);
    return launch_status();
}

MOE_API moe_status moe_route_replay(const int32_t *replay_kT, const uint16_t *x, const uint16_t *w_router,
                                    int T, int d, int E, int k, int score_fn, int renorm, float route_scale,
                                    int32_t *topk_ids, float *topk_gates, int32_t *dev_status, void *stream)
{
    moe_status s = check_route_args(T, d, E, k, score_fn);
    if (s != MOE_OK) return s;
    if (x && score_fn == MOE_SCORE_SOFTMAX && !renorm) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!replay_kT || !topk_ids) return MOE_ERR_NULL;
    if (x && (!w_router || !topk_gates)) return MOE_ERR_NULL;
    if (x && (!aligned16(x) || !aligned16(w_router))) return MOE_ERR_ALIGN;
    const int grid = (T + RT_BT - 1) / RT_BT;
    route_replay_kernel<<<grid, 256, 0, as_stream(stream)>>>(replay_kT, x, w_router, T, d, E, k, score_fn,
                                                              renorm, route_scale, topk_ids, topk_gates,
                                                              dev_status);
    return launch_status();
}
