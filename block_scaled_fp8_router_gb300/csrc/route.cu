// route.cu -- MoE router: fused fp32 logits + warp top-k + gates + capture,
// replay of a captured routing payload, and the router's backward for fixed
// ids (logit gradients through the gates, dx, dW_r).
//
// Router replay (R3) in "RL at 1T Scale: prime-rl Performance Deep Dive",
// section "Router replay": the routing decision made at inference is
// captured into a [num_layers, top_k, seq_len] payload and replayed on the
// trainer.  For the replay to be exact, the decision must be
// bit-reproducible: every logit is one binary32 fma chain in ascending hidden
// index, computed by one thread (a SIMT register-tiled GEMM, not the tensor
// cores, whose accumulation order is not specified).
//
// route_topk_kernel: one cluster of ceil(E/128) CTAs per 64 tokens; each
// 256-thread CTA computes 64 tokens x 128 experts, one 8-token group per
// warp, 8 x 4 fp32 accumulators per thread (three 16-byte shared loads per
// 32 FMAs, the next hidden index's operands loaded while the current FMAs
// run), bf16 tiles of x and W_r (32 deep) read in whole 32-byte sectors and
// widened to fp32 in double-buffered shared memory with conflict-free
// stores while the next tile loads into registers (one barrier per tile).
// Logits stay on chip: each CTA selects its own top-k, CTA 0 merges the
// candidates it receives through distributed shared memory.
#include "common.cuh"

namespace moe {


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

// Derivative of the gates with respect to the chosen logits: lane j < k
// holds its slot's logit my_l and upstream gradient my_dg and returns
// dL/dl_j (rs = route_scale):
//   softmax, renorm:    p_j = exp(l_j) / sum_i exp(l_i), dl_j = rs p_j (dg_j - sum_i dg_i p_i)
//   sigmoid, renorm:    s_j = 1 / (1 + exp(-l_j)), S = sum_i s_i,
//                       dl_j = rs s_j (1 - s_j) (dg_j - sum_i dg_i s_i / S) / S
//   sigmoid, no renorm: dl_j = rs dg_j s_j (1 - s_j)
// (the full softmax over E is not handled here).  s (1 - s) is formed as
// e s^2 with e = exp(-l), which keeps its relative accuracy for large l.
__device__ __forceinline__ float warp_dgate(int lane, int k, float my_l, float my_dg, int score_fn, int renorm,
                                            float route_scale)
{
    const bool mine = lane < k;
    float dl;
    if (score_fn == MOE_SCORE_SOFTMAX) {
        const float m = warp_max(mine ? my_l : -INFINITY);
        const float e = mine ? expf(my_l - m) : 0.0f;
        const float p = __fdiv_rn(e, warp_sum(e));
        const float dot = warp_sum(mine ? my_dg * p : 0.0f);
        dl = route_scale * p * (my_dg - dot);
    } else {
        const float e = mine ? expf(-my_l) : 0.0f;
        const float sg = mine ? __fdiv_rn(1.0f, 1.0f + e) : 0.0f;
        const float ds = e * sg * sg;
        if (renorm) {
            const float S = warp_sum(sg), dot = warp_sum(mine ? my_dg * sg : 0.0f);
            dl = route_scale * ds * __fdiv_rn(my_dg - __fdiv_rn(dot, S), S);
        } else {
            dl = route_scale * my_dg * ds;
        }
    }
    return mine ? dl : 0.0f;
}

// ---- cluster helpers (route_topk runs one cluster per 64 tokens, one CTA
// per 128 experts) ----
__device__ __forceinline__ uint32_t cl_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_size()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_id()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cl_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cl_map(const void *p, uint32_t rank)
{
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(out)
                 : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
    return out;
}
__device__ __forceinline__ void cl_st_f2(uint32_t addr, float a, float b)
{
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}

// k rounds of a warp-wide arg-max under ranks_before over the candidates
// lane l holds (vals[m], idxs[m]) for m < nm (idx < 0 = no candidate); lane j
// ends with the j-th pick in (out_v, out_i) (out_i = -1 if there were fewer).
template <int NM>
__device__ __forceinline__ void warp_topk(const float *vals, const int *idxs, int k, int lane, float &out_v,
                                          int &out_i)
{
    uint32_t taken = 0;
    out_v = 0.0f;
    out_i = -1;
    for (int j = 0; j < k; j++) {
        float bv = 0.0f;
        int bi = -1, bm = -1;
#pragma unroll
        for (int m = 0; m < NM; m++) {
            if ((taken >> m) & 1u) continue;
            const int e = idxs[m];
            if (e < 0) continue;
            if (bi < 0 || ranks_before(vals[m], e, bv, bi)) {
                bv = vals[m];
                bi = e;
                bm = m;
            }
        }
        float wv = bv;
        int wi = bi;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, wv, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, wi, o);
            if (oi >= 0 && (wi < 0 || ranks_before(ov, oi, wv, wi))) {
                wv = ov;
                wi = oi;
            }
        }
        if (wi >= 0 && bi == wi && bm >= 0) taken |= 1u << bm;  // the winning lane retires its entry
        if (lane == j) {
            out_v = wv;
            out_i = wi;
        }
    }
}

constexpr int RC_BT = 64;           // tokens per cluster
constexpr int RC_EC = 128;          // experts per CTA
constexpr int RC_BK = 32;           // hidden indices per shared-memory tile
constexpr int RC_LGS = RC_EC + 4;   // logits row stride (floats)
// tile rows (one per hidden index) gain 8 floats of padding per 8 rows, so
// that the transposing stores of a warp (8 rows x 4 eight-index parts) hit
// 32 distinct banks
__host__ __device__ constexpr int rc_xrow(int i) { return i * RC_BT + (i >> 3) * 8; }
__host__ __device__ constexpr int rc_wrow(int i) { return i * RC_EC + (i >> 3) * 8; }
constexpr int RC_XB = RC_BK * RC_BT + 32;  // floats per x tile buffer
constexpr int RC_WB = RC_BK * RC_EC + 32;  // floats per W_r tile buffer
// shared floats before the candidate arrays: the double-buffered tiles, or
// the logits that replace them after the last tile, whichever is larger
constexpr int RC_TILE_FLOATS = (2 * (RC_XB + RC_WB) > RC_BT * RC_LGS) ? 2 * (RC_XB + RC_WB) : RC_BT * RC_LGS;

// One cluster of ceil(E/128) CTAs per 64 tokens.  CTA r computes the logits
// of experts 128r .. 128r+127 for the 64 tokens (256 threads; warp w owns
// tokens 8w .. 8w+7, lane l experts 4l .. 4l+3: 8 x 4 fp32 fma-chain
// accumulators per thread, three 16-byte shared-memory loads feed 32 fmas,
// the two x loads a broadcast; eight warps per CTA so that one CTA per SM
// already hides the shared-memory latency), keeps them in shared memory,
// selects its own top-k per token and sends those (value, index) candidates
// to CTA 0 of the cluster through distributed shared memory; CTA 0 merges
// them into the top-k over all experts (every member of the global top-k is
// in its own CTA's top-k, and the order is a strict total order, so the merge
// is exact) and writes ids, gates and the capture.
__global__ void __launch_bounds__(256) route_topk_kernel(const uint16_t *__restrict__ x,
                                                         const uint16_t *__restrict__ wr, int T, int d, int E,
                                                         int k, int score_fn, int renorm, float route_scale,
                                                         int32_t *__restrict__ ids, float *__restrict__ gates,
                                                         int32_t *__restrict__ capture,
                                                         float *__restrict__ logits_out)
{
    extern __shared__ float4 smem4[];
    const int ncta = (int)cl_size();
    const int rank = (int)cl_rank();
    // two [RC_BK][RC_BT] x tiles and two [RC_BK][RC_EC] W_r tiles (one is
    // filled while the other is read); the logits [RC_BT][RC_LGS] reuse the
    // same space after the last tile
    float *xs2 = reinterpret_cast<float *>(smem4);
    float *ws2 = xs2 + 2 * RC_XB;
    float *lg = xs2;
    float2 *cand = reinterpret_cast<float2 *>(xs2 + RC_TILE_FLOATS);  // CTA 0: [RC_BT][ncta*k]
    float2 *msum = cand + RC_BT * ncta * k;                           // CTA 0: [RC_BT][ncta]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = (int)cl_id() * RC_BT;
    const int e0 = rank * RC_EC;
    const int tt = warp * 8;                        // my 8 tokens in the tile
    const int ee = lane * 4;                        // my 4 experts of this CTA's 128
    const int nw = blockDim.x >> 5;

    // tile loaders: four lanes read a row's 64 contiguous bytes (whole
    // sectors); one x chunk (token tid >> 2, 8-wide part tid & 3) and two W_r
    // chunks (experts tid >> 2 and 64 + (tid >> 2), part tid & 3)
    const int xt = tid >> 2, xp = tid & 3;
    const int we = tid >> 2, wp = tid & 3;
    float acc[8][4];
#pragma unroll
    for (int a = 0; a < 8; a++)
#pragma unroll
        for (int b = 0; b < 4; b++) acc[a][b] = 0.0f;
    uint4 rx[1], rw[2];
    auto load_tile = [&](int k0) {
        const int t = t0 + xt;
        rx[0] = t < T ? __ldg(reinterpret_cast<const uint4 *>(x + (int64_t)t * d + k0 + xp * 8))
                      : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < 2; r++) {
            const int e = e0 + we + 64 * r;
            rw[r] = e < E ? __ldg(reinterpret_cast<const uint4 *>(wr + (int64_t)e * d + k0 + wp * 8))
                          : make_uint4(0, 0, 0, 0);
        }
    };
    load_tile(0);
    for (int k0 = 0, buf = 0; k0 < d; k0 += RC_BK, buf ^= 1) {
        float *xs = xs2 + buf * RC_XB;
        float *ws = ws2 + buf * RC_WB;
        {
            // rows xp*8 + j: rc_xrow(xp*8 + j) = xp*(8*RC_BT + 8) + j*RC_BT
            float f[8];
            unpack_bf16x8(rx[0], f);
#pragma unroll
            for (int j = 0; j < 8; j++) xs[xp * (8 * RC_BT + 8) + xt + j * RC_BT] = f[j];
#pragma unroll
            for (int r = 0; r < 2; r++) {
                unpack_bf16x8(rw[r], f);
#pragma unroll
                for (int j = 0; j < 8; j++) ws[wp * (8 * RC_EC + 8) + we + 64 * r + j * RC_EC] = f[j];
            }
        }
        // one barrier per tile: it publishes this tile and, since every
        // thread has passed it, the tile read two steps ago is free
        __syncthreads();
        if (k0 + RC_BK < d) load_tile(k0 + RC_BK);
        // operands of hidden index i+1 are loaded while the fmas of i run
        float4 nx0 = *reinterpret_cast<const float4 *>(&xs[tt]);
        float4 nx1 = *reinterpret_cast<const float4 *>(&xs[tt + 4]);
        float4 nw0 = *reinterpret_cast<const float4 *>(&ws[ee]);
#pragma unroll
        for (int i = 0; i < RC_BK; i++) {
            const float4 x0 = nx0, x1 = nx1, w0 = nw0;
            if (i + 1 < RC_BK) {
                nx0 = *reinterpret_cast<const float4 *>(&xs[rc_xrow(i + 1) + tt]);
                nx1 = *reinterpret_cast<const float4 *>(&xs[rc_xrow(i + 1) + tt + 4]);
                nw0 = *reinterpret_cast<const float4 *>(&ws[rc_wrow(i + 1) + ee]);
            }
            const float xa[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const float wb[4] = {w0.x, w0.y, w0.z, w0.w};
#pragma unroll
            for (int a = 0; a < 8; a++)
#pragma unroll
                for (int b = 0; b < 4; b++) acc[a][b] = fmaf(xa[a], wb[b], acc[a][b]);
        }
    }
    __syncthreads();  // the logits overwrite the tiles
#pragma unroll
    for (int a = 0; a < 8; a++)
        *reinterpret_cast<float4 *>(&lg[(tt + a) * RC_LGS + ee]) =
            make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    __syncthreads();
    const int ne = min(RC_EC, E - e0);   // experts of this CTA
    if (logits_out)
        for (int i = tid; i < RC_BT * ne; i += blockDim.x) {
            const int tl = i / ne, el = i - tl * ne;
            if (t0 + tl < T) logits_out[(int64_t)(t0 + tl) * E + e0 + el] = lg[tl * RC_LGS + el];
        }

    // ---- per-CTA top-k of each token over its 128 experts; candidates to CTA 0 ----
    const int nc = ncta * k;
    for (int tl = warp * (RC_BT / nw); tl < (warp + 1) * (RC_BT / nw); tl++) {
        if (t0 + tl >= T) break;
        float vals[4];
        int idx[4];
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const int el = m * 32 + lane;
            vals[m] = el < ne ? lg[tl * RC_LGS + el] : 0.0f;
            idx[m] = el < ne ? e0 + el : -1;
        }
        float v;
        int i;
        warp_topk<4>(vals, idx, k, lane, v, i);
        if (lane < k) cl_st_f2(cl_map(&cand[tl * nc + rank * k + lane], 0), v, __int_as_float(i));
        if (score_fn == MOE_SCORE_SOFTMAX && !renorm) {
            // this CTA's share of the full softmax denominator, as (max, sum exp(l - max))
            float mloc = -INFINITY;
#pragma unroll
            for (int m = 0; m < 4; m++)
                if (idx[m] >= 0) mloc = fmaxf(mloc, vals[m]);
            mloc = warp_max(mloc);
            float sloc = 0.0f;
#pragma unroll
            for (int m = 0; m < 4; m++)
                if (idx[m] >= 0) sloc += expf(vals[m] - mloc);
            sloc = warp_sum(sloc);
            if (lane == 0) cl_st_f2(cl_map(&msum[tl * ncta + rank], 0), mloc, sloc);
        }
    }
    cl_sync();  // every candidate has reached CTA 0; nothing is written remotely after this
    if (rank != 0) return;

    // ---- CTA 0: merge the clusters' candidates, gates, outputs ----
    for (int tl = warp * (RC_BT / nw); tl < (warp + 1) * (RC_BT / nw); tl++) {
        const int t = t0 + tl;
        if (t >= T) break;
        float vals[8];
        int idx[8];
#pragma unroll
        for (int m = 0; m < 8; m++) {
            const int c = m * 32 + lane;
            const float2 cv = c < nc ? cand[tl * nc + c] : make_float2(0.0f, __int_as_float(-1));
            vals[m] = cv.x;
            idx[m] = __float_as_int(cv.y);
        }
        float my_l;
        int my_id;
        warp_topk<8>(vals, idx, k, lane, my_l, my_id);
        float full_max = 0.0f, full_sum = 0.0f;
        if (score_fn == MOE_SCORE_SOFTMAX && !renorm) {
            float M = -INFINITY;
            for (int r = 0; r < ncta; r++) M = fmaxf(M, msum[tl * ncta + r].x);
            float S = 0.0f;
            for (int r = 0; r < ncta; r++) S += msum[tl * ncta + r].y * expf(msum[tl * ncta + r].x - M);
            full_max = M;
            full_sum = S;
        }
        const float g = warp_gate(lane, k, lane < k ? my_l : 0.0f, score_fn, renorm, route_scale, full_max, full_sum);
        if (lane < k) {
            ids[(int64_t)t * k + lane] = my_id;
            gates[(int64_t)t * k + lane] = g;
            if (capture) capture[(int64_t)lane * T + t] = my_id;
        }
    }
}

// V hidden values of a bf16 row, V = 8 (one 16-byte load) or 16 (one
// 32-byte load: a whole sector per lane; the address 32-byte aligned)
template <int V>
struct Bf16Vec {
    uint4 v[V / 8];
};
template <int V>
__device__ __forceinline__ Bf16Vec<V> ldg_bf16(const uint16_t *p)
{
    Bf16Vec<V> r;
    if constexpr (V == 8) {
        r.v[0] = __ldg(reinterpret_cast<const uint4 *>(p));
    } else {
        asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=r"(r.v[0].x), "=r"(r.v[0].y), "=r"(r.v[0].z), "=r"(r.v[0].w), "=r"(r.v[1].x), "=r"(r.v[1].y),
              "=r"(r.v[1].z), "=r"(r.v[1].w)
            : "l"(p));
    }
    return r;
}

// Replay.  CTA = 256 threads for up to 256/TP tokens, TP = threads per token
// (2, 4 or 8, a power of two with TP * 4 >= k); CTA b of the grid takes
// tokens floor(b*T/grid) .. floor((b+1)*T/grid) - 1, the grid a whole number
// of waves of two CTAs per SM, so every SM gets the same number of tokens.
// Copies the layer slab [k, T] to [T, k] and checks the ids; if x is given,
// thread (token, part q) evaluates the router logits of the token's slots
// q*SP .. q*SP+SP-1 (SP = ceil(k/TP)
// <= 4) -- one fma chain per slot in ascending hidden index, as in
// route_topk_kernel -- so every x value it loads feeds SP chains.  x and the
// replayed W_r rows are read straight from L1/L2, V bf16 per load (V = 16
// when both are 32-byte aligned: every load a whole sector), one step
// ahead.  Gates come from warp_gate, the routing kernel's code.
// IdT is the payload's id type: int32 or one byte (the compacted payload).
// BWD: the router backward's first step -- the ids come as [T, k] (replay_kT
// points at them; nothing is copied), the same logits are formed, and the
// kernel writes d_logits (into `gates`) from the upstream d_gates through
// warp_dgate instead of the gates.
template <int TP, int V, typename IdT, bool BWD = false>
__global__ void __launch_bounds__(256, 2) route_replay_kernel(const IdT *__restrict__ replay_kT,
                                                           const uint16_t *__restrict__ x,
                                                           const uint16_t *__restrict__ wr, int T, int d, int E,
                                                           int k, int score_fn, int renorm, float route_scale,
                                                           int32_t *__restrict__ ids,
                                                           float *__restrict__ gates,
                                                           int32_t *__restrict__ dev_status,
                                                           const float *__restrict__ d_gates = nullptr)
{
    constexpr int TPC = 256 / TP;  // tokens per CTA
    __shared__ int32_t sid[TPC * 32];
    __shared__ float slg[TPC * 32];
    __shared__ int sbad[TPC];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = (int)((int64_t)blockIdx.x * T / gridDim.x);
    const int nt = (int)((int64_t)(blockIdx.x + 1) * T / gridDim.x) - t0;  // <= TPC

    if (BWD) {
        for (int idx = tid; idx < nt * k; idx += blockDim.x) sid[idx] = (int32_t)replay_kT[(int64_t)t0 * k + idx];
    } else {
        for (int idx = tid; idx < TPC * k; idx += blockDim.x) {
            const int j = idx / TPC, tl = idx % TPC;
            if (tl < nt) {
                const int32_t v = (int32_t)replay_kT[(int64_t)j * T + t0 + tl];
                sid[tl * k + j] = v;
                ids[(int64_t)(t0 + tl) * k + j] = v;
            }
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

    const int SP = (k + TP - 1) / TP;
    const int tl = tid / TP, q = tid % TP;
    const bool tok_ok = tl < nt;
    const uint16_t *xrow = x + (int64_t)(t0 + (tok_ok ? tl : 0)) * d;
    const uint16_t *wrow[4];
    bool on[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int j = q * SP + u;
        const int32_t e = (tok_ok && u < SP && j < k) ? sid[tl * k + j] : -1;
        on[u] = e >= 0 && e < E;
        wrow[u] = wr + (int64_t)(on[u] ? e : 0) * d;
    }
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (tok_ok) {
        const Bf16Vec<V> zero = {};
        Bf16Vec<V> cx = ldg_bf16<V>(xrow), cw[4];
#pragma unroll
        for (int u = 0; u < 4; u++) cw[u] = on[u] ? ldg_bf16<V>(wrow[u]) : zero;
        for (int i = 0; i < d; i += V) {
            Bf16Vec<V> nx = zero, nw[4];
            const bool more = i + V < d;
            if (more) nx = ldg_bf16<V>(xrow + i + V);
#pragma unroll
            for (int u = 0; u < 4; u++) nw[u] = (more && on[u]) ? ldg_bf16<V>(wrow[u] + i + V) : zero;
#pragma unroll
            for (int h = 0; h < V / 8; h++) {
                float xf[8];
                unpack_bf16x8(cx.v[h], xf);
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    if (!on[u]) continue;
                    float wf[8];
                    unpack_bf16x8(cw[u].v[h], wf);
                    float a = acc[u];
#pragma unroll
                    for (int jj = 0; jj < 8; jj++) a = fmaf(xf[jj], wf[jj], a);
                    acc[u] = a;
                }
            }
            cx = nx;
#pragma unroll
            for (int u = 0; u < 4; u++) cw[u] = nw[u];
        }
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int j = q * SP + u;
        if (tok_ok && u < SP && j < k) slg[tl * k + j] = acc[u];
    }
    __syncthreads();
    for (int t = warp; t < nt; t += 8) {
        const float my_l = lane < k ? slg[t * k + lane] : 0.0f;
        float g;
        if (BWD) {
            const float my_dg = lane < k ? d_gates[(int64_t)(t0 + t) * k + lane] : 0.0f;
            g = warp_dgate(lane, k, my_l, my_dg, score_fn, renorm, route_scale);
        } else {
            g = warp_gate(lane, k, my_l, score_fn, renorm, route_scale, 0.0f, 0.0f);
        }
        if (sbad[t]) g = 0.0f;
        if (lane < k) gates[(int64_t)(t0 + t) * k + lane] = g;
    }
}

// dx[t, c] = sum_j d_logits[t, j] * W_r[ids[t, j], c], the slots in order,
// fp32.  One warp per token; lane l takes columns 8 (l + 32 i) .. + 7, the
// k router rows (L2-resident) read 16 bytes at a time (two chunks per pass
// measured slower).  A slot whose id is
// outside [0, E) is skipped (its d_logit is 0).
__global__ void __launch_bounds__(256) router_dx_kernel(const int32_t *__restrict__ ids,
                                                        const float *__restrict__ d_logits,
                                                        const uint16_t *__restrict__ wr, int T, int d, int E, int k,
                                                        float *__restrict__ dx)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const int32_t my_id = lane < k ? ids[t * k + lane] : -1;
    const float my_dl = lane < k ? d_logits[t * k + lane] : 0.0f;
    for (int c = 8 * lane; c < d; c += 256) {
        float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        for (int j = 0; j < k; j++) {
            const int32_t e = __shfl_sync(0xFFFFFFFFu, my_id, j);
            const float g = __shfl_sync(0xFFFFFFFFu, my_dl, j);
            if (e < 0 || e >= E) continue;
            float w[8];
            unpack_bf16x8(__ldg(reinterpret_cast<const uint4 *>(wr + (int64_t)e * d + c)), w);
#pragma unroll
            for (int i = 0; i < 8; i++) acc[i] = fmaf(g, w[i], acc[i]);
        }
        float4 *o = reinterpret_cast<float4 *>(dx + t * d + c);
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// dw[e, c] = sum over expert e's dispatched rows r (sorted order) of
// d_logits[slot(r)] * x[slot(r) / k, c], fp32, the rows in order.  One CTA
// of 128 threads per (expert, 1024 columns); thread i takes columns
// 8 i .. 8 i + 7 of its chunk.  The rows' (token, d_logit) pairs are staged
// in shared memory 128 at a time (one slot load and division per row for
// the CTA), then every thread walks them with four rows' x loads in flight.
// A slot outside [0, T k) adds nothing; an expert without rows gets zeros.
// Offsets outside [0, T k], or decreasing, are clamped into that range (no
// read past the map) and set MOE_DEV_ROWS.
constexpr int RDW_COLS = 1024;
constexpr int RDW_BATCH = 128;
__global__ void __launch_bounds__(128) router_dw_kernel(const int32_t *__restrict__ sorted_to_slot,
                                                        const int32_t *__restrict__ offsets,
                                                        const float *__restrict__ d_logits,
                                                        const uint16_t *__restrict__ x, int T, int d, int k,
                                                        float *__restrict__ dw, int32_t *dev_status)
{
    __shared__ int32_t s_tok[RDW_BATCH];
    __shared__ float s_g[RDW_BATCH];
    const int e = blockIdx.y;
    const int c = blockIdx.x * RDW_COLS + 8 * threadIdx.x;
    const bool col_ok = c < d;
    const int64_t A = (int64_t)T * k, o0 = __ldg(offsets + e), o1 = __ldg(offsets + e + 1);
    const int64_t r0 = o0 < 0 ? 0 : (o0 > A ? A : o0);
    const int64_t r1 = o1 < r0 ? r0 : (o1 > A ? A : o1);
    if ((r0 != o0 || r1 != o1) && blockIdx.x == 0 && threadIdx.x == 0) dev_flag(dev_status, MOE_DEV_ROWS);
    float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    for (int64_t b0 = r0; b0 < r1; b0 += RDW_BATCH) {
        const int nb = (int)(r1 - b0 < RDW_BATCH ? r1 - b0 : RDW_BATCH);
        __syncthreads();                                   // the previous batch has been read
        if ((int)threadIdx.x < nb) {
            const int32_t slot = __ldg(sorted_to_slot + b0 + threadIdx.x);
            const bool ok = slot >= 0 && slot < A;
            s_tok[threadIdx.x] = ok ? slot / k : -1;
            s_g[threadIdx.x] = ok ? __ldg(d_logits + slot) : 0.0f;
        }
        __syncthreads();
        if (!col_ok) continue;
        for (int i = 0; i < nb; i += 4) {
            float g[4];
            uint4 xv[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int tok = i + u < nb ? s_tok[i + u] : -1;
                g[u] = i + u < nb ? s_g[i + u] : 0.0f;
                xv[u] = tok >= 0 ? __ldg(reinterpret_cast<const uint4 *>(x + (int64_t)tok * d + c))
                                 : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 4; u++) {
                if (i + u >= nb) break;
                float xf[8];
                unpack_bf16x8(xv[u], xf);
#pragma unroll
                for (int j = 0; j < 8; j++) acc[j] = fmaf(g[u], xf[j], acc[j]);
            }
        }
    }
    if (!col_ok) return;
    float4 *o = reinterpret_cast<float4 *>(dw + (int64_t)e * d + c);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
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
    const int ncta = (E + RC_EC - 1) / RC_EC;  // <= 8: a portable cluster size
    const size_t smem = sizeof(float) * (size_t)RC_TILE_FLOATS +
                        sizeof(float2) * ((size_t)RC_BT * ncta * k + (size_t)RC_BT * ncta);
    if (cudaFuncSetAttribute(route_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ncta;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(((T + RC_BT - 1) / RC_BT) * ncta));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = as_stream(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, route_topk_kernel, x, w_router, T, d, E, k, score_fn, renorm, route_scale,
                           topk_ids, topk_gates, capture_kT, logits_out) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_status();
}

namespace moe {

// grid of the replay kernel: ceil(T / tpc) CTAs rounded up to a whole number
// of waves of two CTAs per SM (the kernel's launch bound), at most T
static unsigned replay_grid(int T, int tpc)
{
    const int64_t need = (T + tpc - 1) / tpc, wave = 2LL * sm_count();
    const int64_t g = (need + wave - 1) / wave * wave;
    return (unsigned)(g < T ? g : T);
}

template <int V, typename IdT>
static void replay_launch_tp(const IdT *replay_kT, const uint16_t *x, const uint16_t *w_router, int T, int d, int E,
                             int k, int score_fn, int renorm, float route_scale, int32_t *topk_ids,
                             float *topk_gates, int32_t *dev_status, cudaStream_t st)
{
    if (k <= 8) {
        route_replay_kernel<2, V, IdT><<<replay_grid(T, 128), 256, 0, st>>>(replay_kT, x, w_router, T, d, E, k,
                                                                             score_fn, renorm, route_scale,
                                                                             topk_ids, topk_gates, dev_status);
    } else if (k <= 16) {
        route_replay_kernel<4, V, IdT><<<replay_grid(T, 64), 256, 0, st>>>(replay_kT, x, w_router, T, d, E, k,
                                                                            score_fn, renorm, route_scale,
                                                                            topk_ids, topk_gates, dev_status);
    } else {
        route_replay_kernel<8, V, IdT><<<replay_grid(T, 32), 256, 0, st>>>(replay_kT, x, w_router, T, d, E, k,
                                                                            score_fn, renorm, route_scale,
                                                                            topk_ids, topk_gates, dev_status);
    }
}

template <typename IdT>
static moe_status replay_launch(const IdT *replay_kT, const uint16_t *x, const uint16_t *w_router, int T, int d,
                                int E, int k, int score_fn, int renorm, float route_scale, int32_t *topk_ids,
                                float *topk_gates, int32_t *dev_status, void *stream)
{
    moe_status s = check_route_args(T, d, E, k, score_fn);
    if (s != MOE_OK) return s;
    if (x && score_fn == MOE_SCORE_SOFTMAX && !renorm) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!replay_kT || !topk_ids) return MOE_ERR_NULL;
    if (x && (!w_router || !topk_gates)) return MOE_ERR_NULL;
    if (x && (!aligned16(x) || !aligned16(w_router))) return MOE_ERR_ALIGN;
    cudaStream_t st = as_stream(stream);
    // 32-byte loads when the rows allow them (d is a multiple of 128)
    const bool wide = x && (reinterpret_cast<uintptr_t>(x) & 31u) == 0 &&
                      (reinterpret_cast<uintptr_t>(w_router) & 31u) == 0;
    if (wide)
        replay_launch_tp<16>(replay_kT, x, w_router, T, d, E, k, score_fn, renorm, route_scale, topk_ids,
                             topk_gates, dev_status, st);
    else
        replay_launch_tp<8>(replay_kT, x, w_router, T, d, E, k, score_fn, renorm, route_scale, topk_ids,
                            topk_gates, dev_status, st);
    return launch_status();
}

} // namespace moe

MOE_API moe_status moe_route_replay(const int32_t *replay_kT, const uint16_t *x, const uint16_t *w_router,
                                    int T, int d, int E, int k, int score_fn, int renorm, float route_scale,
                                    int32_t *topk_ids, float *topk_gates, int32_t *dev_status, void *stream)
{
    return replay_launch(replay_kT, x, w_router, T, d, E, k, score_fn, renorm, route_scale, topk_ids, topk_gates,
                         dev_status, stream);
}

MOE_API moe_status moe_route_replay_u8(const uint8_t *replay_kT, const uint16_t *x, const uint16_t *w_router,
                                       int T, int d, int E, int k, int score_fn, int renorm, float route_scale,
                                       int32_t *topk_ids, float *topk_gates, int32_t *dev_status, void *stream)
{
    return replay_launch(replay_kT, x, w_router, T, d, E, k, score_fn, renorm, route_scale, topk_ids, topk_gates,
                         dev_status, stream);
}

namespace moe {

template <int V>
static void router_dlogits_launch(const int32_t *ids, const uint16_t *x, const uint16_t *w_router, int T, int d,
                                  int E, int k, int score_fn, int renorm, float route_scale, const float *d_gates,
                                  float *d_logits, int32_t *dev_status, cudaStream_t st)
{
    // four threads per token (two slot chains each for k <= 8): the
    // backward runs on a layer's T tokens, too few for two per token to
    // keep the SMs' loads in flight
    if (k <= 16)
        route_replay_kernel<4, V, int32_t, true><<<replay_grid(T, 64), 256, 0, st>>>(
            ids, x, w_router, T, d, E, k, score_fn, renorm, route_scale, nullptr, d_logits, dev_status, d_gates);
    else
        route_replay_kernel<8, V, int32_t, true><<<replay_grid(T, 32), 256, 0, st>>>(
            ids, x, w_router, T, d, E, k, score_fn, renorm, route_scale, nullptr, d_logits, dev_status, d_gates);
}

} // namespace moe

MOE_API moe_status moe_router_backward(const uint16_t *x, const uint16_t *w_router, const int32_t *topk_ids,
                                       const float *d_gates, int T, int d, int E, int k, int score_fn, int renorm,
                                       float route_scale, float *d_logits, float *dx,
                                       const int32_t *sorted_to_slot, const int32_t *expert_offsets,
                                       float *dw_router, int32_t *dev_status, void *stream)
{
    moe_status s = check_route_args(T, d, E, k, score_fn);
    if (s != MOE_OK) return s;
    if (score_fn == MOE_SCORE_SOFTMAX && !renorm) return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = as_stream(stream);
    if (T == 0) {   // no tokens (the [T, .] arrays may be NULL): dw_router is all zeros
        if (!dw_router) return MOE_OK;
        if (!aligned16(dw_router)) return MOE_ERR_ALIGN;
        return cudaMemsetAsync(dw_router, 0, sizeof(float) * (size_t)E * d, st) == cudaSuccess ? MOE_OK
                                                                                             : MOE_ERR_CUDA;
    }
    if (!x || !w_router || !topk_ids || !d_gates || !d_logits) return MOE_ERR_NULL;
    if (dw_router && (!sorted_to_slot || !expert_offsets)) return MOE_ERR_NULL;
    if (!aligned16(x) || !aligned16(w_router) || (dx && !aligned16(dx)) || (dw_router && !aligned16(dw_router)))
        return MOE_ERR_ALIGN;
    const bool wide = (reinterpret_cast<uintptr_t>(x) & 31u) == 0 && (reinterpret_cast<uintptr_t>(w_router) & 31u) == 0;
    if (wide)
        router_dlogits_launch<16>(topk_ids, x, w_router, T, d, E, k, score_fn, renorm, route_scale, d_gates, d_logits,
                                  dev_status, st);
    else
        router_dlogits_launch<8>(topk_ids, x, w_router, T, d, E, k, score_fn, renorm, route_scale, d_gates, d_logits,
                                 dev_status, st);
    if (dx) router_dx_kernel<<<(unsigned)(((int64_t)T * 32 + 255) / 256), 256, 0, st>>>(topk_ids, d_logits, w_router, T,
                                                                                      d, E, k, dx);
    if (dw_router)
        router_dw_kernel<<<dim3((unsigned)((d + RDW_COLS - 1) / RDW_COLS), (unsigned)E), 128, 0, st>>>(
            sorted_to_slot, expert_offsets, d_logits, x, T, d, k, dw_router, dev_status);
    return launch_status();
}
