// dispatch.cu -- expert-contiguous permutation of tokens (dispatch) and the
// gate-weighted sum back to token order (combine), the two local halves of
// expert parallelism ("RL at 1T Scale: prime-rl Performance Deep Dive",
// section "Parallelism", "Expert parallelism (EP)"; on one GPU there is no
// all-to-all, only the permutation).
//
// Dispatch is a stable counting sort of the slots s = t*k + j by expert:
//   hist_kernel     one warp per run of consecutive slots (128, or 1024 when
//                   the per-run counts of 128-slot runs would pass 1 MiB):
//                   per-run expert histogram in shared memory -> ws[e][run]
//   scan_kernel     one CTA per expert: exclusive prefix of ws[e][*] over
//                   runs (in place) and the expert total
//   scatter_kernel  one warp per run: exclusive scan of the totals (shared),
//                   per-warp running positions seeded from ws, then 32 slots
//                   at a time: __match_any_sync groups equal experts, a lane's
//                   rank is the number of lower lanes in its group -> the
//                   stable sorted position.  Writes both maps.
//   gather_kernel   one warp per token: the row is read from HBM once
//                   (16-byte vectors) and written to its k sorted positions.
// Combine is one warp per token: for each pair of 16-byte column vectors per
// lane the k source rows are loaded before the fma chain runs over j in slot
// order.
#include <atomic>

#include "common.cuh"

namespace moe {

constexpr int DSP_RUN_SHORT = 128;    // slots per warp run: short runs spread the map
constexpr int DSP_RUN_LONG = 1024;    // kernels over many warps; long runs bound ws
constexpr int DSP_WARPS = 8;

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__global__ void __launch_bounds__(256) hist_kernel(const int32_t *__restrict__ ids, int64_t A, int E,
                                                   int nruns, int run_len, int32_t *__restrict__ ws,
                                                   int32_t *__restrict__ dev_status)
{
    extern __shared__ int32_t hist[];  // [DSP_WARPS][E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *h = hist + warp * E;
    for (int e = lane; e < E; e += 32) h[e] = 0;
    __syncwarp();
    const int run = blockIdx.x * DSP_WARPS + warp;
    bool bad = false;
    if (run < nruns) {
        const int64_t s0 = (int64_t)run * run_len;
        const int64_t s1 = min(s0 + run_len, A);
        for (int64_t s = s0 + lane; s < s1; s += 32) {
            const int32_t e = __ldg(ids + s);
            if (e >= 0 && e < E)
                atomicAdd(h + e, 1);
            else
                bad = true;
        }
        __syncwarp();
        for (int e = lane; e < E; e += 32) ws[(int64_t)e * nruns + run] = h[e];
    }
    if (bad) dev_flag(dev_status, MOE_DEV_BAD_IDS);
}

__global__ void __launch_bounds__(256) scan_kernel(int32_t *__restrict__ ws, int nruns,
                                                   int32_t *__restrict__ counts)
{
    __shared__ int32_t wsum[8];
    const int e = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t *col = ws + (int64_t)e * nruns;
    int32_t carry = 0;
    for (int base = 0; base < nruns; base += 256) {
        const int i = base + tid;
        const int32_t v = i < nruns ? col[i] : 0;
        int32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        int32_t before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < 8; w++) {
            if (w < warp) before += wsum[w];
            total += wsum[w];
        }
        if (i < nruns) col[i] = carry + before + incl - v;
        carry += total;
        __syncthreads();
    }
    if (tid == 0) counts[e] = carry;
}

// exclusive scan of counts[0..E) into off[0..E], by one CTA of 256 threads
__device__ void block_offsets(const int32_t *__restrict__ counts, int E, int32_t *off, int32_t *wsum)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t carry = 0;
    for (int base = 0; base < E; base += 256) {
        const int i = base + tid;
        const int32_t v = i < E ? counts[i] : 0;
        int32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        int32_t before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < 8; w++) {
            if (w < warp) before += wsum[w];
            total += wsum[w];
        }
        if (i < E) off[i] = carry + before + incl - v;
        carry += total;
        __syncthreads();
    }
    if (tid == 0) off[E] = carry;
    __syncthreads();
}

__global__ void __launch_bounds__(256) scatter_kernel(const int32_t *__restrict__ ids, int64_t A, int E,
                                                      int nruns, int run_len, const int32_t *__restrict__ ws,
                                                      const int32_t *__restrict__ counts,
                                                      int32_t *__restrict__ expert_counts,
                                                      int32_t *__restrict__ expert_offsets,
                                                      int32_t *__restrict__ sorted_to_slot,
                                                      int32_t *__restrict__ slot_to_sorted)
{
    extern __shared__ int32_t sm[];
    int32_t *off = sm;                    // [E+1]
    int32_t *wsum = off + E + 1;          // [8]
    int32_t *pos = wsum + 8;              // [DSP_WARPS][E]
    block_offsets(counts, E, off, wsum);
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e <= E; e += blockDim.x) {
            expert_offsets[e] = off[e];
            if (e < E) expert_counts[e] = off[e + 1] - off[e];
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int run = blockIdx.x * DSP_WARPS + warp;
    if (run >= nruns) return;
    int32_t *p = pos + warp * E;
    for (int e = lane; e < E; e += 32) p[e] = off[e] + ws[(int64_t)e * nruns + run];
    __syncwarp();
    const int64_t s0 = (int64_t)run * run_len;
    const int64_t s1 = min(s0 + run_len, A);
    const unsigned lt = lanemask_lt();
    for (int64_t sb = s0; sb < s1; sb += 32) {
        const int64_t s = sb + lane;
        const int32_t e = s < s1 ? __ldg(ids + s) : -1;
        const bool ok = e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, ok ? e : -1);
        int32_t r = -1;
        if (ok) r = p[e] + __popc(peers & lt);
        __syncwarp();
        if (ok && (peers & lt) == 0) p[e] += __popc(peers);
        __syncwarp();
        if (s < s1) {
            slot_to_sorted[s] = r;
            if (ok) sorted_to_slot[r] = (int32_t)s;
        }
    }
}

// rows_sorted[r] = rows[sorted_to_slot[r] / k]: one warp per token reads its
// row once and writes it to the token's k sorted positions.
__global__ void __launch_bounds__(256) gather_kernel(const uint8_t *__restrict__ rows, int64_t row_bytes,
                                                     const float *__restrict__ row_scales, int spr,
                                                     const int32_t *__restrict__ slot_to_sorted, int T, int k,
                                                     uint8_t *__restrict__ rows_sorted,
                                                     float *__restrict__ scales_sorted)
{
    const int lane = threadIdx.x & 31;
    const int64_t nvec = row_bytes >> 4;
    const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t t = gw; t < T; t += nw) {
        const int32_t my_dst = lane < k ? __ldg(slot_to_sorted + t * k + lane) : -1;
        const uint4 *src = reinterpret_cast<const uint4 *>(rows + t * row_bytes);
        for (int64_t v0 = 0; v0 < nvec; v0 += 128) {
            uint4 buf[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int64_t v = v0 + u * 32 + lane;
                if (v < nvec) buf[u] = __ldcs(src + v);
            }
            for (int j = 0; j < k; j++) {
                const int32_t dst = __shfl_sync(0xFFFFFFFFu, my_dst, j);
                if (dst < 0) continue;
                uint4 *out = reinterpret_cast<uint4 *>(rows_sorted + (int64_t)dst * row_bytes);
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const int64_t v = v0 + u * 32 + lane;
                    if (v < nvec) __stcs(out + v, buf[u]);
                }
            }
        }
        for (int c0 = 0; c0 < spr; c0 += 32) {
            const int c = c0 + lane;
            const float sv = c < spr ? __ldg(row_scales + t * spr + c) : 0.0f;
            for (int j = 0; j < k; j++) {
                const int32_t dst = __shfl_sync(0xFFFFFFFFu, my_dst, j);
                if (dst >= 0 && c < spr) scales_sorted[(int64_t)dst * spr + c] = sv;
            }
        }
    }
}

// y[t] = bf16( sum_j g[t,j] * out_sorted[slot_to_sorted[t*k+j]] ), fma chain
// over j in slot order from +0.  One warp per token; each lane owns two
// 16-byte column vectors (v, v + 32) per pass and has all 2 x 8 source loads
// in flight before the first fma (16 x 16 B per lane keeps enough bytes in
// flight to saturate HBM).  k > 8 runs the slots in groups of 8, in order.
// SLOTS: the expert outputs are stored in slot order (row t*k + j), and
// slot_to_sorted only says which slots were routed (>= 0).  Map entries
// outside [0, T*k) are skipped, so a corrupt map never reads outside the
// expert outputs.
template <bool SLOTS>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t *__restrict__ out_sorted,
                                                      const int32_t *__restrict__ slot_to_sorted,
                                                      const float *__restrict__ gates, int T, int k, int d,
                                                      uint16_t *__restrict__ y)
{
    const int lane = threadIdx.x & 31;
    const int nvec = d >> 3;  // 8 bf16 per 16-byte vector
    const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t t = gw; t < T; t += nw) {
        int32_t my_src = lane < k ? __ldg(slot_to_sorted + t * k + lane) : -1;
        // out_sorted holds at most T*k rows: an entry past them (a map not
        // written by moe_dispatch) is read as an unrouted slot
        if ((int64_t)my_src >= (int64_t)T * k) my_src = -1;
        if (SLOTS && my_src >= 0) my_src = (int32_t)(t * k + lane);
        const float my_g = lane < k ? (gates ? __ldg(gates + t * k + lane) : 1.0f) : 0.0f;  // no gates: unit
        for (int v0 = 0; v0 < nvec; v0 += 64) {
            float acc[2][8];
#pragma unroll
            for (int h = 0; h < 2; h++)
#pragma unroll
                for (int i = 0; i < 8; i++) acc[h][i] = 0.0f;
            for (int j0 = 0; j0 < k; j0 += 8) {
                int32_t src[8];
                float g[8];
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    src[u] = __shfl_sync(0xFFFFFFFFu, my_src, (j0 + u) & 31);
                    g[u] = __shfl_sync(0xFFFFFFFFu, my_g, (j0 + u) & 31);
                    if (j0 + u >= k) src[u] = -1;
                }
                uint4 buf[2][8];
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int v = v0 + h * 32 + lane;
#pragma unroll
                    for (int u = 0; u < 8; u++)
                        if (src[u] >= 0 && v < nvec)
                            buf[h][u] = __ldcs(reinterpret_cast<const uint4 *>(out_sorted + (int64_t)src[u] * d) + v);
                }
#pragma unroll
                for (int h = 0; h < 2; h++) {
#pragma unroll
                    for (int u = 0; u < 8; u++) {
                        if (src[u] < 0) continue;
                        float f[8];
                        unpack_bf16x8(buf[h][u], f);
#pragma unroll
                        for (int i = 0; i < 8; i++) acc[h][i] = fmaf(g[u], f[i], acc[h][i]);
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int v = v0 + h * 32 + lane;
                if (v >= nvec) continue;
                uint4 o;
                o.x = pack_bf16x2(acc[h][0], acc[h][1]);
                o.y = pack_bf16x2(acc[h][2], acc[h][3]);
                o.z = pack_bf16x2(acc[h][4], acc[h][5]);
                o.w = pack_bf16x2(acc[h][6], acc[h][7]);
                __stcs(reinterpret_cast<uint4 *>(y + t * d) + v, o);
            }
        }
    }
}

static inline int dsp_run_len(int64_t A, int E)
{
    const int64_t short_runs = (A + DSP_RUN_SHORT - 1) / DSP_RUN_SHORT;
    return (int64_t)E * short_runs * 4 <= (1 << 20) ? DSP_RUN_SHORT : DSP_RUN_LONG;
}
static inline int dsp_nruns(int64_t A, int E)
{
    const int rl = dsp_run_len(A, E);
    return (int)((A + rl - 1) / rl);
}

} // namespace moe

using namespace moe;

MOE_API size_t moe_dispatch_workspace_size(int T, int k, int E)
{
    if (T < 0 || k < 1 || E < 1) return 0;
    const int64_t A = (int64_t)T * k;
    const size_t runs = (size_t)dsp_nruns(A, E);
    const size_t a = sizeof(int32_t) * (size_t)E * (runs > 0 ? runs : 1);  // ws[E][runs]
    const size_t b = sizeof(int32_t) * (size_t)E;                         // totals
    return ((a + 255) & ~(size_t)255) + ((b + 255) & ~(size_t)255);
}

MOE_API moe_status moe_dispatch(const int32_t *topk_ids, int T, int k, int E, const void *rows,
                                int64_t row_bytes, const float *row_scales, int scales_per_row,
                                int32_t *expert_counts, int32_t *expert_offsets, int32_t *sorted_to_slot,
                                int32_t *slot_to_sorted, void *rows_sorted, float *scales_sorted,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    if (T < 0 || k < 1 || k > 32 || E < 1 || E > 1024) return MOE_ERR_SHAPE;
    const int64_t A = (int64_t)T * k;
    if (A >= (1LL << 31)) return MOE_ERR_SHAPE;
    if (!expert_counts || !expert_offsets) return MOE_ERR_NULL;
    const bool with_rows = rows != nullptr || rows_sorted != nullptr;
    if (with_rows) {
        if (!rows || !rows_sorted) return MOE_ERR_NULL;
        if (row_bytes <= 0 || row_bytes % 16 != 0) return MOE_ERR_SHAPE;
        if (!aligned16(rows) || !aligned16(rows_sorted)) return MOE_ERR_ALIGN;
        if (scales_per_row < 0) return MOE_ERR_SHAPE;
        if (scales_per_row > 0 && (!row_scales || !scales_sorted)) return MOE_ERR_NULL;
    }
    if (A > 0 && (!topk_ids || !sorted_to_slot || !slot_to_sorted)) return MOE_ERR_NULL;
    const size_t need = moe_dispatch_workspace_size(T, k, E);
    if (!workspace || workspace_bytes < need) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MOE_ERR_ALIGN;
    cudaStream_t st = as_stream(stream);
    const int nruns = dsp_nruns(A, E);
    const int run_len = dsp_run_len(A, E);
    int32_t *ws = reinterpret_cast<int32_t *>(workspace);
    int32_t *totals =
        reinterpret_cast<int32_t *>(reinterpret_cast<char *>(workspace) +
                                    ((sizeof(int32_t) * (size_t)E * (nruns > 0 ? nruns : 1) + 255) & ~(size_t)255));
    if (A == 0) {
        if (cudaMemsetAsync(totals, 0, sizeof(int32_t) * E, st) != cudaSuccess) return MOE_ERR_CUDA;
    } else {
        const int grid = (nruns + DSP_WARPS - 1) / DSP_WARPS;
        hist_kernel<<<grid, 256, sizeof(int32_t) * DSP_WARPS * E, st>>>(topk_ids, A, E, nruns, run_len, ws,
                                                                        dev_status);
        scan_kernel<<<E, 256, 0, st>>>(ws, nruns, totals);
    }
    const size_t ssm = sizeof(int32_t) * ((size_t)E + 1 + 8 + (size_t)DSP_WARPS * E);
    const int sgrid = A == 0 ? 1 : (nruns + DSP_WARPS - 1) / DSP_WARPS;
    scatter_kernel<<<sgrid, 256, ssm, st>>>(topk_ids, A, E, nruns, run_len, ws, totals, expert_counts,
                                            expert_offsets, sorted_to_slot, slot_to_sorted);
    if (with_rows && T > 0) {
        int64_t grid = ((int64_t)T + 7) / 8;
        const int64_t cap = (int64_t)sm_count() * 8;
        if (grid > cap) grid = cap;
        gather_kernel<<<(unsigned)grid, 256, 0, st>>>(reinterpret_cast<const uint8_t *>(rows), row_bytes,
                                                      row_scales, scales_per_row, slot_to_sorted, T, k,
                                                      reinterpret_cast<uint8_t *>(rows_sorted), scales_sorted);
    }
    return launch_status();
}

MOE_API moe_status moe_combine(const uint16_t *out_sorted, const int32_t *slot_to_sorted, const float *gates,
                               int T, int k, int d, uint16_t *y, void *stream)
{
    if (T < 0 || k < 1 || k > 32 || d <= 0 || d % 8 != 0) return MOE_ERR_SHAPE;
    if (T == 0) return MOE_OK;
    if (!out_sorted || !slot_to_sorted || !gates || !y) return MOE_ERR_NULL;
    if (!aligned16(out_sorted) || !aligned16(y)) return MOE_ERR_ALIGN;
    int64_t grid = ((int64_t)T + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (grid > cap) grid = cap;
    combine_kernel<false><<<(unsigned)grid, 256, 0, as_stream(stream)>>>(out_sorted, slot_to_sorted, gates, T, k, d, y);
    return launch_status();
}

MOE_API moe_status moe_dispatch_backward(const uint16_t *dx_sorted, const int32_t *slot_to_sorted, int T, int k,
                                         int d, uint16_t *dx, void *stream)
{
    if (T < 0 || k < 1 || k > 32 || d <= 0 || d % 8 != 0) return MOE_ERR_SHAPE;
    if (T == 0) return MOE_OK;
    if (!dx_sorted || !slot_to_sorted || !dx) return MOE_ERR_NULL;
    if (!aligned16(dx_sorted) || !aligned16(dx)) return MOE_ERR_ALIGN;
    int64_t grid = ((int64_t)T + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (grid > cap) grid = cap;
    // the combine with unit gates: fma(1, v, acc) is the binary32 sum in slot order
    combine_kernel<false><<<(unsigned)grid, 256, 0, as_stream(stream)>>>(dx_sorted, slot_to_sorted, nullptr, T, k, d,
                                                                         dx);
    return launch_status();
}

MOE_API moe_status moe_combine_slots(const uint16_t *out_slots, const int32_t *slot_to_sorted, const float *gates,
                                     int T, int k, int d, uint16_t *y, void *stream)
{
    if (T < 0 || k < 1 || k > 32 || d <= 0 || d % 8 != 0) return MOE_ERR_SHAPE;
    if (T == 0) return MOE_OK;
    if (!out_slots || !slot_to_sorted || !gates || !y) return MOE_ERR_NULL;
    if (!aligned16(out_slots) || !aligned16(y)) return MOE_ERR_ALIGN;
    int64_t grid = ((int64_t)T + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (grid > cap) grid = cap;
    combine_kernel<true><<<(unsigned)grid, 256, 0, as_stream(stream)>>>(out_slots, slot_to_sorted, gates, T, k, d, y);
    return launch_status();
}

// ---------------------------------------------------------------------------
// moe_dispatch_noalloc: moe_dispatch with its scratch in a static device array
// of this library, for callers that cannot lend a workspace (see moe_r3.h).
// The array is a fixed MOE_DISPATCH_NOALLOC_MAX_SCRATCH bytes on every device
// that loads the library and stays allocated until the process exits.  All
// calls share it, so two calls whose work overlaps on the GPU (different
// streams, or different host threads) race on it.  No word of it needs to
// start at zero: every word the dispatch kernels read was written earlier in
// the same call, so the contents left by the previous call do not matter.

namespace moe {

static __device__ __align__(256) uint8_t g_dispatch_scratch[MOE_DISPATCH_NOALLOC_MAX_SCRATCH];

// Device address of g_dispatch_scratch on the current device.  In host code
// the array's name is only a host-side stand-in; the device address comes
// from cudaGetSymbolAddress, queried once per device (with that device
// current) and kept in a per-device slot.  Concurrent first calls store the
// same value.
static void *dispatch_scratch_address()
{
    static std::atomic<void *> slot[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    if (dev >= 0 && dev < 64) {
        void *p = slot[dev].load(std::memory_order_acquire);
        if (p) return p;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (dev >= 0 && dev < 64) slot[dev].store(p, std::memory_order_release);
    return p;
}

} // namespace moe

MOE_API moe_status moe_dispatch_noalloc(const int32_t *topk_ids, int T, int k, int E, const void *rows,
                                        int64_t row_bytes, const float *row_scales, int scales_per_row,
                                        int32_t *expert_counts, int32_t *expert_offsets, int32_t *sorted_to_slot,
                                        int32_t *slot_to_sorted, void *rows_sorted, float *scales_sorted,
                                        int32_t *dev_status, void *stream)
{
    if (T < 0 || k < 1 || k > 32 || E < 1 || E > 1024) return MOE_ERR_SHAPE;
    if ((int64_t)T * k >= (1LL << 31)) return MOE_ERR_SHAPE;
    if (moe_dispatch_workspace_size(T, k, E) > (size_t)MOE_DISPATCH_NOALLOC_MAX_SCRATCH) return MOE_ERR_WORKSPACE;
    void *scratch = dispatch_scratch_address();
    if (!scratch) return MOE_ERR_CUDA;
    return moe_dispatch(topk_ids, T, k, E, rows, row_bytes, row_scales, scales_per_row, expert_counts,
                        expert_offsets, sorted_to_slot, slot_to_sorted, rows_sorted, scales_sorted, scratch,
                        (size_t)MOE_DISPATCH_NOALLOC_MAX_SCRATCH, dev_status, stream);
}
