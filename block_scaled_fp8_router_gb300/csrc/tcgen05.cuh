// tcgen05.cuh -- building blocks shared by the grouped block-scaled GEMM
// kernels (grouped_ffn.cu, nvfp4_ffn.cu): tile constants, inline-PTX
// wrappers for TMA, mbarriers and the 5th-generation tensor cores (tcgen05
// MMA, TMEM load / alloc / commit), the device-resident tile schedule built
// from the expert offsets, and the host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace moe {
namespace ffn {

constexpr int BM = 128;                 // rows per tile (MMA M)
constexpr int BN = 256;                 // accumulator columns per tile (MMA N)
constexpr int BK = 128;                 // K block = one scale block (bytes of E4M3)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;        // 16 KB
constexpr int B_BYTES = BN * BK;        // 32 KB
constexpr int EPI_WARPS = 16;
constexpr int PRODUCER_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int THREADS = 18 * 32;
constexpr int TMEM_COLS = 512;          // two 256-column fp32 buffers
constexpr int MAX_E = 1024;
constexpr uint64_t TIMEOUT_NS = 1000ull * 1000ull * 1000ull;

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int x, int y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// contiguous bytes (a multiple of 16, both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_load_1d(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// four rows (r0..r3) of a one-row-box tensor map, 128 bytes from column x,
// land as four consecutive 128-byte rows at dst with the map's swizzle, as
// a four-row box would
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *tm, int x, int r0, int r1, int r2, int r3,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3 -> fp32, shapes in idesc
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// arrive once on `bar` when every tcgen05 operation this thread issued so far completes
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 TMEM lanes x 16 consecutive 32-bit columns; thread i gets lane base+i
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v)
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                   "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// 32 TMEM lanes x 32 columns (one load, one wait)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v)
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                   "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
                   "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
                   "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// 2-D tile store from shared memory through a tensor map (bulk async group),
// its lines marked first for eviction from L2: the data is written once and
// not read again by this kernel
__device__ __forceinline__ void tma_store_2d_evict_first(const CUtensorMap *tm, const void *src, int x, int y)
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(x), "r"(y), "r"(smem_u32(src)), "l"(pol)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// this thread's bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// this thread's bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 32 TMEM lanes x 16 columns into r[0..15], completion left to tmem_wait_ld32
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t *r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                   "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}

// wait for this thread's TMEM loads; the 32 registers are tied to the wait
// so that no use of them is scheduled before it
__device__ __forceinline__ void tmem_wait_ld32(uint32_t *r)
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// barrier over the four epilogue warps of TMEM lane quarter q (warps q, q+4,
// q+8, q+12; named barrier 2+q) that also ORs a predicate across them
__device__ __forceinline__ bool quarter_bar_or(int q, bool pred)
{
    uint32_t out;
    asm volatile("{\n\t.reg .pred p, r;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "barrier.cta.red.or.pred r, %2, 128, p;\n\tselp.u32 %0, 1, 0, r;\n\t}"
                 : "=r"(out)
                 : "r"((uint32_t)pred), "r"(2 + q)
                 : "memory");
    return out != 0;
}

// K-major operand tile in shared memory written by TMA with 128-byte
// swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked along
// M/N.  Descriptor: start address >> 4, leading offset (unused for this
// layout) 16 B, stride offset 1024 B between 8-row groups, fixed version
// bits 0b001 at 46, swizzle mode 2 (128 B) at 61.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t desc = 0;
    desc |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    desc |= (uint64_t)(16u >> 4) << 16;
    desc |= (uint64_t)(1024u >> 4) << 32;
    desc |= (uint64_t)1 << 46;
    desc |= (uint64_t)2 << 61;
    return desc;
}

// instruction descriptor: fp32 accumulate, A = B = E4M3, both K-major, N, M
__host__ __device__ constexpr uint32_t idesc_f8(int M, int N)
{
    return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *dev_status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 32; i++)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > TIMEOUT_NS) {
            *abort_flag = 1;
            dev_flag(dev_status, MOE_DEV_TIMEOUT);
            return false;
        }
    }
}

// shared-memory source of a 32 x 16-byte block, no swizzle: 8-row core
// matrices of 128 contiguous bytes, 128 bytes apart
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr)
{
    uint64_t desc = 0;
    desc |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    desc |= (uint64_t)(128u >> 4) << 16;
    desc |= (uint64_t)(128u >> 4) << 32;
    desc |= (uint64_t)1 << 46;
    return desc;
}

__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// ------------------------------------------------------------------ tiles

struct Tile {
    int e, m_blk, n_blk;
    int row0;       // first sorted row
    int rows;       // valid rows in this tile (1..128)
};

template <typename SmemT>
__device__ __forceinline__ Tile decode_tile(const SmemT &s, int E, int n_tiles, int t)
{
    int lo = 0, hi = E;  // largest e with tile_prefix[e] <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s.tile_prefix[mid] <= t) lo = mid; else hi = mid;
    }
    Tile tl;
    tl.e = lo;
    const int rows_e = s.row_lo[lo + 1] - s.row_lo[lo];
    const int m_tiles = (rows_e + BM - 1) / BM;
    const int local = t - s.tile_prefix[lo];
    tl.n_blk = local / m_tiles;
    tl.m_blk = local - tl.n_blk * m_tiles;
    tl.row0 = s.row_lo[lo] + tl.m_blk * BM;
    tl.rows = min(BM, rows_e - tl.m_blk * BM);
    return tl;
}

// per-CTA tile table from the device offsets, by warp 0
template <typename SmemT, typename ParamsT>
__device__ void build_schedule(SmemT &s, const ParamsT &p, int n_tiles)
{
    const int lane = threadIdx.x & 31;
    int32_t carry = 0;
    bool clipped = false;
    for (int base = 0; base <= p.E; base += 32) {
        const int e = base + lane;
        int32_t lo = 0, hi = 0;
        // offsets outside [0, max_rows] are clipped into it (and flagged), so
        // no tile ever addresses a row outside the buffers
        if (e <= p.E) {
            lo = __ldg(p.offsets + e);
            if (lo < 0) { lo = 0; clipped = true; }
            if ((int64_t)lo > p.max_rows) { lo = (int32_t)p.max_rows; clipped = true; }
            s.row_lo[e] = lo;
        }
        if (e < p.E) {
            hi = __ldg(p.offsets + e + 1);
            if (hi < 0) hi = 0;
            if ((int64_t)hi > p.max_rows) hi = (int32_t)p.max_rows;
        }
        const int32_t tiles = (e < p.E && hi > lo) ? ((hi - lo + BM - 1) / BM) * n_tiles : 0;
        int32_t incl = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        if (e <= p.E) s.tile_prefix[e] = carry + incl - tiles;
        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (__any_sync(0xFFFFFFFFu, clipped) && lane == 0 && blockIdx.x == 0) dev_flag(p.dev_status, MOE_DEV_ROWS);
}

// ------------------------------------------------------------------ host

static inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// 2-D uint8 tensor [rows, cols] (row stride = cols bytes), box box_rows x 128 B, 128-byte swizzle
static inline bool make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, const void *base, uint64_t cols,
                     uint64_t rows, uint32_t box_rows)
{
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp32 tensor [rows, cols] (row stride = 4 cols bytes) for 32 x 32 tile
// stores from 128-byte-swizzled shared memory
static inline bool make_map_f32_store(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, void *base, uint64_t cols,
                               uint64_t rows)
{
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

} // namespace ffn
} // namespace moe
