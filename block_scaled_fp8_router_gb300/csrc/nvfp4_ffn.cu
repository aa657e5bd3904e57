// nvfp4_ffn.cu -- the grouped SwiGLU expert FFN in NVFP4 on the block-scaled
// tensor-core MMA (tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X).
//
// NVFP4 is the FP4 variant that "RL at 1T Scale: prime-rl Performance Deep
// Dive" lists as future work for training and inference (closing section).
// Operands are FP4 E2M1 codes (two per byte, element 2i in the low nibble)
// with one E4M3 scale per 16 elements along K and one fp32 scale per
// tensor (x: the token tensor; each expert matrix its own; act: one over all
// routed rows).  The tensor core applies the 16-element block scales itself
// and accumulates the whole K extent in fp32; the epilogue divides by the
// two tensor scales:
//   GEMM1  h = D / (x_enc * w13_enc[e]);  act = silu(g) * u, stored as bf16
//          (the act tensor must exist before its tensor amax, and so its
//          scale, is known; the epilogue takes that amax on the way out);
//   then   act -> NVFP4 by the NVFP4 quantiser's block pass (amax done);
//   GEMM2  out = bf16(D / (act_enc * w2_enc[e])).
//
// Kernel shape: the block-scaled kernel's (one CTA per SM, 576 threads):
// warps 0-15 epilogue, warp 16 producer (TMA operand tiles, the A rows'
// scale words built by its 32 lanes, the B rows' scale images by two 1-D
// bulk copies), warp 17 MMA issuer.  A stage is one 128-byte K block = 256
// FP4 elements: four MMAs of K = 64, each with its own scale words (A: one
// 32-bit word of four E4M3 bytes per row, B likewise) copied from shared
// memory to tensor memory by tcgen05.cp ahead of the MMAs.  One 128 x 256
// fp32 accumulator per tile (256 TMEM columns), read once per tile.
//
// Scale-word images: tcgen05.cp (32x128b, replicated into the four lane
// quadrants) takes 32 rows x 16 bytes whose row r holds the words of tile
// rows r, r+32, r+64, r+96; tile row i then finds its word in lane i,
// column i / 32 of its 4-column group.  For the weights these 512-byte
// images are laid out once per weight update by moe_nvfp4_tile_scales (per
// 128-row group and K block: 4 MMAs x 512 bytes, contiguous), so the
// producer moves them with two bulk copies; the activation rows start
// anywhere, so the producer lanes gather their scale words straight into
// the images with 4-byte cp.async copies (zero-filled past the tile), kept
// F4_SF_AHEAD K blocks in flight: a stage is complete when its TMA bytes
// have landed and, on a second arrival, its gathered words (waited for with
// cp.async.wait_group and fenced to the async proxy, which tcgen05.cp
// reads through).
#include "tcgen05.cuh"
#include "nvfp4_internal.cuh"

namespace moe {
namespace ffn {

constexpr int F4_SFA_STAGE = 2048;      // A: 4 MMAs x 512 bytes
constexpr int F4_SFB_STAGE = 4096;      // B: 2 row groups x 4 MMAs x 512 bytes
constexpr int F4_SF_COL0 = 256;         // TMEM column of stage 0's scale words
constexpr int F4_SF_COLS = 48;          // per stage: A 4 x 4 columns, B 4 x 8
constexpr int F4_SF_AHEAD = 3;          // K blocks of A scale words in flight (< STAGES)
static_assert(F4_SF_AHEAD < STAGES, "a stage's scale words must land before the stage is reused");
static_assert(F4_SF_COL0 + STAGES * F4_SF_COLS <= TMEM_COLS, "NVFP4 scale words in TMEM");

struct SmemF4 {
    uint8_t a[STAGES][A_BYTES];
    uint8_t b[STAGES][B_BYTES];
    uint8_t sfa[STAGES][F4_SFA_STAGE];
    uint8_t sfb[STAGES][F4_SFB_STAGE];
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull;                     // the tile's accumulator is complete
    uint64_t tempty;                    // the epilogue has read it (16 arrivals)
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int32_t tile_prefix[MAX_E + 1];
    int32_t row_lo[MAX_E + 1];
};
constexpr size_t SMEM_F4_BYTES = sizeof(SmemF4) + 1024;
static_assert(SMEM_F4_BYTES <= 227 * 1024, "NVFP4 GEMM shared memory");

struct ParamsF4 {
    const uint8_t *a_sf;        // A rows' E4M3 block scales [max_rows, K/16]
    const uint8_t *b_sf_tiled;  // B scale images (moe_nvfp4_tile_scales layout)
    const float *a_enc;         // A tensor scale (device; GEMM1 x_enc, GEMM2 act_enc)
    const float *b_enc;         // [E] per-expert tensor scales of B
    const int32_t *offsets;     // [E+1]
    uint16_t *act;              // GEMM1 out: act [max_rows, F] bf16
    float *act_amax;            // GEMM1: max |act| over the routed rows (atomicMax on the bits)
    uint16_t *out;              // GEMM2 out [max_rows, d] bf16
    int32_t *dev_status;
    int64_t max_rows;
    int E, d, F;
};

// instruction descriptor of kind::mxf4nvf4: fp32 accumulate, A = B = E2M1
// (format code 1 of the FP4 kinds), both K-major, N, E4M3 (UE4M3) scale
// factors, M; scale-factor ids 0 (scale_vec::4X uses all four bytes of
// each word)
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N)
{
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (0u << 23) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], "
                 "p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
                 : "memory");
}

// 4 bytes global -> shared, asynchronously; src_bytes 0 writes zeros
__device__ __forceinline__ void cp_async4_zfill(void *dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                              const ParamsF4 p)
{
    extern __shared__ uint8_t smem_raw[];
    SmemF4 &s = *reinterpret_cast<SmemF4 *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = MODE == 1 ? p.d : p.F;           // elements
    const int nkb = (K + 255) / 256;                // 128-byte K blocks (the last may be half)
    const int nsf = K / 16;                         // scale bytes per row
    const int n_tiles = MODE == 1 ? p.F / 128 : (p.d + BN - 1) / BN;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; i++) {
            mbar_init(&s.full[i], 2);    // TMA bytes (with lane 0's arrival) + the A scale words' arrival
            mbar_init(&s.empty[i], 1);
        }
        mbar_init(&s.tfull, 1);
        mbar_init(&s.tempty, EPI_WARPS);
        mbar_init(&s.mma_done, 1);
        s.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) build_schedule(s, p, n_tiles);
    if (warp == MMA_WARP) tmem_alloc(&s.tmem_base, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    const int total = s.tile_prefix[p.E];
    volatile int *abort_flag = &s.abort_flag;

    if (warp == PRODUCER_WARP) {
        // ---------------- TMA producer + scale-word images (whole warp) ----------------
        // K block j: wait for its stage, gather its A scale words (cp.async,
        // one commit group per K block), issue its TMA and bulk copies; then
        // complete the stage of K block j - F4_SF_AHEAD, whose words have
        // landed (wait_group), fenced to the async proxy.
        uint32_t j = 0;
        uint32_t issued = 0;
        bool ok = true;
        auto complete_words = [&](uint32_t jj) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.full[jj % STAGES]);
        };
        for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
            const Tile tl = decode_tile(s, p.E, n_tiles, t);
            // scale rows of the tile's A rows lane + 32q (null past the tile)
            const uint8_t *arow[4];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int r = lane + 32 * q;
                arow[q] = r < tl.rows ? p.a_sf + ((int64_t)tl.row0 + r) * nsf : nullptr;
            }
            // the B tile's two 128-row groups (GEMM1: gate and up; GEMM2: two
            // consecutive output blocks, the second absent at a d % 256 tail)
            const int64_t g0 = MODE == 1 ? (int64_t)tl.e * (2 * p.F / 128) + tl.n_blk
                                         : (int64_t)tl.e * (p.d / 128) + tl.n_blk * 2;
            const int64_t g1 = MODE == 1 ? g0 + p.F / 128 : g0 + 1;
            const bool g1_ok = MODE == 1 || (tl.n_blk * 2 + 1) < p.d / 128;
            for (int kb = 0; kb < nkb; kb++, j++) {
                const int st = j % STAGES;
                bool w = true;
                if (lane == 0) w = wait_or_abort(&s.empty[st], ((j / STAGES) & 1) ^ 1, abort_flag, p.dev_status);
                w = __shfl_sync(0xFFFFFFFFu, w, 0);
                if (!w) {
                    ok = false;
                    break;
                }
                // image of MMA ks: row `lane` holds the words of rows lane, +32,
                // +64, +96 (the bytes 16kb + 4ks .. +3 of each row; zeros past
                // the tile or past the row)
                uint8_t *img = s.sfa[st];
#pragma unroll
                for (int ks = 0; ks < 4; ks++) {
                    const int c = 16 * kb + 4 * ks;
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const bool have = arow[q] != nullptr && c < nsf;
                        cp_async4_zfill(img + 512 * ks + 16 * lane + 4 * q, have ? arow[q] + c : p.a_sf, have ? 4u : 0u);
                    }
                }
                cp_async_commit();
                if (lane == 0) {
                    const uint32_t sfb_bytes = g1_ok ? 2u * 2048u : 2048u;
                    mbar_arrive_expect_tx(&s.full[st], A_BYTES + B_BYTES + sfb_bytes);
                    tma_load_2d(s.a[st], &tm_a, kb * BK, tl.row0, &s.full[st]);
                    if (MODE == 1) {
                        const int wrow = tl.e * 2 * p.F + tl.n_blk * 128;
                        tma_load_2d(s.b[st], &tm_b, kb * BK, wrow, &s.full[st]);
                        tma_load_2d(s.b[st] + B_BYTES / 2, &tm_b, kb * BK, wrow + p.F, &s.full[st]);
                    } else {
                        tma_load_2d(s.b[st], &tm_b, kb * BK, tl.e * p.d + tl.n_blk * BN, &s.full[st]);
                    }
                    bulk_load_1d(s.sfb[st], p.b_sf_tiled + (g0 * nkb + kb) * 2048, 2048, &s.full[st]);
                    if (g1_ok) bulk_load_1d(s.sfb[st] + 2048, p.b_sf_tiled + (g1 * nkb + kb) * 2048, 2048, &s.full[st]);
                    issued |= 1u << st;
                }
                if (j >= (uint32_t)F4_SF_AHEAD) {
                    cp_async_wait_group<F4_SF_AHEAD>();
                    complete_words(j - F4_SF_AHEAD);
                }
            }
        }
        // the last K blocks' words (the loop may also have stopped early)
        cp_async_wait_group<0>();
        for (uint32_t jj = j > (uint32_t)F4_SF_AHEAD ? j - F4_SF_AHEAD : 0; jj < j; jj++) complete_words(jj);
        if (lane == 0) {
            for (int i = 0; i < STAGES; i++) {
                if (!(issued & (1u << i)) || j == 0) continue;
                const uint32_t last = j - 1 - ((j - 1 - i) % STAGES);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&s.full[i], (last / STAGES) & 1) && globaltimer_ns() - t0 < TIMEOUT_NS) {}
            }
        }
    } else if (warp == MMA_WARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_nvf4(BM, BN);
            uint32_t j = 0, tcount = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x, tcount++) {
                // the previous tile's accumulator must have been read out
                if (!wait_or_abort(&s.tempty, (tcount & 1) ^ 1, abort_flag, p.dev_status)) break;
                for (int kb = 0; kb < nkb; kb++, j++) {
                    const int st = j % STAGES;
                    if (!wait_or_abort(&s.full[st], (j / STAGES) & 1, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sf_base = tmem + F4_SF_COL0 + F4_SF_COLS * st;
#pragma unroll
                    for (int ks = 0; ks < 4; ks++) {
                        tmem_cp_sf(sf_base + 4 * ks, sf_desc(smem_u32(s.sfa[st] + 512 * ks)));
                        tmem_cp_sf(sf_base + 16 + 8 * ks, sf_desc(smem_u32(s.sfb[st] + 512 * ks)));
                        tmem_cp_sf(sf_base + 16 + 8 * ks + 4, sf_desc(smem_u32(s.sfb[st] + 2048 + 512 * ks)));
                    }
                    const uint64_t adesc = sw128_desc(smem_u32(s.a[st]));
                    const uint64_t bdesc = sw128_desc(smem_u32(s.b[st]));
#pragma unroll
                    for (int ks = 0; ks < 4; ks++)  // K = 64 elements = 32 bytes per MMA: +2 in the >>4 address field
                        mma_nvf4(tmem, adesc + 2 * ks, bdesc + 2 * ks, IDESC, sf_base + 4 * ks, sf_base + 16 + 8 * ks,
                                 (kb > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&s.empty[st]);
                }
                if (ok) mma_commit(&s.tfull);
            }
            mma_commit(&s.mma_done);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&s.mma_done, 0) && globaltimer_ns() - t0 < TIMEOUT_NS) {}
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 0..15): one accumulator read per tile ----------------
        const int q = warp & 3;
        const int cg = warp >> 2;
        const int r_in = q * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        const float a_enc = __ldg(p.a_enc);
        uint32_t tcount = 0;
        bool aborted = false;
        float amax = 0.0f;     // GEMM1: this thread's max |act| (bf16 values) over its tiles
        for (int t = blockIdx.x; t < total; t += gridDim.x, tcount++) {
            const Tile tl = decode_tile(s, p.E, n_tiles, t);
            const bool row_ok = r_in < tl.rows;
            const int64_t row = (int64_t)tl.row0 + r_in;
            // GEMM1: gate columns 32cg.. and up 128+32cg..; GEMM2: 64cg..
            const int col0 = MODE == 1 ? 32 * cg : 64 * cg;
            const int col1 = MODE == 1 ? 128 + 32 * cg : 64 * cg + 32;
            const float inv = __frcp_rn(a_enc * __ldg(p.b_enc + tl.e));
            float acc0[32], acc1[32];
            if (!aborted && !wait_or_abort(&s.tfull, tcount & 1, abort_flag, p.dev_status)) aborted = true;
            if (!aborted) {
                tc_fence_after();
                const uint32_t base = tmem + lane_addr;
                uint32_t r0[32], r1[32];
                tmem_ld16_nowait(base + col0, r0);
                tmem_ld16_nowait(base + col0 + 16, r0 + 16);
                tmem_ld16_nowait(base + col1, r1);
                tmem_ld16_nowait(base + col1 + 16, r1 + 16);
                tmem_wait_ld32(r0);   // one wait for all four loads; the operands
                tmem_wait_ld32(r1);   // order every use of the values after it
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    acc0[i] = __uint_as_float(r0[i]) * inv;
                    acc1[i] = __uint_as_float(r1[i]) * inv;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.tempty);
            }
            if (MODE == 1) {
                if (row_ok && !aborted) {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const float g0 = acc0[2 * i], g1 = acc0[2 * i + 1];
                        w[i] = pack_bf16x2(__fdividef(g0, 1.0f + __expf(-g0)) * acc1[2 * i],
                                           __fdividef(g1, 1.0f + __expf(-g1)) * acc1[2 * i + 1]);
                        amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_f32(w[i] & 0xFFFFu)),
                                                 fabsf(bf16_bits_to_f32(w[i] >> 16))));
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(p.act + row * p.F + tl.n_blk * 128 + 32 * cg);
#pragma unroll
                    for (int i = 0; i < 4; i++) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
            } else {
                const int c_glob = tl.n_blk * BN + 64 * cg;
                if (row_ok && !aborted && c_glob < p.d) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + row * p.d + c_glob);
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        dst[i] = make_uint4(pack_bf16x2(acc0[8 * i], acc0[8 * i + 1]),
                                            pack_bf16x2(acc0[8 * i + 2], acc0[8 * i + 3]),
                                            pack_bf16x2(acc0[8 * i + 4], acc0[8 * i + 5]),
                                            pack_bf16x2(acc0[8 * i + 6], acc0[8 * i + 7]));
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        dst[4 + i] = make_uint4(pack_bf16x2(acc1[8 * i], acc1[8 * i + 1]),
                                                pack_bf16x2(acc1[8 * i + 2], acc1[8 * i + 3]),
                                                pack_bf16x2(acc1[8 * i + 4], acc1[8 * i + 5]),
                                                pack_bf16x2(acc1[8 * i + 6], acc1[8 * i + 7]));
                }
            }
            // the warps share nothing within a tile and leave on their own
            if (aborted || *abort_flag) break;
        }
        if (MODE == 1) {
            // non-negative floats order as their bit patterns
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
            if (lane == 0 && amax > 0.0f) atomicMax(reinterpret_cast<int *>(p.act_amax), __float_as_int(amax));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

// The weight scales' images: s [rows, K/16] E4M3 bytes (rows % 128 == 0) ->
// per 128-row group g and 256-element K block kb, 2048 contiguous bytes:
// [MMA ks 0..3][row r 0..31][q 0..3] words, the word of (g, kb, ks, r, q)
// holding the scale bytes 16 kb + 4 ks .. + 3 of row 128 g + 32 q + r
// (0 past the row's K/16).  One thread per word.
__global__ void nvfp4_tile_scales_kernel(const uint8_t *__restrict__ s, int64_t groups, int nkb, int nsf,
                                         uint32_t *__restrict__ out)
{
    const int64_t nwords = groups * nkb * 512;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nwords; i += (int64_t)gridDim.x * blockDim.x) {
        const int q = (int)(i & 3), r = (int)((i >> 2) & 31), ks = (int)((i >> 7) & 3);
        const int64_t gk = i >> 9;
        const int kb = (int)(gk % nkb);
        const int64_t g = gk / nkb;
        const int64_t row = 128 * g + 32 * q + r;
        const int c0 = 16 * kb + 4 * ks;
        uint32_t w = 0;
        if (c0 < nsf) w = __ldg(reinterpret_cast<const uint32_t *>(s + row * nsf + c0));
        out[i] = w;
    }
}

} // namespace ffn
} // namespace moe

using namespace moe;
using namespace moe::ffn;

MOE_API size_t moe_nvfp4_tiled_scales_size(int64_t rows, int64_t K)
{
    if (rows < 0 || K <= 0 || rows % 128 != 0 || K % 128 != 0) return 0;
    return (size_t)(rows / 128) * (size_t)((K + 255) / 256) * 2048;
}

MOE_API moe_status moe_nvfp4_tile_scales(const uint8_t *s, int64_t rows, int64_t K, uint8_t *s_tiled, void *stream)
{
    if (rows < 0 || K <= 0 || rows % 128 != 0 || K % 128 != 0) return MOE_ERR_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!s || !s_tiled) return MOE_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(s) & 3) != 0 || !aligned16(s_tiled)) return MOE_ERR_ALIGN;
    const int64_t groups = rows / 128;
    const int nkb = (int)((K + 255) / 256);
    const int64_t nwords = groups * nkb * 512;
    int64_t grid = (nwords + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (grid > cap) grid = cap;
    nvfp4_tile_scales_kernel<<<(unsigned)grid, 256, 0, as_stream(stream)>>>(s, groups, nkb, (int)(K / 16),
                                                                           reinterpret_cast<uint32_t *>(s_tiled));
    return launch_status();
}

MOE_API size_t moe_grouped_ffn_nvfp4_workspace_size(int64_t max_rows, int d, int F)
{
    (void)d;
    if (max_rows < 0 || F <= 0) return 0;
    // act bf16 [max_rows, F], its NVFP4 codes [max_rows, F/2] and scales
    // [max_rows, F/16], and the act tensor's (s_enc, amax)
    return align256((size_t)max_rows * F * 2) + align256((size_t)max_rows * (F / 2)) +
           align256((size_t)max_rows * (F / 16)) + 256;
}

MOE_API moe_status moe_grouped_ffn_nvfp4(const uint8_t *xq_sorted, const uint8_t *xs_sorted, const float *x_enc,
                                         const int32_t *expert_offsets, int64_t max_rows, int E, int d, int F,
                                         const uint8_t *w13_q, const uint8_t *w13_sf_tiled, const float *w13_enc,
                                         const uint8_t *w2_q, const uint8_t *w2_sf_tiled, const float *w2_enc,
                                         uint16_t *out_sorted, void *workspace, size_t workspace_bytes,
                                         int32_t *dev_status, void *stream)
{
    if (max_rows < 0 || max_rows >= (1LL << 31) || E < 1 || E > MAX_E || d <= 0 || F <= 0 || d % 128 != 0 ||
        F % 128 != 0)
        return MOE_ERR_SHAPE;
    if ((int64_t)E * 2 * F >= (1LL << 31) || (int64_t)E * d >= (1LL << 31)) return MOE_ERR_SHAPE;
    if (max_rows == 0) return MOE_OK;   // nothing to compute (the workspace may be empty too)
    const size_t need = moe_grouped_ffn_nvfp4_workspace_size(max_rows, d, F);
    if (!workspace || workspace_bytes < need) return MOE_ERR_WORKSPACE;
    if (!xq_sorted || !xs_sorted || !x_enc || !expert_offsets || !w13_q || !w13_sf_tiled || !w13_enc || !w2_q ||
        !w2_sf_tiled || !w2_enc || !out_sorted)
        return MOE_ERR_NULL;
    if (!aligned16(xq_sorted) || (reinterpret_cast<uintptr_t>(xs_sorted) & 7) != 0 || !aligned16(w13_q) ||
        !aligned16(w2_q) || !aligned16(w13_sf_tiled) || !aligned16(w2_sf_tiled) || !aligned16(out_sorted) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return MOE_ERR_ALIGN;
    auto enc = encode_fn();
    if (!enc) return MOE_ERR_CUDA;
    char *ws = reinterpret_cast<char *>(workspace);
    uint16_t *act = reinterpret_cast<uint16_t *>(ws);
    uint8_t *act_q = reinterpret_cast<uint8_t *>(ws + align256((size_t)max_rows * F * 2));
    uint8_t *act_s = act_q + align256((size_t)max_rows * (F / 2));
    float *act_ts = reinterpret_cast<float *>(act_s + align256((size_t)max_rows * (F / 16)));  // [s_enc, amax]
    // FP4 rows are K/2 bytes; 128-byte boxes = 256 elements
    CUtensorMap ma1, mb1, ma2, mb2;
    if (!make_map(enc, &ma1, xq_sorted, d / 2, max_rows, 128) ||
        !make_map(enc, &mb1, w13_q, d / 2, (uint64_t)E * 2 * F, 128) ||
        !make_map(enc, &ma2, act_q, F / 2, max_rows, 128) || !make_map(enc, &mb2, w2_q, F / 2, (uint64_t)E * d, 256))
        return MOE_ERR_CUDA;
    if (cudaFuncSetAttribute(grouped_gemm_nvfp4_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_F4_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(grouped_gemm_nvfp4_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_F4_BYTES) != cudaSuccess)
        return MOE_ERR_CUDA;
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(act_ts, 0, 2 * sizeof(float), st) != cudaSuccess) return MOE_ERR_CUDA;
    ParamsF4 prm{};
    prm.offsets = expert_offsets;
    prm.dev_status = dev_status;
    prm.max_rows = max_rows;
    prm.E = E;
    prm.d = d;
    prm.F = F;
    const int grid = sm_count();
    ParamsF4 p1 = prm;
    p1.a_sf = xs_sorted;
    p1.b_sf_tiled = w13_sf_tiled;
    p1.a_enc = x_enc;
    p1.b_enc = w13_enc;
    p1.act = act;
    p1.act_amax = act_ts + 1;
    grouped_gemm_nvfp4_kernel<1><<<grid, THREADS, SMEM_F4_BYTES, st>>>(ma1, mb1, p1);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    // act -> NVFP4 with the amax GEMM1 took (rows past the routed ones are
    // encoded too and never read)
    if (nvfp4_quant_blocks(act, max_rows, F, act_ts, act_q, act_s, st) != MOE_OK) return MOE_ERR_CUDA;
    ParamsF4 p2 = prm;
    p2.a_sf = act_s;
    p2.b_sf_tiled = w2_sf_tiled;
    p2.a_enc = act_ts;
    p2.b_enc = w2_enc;
    p2.out = out_sorted;
    grouped_gemm_nvfp4_kernel<2><<<grid, THREADS, SMEM_F4_BYTES, st>>>(ma2, mb2, p2);
    return launch_status();
}
