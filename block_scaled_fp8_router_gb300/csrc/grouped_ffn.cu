// grouped_ffn.cu -- per-expert SwiGLU FFN as two grouped block-scaled FP8
// GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Block-scaled FP8 of the DeepSeek-V3 recipe, which the prime-rl post ("RL at
// 1T Scale: prime-rl Performance Deep Dive", section "FP8 training") trains
// with: E4M3 operands, one fp32 scale per 1x128 activation tile and per
// 128x128 weight block.  The scales are arbitrary fp32 (not powers of two),
// so the hardware block-scaled MMA kinds do not apply; instead every
// 128-deep K block is one MMA group whose fp32 partial is read back from
// tensor memory and promoted into an fp32 register accumulator with the
// product of the two scales:
//     acc[r, n] = fma(sa[r, kb] * sb[n/128, kb], P_kb[r, n], acc[r, n]).
//
// Kernel shape (one persistent CTA per SM; the warp roles are listed above
// grouped_gemm_kernel): promotion / epilogue warps that read each K block's
// partial from TMEM and promote it in registers, a TMA producer (A tile
// 128 x 128 B and B tile 256 x 128 B per K block into a 4-stage
// shared-memory ring, 128-byte swizzle), an MMA issuer (4 x tcgen05.mma,
// M=128, N=256, K=32, E4M3 x E4M3 -> fp32, per K block into one of two
// 256-column TMEM buffers, so the epilogue reads block kb while block kb+1
// accumulates) and a scale warp that stages each K block's scales.
// Tiles are (expert, N block, M block) with M fastest, read from the device
// expert offsets (no host sync), so the CTAs working on the same weight tile
// at the same time share it through L2.
//   GEMM1: A = x_sorted [rows, d], B = W13[e] (gate rows n, up rows F + n);
//          one tile = 128 rows x (128 gate + 128 up) columns; the epilogue
//          forms silu(gate) * up for 128 act columns = one 1x128 block and
//          requantises it to E4M3 with its fp32 scale.
//   GEMM2: A = act_q [rows, F], B = W2[e] [d, F]; one tile = 128 x 256
//          output columns, stored as bf16.
// Every mbarrier wait is bounded; on expiry the CTA flags MOE_DEV_TIMEOUT,
// drains its in-flight copies and MMAs, frees TMEM and returns.
//
// Also in this file: the gathered form of the same kernel (GATHER: GEMM1's
// A rows fetched from the token-major codes by tile::gather4, GEMM2's rows
// stored in slot order), grouped_wgrad_kernel (the weight gradients, the
// contraction over each expert's tokens) and grouped_gemm_mx_kernel, the
// power-of-two-scale variant on the hardware block-scaled MMA (each
// described above it).
#include "tcgen05.cuh"

namespace moe {
namespace ffn {

struct Params {
    const float *a_scales;      // [max_rows, K/128]
    const float *b_scales;      // GEMM1 [E, 2F/128, d/128]; GEMM2 [E, d/128, F/128]
    const int32_t *offsets;     // [E+1]
    uint8_t *act_q;             // GEMM1 out [max_rows, F]
    float *act_s;               // GEMM1 out [max_rows, F/128]
    uint16_t *out;              // GEMM2 out [max_rows, d] bf16
    int32_t *dev_status;
    const int32_t *sorted_to_slot;  // gathered form: sorted row -> slot t*top_k + j
    float *h_out;                   // GEMM1, nullable: pre-activations [max_rows, 2F] for the backward
    int64_t max_rows;
    int E, d, F;
    int top_k;
};

// ------------------------------------------------------------------ kernel

// The forward kernel runs twelve warps in three warpgroups:
//   warps 0-7   promotion and tile epilogue (warpgroups 0 and 1, 224
//               registers each after setmaxnreg): warp w reads TMEM lane
//               quadrant w % 4 (32 rows) and column half w / 4 (128 of the
//               256 accumulator columns: GEMM1 64 gate + 64 up columns of the
//               same 64 act columns, GEMM2 one 128-column weight block), so
//               each thread keeps 128 promoted accumulators in registers;
//   warp 8      TMA producer (4-stage ring, as before);
//   warp 9      MMA issuer and TMEM owner;
//   warp 10     scale warp: per K block it copies the rows' scales sa[r, kb]
//               and the two weight-block scales (GEMM1: gate and up blocks;
//               GEMM2: the tile's two 128-column blocks) into a shared-memory
//               ring of FT_SLOTS slots with register-free cp.async copies, so
//               up to FT_SLOTS K blocks of scales are in flight and their L2
//               latency never reaches the promotion warps;
//   warp 11     idle (completes warpgroup 2 for setmaxnreg).
// Per K block a promotion thread reads its 128 columns as two rounds of two
// 32-column TMEM loads (one wait per round) and releases the TMEM buffer as
// soon as the second round has landed in registers, before its FMAs, so the
// MMA of K block kb + 2 waits only for the reads of K block kb.
constexpr int FT_THREADS = 384;
constexpr int FT_EPI_WARPS = 8;
constexpr int FT_PRODUCER = 8;
constexpr int FT_MMA = 9;
constexpr int FT_SCALE = 10;
constexpr int FT_SLOTS = 8;            // scale ring (K blocks whose scales may be in flight)
constexpr int FT_LAUNCH_REGS = 168;    // registers per thread at launch (12 warps, one CTA per SM)
constexpr int FT_EPI_REGS = 224;       // promotion warpgroups after setmaxnreg.inc
constexpr int FT_AUX_REGS = 56;        // warpgroup 2 after setmaxnreg.dec
static_assert(FT_EPI_WARPS * 32 * FT_EPI_REGS + (FT_THREADS - FT_EPI_WARPS * 32) * FT_AUX_REGS <=
                  FT_THREADS * FT_LAUNCH_REGS,
              "register split exceeds the launch allocation");

struct SmemF {
    uint8_t a[STAGES][A_BYTES];
    uint8_t b[STAGES][B_BYTES];
    float sa[FT_SLOTS][BM];             // K block j's row scales in slot j % FT_SLOTS
    float sb[FT_SLOTS][4];              //   and its two weight-block scales
    float red[2][2][BM];                // GEMM1: per-half partial amax (by tile parity)
    uint4 ostage[FT_EPI_WARPS][32 * 4]; // GEMM2: a warp's 32 rows x 32 bf16 columns on their way out
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t sfull[FT_SLOTS];
    uint64_t sempty[FT_SLOTS];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int32_t tile_prefix[MAX_E + 1];     // tiles before expert e
    int32_t row_lo[MAX_E + 1];          // clipped expert row ranges
};
constexpr size_t SMEM_F_BYTES = sizeof(SmemF) + 1024;  // + alignment slack
static_assert(SMEM_F_BYTES <= 227 * 1024, "forward GEMM shared memory");

// 4-byte asynchronous global -> shared copy (no register holds the value)
__device__ __forceinline__ void cp_async4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// one arrival on `bar` once every cp.async this thread issued so far has
// landed (the barrier's expected count includes this arrival)
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

// 32 TMEM lanes x 32 columns into r[0..31], completion left to a tied wait
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t *r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                   "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
                   "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
                   "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}

// ties 32 more registers after a preceding tcgen05.wait::ld (no instruction):
// volatile statements keep their order, so no use of r moves above the wait
__device__ __forceinline__ void tmem_tie32(uint32_t *r)
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// acc[i] = fma(c, v[i], acc[i]) for 64 values, two per packed instruction
// (each lane of the pair rounded as the scalar fmaf)
__device__ __forceinline__ void promote64(float *acc, const uint32_t *v, float c)
{
    const float2 c2 = make_float2(c, c);
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
        const float2 r = __ffma2_rn(c2, make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                    make_float2(acc[i], acc[i + 1]));
        acc[i] = r.x;
        acc[i + 1] = r.y;
    }
}

// barrier over the two promotion warps of TMEM lane quarter q (warps q and
// q + 4; named barrier 1 + q) that also ORs a predicate across them
__device__ __forceinline__ bool pair_bar_or(int q, bool pred)
{
    uint32_t out;
    asm volatile("{\n\t.reg .pred p, r;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "barrier.cta.red.or.pred r, %2, 64, p;\n\tselp.u32 %0, 1, 0, r;\n\t}"
                 : "=r"(out)
                 : "r"((uint32_t)pred), "r"(1 + q)
                 : "memory");
    return out != 0;
}

// GATHER (the gathered form): GEMM1 loads its A rows straight from the
// token-major activation codes (row = sorted_to_slot[r] / top_k, four rows
// per tile::gather4, one per producer lane) and takes their scales from the
// token-major scale array; GEMM2 writes each output row to its slot
// (row sorted_to_slot[r] of a [T*top_k, d] array) instead of its sorted
// position.  A slot outside [0, max_rows) marks its row as not routed: it
// gathers token 0, stores nothing and sets MOE_DEV_ROWS.
template <int MODE, bool GATHER>
__global__ void __launch_bounds__(FT_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                        const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    SmemF &s = *reinterpret_cast<SmemF *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // K extent and N tiling of this GEMM
    const int K = MODE == 1 ? p.d : p.F;
    const int nkb = K / BK;
    const int n_tiles = MODE == 1 ? p.F / 128 : (p.d + BN - 1) / BN;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; i++) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&s.tfull[i], 1);
            mbar_init(&s.tempty[i], FT_EPI_WARPS);
        }
        for (int i = 0; i < FT_SLOTS; i++) {
            mbar_init(&s.sfull[i], 32);
            mbar_init(&s.sempty[i], FT_EPI_WARPS);
        }
        mbar_init(&s.mma_done, 1);
        s.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) build_schedule(s, p, n_tiles);
    if (warp == FT_MMA) tmem_alloc(&s.tmem_base, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    const int total = s.tile_prefix[p.E];
    volatile int *abort_flag = &s.abort_flag;

    if (warp >= FT_EPI_WARPS) {
    setmaxnreg_dec<FT_AUX_REGS>();
    if (warp == FT_PRODUCER) {
        // ---------------- TMA producer ----------------
        // lane 0 alone, or the whole warp when it gathers A rows
        constexpr bool GA = GATHER && MODE == 1;
        if (GA || lane == 0) {
            uint32_t j = 0;
            uint32_t issued = 0;  // per-stage "has an outstanding load" bits
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
                const Tile tl = decode_tile(s, p.E, n_tiles, t);
                int tok[4] = {0, 0, 0, 0};  // token rows of this lane's four A rows (0 past the tile's rows)
                if (GA) {
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int r = 4 * lane + i;
                        if (r < tl.rows) {
                            const int32_t slot = __ldg(p.sorted_to_slot + tl.row0 + r);
                            if (slot >= 0 && (int64_t)slot < p.max_rows) tok[i] = slot / p.top_k;
                        }
                    }
                }
                for (int kb = 0; kb < nkb; kb++, j++) {
                    const int st = j % STAGES;
                    bool w = true;
                    if (lane == 0) w = wait_or_abort(&s.empty[st], ((j / STAGES) & 1) ^ 1, abort_flag, p.dev_status);
                    if (GA) w = __shfl_sync(0xFFFFFFFFu, w, 0);
                    if (!w) {
                        ok = false;
                        break;
                    }
                    if (GA) {
                        if (lane == 0) mbar_arrive_expect_tx(&s.full[st], A_BYTES + B_BYTES);
                        __syncwarp();
                        tma_gather4(s.a[st] + 512 * lane, &tm_a, kb * BK, tok[0], tok[1], tok[2], tok[3], &s.full[st]);
                        if (lane != 0) continue;
                    } else {
                        mbar_arrive_expect_tx(&s.full[st], A_BYTES + B_BYTES);
                        tma_load_2d(s.a[st], &tm_a, kb * BK, tl.row0, &s.full[st]);
                    }
                    if (MODE == 1) {
                        const int wrow = tl.e * 2 * p.F + tl.n_blk * 128;
                        tma_load_2d(s.b[st], &tm_b, kb * BK, wrow, &s.full[st]);
                        tma_load_2d(s.b[st] + B_BYTES / 2, &tm_b, kb * BK, wrow + p.F, &s.full[st]);
                    } else {
                        tma_load_2d(s.b[st], &tm_b, kb * BK, tl.e * p.d + tl.n_blk * BN, &s.full[st]);
                    }
                    issued |= 1u << st;
                }
            }
            // drain: wait for the last load issued into every stage
            for (int i = 0; i < STAGES && lane == 0; i++) {
                if (!(issued & (1u << i)) || j == 0) continue;
                // last use of stage i was at the largest j' < j with j' % STAGES == i
                const uint32_t last = j - 1 - ((j - 1 - i) % STAGES);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&s.full[i], (last / STAGES) & 1) && globaltimer_ns() - t0 < TIMEOUT_NS) {}
            }
        }
    } else if (warp == FT_MMA) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_f8(BM, BN);
            uint32_t j = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
                for (int kb = 0; kb < nkb; kb++, j++) {
                    const int st = j % STAGES;
                    const int buf = j & 1;
                    if (!wait_or_abort(&s.tempty[buf], ((j >> 1) & 1) ^ 1, abort_flag, p.dev_status) ||
                        !wait_or_abort(&s.full[st], (j / STAGES) & 1, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sw128_desc(smem_u32(s.a[st]));
                    const uint64_t bdesc = sw128_desc(smem_u32(s.b[st]));
#pragma unroll
                    for (int ks = 0; ks < BK / 32; ks++)  // K = 32 bytes per MMA: +2 in the >>4 address field
                        mma_f8(tmem + buf * BN, adesc + 2 * ks, bdesc + 2 * ks, IDESC, ks > 0);
                    mma_commit(&s.empty[st]);
                    mma_commit(&s.tfull[buf]);
                }
            }
            mma_commit(&s.mma_done);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&s.mma_done, 0) && globaltimer_ns() - t0 < TIMEOUT_NS) {}
        }
        __syncwarp();
    } else if (warp == FT_SCALE) {
        // ---------------- scale warp ----------------
        // walks the same (tile, K block) sequence as the MMA; lane i copies
        // the scales of rows i, i+32, i+64, i+96, lanes 0 and 1 the two
        // weight-block scales
        const int nkb_a = K / 128;     // A scale row length
        uint32_t j = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
            const Tile tl = decode_tile(s, p.E, n_tiles, t);
            const float *pa[4];        // owned rows' scale rows (null: no row)
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int r = lane + 32 * i;
                pa[i] = nullptr;
                if (r < tl.rows) {
                    int64_t row = (int64_t)tl.row0 + r;
                    if (GATHER && MODE == 1) {
                        const int32_t slot = __ldg(p.sorted_to_slot + row);
                        row = (slot >= 0 && (int64_t)slot < p.max_rows) ? slot / p.top_k : -1;
                    }
                    if (row >= 0) pa[i] = p.a_scales + row * nkb_a;
                }
            }
            const float *pb = nullptr;  // this lane's weight-block scale row (lanes 0, 1)
            if (lane < 2) {
                if (MODE == 1) {
                    pb = p.b_scales + ((int64_t)tl.e * (2 * p.F / 128) + (lane ? p.F / 128 : 0) + tl.n_blk) * nkb;
                } else {
                    const int nbk = tl.n_blk * 2 + lane;
                    if (nbk < p.d / 128) pb = p.b_scales + ((int64_t)tl.e * (p.d / 128) + nbk) * nkb;
                }
            }
            for (int kb = 0; kb < nkb; kb++, j++) {
                const int slot = j % FT_SLOTS;
                if (!wait_or_abort(&s.sempty[slot], ((j / FT_SLOTS) & 1) ^ 1, abort_flag, p.dev_status)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int i = 0; i < 4; i++)
                    if (pa[i]) cp_async4(&s.sa[slot][lane + 32 * i], pa[i] + kb);
                if (lane < 2) {
                    if (pb) cp_async4(&s.sb[slot][lane], pb + kb);
                    else s.sb[slot][lane] = 0.0f;
                }
                cp_async_arrive_noinc(&s.sfull[slot]);
            }
        }
        // no copy may still be in flight when the CTA exits
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    } else {
        setmaxnreg_inc<FT_EPI_REGS>();
        // ---------------- promotion + tile epilogue (warps 0..7) ----------------
        const int q = warp & 3;        // TMEM lane quadrant = rows 32q .. 32q+31
        const int cg = warp >> 2;      // column half 0..1
        const int r_in = q * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        // accumulator columns of this thread: GEMM1 gate 64cg.. and up
        // 128+64cg..; GEMM2 the 128-column run 128cg..
        const int col0 = MODE == 1 ? 64 * cg : 128 * cg;
        const int col1 = MODE == 1 ? 128 + 64 * cg : 128 * cg + 64;
        uint32_t j = 0;
        bool aborted = false;
        bool stop = false;     // GEMM1: abort decided at the row quarter's amax exchange
        int red_par = 0;       // GEMM1: exchange buffer of this tile
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const Tile tl = decode_tile(s, p.E, n_tiles, t);
            bool row_ok = r_in < tl.rows;
            const int64_t row = (int64_t)tl.row0 + r_in;
            // gathered form: GEMM2 stores by slot
            int64_t orow = row;
            if (GATHER && MODE == 2 && row_ok) {
                const int32_t slot = __ldg(p.sorted_to_slot + row);
                if (slot >= 0 && (int64_t)slot < p.max_rows) {
                    orow = slot;
                } else {
                    row_ok = false;
                    dev_flag(p.dev_status, MOE_DEV_ROWS);
                }
            }
            if (GATHER && MODE == 1 && row_ok) {
                const int32_t slot = __ldg(p.sorted_to_slot + row);
                if (slot < 0 || (int64_t)slot >= p.max_rows) {
                    row_ok = false;
                    dev_flag(p.dev_status, MOE_DEV_ROWS);
                }
            }
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; i++) acc[i] = 0.0f;
            for (int kb = 0; kb < nkb; kb++, j++) {
                const int buf = j & 1;
                const int slot = j % FT_SLOTS;
                float c0 = 0.0f, c1 = 0.0f;
                if (!aborted && !wait_or_abort(&s.sfull[slot], (j / FT_SLOTS) & 1, abort_flag, p.dev_status))
                    aborted = true;
                if (!aborted) {
                    const float sa = s.sa[slot][r_in];
                    c0 = sa * s.sb[slot][MODE == 1 ? 0 : cg];
                    c1 = MODE == 1 ? sa * s.sb[slot][1] : c0;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s.sempty[slot]);
                }
                if (!aborted && !wait_or_abort(&s.tfull[buf], (j >> 1) & 1, abort_flag, p.dev_status))
                    aborted = true;
                if (!aborted) {
                    tc_fence_after();
                    const uint32_t base = tmem + lane_addr + buf * BN;
                    uint32_t v[64];
                    tmem_ld32_nowait(base + col0, v);
                    tmem_ld32_nowait(base + col0 + 32, v + 32);
                    tmem_wait_ld32(v);
                    tmem_tie32(v + 32);
                    promote64(acc, v, c0);
                    tmem_ld32_nowait(base + col1, v);
                    tmem_ld32_nowait(base + col1 + 32, v + 32);
                    tmem_wait_ld32(v);
                    tmem_tie32(v + 32);
                    // the partial is in registers: hand the buffer back first
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s.tempty[buf]);
                    promote64(acc + 64, v, c1);
                }
            }
            if (MODE == 1) {
                if (p.h_out != nullptr && row_ok && !aborted) {
                    // the pre-activations, kept for the backward: gate then up columns
                    float4 *hg = reinterpret_cast<float4 *>(p.h_out + row * 2 * p.F + tl.n_blk * 128 + 64 * cg);
                    float4 *hu = reinterpret_cast<float4 *>(p.h_out + row * 2 * p.F + p.F + tl.n_blk * 128 + 64 * cg);
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        hg[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                        hu[i] = make_float4(acc[64 + 4 * i], acc[64 + 4 * i + 1], acc[64 + 4 * i + 2], acc[64 + 4 * i + 3]);
                    }
                }
                // act = silu(gate) * up for 64 of the tile's 128 act columns
                // (fast exponential and reciprocal: act is re-quantised to
                // E4M3 next, 3 mantissa bits, so their few-ulp errors move a
                // code only at a rounding tie)
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 64; i++) {
                    const float g = acc[i];
                    acc[i] = __fdividef(g, 1.0f + __expf(-g)) * acc[64 + i];
                    amax = fmaxf(amax, fabsf(acc[i]));
                }
                // the row's amax over both halves: the two warps of row
                // quarter q meet at their own barrier, which also ORs their
                // abort state so that they leave together; the exchange
                // buffer alternates by tile, so the next tile's writes never
                // meet this tile's reads
                s.red[red_par][cg][r_in] = amax;
                stop = pair_bar_or(q, aborted || *abort_flag);
                amax = fmaxf(s.red[red_par][0][r_in], s.red[red_par][1][r_in]);
                red_par ^= 1;
                const float sc = block_scale(amax);
                // one correctly rounded reciprocal per row, act * (1/sc) per
                // element: the act values are the fast-SiLU ones already, so
                // the requantisation spends no division on them (an exact
                // quotient measured 3-5% slower in this epilogue)
                const float rs = __frcp_rn(sc);
#pragma unroll
                for (int i = 0; i < 64; i++) acc[i] *= rs;
                if (row_ok && !aborted) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.act_q + row * p.F + tl.n_blk * 128 + 64 * cg);
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const float *a = acc + 16 * u + 4 * i;
                            w[i] = (uint32_t)pack_e4m3x2(a[0], a[1]) | ((uint32_t)pack_e4m3x2(a[2], a[3]) << 16);
                        }
                        dst[u] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    if (cg == 0) p.act_s[row * (p.F / 128) + tl.n_blk] = sc;
                }
            } else {
                // bf16 rows leave through a per-warp staging buffer, 32
                // columns at a time: each lane writes its row's 64 bytes, then
                // the warp stores 8 rows x 64 contiguous bytes per instruction
                // (16-byte pieces swizzled by row so that neither side of the
                // staging has bank conflicts)
                const int c_glob = tl.n_blk * BN + 128 * cg;
                if (!aborted && c_glob < p.d) {
                    uint4 *stg = s.ostage[warp];
                    const int sr = lane >> 2, sp = lane & 3;   // row within a group of 8, 16-byte piece
                    int64_t drow[4];
                    bool dok[4];
#pragma unroll
                    for (int m = 0; m < 4; m++) {
                        const int rr = sr + 8 * m;
                        drow[m] = __shfl_sync(0xFFFFFFFFu, orow, rr);
                        dok[m] = __shfl_sync(0xFFFFFFFFu, (int)row_ok, rr) != 0;
                    }
#pragma unroll
                    for (int ch = 0; ch < 4; ch++) {
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const float *a = acc + 32 * ch + 8 * i;
                            stg[lane * 4 + (i ^ ((lane >> 1) & 3))] =
                                make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                                           pack_bf16x2(a[6], a[7]));
                        }
                        __syncwarp();
#pragma unroll
                        for (int m = 0; m < 4; m++) {
                            const int rr = sr + 8 * m;
                            const uint4 v = stg[rr * 4 + (sp ^ ((rr >> 1) & 3))];
                            if (dok[m])
                                *reinterpret_cast<uint4 *>(p.out + drow[m] * p.d + c_glob + 32 * ch + 8 * sp) = v;
                        }
                    }
                }
            }
            // GEMM1 leaves by its row quarter's decision; GEMM2's warps share
            // nothing within a tile and leave on their own (waits are bounded)
            if (MODE == 1 ? stop : (aborted || *abort_flag)) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == FT_MMA) tmem_dealloc(tmem, TMEM_COLS);
}

// Registers per thread the forward kernel was compiled to launch with.  The
// setmaxnreg split inside it assumes exactly FT_LAUNCH_REGS: with fewer, the
// promotion warps' setmaxnreg.inc could not be satisfied and would wait, so
// the host refuses to launch unless the count matches.
template <int MODE, bool GATHER>
static bool forward_kernel_regs_ok()
{
    static const bool ok = [] {
        cudaFuncAttributes a;
        if (cudaFuncGetAttributes(&a, grouped_gemm_kernel<MODE, GATHER>) != cudaSuccess) return false;
        return a.numRegs == FT_LAUNCH_REGS;
    }();
    return ok;
}

// ============================================================================
// Weight gradients: per expert e, out[e] [M, N] fp32 = sum over e's padded
// 128-row blocks kb of (sa[m, kb] * sb[n, kb]) * P_kb(m, n), the same 128-deep
// block MMAs and fp32 promotion as the forward with the contraction over the
// expert's tokens.  A = [M, ld] codes (the 128 x 1 layout of d_out or dh),
// B = [N, ld] (act or x), both scale arrays block-major (saT [ld/128, M],
// sbT [ld/128, N]: a tile's 128 row and 128 column scales of one K block are
// contiguous).  Tiles are (expert, N block, M block), M fastest; experts
// without rows have no tiles (their out is zeroed apart).
// ============================================================================

struct ParamsWG {
    const float *saT;           // [ld/128, M]
    const float *sbT;           // [ld/128, N]
    const int32_t *pad;         // [E+1]
    float *out;                 // [E, M, N]
    int32_t *dev_status;
    int64_t ld;
    int E, M, N;
};

// The contraction runs over an expert's rows (a few 128-row blocks per tile),
// so the tile's output is large next to its MMA work and the kernel is bound
// by its fp32 stores.  128 x 128 tiles keep the promoted accumulator at 32
// values per epilogue thread (under the 18-warp register cap), and four
// 128-column TMEM buffers let the MMAs of the next tile run while the
// epilogue stores this one.  The K block's row and column scales travel with
// it: the producer copies them into a ring of shared-memory slots (its own
// full/empty barriers), so the epilogue reads them at shared-memory latency
// while the stores keep L2 busy.  Each epilogue warp hands its 32 x 32 fp32
// sub-tile to a TMA store (128-byte swizzled staging, conflict-free writes)
// and goes on to the next tile while the copy drains.
constexpr int WG_BN = 128;
constexpr int WG_BUFS = 4;                 // TMEM accumulators (4 x 128 columns)
constexpr int WG_STAGES = 4;
constexpr int WG_B_BYTES = WG_BN * BK;     // 16 KB
constexpr int WG_SLOTS = 8;                // scale slots (K blocks the producer may run ahead of the epilogue)

struct SmemWG {
    uint8_t a[WG_STAGES][A_BYTES];
    uint8_t b[WG_STAGES][WG_B_BYTES];
    float stage[EPI_WARPS][32 * 32];       // a warp's 32 x 32 sub-tile for its TMA store (128-byte swizzle)
    float sa[WG_SLOTS][BM];                // scales of K block j in slot j % WG_SLOTS: the tile's rows
    float sb[WG_SLOTS][WG_BN];             //   and the tile's columns
    uint64_t full[WG_STAGES];
    uint64_t empty[WG_STAGES];
    uint64_t tfull[WG_BUFS];
    uint64_t tempty[WG_BUFS];
    uint64_t sfull[WG_SLOTS];
    uint64_t sempty[WG_SLOTS];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int32_t tile_prefix[MAX_E + 1];
    int32_t pad[MAX_E + 1];
};
constexpr size_t SMEM_WG_BYTES = sizeof(SmemWG) + 1024;
static_assert(SMEM_WG_BYTES <= 227 * 1024, "wgrad shared memory");
static_assert(WG_BUFS * WG_BN <= TMEM_COLS, "wgrad TMEM buffers");

struct TileWG {
    int e, m_blk, n_blk;
    int kb0, nkb;   // first global K block and count
};

// every role walks its tiles in increasing order, so the expert of tile t is
// found by advancing e from the previous tile's
__device__ __forceinline__ TileWG decode_tile_wg(const SmemWG &s, const ParamsWG &p, int t, int &e)
{
    while (e + 1 < p.E && s.tile_prefix[e + 1] <= t) e++;
    TileWG tl;
    tl.e = e;
    const int m_tiles = p.M / BM;
    const int local = t - s.tile_prefix[e];
    tl.n_blk = local / m_tiles;
    tl.m_blk = local - tl.n_blk * m_tiles;
    const int32_t p0 = s.pad[e], p1 = s.pad[e + 1];
    tl.kb0 = p0 / 128;
    tl.nkb = (p1 - p0) / 128;
    return tl;
}

__global__ void __launch_bounds__(THREADS, 1)
    grouped_wgrad_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_out, const ParamsWG p)
{
    extern __shared__ uint8_t smem_raw[];
    SmemWG &s = *reinterpret_cast<SmemWG *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_per_e = (p.M / BM) * (p.N / WG_BN);
    if (threadIdx.x == 0) {
        for (int i = 0; i < WG_STAGES; i++) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < WG_BUFS; i++) {
            mbar_init(&s.tfull[i], 1);
            mbar_init(&s.tempty[i], EPI_WARPS);
        }
        for (int i = 0; i < WG_SLOTS; i++) {
            mbar_init(&s.sfull[i], 1);
            mbar_init(&s.sempty[i], EPI_WARPS);
        }
        mbar_init(&s.mma_done, 1);
        s.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        // tile prefix over experts with rows (warp-wide scan); the scale
        // copies are not bounds-checked, so offsets outside [0, ld] or off
        // the 128-row grid run no tile at all and set MOE_DEV_ROWS
        int32_t carry = 0;
        bool bad = false;
        for (int base = 0; base <= p.E; base += 32) {
            const int e = base + lane;
            int32_t tiles = 0;
            if (e <= p.E) s.pad[e] = __ldg(p.pad + e);
            if (e < p.E) {
                const int32_t p0 = __ldg(p.pad + e), p1 = __ldg(p.pad + e + 1);
                bad |= p0 < 0 || (int64_t)p1 > p.ld || (p0 & 127) != 0 || (p1 & 127) != 0;
                tiles = p1 > p0 ? tiles_per_e : 0;
            }
            int32_t incl = tiles;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            if (e <= p.E) s.tile_prefix[e] = carry + incl - tiles;
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) {
            s.tile_prefix[p.E] = 0;
            if (blockIdx.x == 0) dev_flag(p.dev_status, MOE_DEV_ROWS);
        }
    }
    if (warp == MMA_WARP) tmem_alloc(&s.tmem_base, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    const int total = s.tile_prefix[p.E];
    volatile int *abort_flag = &s.abort_flag;

    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            uint32_t j = 0;
            int ecur = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
                const TileWG tl = decode_tile_wg(s, p, t, ecur);
                for (int kb = 0; kb < tl.nkb; kb++, j++) {
                    const int st = j % WG_STAGES, sl = j % WG_SLOTS;
                    const int64_t kg = tl.kb0 + kb;
                    // both waits come before any copy of block j, so that an
                    // abort leaves exactly blocks 0 .. j-1 issued
                    if (!wait_or_abort(&s.empty[st], ((j / WG_STAGES) & 1) ^ 1, abort_flag, p.dev_status) ||
                        !wait_or_abort(&s.sempty[sl], ((j / WG_SLOTS) & 1) ^ 1, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&s.full[st], A_BYTES + WG_B_BYTES);
                    tma_load_2d(s.a[st], &tm_a, (int)kg * BK, tl.m_blk * BM, &s.full[st]);
                    tma_load_2d(s.b[st], &tm_b, (int)kg * BK, tl.n_blk * WG_BN, &s.full[st]);
                    mbar_arrive_expect_tx(&s.sfull[sl], (BM + WG_BN) * 4);
                    bulk_load_1d(s.sa[sl], p.saT + kg * p.M + (int64_t)tl.m_blk * BM, BM * 4, &s.sfull[sl]);
                    bulk_load_1d(s.sb[sl], p.sbT + kg * p.N + (int64_t)tl.n_blk * WG_BN, WG_BN * 4, &s.sfull[sl]);
                }
            }
            // no copy may still be in flight when the CTA exits: wait for the
            // last block issued into each stage and each scale slot
            for (int i = 0; i < WG_STAGES && (uint32_t)i < j; i++) {
                const uint32_t last = j - 1 - ((j - 1 - i) % WG_STAGES);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&s.full[i], (last / WG_STAGES) & 1) && globaltimer_ns() - t0 < TIMEOUT_NS) {}
            }
            for (int i = 0; i < WG_SLOTS && (uint32_t)i < j; i++) {
                const uint32_t last = j - 1 - ((j - 1 - i) % WG_SLOTS);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&s.sfull[i], (last / WG_SLOTS) & 1) && globaltimer_ns() - t0 < TIMEOUT_NS) {}
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_f8(BM, WG_BN);
            uint32_t j = 0;
            int ecur = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
                const TileWG tl = decode_tile_wg(s, p, t, ecur);
                for (int kb = 0; kb < tl.nkb; kb++, j++) {
                    const int st = j % WG_STAGES;
                    const int buf = j % WG_BUFS;
                    if (!wait_or_abort(&s.tempty[buf], ((j / WG_BUFS) & 1) ^ 1, abort_flag, p.dev_status) ||
                        !wait_or_abort(&s.full[st], (j / WG_STAGES) & 1, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sw128_desc(smem_u32(s.a[st]));
                    const uint64_t bdesc = sw128_desc(smem_u32(s.b[st]));
#pragma unroll
                    for (int ks = 0; ks < BK / 32; ks++)
                        mma_f8(tmem + buf * WG_BN, adesc + 2 * ks, bdesc + 2 * ks, IDESC, ks > 0);
                    mma_commit(&s.empty[st]);
                    mma_commit(&s.tfull[buf]);
                }
            }
            mma_commit(&s.mma_done);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&s.mma_done, 0) && globaltimer_ns() - t0 < TIMEOUT_NS) {}
        }
        __syncwarp();
    } else if (warp < EPI_WARPS) {
        // warp (q, cg): TMEM lanes 32q .. 32q+31 (the tile's rows), columns 32cg .. 32cg+31
        const int q = warp & 3, cg = warp >> 2;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        float *stg = s.stage[warp];
        uint32_t j = 0;
        int ecur = 0;
        bool aborted = false;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const TileWG tl = decode_tile_wg(s, p, t, ecur);
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; i++) acc[i] = 0.0f;
            for (int kb = 0; kb < tl.nkb; kb++, j++) {
                const int buf = j % WG_BUFS, sl = j % WG_SLOTS;
                if (!aborted && (!wait_or_abort(&s.sfull[sl], (j / WG_SLOTS) & 1, abort_flag, p.dev_status) ||
                                 !wait_or_abort(&s.tfull[buf], (j / WG_BUFS) & 1, abort_flag, p.dev_status)))
                    aborted = true;
                if (!aborted) {
                    tc_fence_after();
                    float v[32];
                    tmem_ld32(tmem + lane_addr + buf * WG_BN + 32 * cg, v);
                    const float sa = s.sa[sl][q * 32 + lane];
                    const float4 *sb4 = reinterpret_cast<const float4 *>(&s.sb[sl][32 * cg]);
#pragma unroll
                    for (int i4 = 0; i4 < 8; i4++) {
                        const float4 b = sb4[i4];
                        acc[4 * i4 + 0] = fmaf(sa * b.x, v[4 * i4 + 0], acc[4 * i4 + 0]);
                        acc[4 * i4 + 1] = fmaf(sa * b.y, v[4 * i4 + 1], acc[4 * i4 + 1]);
                        acc[4 * i4 + 2] = fmaf(sa * b.z, v[4 * i4 + 2], acc[4 * i4 + 2]);
                        acc[4 * i4 + 3] = fmaf(sa * b.w, v[4 * i4 + 3], acc[4 * i4 + 3]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&s.tempty[buf]);
                        mbar_arrive(&s.sempty[sl]);
                    }
                }
            }
            if (!aborted) {
                // the previous tile's store has read the staging tile; row
                // `lane` goes in with the 128-byte swizzle (16-byte chunk c of
                // row r at chunk c ^ (r & 7)), then one TMA store of 32 x 32
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; i++)
                    *reinterpret_cast<float4 *>(stg + lane * 32 + 4 * (i ^ (lane & 7))) =
                        make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0)
                    tma_store_2d_evict_first(&tm_out, stg, tl.n_blk * WG_BN + 32 * cg,
                                             tl.e * p.M + tl.m_blk * BM + q * 32);
            }
            // no barrier between the epilogue warps: they share no staging, so
            // each runs ahead until the TMEM ring stops it, and leaves on its
            // own abort (every wait is bounded)
            if (aborted || *abort_flag) break;
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

// zero out[e] of the experts without rows (the GEMM has no tiles for them)
__global__ void wgrad_zero_empty_kernel(const int32_t *__restrict__ pad, int64_t MN, float *__restrict__ out)
{
    const int e = blockIdx.y;
    if (__ldg(pad + e + 1) != __ldg(pad + e)) return;
    float4 *o = reinterpret_cast<float4 *>(out + (int64_t)e * MN);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < MN / 4; i += (int64_t)gridDim.x * blockDim.x)
        o[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

// ============================================================================
// Power-of-two scales (UE8M0): the hardware block-scaled MMA
// ============================================================================
//
// With power-of-two block scales (fp8_block_quant_ue8m0) the scales need no
// software promotion: tcgen05.mma.kind::mxf8f6f4.block_scale multiplies each
// 32-deep K slice by 2^(ea-127) * 2^(eb-127) (one exponent byte per row of A
// and per row of B, read from tensor memory) and accumulates the whole K
// extent in TMEM.  One 128 x 256 fp32 accumulator per tile (256 columns;
// the scale factors of each pipeline stage take 12 more), read once per
// tile by the epilogue warps, which release it before the SwiGLU /
// re-quantisation / store so that the next tile's MMAs start early.
//
// Scale factors: per K block the producer warp writes, for the A tile,
// a 512-byte block of 32 rows x 16 bytes whose row r holds the exponent
// words of A rows r, r+32, r+64, r+96 (each word = the row's exponent byte
// repeated for the four 32-deep slices of the 128-deep block), and one
// such block per 128-row half of the B tile; tcgen05.cp (32x128b, copied
// into all four 32-lane quadrants) moves them to TMEM, where A row i finds
// its word in lane i, column (i / 32) of its 4-column group, and the MMA's
// scale-factor id picks the slice's byte (all four are equal here).

constexpr int SFA_BYTES = 512;          // one 128-row scale-factor block
constexpr int SFB_BYTES = 1024;         // two of them: B rows 0..127, 128..255
constexpr int SF_COL0 = 256;            // TMEM column of stage 0's scale factors
constexpr int SF_COLS_PER_STAGE = 16;   // A: 4 columns, B: 8 (+4 unused)

struct SmemMX {
    uint8_t a[STAGES][A_BYTES];
    uint8_t b[STAGES][B_BYTES];
    uint8_t sfa[STAGES][SFA_BYTES];
    uint8_t sfb[STAGES][SFB_BYTES];
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull;                     // the tile's accumulator is complete
    uint64_t tempty;                    // the epilogue has read it (16 arrivals)
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    float red[2][4][BM];
    int32_t tile_prefix[MAX_E + 1];
    int32_t row_lo[MAX_E + 1];
};
constexpr size_t SMEM_MX_BYTES = sizeof(SmemMX) + 1024;
static_assert(SMEM_MX_BYTES <= 227 * 1024, "block-scaled GEMM shared memory");

struct ParamsMX {
    const uint8_t *a_exp;       // GEMM1: token-major [T, d/128]; GEMM2: sorted [max_rows, F/128]
    const uint8_t *b_exp;       // GEMM1 [E, 2F/128, d/128]; GEMM2 [E, d/128, F/128]
    const int32_t *offsets;     // [E+1]
    const int32_t *sorted_to_slot;
    uint8_t *act_q;             // GEMM1 out [max_rows, F]
    uint8_t *act_e;             // GEMM1 out [max_rows, F/128]
    uint16_t *out;              // GEMM2 out [max_rows, d] bf16
    int32_t *dev_status;
    int64_t max_rows;
    int E, d, F;
    int top_k;
};

// instruction descriptor of the block-scaled kind: fp32 accumulate, A = B =
// E4M3, both K-major, N, UE8M0 scale factors, M, scale-factor ids of A, B
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, uint32_t a_sf_id, uint32_t b_sf_id)
{
    return (b_sf_id << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24) | (a_sf_id << 29);
}

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], "
                 "p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ uint32_t ue8m0_exp_of(float amax)
{
    const uint32_t bits = __float_as_uint(amax);
    const int32_t ef = (int32_t)(bits >> 23);
    if (amax == 0.0f) return 127u;
    if (ef == 0) return 0u;
    const int32_t e = ef - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return (uint32_t)(e < 0 ? 0 : (e > 254 ? 254 : e));
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                           const ParamsMX p)
{
    extern __shared__ uint8_t smem_raw[];
    SmemMX &s = *reinterpret_cast<SmemMX *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = MODE == 1 ? p.d : p.F;
    const int nkb = K / BK;
    const int n_tiles = MODE == 1 ? p.F / 128 : (p.d + BN - 1) / BN;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; i++) {
            mbar_init(&s.full[i], 1);
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
        // ---------------- TMA producer + scale-factor blocks (whole warp) ----------------
        uint32_t j = 0;
        uint32_t issued = 0;
        bool ok = true;
        const int nka = K / 128;
        for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
            const Tile tl = decode_tile(s, p.E, n_tiles, t);
            // exponent rows of A rows lane + 32q (token rows for GEMM1); -1 past the tile
            int64_t arow[4];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int r = lane + 32 * q;
                arow[q] = -1;
                if (r < tl.rows) {
                    const int64_t row = (int64_t)tl.row0 + r;
                    arow[q] = MODE == 1 ? (int64_t)(__ldg(p.sorted_to_slot + row) / p.top_k) : row;
                }
            }
            // exponent rows of the B tile's two 128-row halves
            const int64_t nb0 = MODE == 1 ? (int64_t)tl.e * (2 * p.F / 128) + tl.n_blk
                                          : (int64_t)tl.e * (p.d / 128) + tl.n_blk * 2;
            const int64_t nb1 = MODE == 1 ? nb0 + p.F / 128 : nb0 + 1;
            const bool nb1_ok = MODE == 1 || (tl.n_blk * 2 + 1) < p.d / 128;
            // exponent bytes of K block kb, fetched one block ahead so their
            // latency hides behind the wait for the stage
            auto fetch = [&](int kb, uint32_t *ea, uint32_t &eb0, uint32_t &eb1) {
#pragma unroll
                for (int q = 0; q < 4; q++) ea[q] = arow[q] >= 0 ? (uint32_t)__ldg(p.a_exp + arow[q] * nka + kb) : 0u;
                eb0 = (uint32_t)__ldg(p.b_exp + nb0 * nkb + kb);
                eb1 = nb1_ok ? (uint32_t)__ldg(p.b_exp + nb1 * nkb + kb) : 0u;
            };
            uint32_t ea[4], eb0, eb1;
            fetch(0, ea, eb0, eb1);
            for (int kb = 0; kb < nkb; kb++, j++) {
                const int st = j % STAGES;
                uint32_t na[4] = {0u, 0u, 0u, 0u}, nb0e = 0u, nb1e = 0u;
                if (kb + 1 < nkb) fetch(kb + 1, na, nb0e, nb1e);
                bool w = true;
                if (lane == 0) w = wait_or_abort(&s.empty[st], ((j / STAGES) & 1) ^ 1, abort_flag, p.dev_status);
                w = __shfl_sync(0xFFFFFFFFu, w, 0);
                if (!w) {
                    ok = false;
                    break;
                }
                *reinterpret_cast<uint4 *>(s.sfa[st] + 16 * lane) =
                    make_uint4(ea[0] * 0x01010101u, ea[1] * 0x01010101u, ea[2] * 0x01010101u, ea[3] * 0x01010101u);
                const uint32_t wb0 = eb0 * 0x01010101u, wb1 = eb1 * 0x01010101u;
                *reinterpret_cast<uint4 *>(s.sfb[st] + 16 * lane) = make_uint4(wb0, wb0, wb0, wb0);
                *reinterpret_cast<uint4 *>(s.sfb[st] + SFA_BYTES + 16 * lane) = make_uint4(wb1, wb1, wb1, wb1);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(&s.full[st], A_BYTES + B_BYTES);
                    tma_load_2d(s.a[st], &tm_a, kb * BK, tl.row0, &s.full[st]);
                    if (MODE == 1) {
                        const int wrow = tl.e * 2 * p.F + tl.n_blk * 128;
                        tma_load_2d(s.b[st], &tm_b, kb * BK, wrow, &s.full[st]);
                        tma_load_2d(s.b[st] + B_BYTES / 2, &tm_b, kb * BK, wrow + p.F, &s.full[st]);
                    } else {
                        tma_load_2d(s.b[st], &tm_b, kb * BK, tl.e * p.d + tl.n_blk * BN, &s.full[st]);
                    }
                    issued |= 1u << st;
                }
#pragma unroll
                for (int q = 0; q < 4; q++) ea[q] = na[q];
                eb0 = nb0e;
                eb1 = nb1e;
            }
        }
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
                    const uint32_t sfa_t = tmem + SF_COL0 + SF_COLS_PER_STAGE * st;
                    const uint32_t sfb_t = sfa_t + 4;
                    tmem_cp_sf(sfa_t, sf_desc(smem_u32(s.sfa[st])));
                    tmem_cp_sf(sfb_t, sf_desc(smem_u32(s.sfb[st])));
                    tmem_cp_sf(sfb_t + 4, sf_desc(smem_u32(s.sfb[st] + SFA_BYTES)));
                    const uint64_t adesc = sw128_desc(smem_u32(s.a[st]));
                    const uint64_t bdesc = sw128_desc(smem_u32(s.b[st]));
#pragma unroll
                    for (int ks = 0; ks < BK / 32; ks++)
                        // the four bytes of every scale word are equal (one exponent per
                        // 128-deep block), so scale-factor id 0 serves all four slices
                        mma_mx(tmem, adesc + 2 * ks, bdesc + 2 * ks, idesc_mx(BM, BN, 0, 0), sfa_t, sfb_t,
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
        uint32_t tcount = 0;
        bool aborted = false;
        bool stop = false;     // GEMM1: abort decided at the row quarter's amax exchange
        int red_par = 0;       // GEMM1: exchange buffer of this tile
        for (int t = blockIdx.x; t < total; t += gridDim.x, tcount++) {
            const Tile tl = decode_tile(s, p.E, n_tiles, t);
            const bool row_ok = r_in < tl.rows;
            const int64_t row = (int64_t)tl.row0 + r_in;
            const int col0 = MODE == 1 ? 32 * cg : 64 * cg;
            const int col1 = MODE == 1 ? 128 + 32 * cg : 64 * cg + 32;
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
                    acc0[i] = __uint_as_float(r0[i]);
                    acc1[i] = __uint_as_float(r1[i]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.tempty);
            }
            if (MODE == 1) {
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    const float g = acc0[i];
                    acc0[i] = __fdiv_rn(g, 1.0f + expf(-g)) * acc1[i];
                    amax = fmaxf(amax, fabsf(acc0[i]));
                }
                // the row's amax over the four column groups: the warps of
                // row quarter q meet at their own barrier, which also ORs
                // their abort state so that they leave together; the
                // exchange buffer alternates by tile, so the next tile's
                // writes never meet this tile's reads
                s.red[red_par][cg][r_in] = amax;
                stop = quarter_bar_or(q, aborted || *abort_flag);
                amax = fmaxf(fmaxf(s.red[red_par][0][r_in], s.red[red_par][1][r_in]),
                             fmaxf(s.red[red_par][2][r_in], s.red[red_par][3][r_in]));
                red_par ^= 1;
                const uint32_t e8 = ue8m0_exp_of(amax);
                const float sc = e8 == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(e8 << 23);
                if (row_ok && !aborted) {
                    // sc is a power of two from 2^-127 to 2^127: its reciprocal
                    // is exact, so v * (1/sc) is the correctly rounded v / sc
                    const float rsc = __frcp_rn(sc);
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; i++)
                        w[i] = (uint32_t)pack_e4m3x2(acc0[4 * i] * rsc, acc0[4 * i + 1] * rsc) |
                               ((uint32_t)pack_e4m3x2(acc0[4 * i + 2] * rsc, acc0[4 * i + 3] * rsc) << 16);
                    uint4 *dst = reinterpret_cast<uint4 *>(p.act_q + row * p.F + tl.n_blk * 128 + 32 * cg);
                    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    if (cg == 0) p.act_e[row * (p.F / 128) + tl.n_blk] = (uint8_t)e8;
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
            if (MODE == 1 ? stop : (aborted || *abort_flag)) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

} // namespace ffn
} // namespace moe

using namespace moe;
using namespace moe::ffn;

MOE_API size_t moe_grouped_ffn_workspace_size(int64_t max_rows, int d, int F)
{
    (void)d;
    if (max_rows < 0 || F <= 0) return 0;
    return align256((size_t)max_rows * F) + align256((size_t)max_rows * (F / 128) * sizeof(float));
}

namespace moe {
namespace ffn {

// both GEMMs; GATHER: A rows of GEMM1 from the token-major x (T rows) by
// sorted_to_slot / top_k, outputs of GEMM2 to their slots
template <bool GATHER>
static moe_status ffn_launch(const uint8_t *xq, int64_t x_rows, const float *xs, const int32_t *sorted_to_slot,
                             int top_k, const int32_t *expert_offsets, int64_t max_rows, int E, int d, int F,
                             const uint8_t *w13_q, const float *w13_s, const uint8_t *w2_q, const float *w2_s,
                             uint16_t *out, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                             void *stream, float *h_out = nullptr)
{
    if (max_rows < 0 || max_rows >= (1LL << 31) || E < 1 || E > MAX_E || d <= 0 || F <= 0 || d % 128 != 0 ||
        F % 128 != 0)
        return MOE_ERR_SHAPE;
    if ((int64_t)E * 2 * F >= (1LL << 31) || (int64_t)E * d >= (1LL << 31)) return MOE_ERR_SHAPE;
    if (max_rows == 0) return MOE_OK;   // nothing to compute (the workspace may be empty too)
    const size_t need = moe_grouped_ffn_workspace_size(max_rows, d, F);
    if (!workspace || workspace_bytes < need) return MOE_ERR_WORKSPACE;
    if (!xq || !xs || !expert_offsets || !w13_q || !w13_s || !w2_q || !w2_s || !out) return MOE_ERR_NULL;
    if (GATHER && !sorted_to_slot) return MOE_ERR_NULL;
    if (!aligned16(xq) || !aligned16(w13_q) || !aligned16(w2_q) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return MOE_ERR_ALIGN;
    auto enc = encode_fn();
    if (!enc) return MOE_ERR_CUDA;
    uint8_t *act_q = reinterpret_cast<uint8_t *>(workspace);
    float *act_s = reinterpret_cast<float *>(reinterpret_cast<char *>(workspace) + align256((size_t)max_rows * F));
    CUtensorMap ma1, mb1, ma2, mb2;
    if (!make_map(enc, &ma1, xq, d, x_rows, GATHER ? 1 : 128) || !make_map(enc, &mb1, w13_q, d, (uint64_t)E * 2 * F, 128) ||
        !make_map(enc, &ma2, act_q, F, max_rows, 128) || !make_map(enc, &mb2, w2_q, F, (uint64_t)E * d, 256))
        return MOE_ERR_CUDA;
    Params prm;
    prm.b_scales = nullptr;
    prm.offsets = expert_offsets;
    prm.act_q = act_q;
    prm.act_s = act_s;
    prm.out = out;
    prm.dev_status = dev_status;
    prm.sorted_to_slot = sorted_to_slot;
    prm.h_out = nullptr;
    prm.max_rows = max_rows;
    prm.E = E;
    prm.d = d;
    prm.F = F;
    prm.top_k = top_k;
    if (!forward_kernel_regs_ok<1, GATHER>() || !forward_kernel_regs_ok<2, GATHER>()) return MOE_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(grouped_gemm_kernel<1, GATHER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_F_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(grouped_gemm_kernel<2, GATHER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_F_BYTES) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int grid = sm_count();
    cudaStream_t st = as_stream(stream);
    Params p1 = prm;
    p1.a_scales = xs;
    p1.b_scales = w13_s;
    p1.h_out = h_out;
    grouped_gemm_kernel<1, GATHER><<<grid, FT_THREADS, SMEM_F_BYTES, st>>>(ma1, mb1, p1);
    Params p2 = prm;
    p2.a_scales = act_s;
    p2.b_scales = w2_s;
    grouped_gemm_kernel<2, GATHER><<<grid, FT_THREADS, SMEM_F_BYTES, st>>>(ma2, mb2, p2);
    return launch_status();
}

} // namespace ffn
} // namespace moe

MOE_API moe_status moe_grouped_ffn_fp8(const uint8_t *xq_sorted, const float *xs_sorted,
                                       const int32_t *expert_offsets, int64_t max_rows, int E, int d, int F,
                                       const uint8_t *w13_q, const float *w13_s, const uint8_t *w2_q,
                                       const float *w2_s, uint16_t *out_sorted, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    return ffn_launch<false>(xq_sorted, max_rows, xs_sorted, nullptr, 1, expert_offsets, max_rows, E, d, F, w13_q,
                             w13_s, w2_q, w2_s, out_sorted, workspace, workspace_bytes, dev_status, stream);
}

MOE_API moe_status moe_grouped_ffn_fp8_train(const uint8_t *xq_sorted, const float *xs_sorted,
                                             const int32_t *expert_offsets, int64_t max_rows, int E, int d, int F,
                                             const uint8_t *w13_q, const float *w13_s, const uint8_t *w2_q,
                                             const float *w2_s, uint16_t *out_sorted, float *h_out, void *workspace,
                                             size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    if (max_rows != 0 && !h_out) return MOE_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(h_out) & 15) return MOE_ERR_ALIGN;
    return ffn_launch<false>(xq_sorted, max_rows, xs_sorted, nullptr, 1, expert_offsets, max_rows, E, d, F, w13_q,
                             w13_s, w2_q, w2_s, out_sorted, workspace, workspace_bytes, dev_status, stream, h_out);
}

MOE_API moe_status moe_grouped_gemm_fp8(const uint8_t *a_q, const float *a_s, const int32_t *expert_offsets,
                                        int64_t max_rows, int E, int K, int N, const uint8_t *b_q, const float *b_s,
                                        uint16_t *out, int32_t *dev_status, void *stream)
{
    if (max_rows < 0 || max_rows >= (1LL << 31) || E < 1 || E > MAX_E || K <= 0 || N <= 0 || K % 128 != 0 ||
        N % 128 != 0 || (int64_t)E * N >= (1LL << 31))
        return MOE_ERR_SHAPE;
    if (max_rows == 0) return MOE_OK;
    if (!a_q || !a_s || !expert_offsets || !b_q || !b_s || !out) return MOE_ERR_NULL;
    if (!aligned16(a_q) || !aligned16(b_q) || !aligned16(out)) return MOE_ERR_ALIGN;
    auto enc = encode_fn();
    if (!enc) return MOE_ERR_CUDA;
    CUtensorMap ma, mb;
    if (!make_map(enc, &ma, a_q, K, max_rows, 128) || !make_map(enc, &mb, b_q, K, (uint64_t)E * N, 256))
        return MOE_ERR_CUDA;
    // the GEMM2 form of the kernel with (K, N) in place of (F, d)
    Params prm;
    prm.a_scales = a_s;
    prm.b_scales = b_s;
    prm.offsets = expert_offsets;
    prm.act_q = nullptr;
    prm.act_s = nullptr;
    prm.out = out;
    prm.dev_status = dev_status;
    prm.sorted_to_slot = nullptr;
    prm.h_out = nullptr;
    prm.max_rows = max_rows;
    prm.E = E;
    prm.d = N;
    prm.F = K;
    prm.top_k = 1;
    if (!forward_kernel_regs_ok<2, false>()) return MOE_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(grouped_gemm_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_F_BYTES) != cudaSuccess)
        return MOE_ERR_CUDA;
    grouped_gemm_kernel<2, false><<<sm_count(), FT_THREADS, SMEM_F_BYTES, as_stream(stream)>>>(ma, mb, prm);
    return launch_status();
}

MOE_API moe_status moe_grouped_ffn_fp8_gathered(const uint8_t *xq, const float *xs, int T, int k,
                                                const int32_t *sorted_to_slot, const int32_t *expert_offsets,
                                                int E, int d, int F, const uint8_t *w13_q, const float *w13_s,
                                                const uint8_t *w2_q, const float *w2_s, uint16_t *out_slots,
                                                void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                                void *stream)
{
    if (T < 0 || k < 1 || k > 32 || (int64_t)T * k >= (1LL << 31)) return MOE_ERR_SHAPE;
    if (T == 0) return MOE_OK;
    return ffn_launch<true>(xq, T, xs, sorted_to_slot, k, expert_offsets, (int64_t)T * k, E, d, F, w13_q, w13_s,
                            w2_q, w2_s, out_slots, workspace, workspace_bytes, dev_status, stream);
}

MOE_API size_t moe_grouped_ffn_mx_workspace_size(int64_t max_rows, int d, int F)
{
    (void)d;
    if (max_rows < 0 || F <= 0) return 0;
    return align256((size_t)max_rows * F) + align256((size_t)max_rows * (F / 128));
}

MOE_API moe_status moe_grouped_ffn_mx(const uint8_t *xq_sorted, const uint8_t *x_exp, const int32_t *sorted_to_slot,
                                      int T, int k, const int32_t *expert_offsets, int64_t max_rows, int E, int d,
                                      int F, const uint8_t *w13_q, const uint8_t *w13_exp, const uint8_t *w2_q,
                                      const uint8_t *w2_exp, uint16_t *out_sorted, void *workspace,
                                      size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    if (max_rows < 0 || max_rows >= (1LL << 31) || E < 1 || E > MAX_E || d <= 0 || F <= 0 || d % 128 != 0 ||
        F % 128 != 0 || T < 0 || k < 1 || k > 32)
        return MOE_ERR_SHAPE;
    if ((int64_t)E * 2 * F >= (1LL << 31) || (int64_t)E * d >= (1LL << 31)) return MOE_ERR_SHAPE;
    if (max_rows == 0 || T == 0) return MOE_OK;   // nothing to compute (the workspace may be empty too)
    const size_t need = moe_grouped_ffn_mx_workspace_size(max_rows, d, F);
    if (!workspace || workspace_bytes < need) return MOE_ERR_WORKSPACE;
    if (!xq_sorted || !x_exp || !sorted_to_slot || !expert_offsets || !w13_q || !w13_exp || !w2_q || !w2_exp ||
        !out_sorted)
        return MOE_ERR_NULL;
    if (!aligned16(xq_sorted) || !aligned16(w13_q) || !aligned16(w2_q) || !aligned16(out_sorted) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return MOE_ERR_ALIGN;
    auto enc = encode_fn();
    if (!enc) return MOE_ERR_CUDA;
    uint8_t *act_q = reinterpret_cast<uint8_t *>(workspace);
    uint8_t *act_e = reinterpret_cast<uint8_t *>(workspace) + align256((size_t)max_rows * F);
    CUtensorMap ma1, mb1, ma2, mb2;
    if (!make_map(enc, &ma1, xq_sorted, d, max_rows, 128) || !make_map(enc, &mb1, w13_q, d, (uint64_t)E * 2 * F, 128) ||
        !make_map(enc, &ma2, act_q, F, max_rows, 128) || !make_map(enc, &mb2, w2_q, F, (uint64_t)E * d, 256))
        return MOE_ERR_CUDA;
    ParamsMX prm;
    prm.offsets = expert_offsets;
    prm.sorted_to_slot = sorted_to_slot;
    prm.act_q = act_q;
    prm.act_e = act_e;
    prm.out = out_sorted;
    prm.dev_status = dev_status;
    prm.max_rows = max_rows;
    prm.E = E;
    prm.d = d;
    prm.F = F;
    prm.top_k = k;
    if (cudaFuncSetAttribute(grouped_gemm_mx_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_MX_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(grouped_gemm_mx_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_MX_BYTES) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int grid = sm_count();
    cudaStream_t st = as_stream(stream);
    ParamsMX p1 = prm;
    p1.a_exp = x_exp;
    p1.b_exp = w13_exp;
    grouped_gemm_mx_kernel<1><<<grid, THREADS, SMEM_MX_BYTES, st>>>(ma1, mb1, p1);
    ParamsMX p2 = prm;
    p2.a_exp = act_e;
    p2.b_exp = w2_exp;
    grouped_gemm_mx_kernel<2><<<grid, THREADS, SMEM_MX_BYTES, st>>>(ma2, mb2, p2);
    return launch_status();
}

MOE_API moe_status moe_wgrad_gemm(const uint8_t *a_q, const float *a_sT, const uint8_t *b_q, const float *b_sT,
                                  const int32_t *pad, int E, int M, int N, int64_t ld, float *out,
                                  int32_t *dev_status, void *stream)
{
    // the output rows e * M + m are 32-bit TMA coordinates
    if (E < 1 || E > MAX_E || M <= 0 || N <= 0 || M % BM != 0 || N % 128 != 0 || ld <= 0 || ld % 128 != 0 ||
        ld >= (1LL << 31) || (int64_t)E * M >= (1LL << 31) || (int64_t)N >= (1LL << 31))
        return MOE_ERR_SHAPE;
    if (!a_q || !a_sT || !b_q || !b_sT || !pad || !out) return MOE_ERR_NULL;
    if (!aligned16(a_q) || !aligned16(b_q) || !aligned16(out) || !aligned16(a_sT) || !aligned16(b_sT))
        return MOE_ERR_ALIGN;
    auto enc = encode_fn();
    if (!enc) return MOE_ERR_CUDA;
    CUtensorMap ma, mb;
    CUtensorMap mo;
    if (!make_map(enc, &ma, a_q, ld, M, BM) || !make_map(enc, &mb, b_q, ld, N, WG_BN) ||
        !make_map_f32_store(enc, &mo, out, (uint64_t)N, (uint64_t)E * M))
        return MOE_ERR_CUDA;
    ParamsWG prm;
    prm.saT = a_sT;
    prm.sbT = b_sT;
    prm.pad = pad;
    prm.out = out;
    prm.dev_status = dev_status;
    prm.ld = ld;
    prm.E = E;
    prm.M = M;
    prm.N = N;
    if (cudaFuncSetAttribute(grouped_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_WG_BYTES) != cudaSuccess)
        return MOE_ERR_CUDA;
    cudaStream_t st = as_stream(stream);
    wgrad_zero_empty_kernel<<<dim3(64, (unsigned)E), 256, 0, st>>>(pad, (int64_t)M * N, out);
    grouped_wgrad_kernel<<<sm_count(), THREADS, SMEM_WG_BYTES, st>>>(ma, mb, mo, prm);
    return launch_status();
}
