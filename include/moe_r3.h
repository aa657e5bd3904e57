/*
 * moe_r3.h -- C ABI of libmoe_r3: one GPU's Mixture-of-Experts layer with
 * router replay (R3) and block-scaled FP8 expert GEMMs, for sm_103a (GB300).
 *
 * The method is the one described in "RL at 1T Scale: prime-rl Performance
 * Deep Dive" (prime-rl 0.6.0):
 *   - section "Router replay": the routing decisions made during inference are
 *     captured and replayed on the trainer; the routed-experts payload has
 *     shape [num_layers, top_k, seq_len] and is handled as an opaque tensor;
 *   - section "FP8 training": block-scaled FP8 as proposed by DeepSeek-V3
 *     (E4M3 values, one fp32 scale per 1x128 activation tile and per 128x128
 *     weight block);
 *   - section "Parallelism", "Expert parallelism (EP)": tokens are dispatched
 *     to their experts and combined back.
 * The page leaves the kernel-level contract open; this header states it.
 *
 * Conventions for every entry point
 *   - Tensor pointers are DEVICE pointers owned by the caller, row-major and
 *     dense unless a leading dimension is given.  bf16 travels as uint16_t,
 *     E4M3 as uint8_t (OCP "e4m3fn": bias 7, max 448, no inf).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued on it; no call synchronises the host or
 *     copies device data to the host, and no call allocates or frees memory.
 *     Scratch memory is caller-provided workspace whose size is queried,
 *     except for moe_dispatch_noalloc, whose scratch is a static device array
 *     inside the library (see that call).
 *   - Errors the host can see (NULL pointers, unsupported shapes, misaligned
 *     pointers, short workspace) are returned before anything is launched and
 *     nothing is written.  A failed launch returns MOE_ERR_CUDA.
 *   - Errors only the device can see are OR-ed, as MOE_DEV_* bits, into the
 *     caller-zeroed int32 word `dev_status` (nullable: then not reported).
 *     Kernels never write out of bounds because of them.  Every device wait
 *     is bounded; on expiry the kernel sets MOE_DEV_TIMEOUT and returns.
 *   - Calls are stream-ordered and thread-safe: no call keeps global mutable
 *     state, except moe_dispatch_noalloc, whose calls share one static
 *     scratch array, so the caller must order noalloc calls that could
 *     overlap on the GPU (other streams or threads).
 */
#ifndef MOE_R3_H
#define MOE_R3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status;

/* host return codes */
#define MOE_OK 0
#define MOE_ERR_NULL 1        /* a required pointer is NULL */
#define MOE_ERR_SHAPE 2       /* unsupported sizes (see each call) */
#define MOE_ERR_ALIGN 3       /* a pointer or leading dimension breaks 16-byte alignment */
#define MOE_ERR_WORKSPACE 4   /* workspace NULL or smaller than the queried size */
#define MOE_ERR_CUDA 5        /* a CUDA launch or driver call failed */
#define MOE_ERR_UNSUPPORTED 6 /* valid request this build does not implement */

/* device status bits (OR-ed into *dev_status) */
#define MOE_DEV_BAD_IDS 0x1   /* a replayed / dispatched id is out of [0,E) or repeated in a token */
#define MOE_DEV_TIMEOUT 0x2   /* a bounded device wait expired */
#define MOE_DEV_ROWS 0x4      /* routed rows exceed the max_rows the GEMM was sized for */

/* score functions */
#define MOE_SCORE_SOFTMAX 0
#define MOE_SCORE_SIGMOID 1

/* Limits of this build: 1 <= k <= min(E, 32); 1 <= E <= 1024; d and F
 * multiples of 128; T * k < 2^31. */

const char *moe_status_str(moe_status s);

/* ------------------------------------------------------------------------
 * moe_route_topk -- router logits, top-k selection, gates, optional capture.
 * ("Router replay": this is the decision that inference captures.)
 *
 *   logits[t,e] = sum_{i=0}^{d-1} x[t,i] * w_router[e,i], evaluated as one
 *                 binary32 fused multiply-add chain in ascending i from +0
 *                 (bit-reproducible; denormals honoured);
 *   topk_ids[t,j] = the j-th largest logit's expert; equal logits (-0 == +0)
 *                 go to the lower index; NaN ranks below every number;
 *   topk_gates[t,j] = score(l_j) / sum_{i<k} score(l_i) if renorm (softmax
 *                 over the chosen k; sigmoid normalised over the chosen k),
 *                 else the full softmax over E / the plain sigmoid; then
 *                 times route_scale;
 *   capture_kT[j*T + t] = topk_ids[t,j] (nullable): one layer's [k, T] slab
 *                 of the routed-experts payload [num_layers, top_k, seq_len];
 *   logits_out[t,e] (nullable) = logits.
 * x [T,d] bf16; w_router [E,d] bf16, both 16-byte aligned; topk_ids [T,k]
 * int32; topk_gates [T,k] fp32.  T may be 0 (nothing launched).
 * Errors: NULL, SHAPE, ALIGN.
 * ---------------------------------------------------------------------- */
moe_status moe_route_topk(const uint16_t *x, const uint16_t *w_router, int T, int d, int E, int k,
                          int score_fn, int renorm, float route_scale, int32_t *topk_ids,
                          float *topk_gates, int32_t *capture_kT, float *logits_out, void *stream);

/* ------------------------------------------------------------------------
 * moe_route_replay -- replay one layer of a captured routing payload
 * ("Router replay": decisions captured at inference replace the trainer's
 * own routing).
 *
 *   topk_ids[t,j] = replay_kT[j*T + t], an exact copy in slot order, where
 *   replay_kT = payload + layer*k*T is the layer's [k, T] slab.
 *   A token whose k ids are not all in [0,E) and pairwise distinct sets
 *   MOE_DEV_BAD_IDS; its ids are still copied and its gates are 0.
 *   If x != NULL: topk_gates from the router logits of the replayed experts
 *   (same logits, score function, renormalisation and scale as
 *   moe_route_topk, so replaying a capture reproduces its gates bit for
 *   bit).  If x == NULL, topk_gates may be NULL and is not written.
 * x and w_router 16-byte aligned when x != NULL (with both 32-byte aligned
 * the logits read whole 32-byte sectors per load; same results either way).
 * The full softmax over E (score_fn SOFTMAX, renorm 0) needs every logit
 * and is not replayed from x: UNSUPPORTED.
 * Errors: NULL, SHAPE, ALIGN, UNSUPPORTED.
 * ---------------------------------------------------------------------- */
moe_status moe_route_replay(const int32_t *replay_kT, const uint16_t *x, const uint16_t *w_router,
                            int T, int d, int E, int k, int score_fn, int renorm, float route_scale,
                            int32_t *topk_ids, float *topk_gates, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * moe_route_replay_u8 -- moe_route_replay from a one-byte payload slab
 * ("Router replay": the routed-experts payload moved at one byte per id,
 * see moe_payload_pack_u8).
 *
 *   Identical to moe_route_replay with replay_kT[j*T + t] widened from
 *   uint8_t: same copy, same validation (ids in [0,E), distinct per token,
 *   MOE_DEV_BAD_IDS otherwise), same gates.  replay_kT needs no alignment.
 * Errors: NULL, SHAPE, ALIGN (x, w_router), UNSUPPORTED (as moe_route_replay).
 * ---------------------------------------------------------------------- */
moe_status moe_route_replay_u8(const uint8_t *replay_kT, const uint16_t *x, const uint16_t *w_router,
                               int T, int d, int E, int k, int score_fn, int renorm, float route_scale,
                               int32_t *topk_ids, float *topk_gates, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * moe_router_backward -- gradients of the router for fixed expert ids
 * ("Router replay": the trainer replays the captured ids and still trains
 * the router through the gates it recomputes from their logits).
 *
 *   l[t,j] = the logit of expert topk_ids[t,j], the same binary32 fma chain
 *            as moe_route_topk / moe_route_replay;
 *   d_logits[t,j] = dL/dl[t,j] from d_gates[t,j] = dL/dg[t,j] through the
 *            gate function (rs = route_scale):
 *              softmax, renorm:    p_j = exp(l_j) / sum_i exp(l_i),
 *                                  dl_j = rs p_j (dg_j - sum_i dg_i p_i)
 *              sigmoid, renorm:    s_j = 1 / (1 + exp(-l_j)), S = sum_i s_i,
 *                                  dl_j = rs s_j (1 - s_j) (dg_j - sum_i dg_i s_i / S) / S
 *              sigmoid, no renorm: dl_j = rs dg_j s_j (1 - s_j)
 *            in fp32; a token whose ids are not all in [0,E) and distinct
 *            gets zeros and sets MOE_DEV_BAD_IDS;
 *   dx[t,c] = sum_j d_logits[t,j] * w_router[topk_ids[t,j], c] (nullable;
 *            fp32, the slots in order) -- the router's part of dL/dx;
 *   dw_router[e,c] = sum over expert e's rows of the dispatch that produced
 *            sorted_to_slot / expert_offsets for these ids, in that sorted
 *            order, of d_logits[slot] * x[slot / k, c] (nullable; fp32; an
 *            expert without rows gets zeros).  A slot outside [0, T*k) adds
 *            nothing; offsets outside [0, T*k], or decreasing, are clamped
 *            into that range and set MOE_DEV_ROWS.
 * x [T,d] bf16, w_router [E,d] bf16 (16-byte aligned; 32-byte alignment of
 * both lets the logits read whole sectors), topk_ids [T,k] int32, d_gates,
 * d_logits [T,k] fp32, dx [T,d] fp32, dw_router [E,d] fp32 (16-byte
 * aligned); sorted_to_slot [T*k] and expert_offsets [E+1] are moe_dispatch's
 * maps, needed only with dw_router.  T may be 0: the [T, .] arrays and the
 * maps may then be NULL and dw_router, if given, is zeroed.  The full
 * softmax over E (score_fn SOFTMAX, renorm 0) depends on
 * every expert's logit: UNSUPPORTED.
 * Errors: NULL, SHAPE, ALIGN, UNSUPPORTED.
 * ---------------------------------------------------------------------- */
moe_status moe_router_backward(const uint16_t *x, const uint16_t *w_router, const int32_t *topk_ids,
                               const float *d_gates, int T, int d, int E, int k, int score_fn, int renorm,
                               float route_scale, float *d_logits, float *dx, const int32_t *sorted_to_slot,
                               const int32_t *expert_offsets, float *dw_router, int32_t *dev_status,
                               void *stream);

/* ------------------------------------------------------------------------
 * moe_payload_pack_u8 / moe_payload_unpack_u8 -- the routed-experts payload
 * at one byte per id ("Router replay": the [num_layers, top_k, seq_len]
 * payload is large enough to strain its transport; with E <= 256 every id
 * fits a byte, a 4x smaller payload).
 *
 *   pack:   out[i] = (uint8_t)ids[i] for 0 <= ids[i] < E, i in [0, n).  An id
 *           outside [0, E) is stored as 0xFF and sets MOE_DEV_BAD_IDS in the
 *           caller-zeroed *dev_status (device memory, required).
 *   unpack: out[i] = in[i] widened to int32.
 * Any flat layout: a whole [L, k, T] payload or one [k, T] layer slab, n
 * elements.  Device buffers, caller-owned, need no alignment (16-byte
 * aligned buffers take the vector path).  n may be 0.
 * Errors: pack -- SHAPE (n < 0, E < 1), UNSUPPORTED (E > 256), NULL;
 *         unpack -- SHAPE (n < 0), NULL.
 * ---------------------------------------------------------------------- */
moe_status moe_payload_pack_u8(const int32_t *ids, int64_t n, int E, uint8_t *out, int32_t *dev_status,
                               void *stream);
moe_status moe_payload_unpack_u8(const uint8_t *in, int64_t n, int32_t *out, void *stream);

/* ------------------------------------------------------------------------
 * fp8_block_quant -- block-scaled E4M3 quantisation ("FP8 training",
 * DeepSeek-V3 recipe).
 *
 * Blocks are 1 x 128 (block_rows = 1, activations) or 128 x 128
 * (block_rows = 128, weights).  Per block: amax = max |v|, s = amax / 448
 * (IEEE binary32 division; s = 1 if that is 0), q = E4M3(v / s) with IEEE
 * division, round to nearest even, saturating to +-448, sign of zero kept.
 * src [rows, cols] bf16 with row stride ld_src elements; q [rows, cols]
 * (row stride cols); scales [rows/block_rows, cols/128] fp32.
 * rows may be 0.  Errors: NULL, SHAPE (cols % 128, rows % block_rows),
 * ALIGN (src, q, ld_src not 16-byte aligned).
 * ---------------------------------------------------------------------- */
moe_status fp8_block_quant(const uint16_t *src, int64_t rows, int64_t cols, int64_t ld_src,
                           int block_rows, uint8_t *q, float *scales, void *stream);

/* ------------------------------------------------------------------------
 * fp8_quant_nvfp4 -- NVFP4 quantisation (the FP4 variant listed as future
 * work for training and inference in "RL at 1T Scale", closing section;
 * NVIDIA's NVFP4 format): FP4 E2M1 values, 16-element blocks along each row
 * with E4M3 block scales, one fp32 scale for the tensor.
 *
 *   s_enc = (6 * 448) / amax over the tensor (binary32; 1 if amax is 0),
 *   per block: scale byte = E4M3((amax_block / 6) * s_enc), round to
 *     nearest even, saturating; per element: code = E2M1(x * (s_enc /
 *     scale)), nearest even, saturating to +-6 (0 where the scale byte
 *     decodes to 0); decoded value = e2m1 * scale / s_enc.
 * src [rows, cols] bf16 (row stride cols); q [rows, cols/2] (element 2i in
 * the low nibble of byte i, 2i+1 in the high nibble); scales [rows, cols/16]
 * E4M3 bytes; tensor_scale: two device floats, [0] = s_enc (written), [1] =
 * the tensor amax (written; scratch of the first pass).  Two launches (amax,
 * then the blocks) and a memset on `stream`.
 * rows may be 0.  Errors: NULL, SHAPE (cols % 16), ALIGN (src, q not
 * 16-byte aligned), CUDA.  NaN inputs are outside the contract.
 * ---------------------------------------------------------------------- */
moe_status fp8_quant_nvfp4(const uint16_t *src, int64_t rows, int64_t cols, uint8_t *q, uint8_t *scales,
                           float *tensor_scale, void *stream);

/* ------------------------------------------------------------------------
 * moe_nvfp4_tile_scales -- the E4M3 block scales of an NVFP4 weight matrix
 * (fp8_quant_nvfp4 layout, s [rows, K/16]) rearranged once per weight
 * update into the images the NVFP4 GEMM copies to tensor memory: per
 * 128-row group g and 256-element K block kb, 2048 contiguous bytes
 * [MMA 0..3][r 0..31][q 0..3] of 32-bit words, word (g, kb, m, r, q) =
 * scale bytes 16kb + 4m .. 16kb + 4m + 3 of row 128g + 32q + r (0 past K/16).
 * rows % 128 == 0, K % 128 == 0; s 4-byte aligned, s_tiled 16-byte aligned,
 * moe_nvfp4_tiled_scales_size(rows, K) bytes.
 * Errors: NULL, SHAPE, ALIGN.
 * ---------------------------------------------------------------------- */
size_t moe_nvfp4_tiled_scales_size(int64_t rows, int64_t K);
moe_status moe_nvfp4_tile_scales(const uint8_t *s, int64_t rows, int64_t K, uint8_t *s_tiled, void *stream);

/* ------------------------------------------------------------------------
 * moe_grouped_ffn_nvfp4 -- the grouped SwiGLU expert FFN in NVFP4 (the FP4
 * variant listed as future work for training and inference in "RL at 1T
 * Scale", closing section) on the block-scaled tensor-core MMA
 * (tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X).
 *
 * Operands as fp8_quant_nvfp4 writes them: E2M1 codes two per byte, E4M3
 * scales per 16 elements along K, one fp32 tensor scale s_enc (decoded
 * value = e2m1 * scale / s_enc).  For sorted row r of expert e:
 *   h[r, n]  = sum_k xdec[r, k] * w13dec[e][n, k] (the tensor core applies
 *              the block scales, accumulates in fp32; the epilogue divides
 *              by x_enc * w13_enc[e]);
 *   act[r,c] = bf16( silu(h[r, c]) * h[r, F + c] )  (c < F), materialised
 *              in the workspace with its amax over the routed rows, then
 *              quantised to NVFP4 with one tensor scale (fp8_quant_nvfp4);
 *   out[r,:] = bf16( act_dec[r] W2dec[e]^T ), likewise.
 * xq_sorted [max_rows, d/2], xs_sorted [max_rows, d/16] (moe_dispatch of the
 * token-major codes and scales), x_enc: the token tensor's s_enc (device);
 * w13_q [E, 2F, d/2], w13_sf_tiled = moe_nvfp4_tile_scales of w13's scales
 * [E*2F, d/16], w13_enc [E] (device, one per expert matrix); w2_q
 * [E, d, F/2], w2_sf_tiled of [E*d, F/16], w2_enc [E]; out_sorted
 * [max_rows, d] bf16.  d, F multiples of 128; max_rows bounds
 * expert_offsets[E] as in moe_grouped_ffn_fp8 (clipped, MOE_DEV_ROWS).
 * workspace: moe_grouped_ffn_nvfp4_workspace_size bytes, 256-byte aligned
 * (act in bf16 and NVFP4, and the act tensor's scale).  max_rows may be 0:
 * nothing is launched, and the buffers and the workspace may then be NULL.
 * Errors: NULL, SHAPE, ALIGN, WORKSPACE, CUDA.
 * ---------------------------------------------------------------------- */
size_t moe_grouped_ffn_nvfp4_workspace_size(int64_t max_rows, int d, int F);
moe_status moe_grouped_ffn_nvfp4(const uint8_t *xq_sorted, const uint8_t *xs_sorted, const float *x_enc,
                                 const int32_t *expert_offsets, int64_t max_rows, int E, int d, int F,
                                 const uint8_t *w13_q, const uint8_t *w13_sf_tiled, const float *w13_enc,
                                 const uint8_t *w2_q, const uint8_t *w2_sf_tiled, const float *w2_enc,
                                 uint16_t *out_sorted, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * fp8_block_quant_ue8m0 -- fp8_block_quant with power-of-two block scales
 * (the UE8M0 scale format of MXFP8 and of the hardware block-scaled MMA; a
 * variant of the "FP8 training" recipe, whose scales are arbitrary fp32).
 *
 * Per block (1 x 128 or 128 x 128 as fp8_block_quant): amax = max |v|; the
 * scale is 2^p for the smallest integer p with amax <= 448 * 2^p (p clamped
 * to [-127, 127]; an all-zero block takes p = 0); scale_exp holds p + 127;
 * q = E4M3(v / 2^p), round to nearest even (no code saturates).
 * scale_exp [rows/block_rows, cols/128] uint8.  Errors as fp8_block_quant.
 * ---------------------------------------------------------------------- */
moe_status fp8_block_quant_ue8m0(const uint16_t *src, int64_t rows, int64_t cols, int64_t ld_src,
                                 int block_rows, uint8_t *q, uint8_t *scale_exp, void *stream);

/* ------------------------------------------------------------------------
 * moe_dispatch -- permute token rows into expert-contiguous order
 * ("Expert parallelism": dispatch).
 *
 * Slots s = t*k + j are counting-sorted by expert id in ascending slot order
 * (stable):
 *   expert_counts[e]  = #slots routed to e;
 *   expert_offsets[e] = sum_{e'<e} expert_counts[e'], expert_offsets[E] =
 *                       routed slots;
 *   sorted_to_slot[r] = the slot at sorted position r (r < expert_offsets[E]);
 *   slot_to_sorted[s] = its inverse (-1 for a slot whose id is outside
 *                       [0,E): such slots are not routed and set
 *                       MOE_DEV_BAD_IDS);
 *   rows_sorted[r]    = rows[sorted_to_slot[r] / k]  (row_bytes each),
 *   scales_sorted[r]  = row_scales[sorted_to_slot[r] / k] (scales_per_row
 *                       fp32 each; 0 = no scales, both pointers ignored).
 * rows may be e4m3 codes (row_bytes = d) or bf16 (row_bytes = 2d);
 * row_bytes must be a multiple of 16; rows, rows_sorted 16-byte aligned.
 * rows / rows_sorted may be NULL to build the maps only.
 * Sorted positions >= expert_offsets[E] are left unwritten.
 * workspace: moe_dispatch_workspace_size(T, k, E) bytes, 256-byte aligned.
 * Errors: NULL, SHAPE, ALIGN, WORKSPACE.
 * ---------------------------------------------------------------------- */
size_t moe_dispatch_workspace_size(int T, int k, int E);
moe_status moe_dispatch(const int32_t *topk_ids, int T, int k, int E, const void *rows,
                        int64_t row_bytes, const float *row_scales, int scales_per_row,
                        int32_t *expert_counts, int32_t *expert_offsets, int32_t *sorted_to_slot,
                        int32_t *slot_to_sorted, void *rows_sorted, float *scales_sorted,
                        void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * moe_dispatch_noalloc -- moe_dispatch without a caller workspace.
 *
 * The page describes no such call; it exists for callers of this library
 * that cannot allocate device memory when they dispatch: a process that
 * plans its whole device-memory budget up front and has no spare buffer to
 * lend, or a latency-critical path that must not call cudaMalloc (which may
 * synchronise the device).  Arguments, results and errors are those of
 * moe_dispatch, without `workspace` / `workspace_bytes`: the scratch lives
 * in a static device array of MOE_DISPATCH_NOALLOC_MAX_SCRATCH bytes inside
 * the library, held on every GPU that loads the library until the process
 * exits.  A request whose moe_dispatch_workspace_size(T, k, E) exceeds that
 * limit returns MOE_ERR_WORKSPACE before anything is launched (4 MiB covers,
 * e.g., E = 256 with T*k up to 4M slots, or E = 1024 with T*k up to 1M).
 * Nothing is allocated or freed: no cudaMalloc, no cudaFree, no allocating
 * library routine.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current) and keeps it, so
 * make that first call before any stream capture.  Every call shares the one
 * array: calls whose work overlaps on the GPU (other streams or threads)
 * race on it and must be ordered by the caller.  No part of the array needs
 * to start zeroed; the contents a previous call left are never read.
 * ---------------------------------------------------------------------- */
#define MOE_DISPATCH_NOALLOC_MAX_SCRATCH (4u << 20)
moe_status moe_dispatch_noalloc(const int32_t *topk_ids, int T, int k, int E, const void *rows,
                                int64_t row_bytes, const float *row_scales, int scales_per_row,
                                int32_t *expert_counts, int32_t *expert_offsets, int32_t *sorted_to_slot,
                                int32_t *slot_to_sorted, void *rows_sorted, float *scales_sorted,
                                int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * moe_grouped_ffn_fp8 -- per-expert SwiGLU FFN as two grouped block-scaled
 * FP8 GEMMs on the tensor cores ("FP8 training", DeepSeek-V3 recipe).
 *
 * For every expert e and sorted row r in [expert_offsets[e],
 * expert_offsets[e+1]) (offsets read on the device; no host sync):
 *   h[r,n]   = sum_kb (xs_sorted[r,kb] * w13_s[e,n/128,kb]) * P_kb(r,n),
 *              P_kb = the 128-deep block product of E4M3 codes accumulated
 *              in fp32, promoted into an fp32 accumulator block by block;
 *   act[r,c] = silu(h[r,c]) * h[r,F+c]   (c < F; w13 rows 0..F-1 gate,
 *              F..2F-1 up; silu from the fast exponential and reciprocal),
 *              requantised 1x128 along F with fp8_block_quant's scale rule,
 *              codes E4M3(act * RN(1/s));
 *   out_sorted[r,:] = bf16 (round to nearest even) of act_q[r,:] W2[e]^T by
 *              the same block promotion.
 * xq_sorted [max_rows, d] e4m3, xs_sorted [max_rows, d/128] fp32;
 * w13_q [E, 2F, d], w13_s [E, 2F/128, d/128]; w2_q [E, d, F],
 * w2_s [E, d/128, F/128]; out_sorted [max_rows, d] bf16.  max_rows bounds
 * expert_offsets[E]: offsets outside [0, max_rows] are clipped into it and
 * set MOE_DEV_ROWS, so rows outside the buffers are never read or written.
 * workspace: moe_grouped_ffn_workspace_size(max_rows, d, F) bytes (holds
 * act_q and its scales), 256-byte aligned.  max_rows may be 0: nothing is
 * launched, and the buffers and the workspace may then be NULL.
 * Errors: NULL, SHAPE, ALIGN, WORKSPACE, CUDA.
 * ---------------------------------------------------------------------- */
size_t moe_grouped_ffn_workspace_size(int64_t max_rows, int d, int F);
moe_status moe_grouped_ffn_fp8(const uint8_t *xq_sorted, const float *xs_sorted,
                               const int32_t *expert_offsets, int64_t max_rows, int E, int d, int F,
                               const uint8_t *w13_q, const float *w13_s, const uint8_t *w2_q,
                               const float *w2_s, uint16_t *out_sorted, void *workspace,
                               size_t workspace_bytes, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * moe_grouped_ffn_fp8_gathered -- moe_grouped_ffn_fp8 with the dispatch
 * row gather fused into GEMM1's operand load and the un-permute fused into
 * GEMM2's store ("FP8 inference": FP8 with DeepEP dispatch/combine and
 * DeepGEMM kernels; "Expert parallelism": dispatch and combine).
 *
 *   Same arithmetic as moe_grouped_ffn_fp8 for sorted row r of expert e, but
 *   the row's codes and scales are read from the token-major quantised
 *   activations, xq[t] and xs[t] with t = sorted_to_slot[r] / k (tile::gather4
 *   TMA loads, four rows per copy), and its output goes to
 *   out_slots[sorted_to_slot[r], :] -- slot order, row t*k + j -- so the
 *   permuted activation copy of moe_dispatch (its rows output) is not needed
 *   and moe_combine_slots reads each token's k rows contiguously.
 * xq [T, d] e4m3, xs [T, d/128] fp32, sorted_to_slot and expert_offsets from
 * moe_dispatch (maps only); out_slots [T*k, d] bf16 (rows of unrouted slots
 * are not written; a sorted_to_slot entry outside [0, T*k) marks its row as
 * not routed: nothing is stored for it and MOE_DEV_ROWS is set);
 * workspace: moe_grouped_ffn_workspace_size(T*k, d, F).
 * Errors: NULL, SHAPE, ALIGN, WORKSPACE, CUDA.
 * ---------------------------------------------------------------------- */
moe_status moe_grouped_ffn_fp8_gathered(const uint8_t *xq, const float *xs, int T, int k,
                                        const int32_t *sorted_to_slot, const int32_t *expert_offsets, int E,
                                        int d, int F, const uint8_t *w13_q, const float *w13_s,
                                        const uint8_t *w2_q, const float *w2_s, uint16_t *out_slots,
                                        void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                        void *stream);

/* ------------------------------------------------------------------------
 * moe_grouped_ffn_mx -- the grouped SwiGLU FFN with power-of-two (UE8M0)
 * block scales on the hardware block-scaled MMA
 * (tcgen05.mma.kind::mxf8f6f4.block_scale): a variant of the "FP8
 * training" recipe whose scales are powers of two, so no per-block software
 * promotion is needed.
 *
 *   h[r,n] = sum over K of (xq * 2^(x_exp-127)) (w13_q * 2^(w13_exp-127)),
 *            accumulated in fp32 by the tensor core; act = silu(gate) * up,
 *            re-quantised 1x128 along F with power-of-two scales (the rule of
 *            fp8_block_quant_ue8m0); out_sorted = bf16 of act_q W2^T likewise.
 * xq_sorted [max_rows, d] e4m3 (moe_dispatch rows); x_exp [T, d/128] uint8,
 * token-major (row r's exponents are x_exp[sorted_to_slot[r] / k]);
 * w13_q [E, 2F, d], w13_exp [E, 2F/128, d/128]; w2_q [E, d, F],
 * w2_exp [E, d/128, F/128]; workspace moe_grouped_ffn_mx_workspace_size
 * bytes (act_q and its exponents), 256-byte aligned.  max_rows or T may be
 * 0: nothing is launched, and the buffers and the workspace may then be NULL.
 * Errors: NULL, SHAPE, ALIGN, WORKSPACE, CUDA.
 * ---------------------------------------------------------------------- */
size_t moe_grouped_ffn_mx_workspace_size(int64_t max_rows, int d, int F);
moe_status moe_grouped_ffn_mx(const uint8_t *xq_sorted, const uint8_t *x_exp, const int32_t *sorted_to_slot,
                              int T, int k, const int32_t *expert_offsets, int64_t max_rows, int E, int d, int F,
                              const uint8_t *w13_q, const uint8_t *w13_exp, const uint8_t *w2_q,
                              const uint8_t *w2_exp, uint16_t *out_sorted, void *workspace,
                              size_t workspace_bytes, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Backward of the expert path under replay ("Router replay": the trainer
 * replays the captured routing and trains through the layer; "FP8 training":
 * its GEMMs are block-scaled FP8).  With the ids fixed, given dy [T, d]:
 *   moe_combine_backward   d_out[r] = g[t,j] * dy[t] (binary32 product),
 *                          quantised 1x128 along d as fp8_block_quant, to the
 *                          slot's sorted row r = slot_to_sorted[t*k+j];
 *                          d_gates[t,j] = <dy[t], out_sorted[r]> (fp32
 *                          accumulation in a fixed order), 0 for an
 *                          unrouted slot.  For d <= 8192 the rows are
 *                          staged by bulk copies and every wait is bounded:
 *                          one that runs out ORs MOE_DEV_TIMEOUT into
 *                          dev_status (nullable) and the call's outputs are
 *                          then incomplete.
 *   moe_grouped_gemm_fp8   with W2 transposed: d_act = d_out W2 (bf16).
 *   moe_swiglu_backward    from the saved pre-activations h = [g | u]:
 *                          d_g = d_act * u * s(g) * (1 + g (1 - s(g))),
 *                          d_u = d_act * g * s(g) (s the logistic sigmoid,
 *                          from the fast exponential and reciprocal as the
 *                          forward's silu), quantised 1x128 along 2F.
 *   moe_grouped_gemm_fp8   with W13 transposed: dx_sorted = dh W13 (bf16).
 *   moe_dispatch_backward  dx[t] = bf16(sum_j dx_sorted[r(t,j)]), a binary32
 *                          sum in slot order.
 * moe_grouped_ffn_fp8_train is moe_grouped_ffn_fp8 that also writes h
 * [max_rows, 2F] fp32 (GEMM1's promoted accumulators, gate columns then up
 * columns).  fp8_weight_transpose turns [E, R, C] codes with [E, R/128,
 * C/128] scales into [E, C, R] / [E, C/128, R/128] (block quantisation
 * commutes with transposition), once per weight update.
 * moe_grouped_gemm_fp8 is the block-scaled grouped GEMM with bf16 output:
 * out[r, :] = bf16(a[r] b[e]^T) for the rows of expert e, a [max_rows, K]
 * e4m3 with [max_rows, K/128] fp32 scales, b [E, N, K] with [E, N/128,
 * K/128]; K, N multiples of 128 (the forward's GEMM2 is K = F, N = d).
 * Weight gradients (same section): dW2[e] = d_out^T act and dW13[e] =
 * dh^T x over expert e's rows, with both operands re-quantised 128 x 1 (one
 * fp32 scale, amax/448, per channel per 128-row block of the expert) because
 * the contraction runs over tokens:
 *   moe_wgrad_pad_offsets  pad[e] = sum of the 128-rounded row counts of the
 *                          experts before e (device, [E+1]).
 *   moe_wgrad_quant        one operand in the channel-major layout q [C, ld]
 *                          (expert e's rows at columns pad[e].., zero codes in
 *                          the padding), scales [C, ld/128] or, with
 *                          scales_kb_major, [ld/128, C]; ld is a host-known
 *                          bound of pad[E] (multiple of 128, e.g.
 *                          (ceil(A/128) + E) * 128).  src selects the operand
 *                          0: g * dy (d_out, C = d), 1: silu(g) * u from h
 *                          (act, C = F, silu as the forward's GEMM1 epilogue
 *                          forms it), 2: dh from d_act and h (C = 2F, as
 *                          moe_swiglu_backward forms it),
 *                          3: x (C = d); rows map to tokens by
 *                          sorted_to_slot / k.  C a multiple of 128; q and
 *                          the source buffers 16-byte aligned.
 *                          expert_offsets and pad are read as given (the
 *                          outputs of moe_dispatch and moe_wgrad_pad_offsets
 *                          for these rows): the source rows they name must
 *                          exist; no store leaves q [C, ld] or its scales.
 *   moe_wgrad_gemm         out[e] [M, N] fp32 = sum over e's blocks kb of
 *                          (a_sT[kb, m] * b_sT[kb, n]) * P_kb(m, n) (the
 *                          forward's per-block promotion), a [M, ld], b [N,
 *                          ld], both scale arrays kb-major [ld/128, *] (as
 *                          moe_wgrad_quant writes them with scales_kb_major);
 *                          M, N multiples of 128, E * M < 2^31; experts
 *                          without rows get zeros; pad entries outside
 *                          [0, ld] or not multiples of 128 run no tile and
 *                          set MOE_DEV_ROWS.
 * The router's own gradients, from the d_gates that moe_combine_backward
 * returns, are moe_router_backward's.
 * Errors: NULL, SHAPE, ALIGN, CUDA (WORKSPACE for the _train call).
 * ---------------------------------------------------------------------- */
moe_status moe_grouped_ffn_fp8_train(const uint8_t *xq_sorted, const float *xs_sorted,
                                     const int32_t *expert_offsets, int64_t max_rows, int E, int d, int F,
                                     const uint8_t *w13_q, const float *w13_s, const uint8_t *w2_q,
                                     const float *w2_s, uint16_t *out_sorted, float *h_out, void *workspace,
                                     size_t workspace_bytes, int32_t *dev_status, void *stream);
moe_status moe_grouped_gemm_fp8(const uint8_t *a_q, const float *a_s, const int32_t *expert_offsets,
                                int64_t max_rows, int E, int K, int N, const uint8_t *b_q, const float *b_s,
                                uint16_t *out, int32_t *dev_status, void *stream);
moe_status fp8_weight_transpose(const uint8_t *q, const float *s, int64_t E, int64_t R, int64_t C, uint8_t *qt,
                                float *st, void *stream);
moe_status moe_combine_backward(const uint16_t *dy, const float *gates, const uint16_t *out_sorted,
                                const int32_t *slot_to_sorted, int T, int k, int d, int64_t A, uint8_t *d_out_q,
                                float *d_out_s, float *d_gates, int32_t *dev_status, void *stream);
moe_status moe_swiglu_backward(const uint16_t *d_act, const float *h, int64_t rows, int F, uint8_t *dh_q,
                               float *dh_s, void *stream);
moe_status moe_dispatch_backward(const uint16_t *dx_sorted, const int32_t *slot_to_sorted, int T, int k, int d,
                                 uint16_t *dx, void *stream);
moe_status moe_wgrad_pad_offsets(const int32_t *expert_offsets, int E, int32_t *pad, void *stream);
moe_status moe_wgrad_quant(int src, const uint16_t *dy, const float *gates, const uint16_t *x,
                           const int32_t *sorted_to_slot, int k, const float *h, const uint16_t *d_act, int F,
                           const int32_t *expert_offsets, const int32_t *pad, int E, int64_t C, int64_t ld,
                           int scales_kb_major, uint8_t *q, float *scales, void *stream);
moe_status moe_wgrad_gemm(const uint8_t *a_q, const float *a_sT, const uint8_t *b_q, const float *b_sT,
                          const int32_t *pad, int E, int M, int N, int64_t ld, float *out, int32_t *dev_status,
                          void *stream);

/* ------------------------------------------------------------------------
 * moe_combine -- gate-weighted sum back to token order ("Expert
 * parallelism": combine).
 *
 *   y[t,c] = bf16( sum_{j=0}^{k-1} gates[t,j] * out_sorted[slot_to_sorted[t*k+j], c] ),
 *   one binary32 fused multiply-add chain over j in slot order from +0,
 *   rounded to nearest even; slots with slot_to_sorted = -1 are skipped.
 *   slot_to_sorted should come from moe_dispatch unchanged; an entry outside
 *   [0, T*k) is skipped like -1, so no read leaves out_sorted's T*k rows.
 * out_sorted [*, d] bf16, y [T, d] bf16; d a multiple of 8; out_sorted and y
 * 16-byte aligned.  Errors: NULL, SHAPE, ALIGN.
 * ---------------------------------------------------------------------- */
moe_status moe_combine(const uint16_t *out_sorted, const int32_t *slot_to_sorted, const float *gates,
                       int T, int k, int d, uint16_t *y, void *stream);

/* ------------------------------------------------------------------------
 * moe_combine_slots -- moe_combine over expert outputs stored in slot order
 * (as moe_grouped_ffn_fp8_gathered writes them).
 *
 *   y[t,c] = bf16( sum_j gates[t,j] * out_slots[t*k+j, c] ) over the slots
 *   with slot_to_sorted[t*k+j] >= 0, the same fma chain in slot order as
 *   moe_combine (so both give the same bits for the same expert outputs).
 * out_slots [T*k, d] bf16; other arguments as moe_combine.
 * Errors: NULL, SHAPE, ALIGN.
 * ---------------------------------------------------------------------- */
moe_status moe_combine_slots(const uint16_t *out_slots, const int32_t *slot_to_sorted, const float *gates,
                             int T, int k, int d, uint16_t *y, void *stream);

/* ------------------------------------------------------------------------
 * moe_debug_bounded_wait -- exercises the bounded device wait that every
 * pipelined kernel uses: one CTA waits on an mbarrier that nothing arrives
 * at, for at most timeout_ns, then sets MOE_DEV_TIMEOUT in *dev_status and
 * returns.  For fault-handling tests; no counterpart in the method.
 * timeout_ns in [0, 10^10] (ten seconds at most).
 * Errors: NULL (dev_status), SHAPE (timeout_ns out of range), CUDA.
 * ---------------------------------------------------------------------- */
moe_status moe_debug_bounded_wait(int64_t timeout_ns, int32_t *dev_status, void *stream);

/* Number of SMs of the current CUDA device (the figure the persistent
 * kernels size their grids by); 1 if the device cannot be queried. */
int moe_device_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_R3_H */
