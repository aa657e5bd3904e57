// payload.cu -- the routed-experts payload at one byte per id.
//
// Router replay ("RL at 1T Scale: prime-rl Performance Deep Dive", section
// "Router replay") moves the captured [num_layers, top_k, seq_len] id tensor
// from inference to the trainer as an opaque payload whose size is the
// problem the section describes.  With E <= 256 every valid id fits one
// byte, so the payload shrinks 4x against int32.  Both directions are
// streaming copies: each thread moves 16 ids per step (four 16-byte loads
// and one 16-byte store when packing, the reverse when unpacking) on a grid
// of a few CTAs per SM, with a scalar path for a ragged tail or unaligned
// buffers.  Out-of-range ids are stored as 0xFF and flagged in the caller's
// device status word.
#include "common.cuh"

namespace moe {
namespace payload {

constexpr int V = 16;        // ids per thread step
constexpr int THREADS = 256;

__device__ __forceinline__ uint32_t id_byte(int32_t v, int E, bool &bad)
{
    const bool ok = v >= 0 && v < E;
    bad |= !ok;
    return ok ? (uint32_t)v : 0xFFu;
}

__global__ void __launch_bounds__(THREADS) pack_u8_kernel(const int32_t *__restrict__ ids, int64_t n, int E,
                                                          uint8_t *__restrict__ out, int32_t *dev_status,
                                                          bool vec)
{
    const int64_t steps = (n + V - 1) / V;
    bool bad = false;
    for (int64_t c = blockIdx.x * (int64_t)THREADS + threadIdx.x; c < steps; c += (int64_t)gridDim.x * THREADS) {
        const int64_t i0 = c * V;
        if (vec && i0 + V <= n) {
            const int4 *src = reinterpret_cast<const int4 *>(ids + i0);
            int4 v[4];
#pragma unroll
            for (int q = 0; q < 4; q++) v[q] = __ldcs(src + q);
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; q++)
                w[q] = id_byte(v[q].x, E, bad) | (id_byte(v[q].y, E, bad) << 8) |
                       (id_byte(v[q].z, E, bad) << 16) | (id_byte(v[q].w, E, bad) << 24);
            __stcs(reinterpret_cast<uint4 *>(out + i0), make_uint4(w[0], w[1], w[2], w[3]));
        } else {
            const int64_t i1 = i0 + V < n ? i0 + V : n;
            for (int64_t i = i0; i < i1; i++) out[i] = (uint8_t)id_byte(ids[i], E, bad);
        }
    }
    if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) dev_flag(dev_status, MOE_DEV_BAD_IDS);
}

__global__ void __launch_bounds__(THREADS) unpack_u8_kernel(const uint8_t *__restrict__ in, int64_t n,
                                                            int32_t *__restrict__ out, bool vec)
{
    const int64_t steps = (n + V - 1) / V;
    for (int64_t c = blockIdx.x * (int64_t)THREADS + threadIdx.x; c < steps; c += (int64_t)gridDim.x * THREADS) {
        const int64_t i0 = c * V;
        if (vec && i0 + V <= n) {
            const uint4 b = __ldcs(reinterpret_cast<const uint4 *>(in + i0));
            const uint32_t w[4] = {b.x, b.y, b.z, b.w};
            int4 *dst = reinterpret_cast<int4 *>(out + i0);
#pragma unroll
            for (int q = 0; q < 4; q++)
                __stcs(dst + q, make_int4((int)(w[q] & 0xFF), (int)((w[q] >> 8) & 0xFF), (int)((w[q] >> 16) & 0xFF),
                                          (int)(w[q] >> 24)));
        } else {
            const int64_t i1 = i0 + V < n ? i0 + V : n;
            for (int64_t i = i0; i < i1; i++) out[i] = (int32_t)in[i];
        }
    }
}

static unsigned grid_for(int64_t n)
{
    const int64_t steps = (n + V - 1) / V;
    const int64_t want = (steps + THREADS - 1) / THREADS;
    const int64_t cap = (int64_t)sm_count() * 8;
    return (unsigned)(want < cap ? want : cap);
}

} // namespace payload
} // namespace moe

using namespace moe;
using namespace moe::payload;

MOE_API moe_status moe_payload_pack_u8(const int32_t *ids, int64_t n, int E, uint8_t *out, int32_t *dev_status,
                                       void *stream)
{
    if (n < 0 || E < 1) return MOE_ERR_SHAPE;
    if (E > 256) return MOE_ERR_UNSUPPORTED;
    if (n == 0) return MOE_OK;
    if (!ids || !out || !dev_status) return MOE_ERR_NULL;
    const bool vec = aligned16(ids) && aligned16(out);
    pack_u8_kernel<<<grid_for(n), THREADS, 0, as_stream(stream)>>>(ids, n, E, out, dev_status, vec);
    return launch_status();
}

MOE_API moe_status moe_payload_unpack_u8(const uint8_t *in, int64_t n, int32_t *out, void *stream)
{
    if (n < 0) return MOE_ERR_SHAPE;
    if (n == 0) return MOE_OK;
    if (!in || !out) return MOE_ERR_NULL;
    const bool vec = aligned16(in) && aligned16(out);
    unpack_u8_kernel<<<grid_for(n), THREADS, 0, as_stream(stream)>>>(in, n, out, vec);
    return launch_status();
}
