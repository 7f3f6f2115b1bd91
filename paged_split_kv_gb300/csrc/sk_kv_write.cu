// KV write: the standard-page writer of vLLM RFC 59111 ("NixlConnector:
// convert standard KV pages to ROCm AITER shuffled pages on the decode side",
// Background): per KV head, a token's K and V rows sit side by side in one
// page row, so token t with slot = slot_mapping[t] fills row slot % page of
// block slot / page with K[t][h] (elements [0, D)) and V[t][h] ([D, 2D)).
// A negative slot writes nothing; a slot past the last block writes nothing
// and sets SK_DEV_BAD_BLOCK.  e4m3 pages receive each value divided by its
// tensor's scale (IEEE binary32 division; a multiply by the exact reciprocal
// when the scale is a power of two, which rounds identically) and converted to
// the nearest e4m3fn code, ties to even, saturating at +-448.
//
// Pure data movement, bound by HBM: one warp per (token, head) row.  Lanes
// 0-15 read K and lanes 16-31 read V, 16 bytes each (read-once loads that do
// not allocate in L1), and the warp writes the page row as one contiguous
// 512-byte store (256 bytes of codes for e4m3); lane l's bytes land at byte
// 16 l (bf16) or 8 l (e4m3) of the row either way.  Each warp takes four rows
// at a time, loads first, so about 2 KB per warp is in flight.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <cmath>

#include "sk_internal.cuh"

namespace sk {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerWarp = 4;

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Two bf16 values (one packed word) divided by `scale` -> two e4m3fn codes
// (low byte from the low half), nearest even, saturated.  With RECIP the
// caller guarantees scale = 2^k and inv = 2^-k exactly, so x * inv is the
// correctly rounded x / scale (both round the same real number).
template <bool RECIP>
__device__ __forceinline__ uint32_t quant2(uint32_t w, float scale, float inv)
{
    const float a = __uint_as_float(w << 16), b = __uint_as_float(w & 0xFFFF0000u);
    const float lo = RECIP ? a * inv : __fdiv_rn(a, scale);
    const float hi = RECIP ? b * inv : __fdiv_rn(b, scale);
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <bool FP8, bool RECIP>
__global__ void __launch_bounds__(kThreads)
kv_write_kernel(const uint16_t *__restrict__ key, const uint16_t *__restrict__ value,
                const int64_t *__restrict__ slot_mapping, long long rows, int H, long long num_slots,
                void *__restrict__ pages, float k_scale, float v_scale, int *status)
{
    wait_prior_grid();    // K, V and the slots may come from the kernels before this one
    const int lane = threadIdx.x & 31;
    const long long warp0 = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const long long nwarps = (long long)gridDim.x * (kThreads / 32);
    const bool is_v = lane >= 16;
    const uint16_t *src_base = (is_v ? value : key) + (lane & 15) * 8;
    const float sc = is_v ? v_scale : k_scale;
    const float inv = RECIP ? 1.f / sc : 0.f;     // exact for a power of two
    for (long long r0 = warp0 * kRowsPerWarp; r0 < rows; r0 += nwarps * kRowsPerWarp) {
        uint4 v[kRowsPerWarp];
        long long dst_row[kRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const long long r = r0 + i;
            dst_row[i] = -1;
            if (r < rows) {
                const long long t = r / H;
                const long long h = r - t * H;
                const long long slot = __ldg(slot_mapping + t);
                if (slot >= num_slots) {
                    if (lane == 0)
                        atomicOr(status, SK_DEV_BAD_BLOCK);
                } else if (slot >= 0) {
                    const long long blk = slot / kPage, off = slot - blk * kPage;
                    dst_row[i] = (blk * H + h) * kPage + off;
                    v[i] = ld_stream(src_base + r * kHeadDim);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            if (dst_row[i] < 0)
                continue;
            if constexpr (FP8) {
                uint2 q;
                q.x = quant2<RECIP>(v[i].x, sc, inv) | (quant2<RECIP>(v[i].y, sc, inv) << 16);
                q.y = quant2<RECIP>(v[i].z, sc, inv) | (quant2<RECIP>(v[i].w, sc, inv) << 16);
                *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(pages) + dst_row[i] * (2 * kHeadDim) + lane * 8) = q;
            } else {
                *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(pages) + dst_row[i] * (2 * kHeadDim) + lane * 8) = v[i];
            }
        }
    }
}

}  // namespace

cudaError_t launch_kv_write(const uint16_t *key, const uint16_t *value, const int64_t *slot_mapping,
                            int num_tokens, int num_kv_heads, long long num_blocks, void *pages,
                            int kv_dtype, float k_scale, float v_scale, int *status, int num_sms,
                            cudaStream_t stream)
{
    const long long rows = (long long)num_tokens * num_kv_heads;
    if (rows == 0)
        return cudaSuccess;
    const long long warps = (rows + kRowsPerWarp - 1) / kRowsPerWarp;
    long long blocks = (warps + kThreads / 32 - 1) / (kThreads / 32);
    const long long cap = (long long)(num_sms > 0 ? num_sms : 1) * 8;   // 8 CTAs of 256 per SM
    blocks = blocks < cap ? blocks : cap;
    const long long num_slots = num_blocks * kPage;
    // a power-of-two scale with a normal reciprocal: multiply instead of divide
    auto exact_recip = [](float sc) {
        int e = 0;
        const float m = frexpf(sc, &e);
        const float r = 1.f / sc;
        return m == 0.5f && r * sc == 1.f && std::isnormal(r) && std::isnormal(sc);
    };
    const dim3 grid((unsigned)blocks);
    auto kernel = kv_dtype != SK_KV_FP8_E4M3                     ? kv_write_kernel<false, false>
                  : (exact_recip(k_scale) && exact_recip(v_scale)) ? kv_write_kernel<true, true>
                                                                   : kv_write_kernel<true, false>;
    return launch_pdl(kernel, grid, dim3(kThreads), 0, stream, key, value, slot_mapping, rows, num_kv_heads, num_slots,
                      pages, k_scale, v_scale, status);
}

}  // namespace sk
