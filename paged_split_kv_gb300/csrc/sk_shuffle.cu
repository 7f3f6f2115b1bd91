// Standard -> shuffled page conversion: the per-block view/permute of vLLM RFC
// 59111 ("NixlConnector: convert standard KV pages to ROCm AITER shuffled pages
// on the decode side", Proposed Change, Convert).  With x = 16 / element size
// (8 for bf16, 16 for e4m3), for every listed block, head h, token row n and
// dimension d:
//   k_shuf[blk][h][d / x][n][d % x] = K[blk][h][n][d]
//   v_shuf[blk][h][n / x][d][n % x] = V[blk][h][n][d]
// An id outside [0, num_blocks) is skipped and sets SK_DEV_BAD_BLOCK.
//
// Pure data movement, bound by HBM.  One warp per (block, head): the page's 16
// token rows (8 KB bf16, 4 KB e4m3) come in as coalesced 16-byte loads into
// shared memory (rows padded by 16 bytes, so the column-wise reads below hit
// every bank once per eight lanes).  K leaves as a transpose of 16-byte units
// (each unit of x elements stays whole); V needs an element transpose, done
// with byte permutes on 32-bit words: bf16 pairs rows two by two, e4m3 takes
// 4 x 4 byte blocks.  Every global store is a 16-byte vector.
#include <cuda_runtime.h>
#include <stdint.h>

#include "sk_internal.cuh"

namespace sk {
namespace {

constexpr int kWarps = 4;

__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Word c of out: byte c of each of a, b, c, d (a 4 x 4 byte transpose).
__device__ __forceinline__ void transpose4x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t (&out)[4])
{
    const uint32_t ab_lo = __byte_perm(a, b, 0x5140), ab_hi = __byte_perm(a, b, 0x7362);
    const uint32_t cd_lo = __byte_perm(c, d, 0x5140), cd_hi = __byte_perm(c, d, 0x7362);
    out[0] = __byte_perm(ab_lo, cd_lo, 0x5410);
    out[1] = __byte_perm(ab_lo, cd_lo, 0x7632);
    out[2] = __byte_perm(ab_hi, cd_hi, 0x5410);
    out[3] = __byte_perm(ab_hi, cd_hi, 0x7632);
}

template <bool FP8>
__global__ void __launch_bounds__(32 * kWarps)
std_to_shuffled_kernel(const uint8_t *__restrict__ pages, const int32_t *__restrict__ ids, long long num_units,
                       int H, long long num_blocks, uint8_t *__restrict__ k_out, uint8_t *__restrict__ v_out,
                       int *status)
{
    constexpr int kRowBytes = FP8 ? 256 : 512;          // one token row: K | V
    constexpr int kRowS = kRowBytes + 16;               // padded row in shared memory
    constexpr int kHeadBytes = kPage * kRowBytes;       // one page of one head
    constexpr int kUnitsPerRow = kRowBytes / 16;
    constexpr int kKUnits = kHeadBytes / 32;            // 16-byte units of K (half the page)
    __shared__ __align__(16) uint8_t buf[kWarps][kPage * kRowS];
    wait_prior_grid();    // the pages may come from the kernels before this one
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *sb = buf[warp];
    for (long long u = (long long)blockIdx.x * kWarps + warp; u < num_units; u += (long long)gridDim.x * kWarps) {
        const long long i = u / H;
        const long long h = u - i * H;
        const long long blk = ids != nullptr ? (long long)__ldg(ids + i) : i;
        if (blk < 0 || blk >= num_blocks) {
            if (lane == 0)
                atomicOr(status, SK_DEV_BAD_BLOCK);
            continue;
        }
        const long long bh = blk * H + h;
        const uint8_t *src = pages + bh * kHeadBytes;
#pragma unroll
        for (int it = 0; it < kHeadBytes / 16 / 32; ++it) {
            const int q = it * 32 + lane;
            const uint4 val = ld_stream16(src + q * 16);
            *reinterpret_cast<uint4 *>(sb + (q / kUnitsPerRow) * kRowS + (q % kUnitsPerRow) * 16) = val;
        }
        __syncwarp();
        // K: output unit o = (d / x) * 16 + n holds row n's unit d / x
        uint8_t *kdst = k_out + bh * (kHeadBytes / 2);
#pragma unroll
        for (int it = 0; it < kKUnits / 32; ++it) {
            const int o = it * 32 + lane;
            *reinterpret_cast<uint4 *>(kdst + o * 16) =
                *reinterpret_cast<const uint4 *>(sb + (o % kPage) * kRowS + (o / kPage) * 16);
        }
        uint8_t *vdst = v_out + bh * (kHeadBytes / 2);
        if constexpr (!FP8) {
            // vector (ng, d) holds V[8 ng + j][d], j < 8; a lane takes the dimension pair (2p, 2p + 1)
#pragma unroll
            for (int ng = 0; ng < 2; ++ng) {
#pragma unroll
                for (int it = 0; it < 2; ++it) {
                    const int p = it * 32 + lane;
                    uint32_t w[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        w[j] = *reinterpret_cast<const uint32_t *>(sb + (8 * ng + j) * kRowS + 256 + p * 4);
                    uint4 a, b;     // dimension 2p (low halves), 2p + 1 (high halves)
                    a.x = __byte_perm(w[0], w[1], 0x5410);
                    a.y = __byte_perm(w[2], w[3], 0x5410);
                    a.z = __byte_perm(w[4], w[5], 0x5410);
                    a.w = __byte_perm(w[6], w[7], 0x5410);
                    b.x = __byte_perm(w[0], w[1], 0x7632);
                    b.y = __byte_perm(w[2], w[3], 0x7632);
                    b.z = __byte_perm(w[4], w[5], 0x7632);
                    b.w = __byte_perm(w[6], w[7], 0x7632);
                    uint4 *dst = reinterpret_cast<uint4 *>(vdst + (ng * kHeadDim + 2 * p) * 16);
                    dst[0] = a;
                    dst[1] = b;
                }
            }
        } else {
            // vector d holds V[j][d], j < 16; a lane takes dimensions 4 lane .. 4 lane + 3
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                w[j] = *reinterpret_cast<const uint32_t *>(sb + j * kRowS + kHeadDim + lane * 4);
            uint32_t o[4][4];       // o[g][c]: bytes of rows 4g..4g+3 for dimension 4 lane + c
#pragma unroll
            for (int g = 0; g < 4; ++g)
                transpose4x4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3], o[g]);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4 *>(vdst + (4 * lane + c) * 16) = make_uint4(o[0][c], o[1][c], o[2][c], o[3][c]);
        }
        __syncwarp();     // the buffer is refilled by the next unit
    }
}

}  // namespace

cudaError_t launch_std_to_shuffled(const void *pages, int kv_dtype, const int32_t *ids, int num_ids,
                                   long long num_blocks, int num_kv_heads, void *k_out, void *v_out,
                                   int *status, int num_sms, cudaStream_t stream)
{
    const long long units = (ids != nullptr ? (long long)num_ids : num_blocks) * num_kv_heads;
    if (units == 0)
        return cudaSuccess;
    long long blocks = (units + kWarps - 1) / kWarps;
    const long long cap = (long long)(num_sms > 0 ? num_sms : 1) * 16;
    blocks = blocks < cap ? blocks : cap;
    const auto *src = static_cast<const uint8_t *>(pages);
    auto *ko = static_cast<uint8_t *>(k_out);
    auto *vo = static_cast<uint8_t *>(v_out);
    auto kernel = kv_dtype == SK_KV_FP8_E4M3 ? std_to_shuffled_kernel<true> : std_to_shuffled_kernel<false>;
    return launch_pdl(kernel, dim3((unsigned)blocks), dim3(32 * kWarps), 0, stream, src, ids, units, num_kv_heads,
                      num_blocks, ko, vo, status);
}

}  // namespace sk
