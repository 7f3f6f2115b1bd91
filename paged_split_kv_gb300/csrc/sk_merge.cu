// Segment merge: the reduce of SGLang PR 39172 (Modifications, third item:
// it reads only its own token's segment count).
//
// For one (token, query head) row with n segments, over the segments with
// l > 0:  M = max_g m_g,  Lambda = sum_g l_g e^(m_g - M),
//         out = sum_g o_g e^(m_g - M) / Lambda   (bf16, nearest even),
//         lse = M + ln Lambda;  no contributing segment: out = 0, lse = -inf.
//
// WPR warps per row: one (four rows per CTA) for the plan's per-token counts,
// four (one row per CTA) when the fixed split gives every row 16 or more
// segments, as the bs == 1 bypass does.  Lanes first load the (m, l) of up to
// 64 segments into registers (lane i: segments i and i + 32), so M, the
// segment weights and Lambda come out of one load round; the weighted sum of
// the o vectors then runs over the warp's share of the segments, each lane
// owning 4 of the 128 dimensions (one coalesced 512-byte read per segment).
// The first 8 (one warp a row) or 16 (four) of a warp's o vectors are loaded
// with the (m, l), so up to 8 segments (64 with four warps a row) cost one
// round trip to L2; the rest follow in batches of the same size whose loads are
// all in flight before the first is used (an unrolled loop that left the
// compiler to interleave loads with the weight shuffles took 11.2 instead of
// 10.0 us per merge on a batch whose longest rows have 27 segments).  Sixteen
// vectors a warp cut that batch's merge to 9.3 us, but the extra registers cost
// the uniform batch 1.1 us.
// More than 64 segments take a strided path with the same arithmetic.  With
// WPR = 4 the partial sums meet in shared memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "sk_internal.cuh"

namespace sk {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kThreads = 128;

__device__ __forceinline__ float seg_weight(float m, float l, float M)
{
    return l > 0.f ? expf(m - M) : 0.f;
}

template <int WPR>
__global__ void __launch_bounds__(kThreads)
merge_kernel(const float *__restrict__ part_o, const float *__restrict__ part_m,
             const float *__restrict__ part_l, const int32_t *__restrict__ tok_nseg,
             int fixed_nseg, long long rows, int H_q, int seg_max, uint16_t *__restrict__ out,
             float *__restrict__ lse)
{
    constexpr int kRowsPerCta = (kThreads / 32) / WPR;
    // o vectors a warp loads together with (m, l): 8 (16 with four warps a row, all of a
    // warp's segments when the fixed split gives 64), so few segments cost one round trip
    constexpr int kPre = WPR > 1 ? 16 : 8;
    __shared__ float4 acc_s[kThreads / 32][32];
    wait_prior_grid();    // the partials come from the attention kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = warp % WPR;                       // this warp's share of the row's segments
    const long long row = (long long)blockIdx.x * kRowsPerCta + warp / WPR;
    const bool live = row < rows;
    const int t = live ? (int)(row / H_q) : 0;
    const int hq = live ? (int)(row - (long long)t * H_q) : 0;
    int n = live ? (tok_nseg ? __ldg(tok_nseg + t) : fixed_nseg) : 0;
    n = n < 0 ? 0 : (n > seg_max ? seg_max : n);
    const long long base = (long long)t * seg_max * H_q + hq;   // slot of segment 0; segments H_q apart

    float M = -CUDART_INF_F, lam = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto load_o = [&](int g) {
        return __ldg(reinterpret_cast<const float4 *>(part_o + (base + (long long)g * H_q) * kHeadDim) + lane);
    };
    auto fma4 = [&](const float4 og, float wg) {
        acc.x = fmaf(og.x, wg, acc.x);
        acc.y = fmaf(og.y, wg, acc.y);
        acc.z = fmaf(og.z, wg, acc.z);
        acc.w = fmaf(og.w, wg, acc.w);
    };
    auto add = [&](int g, float wg) { fma4(load_o(g), wg); };
    if (n <= 64) {
        // the first kPre of this warp's segments' o vectors are loaded with their (m, l),
        // so a row with few segments costs one round trip to L2
        float4 opre[kPre];
#pragma unroll
        for (int k = 0; k < kPre; ++k) {
            const int g = sub + k * WPR;
            opre[k] = g < n ? load_o(g) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float m0 = -CUDART_INF_F, l0 = 0.f, m1 = -CUDART_INF_F, l1 = 0.f;
        if (lane < n) {
            m0 = __ldg(part_m + base + (long long)lane * H_q);
            l0 = __ldg(part_l + base + (long long)lane * H_q);
        }
        if (lane + 32 < n) {
            m1 = __ldg(part_m + base + (long long)(lane + 32) * H_q);
            l1 = __ldg(part_l + base + (long long)(lane + 32) * H_q);
        }
        M = fmaxf(l0 > 0.f ? m0 : -CUDART_INF_F, l1 > 0.f ? m1 : -CUDART_INF_F);
        for (int o = 16; o > 0; o >>= 1)
            M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        if (M != -CUDART_INF_F) {
            const float w0 = seg_weight(m0, l0, M), w1 = seg_weight(m1, l1, M);
            lam = l0 * w0 + l1 * w1;
            for (int o = 16; o > 0; o >>= 1)
                lam += __shfl_xor_sync(kFull, lam, o);
#pragma unroll
            for (int k = 0; k < kPre; ++k) {
                const int g = sub + k * WPR;           // g < 64; a zero vector when g >= n
                fma4(opre[k], __shfl_sync(kFull, g < 32 ? w0 : w1, g & 31));
            }
            // the rest in batches whose loads are all issued before the first of them is used
            for (int g0 = sub + kPre * WPR; g0 < n; g0 += kPre * WPR) {
                float4 ob[kPre];
#pragma unroll
                for (int k = 0; k < kPre; ++k) {
                    const int g = g0 + k * WPR;
                    ob[k] = g < n ? load_o(g) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int k = 0; k < kPre; ++k) {
                    const int g = g0 + k * WPR;       // < 64; a zero vector when g >= n
                    fma4(ob[k], __shfl_sync(kFull, g < 32 ? w0 : w1, g & 31));
                }
            }
        }
    } else {
        for (int g = lane; g < n; g += 32) {
            const long long k = base + (long long)g * H_q;
            if (__ldg(part_l + k) > 0.f)
                M = fmaxf(M, __ldg(part_m + k));
        }
        for (int o = 16; o > 0; o >>= 1)
            M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        if (M != -CUDART_INF_F) {
            for (int c0 = 0; c0 < n; c0 += 32) {
                float wl = 0.f;
                if (c0 + lane < n) {
                    const long long k = base + (long long)(c0 + lane) * H_q;
                    const float lg = __ldg(part_l + k);
                    wl = seg_weight(__ldg(part_m + k), lg, M);
                    lam = fmaf(lg, wl, lam);
                }
                const int cn = min(32, n - c0);
#pragma unroll 8
                for (int i = sub; i < cn; i += WPR)
                    add(c0 + i, __shfl_sync(kFull, wl, i));
            }
            for (int o = 16; o > 0; o >>= 1)
                lam += __shfl_xor_sync(kFull, lam, o);
        }
    }

    if constexpr (WPR > 1) {
        acc_s[warp][lane] = acc;
        __syncthreads();
        if (sub != 0)
            return;
#pragma unroll
        for (int w = 1; w < WPR; ++w) {
            const float4 v = acc_s[warp + w][lane];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
    }
    if (!live)
        return;
    const float inv = lam > 0.f ? 1.f / lam : 0.f;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t *>(&lo);
    packed.y = *reinterpret_cast<const uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(out + row * kHeadDim)[lane] = packed;
    if (lse != nullptr && lane == 0)
        lse[row] = lam > 0.f ? M + logf(lam) : -CUDART_INF_F;
}

}  // namespace

cudaError_t launch_merge(const float *part_o, const float *part_m, const float *part_l,
                         const int32_t *tok_nseg, int fixed_nseg, int num_tokens, int H_q,
                         int seg_max, uint16_t *out, float *lse, cudaStream_t stream)
{
    const long long rows = (long long)num_tokens * H_q;
    if (rows == 0)
        return cudaSuccess;
    if (tok_nseg == nullptr && fixed_nseg >= 16) {
        if (rows > 0x7FFFFFFFLL)
            return cudaErrorInvalidValue;
        return launch_pdl(merge_kernel<4>, dim3((unsigned)rows), dim3(kThreads), 0, stream, part_o, part_m, part_l,
                          tok_nseg, fixed_nseg, rows, H_q, seg_max, out, lse);
    } else {
        const long long grid = (rows + kThreads / 32 - 1) / (kThreads / 32);
        if (grid > 0x7FFFFFFFLL)
            return cudaErrorInvalidValue;
        return launch_pdl(merge_kernel<1>, dim3((unsigned)grid), dim3(kThreads), 0, stream, part_o, part_m, part_l,
                          tok_nseg, fixed_nseg, rows, H_q, seg_max, out, lse);
    }
}

}  // namespace sk
