// Segment merge: the reduce of SGLang PR 39172 (Modifications, third item:
// it reads only its own token's segment count).
//
// One warp per (token, query head) row; each lane owns 4 of the 128
// dimensions, so every segment's o vector is one coalesced 512 B read.  The
// log-sum-exp combination:
//   M = max_g m_g,  Lambda = sum_g l_g e^(m_g - M),
//   out = sum_g o_g e^(m_g - M) / Lambda, lse = M + ln Lambda,
// over the segments with l > 0; no such segment gives out = 0, lse = -inf.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "sk_internal.cuh"

namespace sk {
namespace {

constexpr int kRowsPerCta = 8;

__global__ void __launch_bounds__(kRowsPerCta * 32)
merge_kernel(const float *__restrict__ part_o, const float *__restrict__ part_m,
             const float *__restrict__ part_l, const int32_t *__restrict__ tok_nseg,
             int fixed_nseg, int num_tokens, int H_q, int seg_max, uint16_t *__restrict__ out,
             float *__restrict__ lse)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kRowsPerCta + warp;
    if (row >= (long long)num_tokens * H_q)
        return;
    const int t = (int)(row / H_q), hq = (int)(row - (long long)t * H_q);
    int n = tok_nseg ? __ldg(tok_nseg + t) : fixed_nseg;
    n = n < 0 ? 0 : (n > seg_max ? seg_max : n);

    const long long base = (long long)t * seg_max * H_q + hq;   // slot of segment 0
    float M = -CUDART_INF_F;
    for (int g = lane; g < n; g += 32) {
        const long long k = base + (long long)g * H_q;
        if (__ldg(part_l + k) > 0.f)
            M = fmaxf(M, __ldg(part_m + k));
    }
    for (int o = 16; o > 0; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

    float Lam = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -CUDART_INF_F) {
        for (int g = 0; g < n; ++g) {
            const long long k = base + (long long)g * H_q;
            const float lg = __ldg(part_l + k);
            if (!(lg > 0.f))
                continue;
            const float f = expf(__ldg(part_m + k) - M);
            Lam = fmaf(lg, f, Lam);
            const float4 og = __ldg(reinterpret_cast<const float4 *>(part_o + k * kHeadDim) + lane);
            acc.x = fmaf(og.x, f, acc.x);
            acc.y = fmaf(og.y, f, acc.y);
            acc.z = fmaf(og.z, f, acc.z);
            acc.w = fmaf(og.w, f, acc.w);
        }
    }
    const float inv = Lam > 0.f ? 1.f / Lam : 0.f;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t *>(&lo);
    packed.y = *reinterpret_cast<const uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(out + row * kHeadDim)[lane] = packed;
    if (lse != nullptr && lane == 0)
        lse[row] = Lam > 0.f ? M + logf(Lam) : -CUDART_INF_F;
}

}  // namespace

cudaError_t launch_merge(const float *part_o, const float *part_m, const float *part_l,
                         const int32_t *tok_nseg, int fixed_nseg, int num_tokens, int H_q,
                         int seg_max, uint16_t *out, float *lse, cudaStream_t stream)
{
    const long long rows = (long long)num_tokens * H_q;
    if (rows == 0)
        return cudaSuccess;
    const unsigned grid = (unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta);
    merge_kernel<<<grid, kRowsPerCta * 32, 0, stream>>>(part_o, part_m, part_l, tok_nseg, fixed_nseg,
                                                        num_tokens, H_q, seg_max, out, lse);
    return cudaGetLastError();
}

}  // namespace sk
