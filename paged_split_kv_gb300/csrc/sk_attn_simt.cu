// Split-KV paged attention on CUDA cores.
//
// One CTA per (sequence, segment, KV head) work item (SGLang PR 39172,
// Modifications, second item).  This kernel serves work items with few query
// rows (decode with a small GQA group), where the arithmetic per KV byte is a
// handful of FMAs and the tensor cores buy nothing; it also accepts any row
// count by walking the rows in chunks of kRows.
//
// Work split inside the CTA: 4 warps take pages round-robin; inside a warp
// each half-warp owns one token and each lane 8 of the 128 dimensions, so a
// token row (K or V, 256 B bf16 / 128 B fp8) is read as one coalesced 16 B (or
// 8 B) access per lane straight from the page in HBM.  Scores are reduced
// across the 16 lanes of a half-warp with shuffles; the online softmax runs in
// the log2 domain, one max update per page.  At the end the two half-warps and
// the four warps are merged through shared memory and the segment partial
// (m, l, o) of every query row is written.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "sk_internal.cuh"

namespace sk {
namespace {

constexpr int kWarpsPerCta = 4;
constexpr int kThreads = kWarpsPerCta * 32;
constexpr int kRows = 4;            // query rows per pass
constexpr int kSteps = kPage / 2;   // half-warp token pairs per page

__device__ __forceinline__ void bf16x8_to_float(const uint4 &u, float *f)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void e4m3x8_to_float(const uint2 &u, float *f)
{
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[i] >> (16 * k)) & 0xFFFF);
            const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
            const float2 ff = __half22float2(*reinterpret_cast<const __half2 *>(&h));
            f[4 * i + 2 * k] = ff.x;
            f[4 * i + 2 * k + 1] = ff.y;
        }
    }
}

template <int KV_FP8>
struct RowLoad;

template <>
struct RowLoad<0> {   // bf16: 256 elements * 2 B per token row
    using Vec = uint4;
    static __device__ __forceinline__ Vec load(const void *base, long long elem)
    {
        return __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + elem));
    }
    static __device__ __forceinline__ void cvt(const Vec &v, float *f) { bf16x8_to_float(v, f); }
};

template <>
struct RowLoad<1> {   // e4m3: 256 elements * 1 B per token row
    using Vec = uint2;
    static __device__ __forceinline__ Vec load(const void *base, long long elem)
    {
        return __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint8_t *>(base) + elem));
    }
    static __device__ __forceinline__ void cvt(const Vec &v, float *f) { e4m3x8_to_float(v, f); }
};

template <int KV_FP8>
__global__ void __launch_bounds__(kThreads)
attn_simt_kernel(const AttnParams p)
{
    using LD = RowLoad<KV_FP8>;
    __shared__ float sm_m[kWarpsPerCta][kRows];
    __shared__ float sm_l[kWarpsPerCta][kRows];
    __shared__ float sm_o[kWarpsPerCta][kRows][kHeadDim];

    const int item = blockIdx.x / p.H_kv;
    const int h = blockIdx.x - item * p.H_kv;
    WorkItem w;
    if (item >= p.num_items || !decode_work_item(p, item, w))
        return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane >> 4, hl = lane & 15;
    const int R = p.G * w.q_len;
    const long long head_stride = (long long)kPage * 2 * kHeadDim;   // elements per page-head
    const int32_t *bt_row = p.block_table + (long long)w.s * p.bt_stride;

    for (int r0 = 0; r0 < R; r0 += kRows) {
        float qf[kRows][8];
        int vis_end[kRows];
        int chunk_end = w.k0;
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
            const int r = r0 + rr;
            if (r < R) {
                const int j = r / p.G, i = r - j * p.G;
                const uint16_t *qp = p.q + ((long long)(w.tok0 + j) * p.H_q + h * p.G + i) * kHeadDim + hl * 8;
                bf16x8_to_float(__ldg(reinterpret_cast<const uint4 *>(qp)), qf[rr]);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    qf[rr][e] *= p.score_scale_log2;
                const int n = visible_keys(w.L, w.q_len, j, p.causal);
                vis_end[rr] = min(w.k1, n);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    qf[rr][e] = 0.f;
                vis_end[rr] = w.k0;
            }
            chunk_end = max(chunk_end, vis_end[rr]);
        }

        float m[kRows], l[kRows], o[kRows][8];
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
            m[rr] = -CUDART_INF_F;
            l[rr] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                o[rr][e] = 0.f;
        }

        for (int pg = w.k0 / kPage + warp; pg * kPage < chunk_end; pg += kWarpsPerCta) {
            const int blk = __ldg(bt_row + pg);
            if (blk < 0 || blk >= p.num_blocks) {
                if (lane == 0)
                    atomicOr(p.status, SK_DEV_BAD_BLOCK);
                continue;
            }
            const long long base = ((long long)blk * p.H_kv + h) * head_stride;

            typename LD::Vec kv_raw[kSteps];
#pragma unroll
            for (int st = 0; st < kSteps; ++st)
                kv_raw[st] = LD::load(p.kv, base + (long long)(2 * st + half) * (2 * kHeadDim) + hl * 8);

            float sc[kSteps][kRows];
#pragma unroll
            for (int st = 0; st < kSteps; ++st) {
                float kf[8];
                LD::cvt(kv_raw[st], kf);
                const int tok = pg * kPage + 2 * st + half;
#pragma unroll
                for (int rr = 0; rr < kRows; ++rr) {
                    float d = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        d = fmaf(qf[rr][e], kf[e], d);
                    d += __shfl_xor_sync(0xffffffffu, d, 8);
                    d += __shfl_xor_sync(0xffffffffu, d, 4);
                    d += __shfl_xor_sync(0xffffffffu, d, 2);
                    d += __shfl_xor_sync(0xffffffffu, d, 1);
                    sc[st][rr] = (tok >= w.k0 && tok < vis_end[rr]) ? d : -CUDART_INF_F;
                }
            }
            // V rows of the page (issued before the softmax math to overlap latency)
#pragma unroll
            for (int st = 0; st < kSteps; ++st)
                kv_raw[st] = LD::load(p.kv, base + (long long)(2 * st + half) * (2 * kHeadDim) + kHeadDim + hl * 8);

#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) {
                float pm = sc[0][rr];
#pragma unroll
                for (int st = 1; st < kSteps; ++st)
                    pm = fmaxf(pm, sc[st][rr]);
                pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
                const float m_new = fmaxf(m[rr], pm);
                if (m_new != -CUDART_INF_F && m_new != m[rr]) {
                    const float alpha = exp2f(m[rr] - m_new);   // m = -inf -> 0
                    l[rr] *= alpha;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        o[rr][e] *= alpha;
                    m[rr] = m_new;
                }
            }
#pragma unroll
            for (int st = 0; st < kSteps; ++st) {
                float vf[8];
                LD::cvt(kv_raw[st], vf);
#pragma unroll
                for (int rr = 0; rr < kRows; ++rr) {
                    if (sc[st][rr] != -CUDART_INF_F) {
                        const float pw = exp2f(sc[st][rr] - m[rr]);
                        l[rr] += pw;
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            o[rr][e] = fmaf(pw, vf[e], o[rr][e]);
                    }
                }
            }
        }

        // merge the two half-warps (same m), then the warps through shared memory
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
            l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 16);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                o[rr][e] += __shfl_xor_sync(0xffffffffu, o[rr][e], 16);
            if (lane == 0) {
                sm_m[warp][rr] = m[rr];
                sm_l[warp][rr] = l[rr];
            }
            if (half == 0) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    sm_o[warp][rr][hl * 8 + e] = o[rr][e];
            }
        }
        __syncthreads();
        // thread -> dimension d; loop over the chunk's rows
        const int d = threadIdx.x;
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
            const int r = r0 + rr;
            if (r >= R)
                break;
            float M = -CUDART_INF_F;
#pragma unroll
            for (int wi = 0; wi < kWarpsPerCta; ++wi)
                M = fmaxf(M, sm_m[wi][rr]);
            float Lsum = 0.f, O = 0.f;
            if (M != -CUDART_INF_F) {
#pragma unroll
                for (int wi = 0; wi < kWarpsPerCta; ++wi) {
                    const float mw = sm_m[wi][rr];
                    if (mw != -CUDART_INF_F) {
                        const float f = exp2f(mw - M);
                        Lsum = fmaf(sm_l[wi][rr], f, Lsum);
                        O = fmaf(sm_o[wi][rr][d], f, O);
                    }
                }
            }
            const int j = r / p.G, i = r - j * p.G;
            const long long slot = ((long long)(w.tok0 + j) * p.seg_max + w.g) * p.H_q + h * p.G + i;
            p.part_o[slot * kHeadDim + d] = O * p.v_scale;
            if (d == 0) {
                p.part_m[slot] = M == -CUDART_INF_F ? -CUDART_INF_F : M * 0.69314718055994531f;
                p.part_l[slot] = Lsum;
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_attn_simt(const AttnParams &p, int kv_dtype, cudaStream_t stream)
{
    const dim3 grid((unsigned)p.num_items * (unsigned)p.H_kv);
    if (kv_dtype == SK_KV_FP8_E4M3)
        attn_simt_kernel<1><<<grid, kThreads, 0, stream>>>(p);
    else
        attn_simt_kernel<0><<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sk
