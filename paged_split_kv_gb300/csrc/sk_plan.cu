// Plan kernel: the length-aware segment plan of SGLang PR 39172 ("[AMD]
// gfx950 assembly attention: length-aware split-KV for dynamic workload",
// Modifications, first item).
//
// One CTA of 1024 threads does the whole batch (bs <= 32767), entirely on the
// device, so the call never reads anything back and can be captured in a
// CUDA graph.  The page's rule -- the smallest T with total segments <= B and
// per-sequence segments <= seg_max -- is monotone in T (both counts only fall
// as T grows), so T is found by binary search over [1, max tiles] instead of
// trying every T; each probe is one block-wide sum.
#include <cuda_runtime.h>
#include <stdint.h>

#include "sk_internal.cuh"

namespace sk {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kWarps = kPlanThreads / 32;

__device__ long long block_sum(long long v, long long *scratch)
{
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0)
        scratch[warp] = v;
    __syncthreads();
    long long r = 0;
    if (warp == 0) {
        r = lane < kWarps ? scratch[lane] : 0;
        for (int o = 16; o > 0; o >>= 1)
            r += __shfl_xor_sync(0xffffffffu, r, o);
        if (lane == 0)
            scratch[kWarps] = r;
    }
    __syncthreads();
    return scratch[kWarps];
}

__device__ long long block_max(long long v, long long *scratch)
{
    for (int o = 16; o > 0; o >>= 1) {
        long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0)
        scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        long long r = lane < kWarps ? scratch[lane] : 0;
        for (int o = 16; o > 0; o >>= 1) {
            long long w = __shfl_xor_sync(0xffffffffu, r, o);
            r = w > r ? w : r;
        }
        if (lane == 0)
            scratch[kWarps] = r;
    }
    __syncthreads();
    return scratch[kWarps];
}

__device__ __forceinline__ long long tiles_of(int L)
{
    return L > 0 ? ((long long)L + kTile - 1) / kTile : 0;
}

__global__ void __launch_bounds__(kPlanThreads, 1)
plan_kernel(const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ cu_q, int bs,
            int num_tokens, int budget, int seg_max, int32_t *__restrict__ plan, int plan_capacity,
            int32_t *__restrict__ tok_nseg, int *status)
{
    __shared__ long long red[kWarps + 1];
    __shared__ long long scan[kPlanThreads];
    const int tid = threadIdx.x;

    // 1. largest tile count and number of non-empty sequences
    long long my_max = 0, my_nonempty = 0;
    for (int s = tid; s < bs; s += kPlanThreads) {
        const long long t = tiles_of(__ldg(seq_lens + s));
        my_max = t > my_max ? t : my_max;
        my_nonempty += t > 0;
    }
    const long long max_tiles = block_max(my_max, red);
    const long long nonempty = block_sum(my_nonempty, red);

    // 2. T: the smallest feasible t, or one segment per non-empty sequence
    long long T;
    const long long hi_all = max_tiles > 0 ? max_tiles : 1;
    if (nonempty > budget) {
        T = hi_all;
    } else {
        // t = hi_all is feasible (total = nonempty <= budget, per-sequence 1 <= seg_max).
        long long lo = 1, hi = hi_all;
        const long long per_seq_lo = (max_tiles + seg_max - 1) / seg_max;
        lo = per_seq_lo > lo ? per_seq_lo : lo;
        if (lo > hi)
            lo = hi;
        while (lo < hi) {
            const long long mid = lo + (hi - lo) / 2;
            long long part = 0;
            for (int s = tid; s < bs; s += kPlanThreads)
                part += (tiles_of(__ldg(seq_lens + s)) + mid - 1) / mid;
            const long long total = block_sum(part, red);
            const bool ok = total <= budget && (max_tiles + mid - 1) / mid <= seg_max;
            if (ok)
                hi = mid;
            else
                lo = mid + 1;
        }
        T = lo;
    }

    // 3. exclusive prefix sum of nseg_s over a contiguous chunk per thread
    const int chunk = (bs + kPlanThreads - 1) / kPlanThreads;
    const int s_begin = tid * chunk;
    const int s_end = min(bs, s_begin + chunk);
    long long mine = 0;
    for (int s = s_begin; s < s_end; ++s)
        mine += (tiles_of(__ldg(seq_lens + s)) + T - 1) / T;
    scan[tid] = mine;
    __syncthreads();
    for (int off = 1; off < kPlanThreads; off <<= 1) {
        const long long add = tid >= off ? scan[tid - off] : 0;
        __syncthreads();
        scan[tid] += add;
        __syncthreads();
    }
    long long base = scan[tid] - mine;
    const long long total_items = scan[kPlanThreads - 1];

    // 4. work list, -1 tail, per-token counts
    if (tid == 0)
        plan[0] = (int32_t)T;
    for (int s = s_begin; s < s_end; ++s) {
        const int n = (int)((tiles_of(__ldg(seq_lens + s)) + T - 1) / T);
        for (int g = 0; g < n; ++g) {
            const long long slot = 1 + base + g;
            if (slot < plan_capacity)
                plan[slot] = (int32_t)(((uint32_t)s << 16) | (uint32_t)g);
        }
        base += n;
        const int a = __ldg(cu_q + s), b = __ldg(cu_q + s + 1);
        if (a < 0 || b < a || b > num_tokens) {
            atomicOr(status, SK_DEV_BAD_SEQ);
            continue;
        }
        for (int t = a; t < b; ++t)
            tok_nseg[t] = n;
    }
    if (1 + total_items > plan_capacity && tid == 0)
        atomicOr(status, SK_DEV_BAD_SEQ);
    for (long long k = 1 + total_items + tid; k < plan_capacity; k += kPlanThreads)
        plan[k] = -1;
}

}  // namespace

cudaError_t launch_plan(const int32_t *seq_lens, const int32_t *cu_q, int bs, int num_tokens,
                        int budget, int seg_max, int32_t *plan, int plan_capacity,
                        int32_t *tok_nseg, int *status, cudaStream_t stream)
{
    plan_kernel<<<1, kPlanThreads, 0, stream>>>(seq_lens, cu_q, bs, num_tokens, budget, seg_max,
                                                plan, plan_capacity, tok_nseg, status);
    return cudaGetLastError();
}

}  // namespace sk
