// Plan kernel: the length-aware segment plan of SGLang PR 39172 ("[AMD]
// gfx950 assembly attention: length-aware split-KV for dynamic workload",
// Modifications, first item).
//
// One CTA does the whole batch (bs <= 32767), entirely on the device, so the
// call never reads anything back and can be captured in a CUDA graph.  The
// page's rule -- the smallest T with total segments <= B and per-sequence
// segments <= seg_max -- is monotone in T (both counts only fall as T grows),
// so T is found by binary search instead of trying every T.  The search runs
// between two bounds that follow from ceil(x) in [x, x + 1): with S tiles in
// n non-empty sequences, no T < S / B fits (the total is at least S / T), and
// every T >= S / (B - n) does (the total is below S / T + n).
//
// The CTA has one warp per 32 sequences (at most 1024 threads); tile counts
// sit in shared memory for batches up to kCacheSeqs, so a probe is one pass
// over them and one barrier (partial sums double-buffered by probe parity).
// A batch of at most 32 sequences is searched by its one warp 32 candidates
// at a time (each lane sums the batch for its own T), two or three rounds
// where bisection would take about log2 of the range.
#include <cuda_runtime.h>
#include <stdint.h>

#include "sk_internal.cuh"

namespace sk {
namespace {

constexpr int kPlanMaxThreads = 1024;
constexpr int kCacheSeqs = 8192;
constexpr uint32_t kFull = 0xffffffffu;

__device__ __forceinline__ long long tiles_of(int L)
{
    return L > 0 ? ((long long)L + kTile - 1) / kTile : 0;
}

__device__ __forceinline__ long long warp_sum(long long v)
{
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ uint32_t warp_sum32(uint32_t v)
{
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ long long warp_max(long long v)
{
    for (int o = 16; o > 0; o >>= 1) {
        const long long w = __shfl_xor_sync(kFull, v, o);
        v = w > v ? w : v;
    }
    return v;
}

__global__ void __launch_bounds__(kPlanMaxThreads, 1)
plan_kernel(const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ cu_q, int bs,
            int num_tokens, int budget, int seg_max, int32_t *__restrict__ plan, int plan_capacity,
            int32_t *__restrict__ tok_nseg, int *status)
{
    __shared__ int32_t tiles_s[kCacheSeqs];
    __shared__ long long part[2][32];
    __shared__ uint32_t part32[2][32];
    __shared__ long long part3[3][32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthr = blockDim.x, nwarps = nthr >> 5;
    const bool cached = bs <= kCacheSeqs;
    wait_prior_grid();    // the lengths may come from a kernel before this one
    // tile counts are below 2^26 (lengths are int32), so they and T fit in 32 bits
    auto tiles_at = [&](int s) -> uint32_t {
        return cached ? (uint32_t)tiles_s[s] : (uint32_t)tiles_of(__ldg(seq_lens + s));
    };

    // the query-token range of this thread's sequence, fetched with the lengths (one
    // sequence per thread whenever bs <= 1024)
    const bool one_seq = bs <= nthr;
    int cu_a = 0, cu_b = 0;
    if (one_seq && tid < bs) {
        cu_a = __ldg(cu_q + tid);
        cu_b = __ldg(cu_q + tid + 1);
    }
    // the ends of cu_seqlens_q for the coverage check at the end, loaded with everything else
    const int cu_first = __ldg(cu_q), cu_last = __ldg(cu_q + bs);

    // 1. tile counts; largest, number of non-empty sequences, total
    long long my_max = 0, my_nonempty = 0, my_sum = 0;
    for (int s = tid; s < bs; s += nthr) {
        const long long t = tiles_of(__ldg(seq_lens + s));
        if (cached)
            tiles_s[s] = (int32_t)t;              // < 2^26: lengths are int32
        my_max = t > my_max ? t : my_max;
        my_nonempty += t > 0;
        my_sum += t;
    }
    my_max = warp_max(my_max);
    my_nonempty = warp_sum(my_nonempty);
    my_sum = warp_sum(my_sum);
    if (lane == 0) {
        part3[0][warp] = my_max;
        part3[1][warp] = my_nonempty;
        part3[2][warp] = my_sum;
    }
    __syncthreads();
    long long max_tiles = 0, nonempty = 0, total_tiles = 0;
    for (int k = 0; k < nwarps; ++k) {
        max_tiles = part3[0][k] > max_tiles ? part3[0][k] : max_tiles;
        nonempty += part3[1][k];
        total_tiles += part3[2][k];
    }

    // 2. T: the smallest feasible t, or one segment per non-empty sequence
    long long T;
    const long long hi_all = max_tiles > 0 ? max_tiles : 1;
    if (nonempty > budget) {
        T = hi_all;
    } else {
        // t = hi_all is feasible (total = nonempty <= budget, per-sequence 1 <= seg_max)
        long long lo = (max_tiles + seg_max - 1) / seg_max;
        const long long by_total = budget > 0 ? (total_tiles + budget - 1) / budget : 0;
        lo = by_total > lo ? by_total : lo;
        lo = lo < 1 ? 1 : lo;
        long long hi = hi_all;
        if (budget > nonempty) {
            const long long fits = (total_tiles + (budget - nonempty) - 1) / (budget - nonempty);
            const long long h2 = fits > lo ? fits : lo;
            hi = h2 < hi ? h2 : hi;
        }
        if (lo > hi)
            lo = hi;
        // Every probe has mid >= S / B, so its total is below S / mid + bs <= B + bs < 2^32
        // (B < 2^31: plan_capacity > B is an int; bs < 2^15).
        // ceil(max / mid) <= seg_max is max <= seg_max * mid.
        if (nwarps == 1) {
            // One warp holds the whole batch (bs <= 32): each lane tests its own candidate,
            // lo + l * step with the last one at hi, so every round cuts the range 31-fold.
            // Feasibility is monotone, so the feasible lanes are a suffix and the first of
            // them bounds T from above, its left neighbour from below.
            const uint32_t my_t = tid < bs ? tiles_at(tid) : 0u;   // the sum is < 2^31 (bs <= 32, tiles < 2^26)
            while (lo < hi) {
                const long long step = (hi - lo + 30) / 31;
                const long long c = lo + step * lane < hi ? lo + step * lane : hi;
                const uint32_t c32 = (uint32_t)c;
                uint32_t sum = 0;
                for (int s = 0; s < bs; ++s)
                    sum += (__shfl_sync(kFull, my_t, s) + c32 - 1u) / c32;
                const bool ok = sum <= (uint32_t)budget && max_tiles <= (long long)seg_max * c;
                const int k = __ffs(__ballot_sync(kFull, ok)) - 1;   // lane 31 tests hi: k >= 0
                const long long c_k = lo + step * k < hi ? lo + step * k : hi;
                if (k > 0)
                    lo = lo + step * (k - 1) + 1;                  // lane k - 1 was below hi, infeasible
                hi = c_k;
                if (k == 0)
                    lo = hi;
            }
        }
        int parity = 0;
        while (lo < hi) {
            const long long mid = lo + (hi - lo) / 2;
            const uint32_t m32 = (uint32_t)mid;
            uint32_t sum = 0;
            for (int s = tid; s < bs; s += nthr)
                sum += (tiles_at(s) + m32 - 1u) / m32;
            sum = warp_sum32(sum);
            if (lane == 0)
                part32[parity][warp] = sum;
            __syncthreads();
            long long total = 0;
            for (int k = 0; k < nwarps; ++k)
                total += part32[parity][k];
            parity ^= 1;
            const bool ok = total <= budget && max_tiles <= (long long)seg_max * mid;
            if (ok)
                hi = mid;
            else
                lo = mid + 1;
        }
        T = lo;
    }

    // 3. exclusive prefix sum of nseg_s over a contiguous chunk of sequences per thread
    const int chunk = (bs + nthr - 1) / nthr;
    const int s_begin = tid * chunk;
    const int s_end = min(bs, s_begin + chunk);
    const uint32_t T32 = (uint32_t)T;
    long long mine = 0;
    for (int s = s_begin; s < s_end; ++s)
        mine += (tiles_at(s) + T32 - 1u) / T32;
    long long incl = mine;
    for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o)
            incl += v;
    }
    __syncthreads();                       // every probe has read its partials
    if (lane == 31)
        part[0][warp] = incl;
    __syncthreads();
    long long base = incl - mine, total_items = 0;
    for (int k = 0; k < nwarps; ++k) {
        const long long v = part[0][k];
        base += k < warp ? v : 0;
        total_items += v;
    }

    // 4. work list, -1 tail, per-token counts
    if (tid == 0)
        plan[0] = (int32_t)T;
    for (int s = s_begin; s < s_end; ++s) {
        const int n = (int)((tiles_at(s) + T32 - 1u) / T32);
        for (int g = 0; g < n; ++g) {
            const long long slot = 1 + base + g;
            if (slot < plan_capacity)
                plan[slot] = (int32_t)(((uint32_t)s << 16) | (uint32_t)g);
        }
        base += n;
        const int a = one_seq ? cu_a : __ldg(cu_q + s), b = one_seq ? cu_b : __ldg(cu_q + s + 1);
        if (a < 0 || b < a || b > num_tokens) {
            atomicOr(status, SK_DEV_BAD_SEQ);
            continue;
        }
        for (int t = a; t < b; ++t)
            tok_nseg[t] = n;
    }
    if (1 + total_items > plan_capacity && tid == 0)
        atomicOr(status, SK_DEV_BAD_SEQ);
    // cu_seqlens_q must cover [0, num_tokens) exactly: cu[0] == 0 and cu[bs] == num_tokens.  Tokens
    // outside [cu[0], cu[bs]) belong to no sequence; they get 0 segments (the merge writes 0 for
    // them), and the status word reports the inconsistency.
    {
        const int first = cu_first, last = cu_last;
        if (tid == 0 && (first != 0 || last != num_tokens))
            atomicOr(status, SK_DEV_BAD_SEQ);
        const int lo_end = min(max(first, 0), num_tokens), hi_begin = min(max(last, 0), num_tokens);
        for (int t = tid; t < lo_end; t += nthr)
            tok_nseg[t] = 0;
        for (int t = max(hi_begin, lo_end) + tid; t < num_tokens; t += nthr)
            tok_nseg[t] = 0;
    }
    for (long long k = 1 + total_items + tid; k < plan_capacity; k += nthr)
        plan[k] = -1;
}

}  // namespace

cudaError_t launch_plan(const int32_t *seq_lens, const int32_t *cu_q, int bs, int num_tokens,
                        int budget, int seg_max, int32_t *plan, int plan_capacity,
                        int32_t *tok_nseg, int *status, cudaStream_t stream)
{
    const int warps = (bs + 31) / 32;
    const int threads = 32 * (warps < 1 ? 1 : warps > kPlanMaxThreads / 32 ? kPlanMaxThreads / 32 : warps);
    return launch_pdl(plan_kernel, dim3(1), dim3(threads), 0, stream, seq_lens, cu_q, bs, num_tokens, budget,
                      seg_max, plan, plan_capacity, tok_nseg, status);
}

}  // namespace sk
