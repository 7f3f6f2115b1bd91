// Internal declarations shared by the libsk translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sk.h"

namespace sk {

constexpr int kTile = 64;        // tokens per plan tile
constexpr int kHeadDim = 128;
constexpr int kPage = 16;

// Everything the attention kernels need, resolved on the host.
struct AttnParams {
    const uint16_t *q;           // bf16 bits [NT, H_q, D]
    const void *kv;              // [NB, H_kv, 16, 2D] bf16 bits or e4m3 codes
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *cu_q;
    const int32_t *plan;         // NULL: fixed split
    float *part_o, *part_m, *part_l;
    int *status;                 // device status word
    int64_t num_blocks;
    int bt_stride;
    int bs, num_tokens, max_q_len;
    int H_q, H_kv, G;
    int seg_max;
    int fixed_nseg;              // segments per sequence when plan == NULL
    int num_items;               // work items the grid covers (per KV head)
    int row_blocks;              // CTAs per (work item, KV head), each taking up to 64 of its rows
    int causal;
    float score_scale_log2;      // sm_scale * k_scale * log2(e)
    float v_scale;               // applied to o (1 for bf16)
    long long wait_limit;        // clock cycles an abortable mbarrier wait may take (sk_set_wait_limit)
};

// A decoded work item.
struct WorkItem {
    int s, g;                    // sequence, segment
    int k0, k1;                  // key range [k0, k1) of the segment (k1 <= L_s; may be empty)
    int L, q_len, tok0;          // sequence length, query tokens, first query token
};

// Decodes work item `item` (SGLang PR 39172, Modifications: the prologue
// reads plan[1+i], exits on -1, tiles per segment come from plan[0]).
// Returns false when the CTA has nothing to do.
__device__ __forceinline__ bool decode_work_item(const AttnParams &p, int item, WorkItem &w)
{
    int T;
    if (p.plan != nullptr) {
        const int code = __ldg(p.plan + 1 + item);
        if (code < 0)
            return false;
        w.s = code >> 16;
        w.g = code & 0xFFFF;
        T = __ldg(p.plan) * kTile;
    } else {
        w.s = item / p.fixed_nseg;
        w.g = item - w.s * p.fixed_nseg;
        if (w.s >= p.bs)
            return false;
        const int L = __ldg(p.seq_lens + w.s);
        const int tiles = (L + kTile - 1) / kTile;
        int per = (tiles + p.fixed_nseg - 1) / p.fixed_nseg;
        per = per < 1 ? 1 : per;
        T = per * kTile;
    }
    if (w.s >= p.bs || w.g >= p.seg_max) {
        atomicOr(p.status, SK_DEV_BAD_SEQ);
        return false;
    }
    w.L = __ldg(p.seq_lens + w.s);
    w.tok0 = __ldg(p.cu_q + w.s);
    w.q_len = __ldg(p.cu_q + w.s + 1) - w.tok0;
    const long long k0 = (long long)w.g * T;
    long long k1 = k0 + T;
    if (k1 > w.L)
        k1 = w.L;
    w.k0 = (int)(k0 < w.L ? k0 : w.L);
    w.k1 = (int)(k1 > w.k0 ? k1 : w.k0);
    if (w.q_len < 0 || w.q_len > p.max_q_len || w.tok0 < 0 || w.tok0 + w.q_len > p.num_tokens ||
        w.L < 0 || (long long)w.L > (long long)p.bt_stride * kPage) {
        atomicOr(p.status, SK_DEV_BAD_SEQ);
        return false;
    }
    return true;
}

// Keys [0, n) that query token j (of q_len) of a sequence of length L sees.
__device__ __forceinline__ int visible_keys(int L, int q_len, int j, int causal)
{
    if (!causal)
        return L;
    int n = L - q_len + j + 1;
    n = n < L ? n : L;
    return n > 0 ? n : 0;
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// launch_pdl, so it may begin while the kernel before it on the stream is still
// finishing (its launch latency then overlaps that kernel's tail).  Each kernel
// calls wait_prior_grid() before it reads anything an earlier kernel may have
// written; the call waits until that kernel has completed and its writes are
// visible, and returns at once when there is no such kernel.
__device__ __forceinline__ void wait_prior_grid()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Address of the current device's status word (looked up once per device).
int device_status_word(int **out);
// Default limit of the attention kernel's abortable waits: about two seconds of SM clock.
constexpr long long kDefaultWaitLimit = 4000000000LL;
// The limit in force (sk_set_wait_limit).
long long wait_limit();
// Records `msg` as this thread's last error and returns `code`.
int set_error(int code, const char *msg);

// Host halves of sk_paged_decode_attn and sk_merge_segments, so that a composite call can check
// every argument before it launches anything.  prepare_attn validates and resolves the kernel
// parameters (*rp_out = 0: nothing to launch); launch_prepared_attn launches them; check_merge
// validates a merge call.  All return an sk_status.
int prepare_attn(const void *q, const void *kv_pages, int kv_dtype, float k_scale, float v_scale,
                 const int32_t *block_table, int block_table_stride, int num_blocks, int page_size,
                 const int32_t *seq_lens, const int32_t *cu_seqlens_q, const int32_t *plan,
                 int plan_capacity, int bs, int num_tokens, int max_q_len, int num_q_heads,
                 int num_kv_heads, int head_dim, float sm_scale, int causal, int num_sms, int seg_max,
                 float *part_o, float *part_m, float *part_l, AttnParams *params, int *rp_out);
int launch_prepared_attn(const AttnParams &p, int kv_dtype, int rp, void *stream);
int check_merge(const float *part_o, const float *part_m, const float *part_l, const int32_t *tok_nseg,
                int fixed_nseg, int num_tokens, int num_q_heads, int head_dim, int seg_max, const void *out);

// Launchers (each returns a cudaError_t from the launch).
cudaError_t launch_plan(const int32_t *seq_lens, const int32_t *cu_q, int bs, int num_tokens,
                        int budget, int seg_max, int32_t *plan, int plan_capacity,
                        int32_t *tok_nseg, int *status, cudaStream_t stream);
// Tensor-core kernel: attn_tc_rows() gives the row tile (16, 32, 64) it would
// use for a call, or 0 when it cannot take the call.
int attn_tc_rows(int kv_dtype, int rows_max, long long num_blocks, int H_kv);
constexpr int kMaxRowBlocks = 1024;   // rows per work item up to 1024 * 64
cudaError_t launch_attn_tc(const AttnParams &p, int kv_dtype, int rp, cudaStream_t stream);
cudaError_t launch_kv_write(const uint16_t *key, const uint16_t *value, const int64_t *slot_mapping,
                            int num_tokens, int num_kv_heads, long long num_blocks, void *pages,
                            int kv_dtype, float k_scale, float v_scale, int *status, int num_sms,
                            cudaStream_t stream);
cudaError_t launch_std_to_shuffled(const void *pages, int kv_dtype, const int32_t *ids, int num_ids,
                                   long long num_blocks, int num_kv_heads, void *k_out, void *v_out,
                                   int *status, int num_sms, cudaStream_t stream);
cudaError_t launch_merge(const float *part_o, const float *part_m, const float *part_l,
                         const int32_t *tok_nseg, int fixed_nseg, int num_tokens, int H_q,
                         int seg_max, uint16_t *out, float *lse, cudaStream_t stream);

}  // namespace sk
