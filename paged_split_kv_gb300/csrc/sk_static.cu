// sk_paged_decode_attention_static: the whole attention call (plan,
// split-KV attention, merge) for callers that cannot allocate device memory.
//
// Who needs it: a host that owns every byte of device memory through its own
// allocator and does not let plug-in libraries call cudaMalloc (an inference
// engine that carves its memory pool at start-up), and plain C callers that
// have no caching allocator and cannot afford cudaMalloc/cudaFree (which may
// synchronise the device) inside a serving step.  They pass only inputs and
// outputs; the scratch the method needs between its kernels -- the plan, the
// per-token segment counts and the segment partials -- lives in one
// file-scope device array of fixed size.
//
// The array is kStaticScratchBytes (32 MiB) on every GPU that loads the
// library, held until the process exits.  Every call shares it: two calls
// whose kernels overlap on the GPU (different streams, or different host
// threads on the same device) race on it and must be serialised by the
// caller.  The array keeps the previous call's contents; nothing in it needs
// to start at zero, because the plan kernel writes the whole plan and every
// per-token count, the attention kernel writes every partial the merge later
// reads, and the merge reads only those.
//
// The first call on a device looks up the array's device address with
// cudaGetSymbolAddress (once per device, with that device current); make that
// first call before any stream capture.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "sk.h"
#include "sk_internal.cuh"

namespace sk {
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;
constexpr int kMaxStaticDevices = 64;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

unsigned char *g_scratch_addr[kMaxStaticDevices];
std::mutex g_scratch_mutex;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

const char *const kCapacityMsg =
    "sk_paged_decode_attention_static: the call needs more scratch than the 32 MiB static array "
    "(num_tokens * seg_max * num_q_heads * (head_dim + 2) * 4 bytes plus the plan); lower seg_max "
    "or split the batch";

// Device address of g_static_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, never a device pointer.
int scratch_address(unsigned char **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return set_error(SK_ERR_CUDA, "sk_paged_decode_attention_static: cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxStaticDevices)
        return set_error(SK_ERR_UNSUPPORTED, "sk_paged_decode_attention_static: device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || p == nullptr)
            return set_error(SK_ERR_CUDA, "sk_paged_decode_attention_static: cudaGetSymbolAddress failed");
        g_scratch_addr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_scratch_addr[dev];
    return SK_OK;
}

}  // namespace
}  // namespace sk

using namespace sk;

extern "C" size_t sk_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" int sk_paged_decode_attention_static(
    const void *q, const void *kv_pages, int kv_dtype, float k_scale, float v_scale,
    const int32_t *block_table, int block_table_stride, int num_blocks, int page_size,
    const int32_t *seq_lens, const int32_t *cu_seqlens_q, int use_plan, int bs, int num_tokens,
    int max_q_len, int num_q_heads, int num_kv_heads, int head_dim, float sm_scale, int causal,
    int num_sms, int seg_max, void *out, float *lse, void *stream)
{
    if (out == nullptr)
        return set_error(SK_ERR_INVALID, "sk_paged_decode_attention_static: null out");
    if (bs < 1 || bs > 32767 || num_tokens < 0 || num_q_heads < 1 || num_kv_heads < 1 ||
        num_sms < 1 || seg_max < 1 || seg_max > 0xFFFF || head_dim != kHeadDim)
        return set_error(SK_ERR_INVALID, "sk_paged_decode_attention_static: bad sizes");

    // scratch layout: plan | tok_nseg | part_m | part_l | part_o, each 256-byte aligned
    const int capacity = sk_plan_capacity(bs, num_kv_heads, num_sms);
    if (capacity < 0)
        return capacity;
    // rows = num_tokens * seg_max * num_q_heads, each (head_dim + 2) * 4 bytes of partials; the
    // bound is checked by division first, so none of the products below can wrap
    const size_t per_row = (size_t)(head_dim + 2) * 4;
    const size_t heads_segs = (size_t)seg_max * (size_t)num_q_heads;    // < 2^47
    if (num_tokens > 0 && heads_segs > kStaticScratchBytes / per_row / (size_t)num_tokens)
        return set_error(SK_ERR_CAPACITY, kCapacityMsg);
    const size_t rows = (size_t)num_tokens * heads_segs;
    const size_t off_plan = 0;
    const size_t off_tok = align256(off_plan + (use_plan ? (size_t)capacity * 4 : 0));
    const size_t off_m = align256(off_tok + (use_plan ? (size_t)num_tokens * 4 : 0));
    const size_t off_l = align256(off_m + rows * 4);
    const size_t off_o = align256(off_l + rows * 4);
    const size_t need = off_o + rows * (size_t)head_dim * 4;
    if (need > kStaticScratchBytes)
        return set_error(SK_ERR_CAPACITY, kCapacityMsg);

    unsigned char *base = nullptr;
    int rc = scratch_address(&base);
    if (rc != SK_OK)
        return rc;
    int32_t *plan = use_plan ? reinterpret_cast<int32_t *>(base + off_plan) : nullptr;
    int32_t *tok = use_plan ? reinterpret_cast<int32_t *>(base + off_tok) : nullptr;
    float *part_m = reinterpret_cast<float *>(base + off_m);
    float *part_l = reinterpret_cast<float *>(base + off_l);
    float *part_o = reinterpret_cast<float *>(base + off_o);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // every argument is checked before the first launch
    if (use_plan && (seq_lens == nullptr || cu_seqlens_q == nullptr))
        return set_error(SK_ERR_INVALID, "sk_paged_decode_attention_static: null seq_lens or cu_seqlens_q");
    AttnParams params;
    int rp = 0;
    rc = prepare_attn(q, kv_pages, kv_dtype, k_scale, v_scale, block_table, block_table_stride, num_blocks,
                      page_size, seq_lens, cu_seqlens_q, plan, capacity, bs, num_tokens, max_q_len, num_q_heads,
                      num_kv_heads, head_dim, sm_scale, causal, num_sms, seg_max, part_o, part_m, part_l, &params,
                      &rp);
    if (rc != SK_OK)
        return rc;
    const int fixed = use_plan ? 0 : sk_fixed_nseg(bs, num_kv_heads, num_sms, seg_max);
    rc = check_merge(part_o, part_m, part_l, tok, fixed, num_tokens, num_q_heads, head_dim, seg_max, out);
    if (rc != SK_OK)
        return rc;

    if (use_plan) {
        int *status = nullptr;
        rc = device_status_word(&status);
        if (rc != SK_OK)
            return rc;
        // built on every call: the caller's lengths may have changed in place
        const int budget = num_sms / num_kv_heads;   // B of the plan rule
        cudaError_t e = launch_plan(seq_lens, cu_seqlens_q, bs, num_tokens, budget, seg_max, plan,
                                    capacity, tok, status, st);
        if (e != cudaSuccess)
            return set_error(SK_ERR_CUDA, "sk_paged_decode_attention_static: plan kernel launch failed");
    }
    if (rp > 0) {
        rc = launch_prepared_attn(params, kv_dtype, rp, stream);
        if (rc != SK_OK)
            return rc;
    }
    return sk_merge_segments(part_o, part_m, part_l, tok, fixed, num_tokens, num_q_heads, head_dim,
                             seg_max, out, lse, stream);
}
