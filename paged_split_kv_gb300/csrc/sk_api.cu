// C ABI of libsk: argument validation, the plan cache, the device status
// word and kernel dispatch.  See include/sk.h for the contract of each call.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "sk.h"
#include "sk_internal.cuh"

namespace sk {

// One status word per device; kernels OR SK_DEV_* bits into it.
__device__ int g_device_status;

namespace {

thread_local char g_msg[512];

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(SK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
int *g_status_ptr[kMaxDevices];
std::mutex g_status_mutex;

// Address of this device's status word (looked up once per device).
// SM count of the current device, read once per device.
int sm_count(int *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(SK_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    static std::atomic<int> cached[kMaxDevices];
    int v = cached[dev].load();
    if (v == 0) {
        e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        cached[dev].store(v);
    }
    *out = v;
    return SK_OK;
}

int status_ptr(int **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(SK_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (g_status_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_status);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(status)");
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    *out = g_status_ptr[dev];
    return SK_OK;
}

// ---------------------------------------------------------------- plan cache
struct PlanKey {
    const void *seq_lens;
    uint64_t seq_lens_version;
    const void *cu_q;
    uint64_t cu_q_version;
    int bs, num_tokens, num_kv_heads, num_sms, seg_max;
    const void *plan;
    int plan_capacity;
    const void *tok_nseg;
    int capturing;
    int device;
};

bool same_key(const PlanKey &a, const PlanKey &b)
{
    return a.seq_lens == b.seq_lens && a.seq_lens_version == b.seq_lens_version && a.cu_q == b.cu_q &&
           a.cu_q_version == b.cu_q_version && a.bs == b.bs && a.num_tokens == b.num_tokens &&
           a.num_kv_heads == b.num_kv_heads && a.num_sms == b.num_sms && a.seg_max == b.seg_max &&
           a.plan == b.plan && a.plan_capacity == b.plan_capacity && a.tok_nseg == b.tok_nseg &&
           a.capturing == b.capturing && a.device == b.device;
}

constexpr int kCacheSlots = 8;
PlanKey g_cache[kCacheSlots];
int g_cache_used = 0;
int g_cache_next = 0;
std::mutex g_cache_mutex;
std::atomic<long long> g_plan_launches{0};

}  // namespace

int device_status_word(int **out) { return status_ptr(out); }

namespace {
std::atomic<long long> g_wait_limit{kDefaultWaitLimit};
thread_local int g_last_device_status = 0;

// Plan buffer length: the plan's T, then up to max(B, bs) work items, B = floor(num_sms /
// num_kv_heads) (SGLang PR 39172, Modifications: the total segment count is capped at
// num_CUs / kv_heads, and a batch with more non-empty sequences than that takes one each).
long long capacity_of(int bs, int num_kv_heads, int num_sms)
{
    const long long budget = (long long)num_sms / num_kv_heads;
    return 1 + (budget > bs ? budget : bs);
}
}  // namespace

long long wait_limit() { return g_wait_limit.load(); }

int set_error(int code, const char *msg) { return fail(code, "%s", msg); }

}  // namespace sk

using namespace sk;

extern "C" {

int sk_tile_tokens(void) { return kTile; }

int sk_fixed_nseg(int bs, int num_kv_heads, int num_sms, int seg_max)
{
    long long denom = (long long)bs * num_kv_heads;
    long long q = denom > 0 && num_sms > 0 ? (long long)num_sms / denom : 0;
    long long p = 0;
    if (q >= 1) {
        p = 1;
        while (p * 2 <= q)
            p *= 2;
    }
    if (p > seg_max)
        p = seg_max;
    return p < 1 ? 1 : (int)p;
}

const char *sk_last_error(void) { return g_msg; }

int sk_plan_capacity(int bs, int num_kv_heads, int num_sms)
{
    if (bs < 1 || bs > 32767 || num_kv_heads < 1 || num_sms < 1)
        return fail(SK_ERR_INVALID, "sk_plan_capacity: bs=%d num_kv_heads=%d num_sms=%d", bs, num_kv_heads,
                    num_sms);
    const long long c = capacity_of(bs, num_kv_heads, num_sms);
    if (c > 0x7FFFFFFFLL)
        return fail(SK_ERR_INVALID, "sk_plan_capacity: capacity overflows int");
    return (int)c;
}

long long sk_set_wait_limit(long long cycles)
{
    return g_wait_limit.exchange(cycles < 0 ? kDefaultWaitLimit : cycles);
}

int sk_last_device_status(void) { return g_last_device_status; }

void sk_plan_cache_reset(void)
{
    std::lock_guard<std::mutex> lock(g_cache_mutex);
    g_cache_used = 0;
    g_cache_next = 0;
}

long long sk_plan_launch_count(void) { return g_plan_launches.load(); }

int sk_build_plan(const int32_t *seq_lens, uint64_t seq_lens_version, const int32_t *cu_seqlens_q,
                  uint64_t cu_seqlens_q_version, int bs, int num_tokens, int num_kv_heads,
                  int num_sms, int seg_max, int32_t *plan, int plan_capacity, int32_t *tok_nseg,
                  void *stream)
{
    if (seq_lens == nullptr || cu_seqlens_q == nullptr || plan == nullptr)
        return fail(SK_ERR_INVALID, "sk_build_plan: null seq_lens, cu_seqlens_q or plan");
    if (bs < 1 || bs > 32767)
        return fail(SK_ERR_INVALID, "sk_build_plan: bs=%d outside [1, 32767]", bs);
    if (num_tokens < 0 || (num_tokens > 0 && tok_nseg == nullptr))
        return fail(SK_ERR_INVALID, "sk_build_plan: num_tokens=%d with tok_nseg=%p", num_tokens,
                    (void *)tok_nseg);
    if (num_kv_heads < 1 || num_sms < 1)
        return fail(SK_ERR_INVALID, "sk_build_plan: num_kv_heads=%d num_sms=%d", num_kv_heads, num_sms);
    if (seg_max < 1 || seg_max > 0xFFFF)
        return fail(SK_ERR_INVALID, "sk_build_plan: seg_max=%d outside [1, 65535]", seg_max);
    const int budget = num_sms / num_kv_heads;
    if (plan_capacity < capacity_of(bs, num_kv_heads, num_sms))
        return fail(SK_ERR_CAPACITY, "sk_build_plan: plan_capacity=%d < 1 + max(B=%d, bs=%d)",
                    plan_capacity, budget, bs);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cap);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamIsCapturing");
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");

    PlanKey key{seq_lens, seq_lens_version, cu_seqlens_q, cu_seqlens_q_version, bs, num_tokens,
                num_kv_heads, num_sms, seg_max, plan, plan_capacity, tok_nseg,
                cap != cudaStreamCaptureStatusNone ? 1 : 0, dev};
    {
        std::lock_guard<std::mutex> lock(g_cache_mutex);
        for (int i = 0; i < g_cache_used; ++i)
            if (same_key(g_cache[i], key))
                return SK_CACHED;
    }
    int *status = nullptr;
    int rc = status_ptr(&status);
    if (rc != SK_OK)
        return rc;
    e = launch_plan(seq_lens, cu_seqlens_q, bs, num_tokens, budget, seg_max, plan, plan_capacity,
                    tok_nseg, status, st);
    if (e != cudaSuccess)
        return cuda_fail(e, "plan kernel launch");
    g_plan_launches.fetch_add(1);
    {
        std::lock_guard<std::mutex> lock(g_cache_mutex);
        // a plan buffer holds one plan: drop entries that wrote to the same buffers
        int w = 0;
        for (int i = 0; i < g_cache_used; ++i)
            if (g_cache[i].plan != plan && g_cache[i].tok_nseg != tok_nseg)
                g_cache[w++] = g_cache[i];
        g_cache_used = w;
        if (g_cache_used < kCacheSlots) {
            g_cache[g_cache_used++] = key;
        } else {
            g_cache[g_cache_next] = key;
            g_cache_next = (g_cache_next + 1) % kCacheSlots;
        }
    }
    return SK_OK;
}

}  // extern "C"

namespace sk {

// Checks the arguments of an attention call and resolves the kernel's parameters; launches
// nothing.  *rp_out is the row tile of the launch, 0 when there is nothing to launch.
int prepare_attn(const void *q, const void *kv_pages, int kv_dtype, float k_scale, float v_scale,
                 const int32_t *block_table, int block_table_stride, int num_blocks, int page_size,
                 const int32_t *seq_lens, const int32_t *cu_seqlens_q, const int32_t *plan,
                 int plan_capacity, int bs, int num_tokens, int max_q_len, int num_q_heads,
                 int num_kv_heads, int head_dim, float sm_scale, int causal, int num_sms, int seg_max,
                 float *part_o, float *part_m, float *part_l, AttnParams *params, int *rp_out)
{
    if (q == nullptr || kv_pages == nullptr || block_table == nullptr || seq_lens == nullptr ||
        cu_seqlens_q == nullptr || part_o == nullptr || part_m == nullptr || part_l == nullptr)
        return fail(SK_ERR_INVALID, "sk_paged_decode_attn: null pointer argument");
    if (kv_dtype != SK_KV_BF16 && kv_dtype != SK_KV_FP8_E4M3)
        return fail(SK_ERR_INVALID, "sk_paged_decode_attn: kv_dtype=%d", kv_dtype);
    if (head_dim != kHeadDim)
        return fail(SK_ERR_UNSUPPORTED, "sk_paged_decode_attn: head_dim=%d (only 128)", head_dim);
    if (page_size != kPage)
        return fail(SK_ERR_UNSUPPORTED, "sk_paged_decode_attn: page_size=%d (only 16)", page_size);
    if (bs < 1 || bs > 32767)
        return fail(SK_ERR_INVALID, "sk_paged_decode_attn: bs=%d outside [1, 32767]", bs);
    if (num_tokens < 0 || max_q_len < 0 || (num_tokens > 0 && max_q_len < 1) || block_table_stride < 1 ||
        num_blocks < 1)
        return fail(SK_ERR_INVALID,
                    "sk_paged_decode_attn: num_tokens=%d max_q_len=%d stride=%d num_blocks=%d",
                    num_tokens, max_q_len, block_table_stride, num_blocks);
    if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0)
        return fail(SK_ERR_INVALID, "sk_paged_decode_attn: %d query heads, %d kv heads", num_q_heads,
                    num_kv_heads);
    if (num_sms < 1 || seg_max < 1 || seg_max > 0xFFFF)
        return fail(SK_ERR_INVALID, "sk_paged_decode_attn: num_sms=%d seg_max=%d", num_sms, seg_max);
    if (!(sm_scale > 0.f) || (kv_dtype == SK_KV_FP8_E4M3 && !(k_scale > 0.f && v_scale > 0.f)))
        return fail(SK_ERR_INVALID, "sk_paged_decode_attn: scales must be positive");
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_pages) |
         reinterpret_cast<uintptr_t>(part_o)) & 15)
        return fail(SK_ERR_INVALID, "sk_paged_decode_attn: q, kv_pages and part_o must be 16-byte aligned");
    int num_items;
    int fixed = 0;
    if (plan != nullptr) {
        const long long need = capacity_of(bs, num_kv_heads, num_sms);
        if (plan_capacity < need)
            return fail(SK_ERR_CAPACITY, "sk_paged_decode_attn: plan_capacity=%d < %lld", plan_capacity,
                        need);
        num_items = plan_capacity - 1;
    } else {
        fixed = sk_fixed_nseg(bs, num_kv_heads, num_sms, seg_max);
        num_items = bs * fixed;
    }
    const long long rows_ll = (long long)(num_q_heads / num_kv_heads) * max_q_len;
    const int rows_max = rows_ll > 0x7FFFFFFFLL ? 0x7FFFFFFF : (int)rows_ll;
    const int rp = attn_tc_rows(kv_dtype, rows_max, num_blocks, num_kv_heads);
    if (num_tokens > 0 && rp == 0)
        return fail(SK_ERR_UNSUPPORTED,
                    "sk_paged_decode_attn: %d rows per work item (G * max_q_len) or %d blocks x %d heads "
                    "exceed the kernel's limits (65536 rows; 2^30 block-heads)",
                    rows_max, num_blocks, num_kv_heads);
    const int row_blocks = rp > 0 ? (rows_max + rp - 1) / rp : 1;
    if ((long long)num_items * num_kv_heads * row_blocks > 0x7FFFFFFFLL)
        return fail(SK_ERR_INVALID, "sk_paged_decode_attn: grid too large");
    *rp_out = 0;
    if (num_tokens == 0)
        return SK_OK;

    int *status = nullptr;
    int rc = status_ptr(&status);
    if (rc != SK_OK)
        return rc;

    AttnParams &p = *params;
    p.q = static_cast<const uint16_t *>(q);
    p.kv = kv_pages;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.cu_q = cu_seqlens_q;
    p.plan = plan;
    p.part_o = part_o;
    p.part_m = part_m;
    p.part_l = part_l;
    p.status = status;
    p.num_blocks = num_blocks;
    p.bt_stride = block_table_stride;
    p.bs = bs;
    p.num_tokens = num_tokens;
    p.max_q_len = max_q_len;
    p.H_q = num_q_heads;
    p.H_kv = num_kv_heads;
    p.G = num_q_heads / num_kv_heads;
    p.seg_max = seg_max;
    p.fixed_nseg = fixed;
    p.num_items = num_items;
    p.causal = causal ? 1 : 0;
    const float log2e = 1.4426950408889634f;
    p.score_scale_log2 = sm_scale * (kv_dtype == SK_KV_FP8_E4M3 ? k_scale : 1.f) * log2e;
    p.v_scale = kv_dtype == SK_KV_FP8_E4M3 ? v_scale : 1.f;
    p.wait_limit = wait_limit();

    p.row_blocks = row_blocks;
    *rp_out = rp;
    return SK_OK;
}

// Checks the arguments of a merge call; launches nothing.
int check_merge(const float *part_o, const float *part_m, const float *part_l, const int32_t *tok_nseg,
                int fixed_nseg, int num_tokens, int num_q_heads, int head_dim, int seg_max, const void *out)
{
    if (part_o == nullptr || part_m == nullptr || part_l == nullptr || out == nullptr)
        return fail(SK_ERR_INVALID, "sk_merge_segments: null pointer argument");
    if (head_dim != kHeadDim)
        return fail(SK_ERR_UNSUPPORTED, "sk_merge_segments: head_dim=%d (only 128)", head_dim);
    if (num_tokens < 0 || num_q_heads < 1 || seg_max < 1 || seg_max > 0xFFFF)
        return fail(SK_ERR_INVALID, "sk_merge_segments: num_tokens=%d num_q_heads=%d seg_max=%d",
                    num_tokens, num_q_heads, seg_max);
    if (tok_nseg == nullptr && (fixed_nseg < 0 || fixed_nseg > seg_max))
        return fail(SK_ERR_INVALID, "sk_merge_segments: fixed_nseg=%d outside [0, seg_max]", fixed_nseg);
    if ((reinterpret_cast<uintptr_t>(part_o) & 15) || (reinterpret_cast<uintptr_t>(out) & 7))
        return fail(SK_ERR_INVALID, "sk_merge_segments: part_o must be 16-byte and out 8-byte aligned");
    return SK_OK;
}

int launch_prepared_attn(const AttnParams &p, int kv_dtype, int rp, void *stream)
{
    cudaError_t e = launch_attn_tc(p, kv_dtype, rp, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "attention kernel launch");
    return SK_OK;
}

}  // namespace sk

extern "C" {

int sk_paged_decode_attn(const void *q, const void *kv_pages, int kv_dtype, float k_scale,
                         float v_scale, const int32_t *block_table, int block_table_stride,
                         int num_blocks, int page_size, const int32_t *seq_lens,
                         const int32_t *cu_seqlens_q, const int32_t *plan, int plan_capacity,
                         int bs, int num_tokens, int max_q_len, int num_q_heads, int num_kv_heads,
                         int head_dim, float sm_scale, int causal, int num_sms, int seg_max,
                         float *part_o, float *part_m, float *part_l, void *stream)
{
    AttnParams p;
    int rp = 0;
    const int rc = prepare_attn(q, kv_pages, kv_dtype, k_scale, v_scale, block_table, block_table_stride,
                                num_blocks, page_size, seq_lens, cu_seqlens_q, plan, plan_capacity, bs,
                                num_tokens, max_q_len, num_q_heads, num_kv_heads, head_dim, sm_scale,
                                causal, num_sms, seg_max, part_o, part_m, part_l, &p, &rp);
    if (rc != SK_OK || rp == 0)
        return rc;
    return launch_prepared_attn(p, kv_dtype, rp, stream);
}

int sk_merge_segments(const float *part_o, const float *part_m, const float *part_l,
                      const int32_t *tok_nseg, int fixed_nseg, int num_tokens, int num_q_heads,
                      int head_dim, int seg_max, void *out, float *lse, void *stream)
{
    const int rc = check_merge(part_o, part_m, part_l, tok_nseg, fixed_nseg, num_tokens, num_q_heads,
                               head_dim, seg_max, out);
    if (rc != SK_OK)
        return rc;
    cudaError_t e = launch_merge(part_o, part_m, part_l, tok_nseg, fixed_nseg, num_tokens, num_q_heads,
                                 seg_max, static_cast<uint16_t *>(out), lse,
                                 static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "merge kernel launch");
    return SK_OK;
}

int sk_reshape_and_cache(const void *key, const void *value, const int64_t *slot_mapping,
                         int num_tokens, int num_kv_heads, int head_dim, void *kv_pages, int kv_dtype,
                         float k_scale, float v_scale, int num_blocks, int page_size, void *stream)
{
    if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 1)
        return fail(SK_ERR_INVALID, "sk_reshape_and_cache: num_tokens=%d num_kv_heads=%d num_blocks=%d",
                    num_tokens, num_kv_heads, num_blocks);
    if (kv_dtype != SK_KV_BF16 && kv_dtype != SK_KV_FP8_E4M3)
        return fail(SK_ERR_INVALID, "sk_reshape_and_cache: kv_dtype=%d", kv_dtype);
    if (head_dim != kHeadDim)
        return fail(SK_ERR_UNSUPPORTED, "sk_reshape_and_cache: head_dim=%d (only 128)", head_dim);
    if (page_size != kPage)
        return fail(SK_ERR_UNSUPPORTED, "sk_reshape_and_cache: page_size=%d (only 16)", page_size);
    if (kv_dtype == SK_KV_FP8_E4M3 && !(k_scale > 0.f && v_scale > 0.f && k_scale < INFINITY && v_scale < INFINITY))
        return fail(SK_ERR_INVALID, "sk_reshape_and_cache: scales must be positive and finite");
    if (num_tokens == 0)
        return SK_OK;
    if (key == nullptr || value == nullptr || slot_mapping == nullptr || kv_pages == nullptr)
        return fail(SK_ERR_INVALID, "sk_reshape_and_cache: null pointer argument");
    if ((reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value) |
         reinterpret_cast<uintptr_t>(kv_pages)) & 15)
        return fail(SK_ERR_INVALID, "sk_reshape_and_cache: key, value and kv_pages must be 16-byte aligned");
    int *status = nullptr;
    int rc = status_ptr(&status);
    if (rc != SK_OK)
        return rc;
    int sms = 0;
    rc = sm_count(&sms);
    if (rc != SK_OK)
        return rc;
    cudaError_t e = launch_kv_write(static_cast<const uint16_t *>(key), static_cast<const uint16_t *>(value),
                                    slot_mapping, num_tokens, num_kv_heads, num_blocks, kv_pages, kv_dtype,
                                    k_scale, v_scale, status, sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "kv write kernel launch");
    return SK_OK;
}

int sk_std_to_shuffled(const void *kv_pages, int kv_dtype, const int32_t *block_ids, int num_ids,
                       int num_blocks, int num_kv_heads, int head_dim, int page_size, void *k_shuf,
                       void *v_shuf, void *stream)
{
    if (num_blocks < 1 || num_kv_heads < 1 || (block_ids != nullptr && num_ids < 0))
        return fail(SK_ERR_INVALID, "sk_std_to_shuffled: num_blocks=%d num_kv_heads=%d num_ids=%d", num_blocks,
                    num_kv_heads, num_ids);
    if (kv_dtype != SK_KV_BF16 && kv_dtype != SK_KV_FP8_E4M3)
        return fail(SK_ERR_INVALID, "sk_std_to_shuffled: kv_dtype=%d", kv_dtype);
    if (head_dim != kHeadDim)
        return fail(SK_ERR_UNSUPPORTED, "sk_std_to_shuffled: head_dim=%d (only 128)", head_dim);
    if (page_size != kPage)
        return fail(SK_ERR_UNSUPPORTED, "sk_std_to_shuffled: page_size=%d (only 16)", page_size);
    if (kv_pages == nullptr || k_shuf == nullptr || v_shuf == nullptr)
        return fail(SK_ERR_INVALID, "sk_std_to_shuffled: null pointer argument");
    if ((reinterpret_cast<uintptr_t>(kv_pages) | reinterpret_cast<uintptr_t>(k_shuf) |
         reinterpret_cast<uintptr_t>(v_shuf)) & 15)
        return fail(SK_ERR_INVALID, "sk_std_to_shuffled: kv_pages, k_shuf and v_shuf must be 16-byte aligned");
    if (block_ids != nullptr && num_ids == 0)
        return SK_OK;
    int *status = nullptr;
    int rc = status_ptr(&status);
    if (rc != SK_OK)
        return rc;
    int sms = 0;
    rc = sm_count(&sms);
    if (rc != SK_OK)
        return rc;
    cudaError_t e = launch_std_to_shuffled(kv_pages, kv_dtype, block_ids, num_ids, num_blocks, num_kv_heads, k_shuf,
                                           v_shuf, status, sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "shuffle kernel launch");
    return SK_OK;
}

int sk_get_device_status(void *stream, int clear)
{
    int *status = nullptr;
    int rc = status_ptr(&status);
    if (rc != SK_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int value = 0;
    cudaError_t e = cudaMemcpyAsync(&value, status, sizeof value, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && clear)
        e = cudaMemsetAsync(status, 0, sizeof(int), st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the device status word");
    g_last_device_status = value;
    if (value & SK_DEV_TIMEOUT)
        return fail(SK_ERR_TIMEOUT, "a bounded wait inside a kernel expired (device status 0x%x)", value);
    return value;
}

}  // extern "C"
