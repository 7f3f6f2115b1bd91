/*
 * sk.h -- C ABI of libsk: length-aware split-KV paged decode/verify attention
 * for one GB300 (sm_103a).
 *
 * The method (SGLang PR 39172, "[AMD] gfx950 assembly attention: length-aware
 * split-KV for dynamic workload") runs in three device steps per attention
 * call:
 *   1. sk_build_plan        picks one segment length T from the batch's
 *                           sequence lengths and writes a compact work list
 *                           of (sequence, segment) items plus a per-query-
 *                           token segment count (Modifications, first item).
 *   2. sk_paged_decode_attn one CTA per (sequence, segment, kv head) work item
 *                           gathers K/V from standard pages and emits a
 *                           partial softmax state per query row
 *                           (Modifications, second item).
 *   3. sk_merge_segments    merges each token's segments by log-sum-exp,
 *                           reading only that token's segment count
 *                           (Modifications, third item).
 * A NULL plan selects the fixed split of the Motivation section (used for
 * bs == 1, where it already gives 64 segments).
 *
 * Conventions for every call:
 *  - Pointers marked "device" are device memory owned by the caller; the
 *    library keeps no reference after the call returns.  It allocates no
 *    device memory of its own: its only device storage is one status word
 *    per device and the fixed scratch array of
 *    sk_paged_decode_attention_static (both static __device__ variables).
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  No call synchronises, so the whole path can be
 *    captured into a CUDA graph.  Every kernel is launched with programmatic
 *    stream serialization: it may start while the kernel before it on the
 *    stream finishes, and waits for that kernel's completion (and its writes)
 *    before it reads anything, so stream order is kept.
 *  - Invalid arguments are caught on the host before anything is launched
 *    and return a negative sk_status; sk_last_error() then describes the
 *    problem.  Conditions only the device can see (a block id outside
 *    [0, num_blocks), a query length above max_q_len, an inconsistent
 *    cu_seqlens_q, a wait that timed out) set bits in the device status word
 *    and the affected work is skipped; read them with sk_get_device_status().
 *    cu_seqlens_q must be non-decreasing with cu[0] == 0 and cu[bs] ==
 *    num_tokens; otherwise SK_DEV_BAD_SEQ is set, tokens outside [cu[0],
 *    cu[bs]) get 0 segments from the plan (output 0, lse -inf), and on the
 *    fixed split their outputs are undefined.
 *  - Supported shapes: head_dim == 128, page_size == 16, 1 <= bs <= 32767
 *    (so seq << 16 stays positive), num_q_heads % num_kv_heads == 0.
 */
#ifndef SK_H_
#define SK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SK_OK = 0,
    SK_CACHED = 1,            /* sk_build_plan: cache hit, nothing launched */
    SK_ERR_INVALID = -1,      /* bad pointer, size or stride */
    SK_ERR_CAPACITY = -2,     /* plan_capacity too small */
    SK_ERR_UNSUPPORTED = -3,  /* shape outside the supported set */
    SK_ERR_CUDA = -4,         /* a CUDA runtime call failed */
    SK_ERR_TIMEOUT = -5       /* sk_get_device_status: a bounded wait inside a kernel expired */
} sk_status;

typedef enum {
    SK_KV_BF16 = 0,           /* pages hold bf16 */
    SK_KV_FP8_E4M3 = 1        /* pages hold OCP e4m3fn codes (vLLM RFC 59111, Proposed Change:
                                 OCP e4m3fn, not MI300's fnuz), value = code * scale */
} sk_kv_dtype;

/* Bits of the device status word (sk_get_device_status). */
#define SK_DEV_BAD_BLOCK 0x1   /* a block-table entry outside [0, num_blocks) was skipped */
#define SK_DEV_BAD_SEQ 0x2     /* q_len > max_q_len, L > block_table_stride * page, or bad cu_seqlens_q */
#define SK_DEV_TIMEOUT 0x4     /* a bounded wait inside a kernel expired; its work item was abandoned */
#define SK_DEV_INTERNAL 0x8    /* a kernel precondition failed (e.g. shared-memory alignment); item skipped */

/* Tokens per plan tile.  The plan counts segment lengths in tiles:
 * plan[0] = tiles per segment, so a segment spans plan[0] * sk_tile_tokens()
 * tokens (SGLang PR 39172, Modifications: "tiles per segment come from
 * plan[0]").  Returns 64. */
int sk_tile_tokens(void);

/* Smallest valid plan_capacity for a batch: 1 + max(B, bs) with
 * B = floor(num_sms / num_kv_heads), the plan's budget of work items (SGLang PR
 * 39172, Modifications: total segments capped at num_CUs / kv_heads; a batch
 * with more non-empty sequences than B takes one segment each, so up to bs
 * items).  Host-only arithmetic; SK_ERR_INVALID for bs outside [1, 32767] or
 * a non-positive head or SM count. */
int sk_plan_capacity(int bs, int num_kv_heads, int num_sms);

/* Segment count of the fixed split (SGLang PR 39172, Motivation):
 * max(1, min(seg_max, pow2floor(num_sms / (bs * num_kv_heads)))), pow2floor
 * of a value below 1 being 0.  Host-only arithmetic. */
int sk_fixed_nseg(int bs, int num_kv_heads, int num_sms, int seg_max);

/* Build the length-aware plan on the device (SGLang PR 39172, Modifications).
 *
 *   tiles_s = ceil(seq_lens[s] / sk_tile_tokens())
 *   B       = floor(num_sms / num_kv_heads)
 *   T       = smallest t >= 1 with sum_s ceil(tiles_s / t) <= B and
 *             max_s ceil(tiles_s / t) <= seg_max; if no t qualifies (more
 *             non-empty sequences than B) T = max_s tiles_s, one segment per
 *             non-empty sequence; T = 1 when every sequence is empty.
 *
 * Outputs (device, caller-owned):
 *   plan     int32[plan_capacity]: plan[0] = T; plan[1+k] = (s << 16) | g for
 *            every segment g < ceil(tiles_s / T) of every sequence s, in
 *            (s ascending, g ascending) order; -1 in every later slot.
 *   tok_nseg int32[num_tokens]: tok_nseg[t] = segment count of t's sequence.
 * Inputs (device): seq_lens int32[bs] (KV length including this step's query
 *   tokens), cu_seqlens_q int32[bs+1] (query-token offsets, cu[bs] ==
 *   num_tokens).
 * plan_capacity must be >= sk_plan_capacity(bs, num_kv_heads, num_sms) =
 * 1 + max(B, bs); larger values are allowed.
 *
 * Plan cache: the plan is built once per forward and reused by every layer.
 * The cache key is (seq_lens, seq_lens_version, cu_seqlens_q,
 * cu_seqlens_q_version, bs, num_tokens, num_kv_heads, num_sms, seg_max, plan,
 * plan_capacity, tok_nseg, whether `stream` is capturing).  A hit returns
 * SK_CACHED and launches nothing: the caller's plan/tok_nseg buffers still hold
 * the result.  The version arguments let a caller mark in-place changes (the
 * Python binding passes tensor._version).  sk_plan_cache_reset() clears the
 * cache; call it at the start of every forward.
 * Returns SK_OK (plan kernel enqueued), SK_CACHED, or a negative sk_status. */
int sk_build_plan(const int32_t *seq_lens, uint64_t seq_lens_version,
                  const int32_t *cu_seqlens_q, uint64_t cu_seqlens_q_version,
                  int bs, int num_tokens, int num_kv_heads, int num_sms, int seg_max,
                  int32_t *plan, int plan_capacity, int32_t *tok_nseg, void *stream);

/* Clear the plan cache (SGLang PR 39172, Modifications: the cache is cleared
 * at the start of every forward). */
void sk_plan_cache_reset(void);

/* Number of plan kernels launched by this process so far (cache misses). */
long long sk_plan_launch_count(void);

/* Split-KV paged attention (SGLang PR 39172, Modifications, second item).
 *
 * Grid: with a plan, (plan_capacity - 1) * num_kv_heads * row_blocks CTAs,
 * row_blocks = ceil(G * max_q_len / 64) when that exceeds 64 rows (else 1);
 * CTA b takes row block b % row_blocks (rows [64 rb, 64 rb + 64) of the item)
 * of work item i = (b / row_blocks) / num_kv_heads and KV head
 * h = (b / row_blocks) % num_kv_heads, reads w = plan[1+i], and exits at once
 * when w == -1 or the block is past the item's rows.  Sequence s = w >> 16,
 * segment g = w & 0xFFFF covers keys [g*T, min((g+1)*T, L_s)) with
 * T = plan[0] * sk_tile_tokens().  With plan == NULL the fixed split runs:
 * nseg = sk_fixed_nseg(bs, num_kv_heads, num_sms, seg_max) segments per
 * sequence of ceil(tiles_s / nseg) tiles each (trailing ones may be empty);
 * the grid is bs * nseg * num_kv_heads.
 *
 * Layouts (device):
 *   q            bf16 [num_tokens, num_q_heads, head_dim], token-major via
 *                cu_seqlens_q.  Query head hq uses KV head hq / G, G =
 *                num_q_heads / num_kv_heads.
 *   kv_pages     [num_blocks, num_kv_heads, page_size, 2*head_dim]: standard
 *                pages (vLLM RFC 59111, Background): per head, each token
 *                row holds K in [0, D) and V in [D, 2D).  bf16 or e4m3fn.
 *   block_table  int32 [bs, block_table_stride]; key p of sequence s lives in
 *                block block_table[s*stride + p/page_size], row p % page_size.
 *   seq_lens, cu_seqlens_q as for sk_build_plan; plan as written by it.
 * Masking: with causal != 0, query token j of sequence s (q_s tokens) sees
 *   keys p <= L_s - q_s + j; otherwise all L_s keys.
 * Scores: sm_scale * k_scale * <q, k>; values are multiplied by v_scale (the
 *   two scales apply to fp8 pages only and are ignored for bf16).
 * max_q_len: an upper bound on every q_s (at least 1 when num_tokens > 0); it
 *   sizes the kernel's row tile and row blocks (rows per work item = G * q_s).
 *   G * max_q_len above 65536, or num_blocks * num_kv_heads above 2^30, is
 *   SK_ERR_UNSUPPORTED.
 * Outputs (device, fp32): for every query token t of the item's sequence,
 *   every query head hq of KV head h, and the item's segment g:
 *     part_m[(t*seg_max + g)*num_q_heads + hq]  reference value m (score units)
 *     part_l[same]                               l = sum_p exp(score_p - m)
 *     part_o[same * head_dim + d]                o = v_scale * sum_p exp(score_p - m) * V_p[d]
 *   over the keys of the segment that the row sees.  A row that sees none of
 *   them gets (m, l, o) = (-inf, 0, 0).  m is not required to be the maximum
 *   score; m + log(l) and o / l are the segment's unique log-sum-exp and output.
 *   Arrays are [num_tokens, seg_max, num_q_heads(, head_dim)]; only segments
 *   that exist are written.
 * q, kv_pages and part_o must be 16-byte aligned (SK_ERR_INVALID otherwise).
 * Returns SK_OK or a negative sk_status. */
int sk_paged_decode_attn(const void *q, const void *kv_pages, int kv_dtype, float k_scale,
                         float v_scale, const int32_t *block_table, int block_table_stride,
                         int num_blocks, int page_size, const int32_t *seq_lens,
                         const int32_t *cu_seqlens_q, const int32_t *plan, int plan_capacity,
                         int bs, int num_tokens, int max_q_len, int num_q_heads, int num_kv_heads,
                         int head_dim, float sm_scale, int causal, int num_sms, int seg_max,
                         float *part_o, float *part_m, float *part_l, void *stream);

/* Merge segment partials by log-sum-exp (SGLang PR 39172, Modifications,
 * third item: the reduce reads only its token's segment count).
 * For token t and query head hq with n = tok_nseg[t] (or fixed_nseg when
 * tok_nseg == NULL) segments, over segments with l > 0:
 *   M = max m_g,  Lambda = sum l_g exp(m_g - M),
 *   out = sum o_g exp(m_g - M) / Lambda   (bf16, round to nearest even),
 *   lse = M + log(Lambda)                  (fp32, optional).
 * No contributing segment: out = 0, lse = -inf.
 * out bf16 [num_tokens, num_q_heads, head_dim]; lse fp32 [num_tokens,
 * num_q_heads] or NULL.  Partials as written by sk_paged_decode_attn.
 * part_o must be 16-byte and out 8-byte aligned (SK_ERR_INVALID otherwise).
 * Returns SK_OK or a negative sk_status. */
int sk_merge_segments(const float *part_o, const float *part_m, const float *part_l,
                      const int32_t *tok_nseg, int fixed_nseg, int num_tokens, int num_q_heads,
                      int head_dim, int seg_max, void *out, float *lse, void *stream);

/* KV write: store this step's K and V rows into standard pages through a
 * slot mapping (the writer of the backends that keep standard pages, vLLM RFC
 * 59111, Background: per head, a token row holds K and V side by side).
 *
 * For token t and KV head h with slot = slot_mapping[t] >= 0:
 *   kv_pages[slot / page_size][h][slot % page_size][0 : D)  = K[t][h][:]
 *   kv_pages[slot / page_size][h][slot % page_size][D : 2D) = V[t][h][:]
 * bf16 pages receive the input bits unchanged.  e4m3fn pages
 * (kv_dtype == SK_KV_FP8_E4M3) receive each value divided by k_scale (K) or
 * v_scale (V) in IEEE binary32 and rounded to the nearest e4m3fn code, ties
 * to even, magnitudes above 448 (and infinities) saturated to 448, NaN kept
 * as NaN; sk_paged_decode_attn then multiplies the codes back by the same
 * scales.
 * A negative slot writes nothing for that token.  A slot at or past
 * num_blocks * page_size writes nothing and sets SK_DEV_BAD_BLOCK in the
 * device status word.  Two tokens with the same slot leave that row
 * undefined (either token's values).
 *
 * Layouts (device, caller-owned): key, value bf16 [num_tokens, num_kv_heads,
 * head_dim]; slot_mapping int64 [num_tokens]; kv_pages [num_blocks,
 * num_kv_heads, page_size, 2*head_dim] of bf16 or e4m3fn, written in place.
 * key, value and kv_pages must be 16-byte aligned; head_dim must be 128 and
 * page_size 16.  Asynchronous on `stream`, no allocation, capture safe.
 * Returns SK_OK or a negative sk_status. */
int sk_reshape_and_cache(const void *key, const void *value, const int64_t *slot_mapping,
                         int num_tokens, int num_kv_heads, int head_dim, void *kv_pages, int kv_dtype,
                         float k_scale, float v_scale, int num_blocks, int page_size, void *stream);

/* Standard -> shuffled page conversion (vLLM RFC 59111, Proposed Change,
 * Convert: the per-block view/permute that turns standard pages into ROCm
 * AITER's shuffled pages).  With x = 16 / element size (8 for bf16, 16 for
 * e4m3fn), for every block blk listed in block_ids (all num_blocks blocks when
 * block_ids == NULL, num_ids then ignored), head h, token row n, dimension d:
 *   k_shuf[blk][h][d / x][n][d % x] = kv_pages[blk][h][n][d]
 *   v_shuf[blk][h][n / x][d][n % x] = kv_pages[blk][h][n][D + d]
 * Other blocks of k_shuf and v_shuf are left alone.  An id outside
 * [0, num_blocks) is skipped and sets SK_DEV_BAD_BLOCK in the device status.
 *
 * Layouts (device, caller-owned): kv_pages [num_blocks, num_kv_heads,
 * page_size, 2*head_dim] (kv_dtype bf16 or e4m3fn, bytes copied as they are);
 * k_shuf [num_blocks, num_kv_heads, head_dim / x, page_size, x];
 * v_shuf [num_blocks, num_kv_heads, page_size / x, head_dim, x]; block_ids
 * int32 [num_ids] or NULL.  All three arrays 16-byte aligned; head_dim 128,
 * page_size 16.  Asynchronous on `stream`, no allocation, capture safe.
 * Returns SK_OK or a negative sk_status. */
int sk_std_to_shuffled(const void *kv_pages, int kv_dtype, const int32_t *block_ids, int num_ids,
                       int num_blocks, int num_kv_heads, int head_dim, int page_size, void *k_shuf,
                       void *v_shuf, void *stream);

/* The whole attention call -- plan (use_plan != 0) or fixed split, split-KV
 * attention, merge -- without any device allocation, for callers that cannot
 * allocate: a host engine that owns all device memory through its own
 * allocator and forbids plug-ins to call cudaMalloc, or a C caller without a
 * caching allocator that cannot afford cudaMalloc/cudaFree (which may
 * synchronise the device) in a serving step.  The pages have no counterpart
 * to this call; it exists for those callers only.
 *
 * The caller passes inputs and outputs as for sk_build_plan,
 * sk_paged_decode_attn and sk_merge_segments (same meanings and layouts;
 * out bf16 [num_tokens, num_q_heads, 128], lse fp32 or NULL).  The plan,
 * per-token segment counts and segment partials live in one file-scope
 * device array of sk_static_scratch_bytes() = 32 MiB per GPU that loads the
 * library, held until exit.  A call needs about
 * num_tokens * seg_max * num_q_heads * 520 bytes plus the plan; larger calls
 * return SK_ERR_CAPACITY and launch nothing.  The plan is rebuilt on every
 * call (no plan cache).  All calls share the array and it keeps the last
 * call's contents (nothing in it needs to start at zero); calls whose kernels
 * overlap on the GPU race on it, so serialise them.  The first call on a
 * device looks up the array's address (cudaGetSymbolAddress, once per
 * device); make that first call before any stream capture.
 * Returns SK_OK or a negative sk_status. */
int sk_paged_decode_attention_static(const void *q, const void *kv_pages, int kv_dtype,
                                     float k_scale, float v_scale, const int32_t *block_table,
                                     int block_table_stride, int num_blocks, int page_size,
                                     const int32_t *seq_lens, const int32_t *cu_seqlens_q,
                                     int use_plan, int bs, int num_tokens, int max_q_len,
                                     int num_q_heads, int num_kv_heads, int head_dim,
                                     float sm_scale, int causal, int num_sms, int seg_max,
                                     void *out, float *lse, void *stream);

/* Size in bytes of the static scratch array used by
 * sk_paged_decode_attention_static. */
size_t sk_static_scratch_bytes(void);

/* Synchronise `stream`, read the device status word of the current device
 * and clear it when `clear` != 0.
 * Returns SK_ERR_TIMEOUT when SK_DEV_TIMEOUT is set (a bounded wait expired and
 * its work item was abandoned, so some partials and outputs of the calls since
 * the last clear are missing); otherwise the mask of SK_DEV_* bits, 0 when
 * clean; another negative sk_status if a CUDA call fails.  The whole mask read
 * by the last call on this thread, timeout bit included, is
 * sk_last_device_status(). */
int sk_get_device_status(void *stream, int clear);

/* The mask of SK_DEV_* bits that the last sk_get_device_status call on this
 * thread read (0 before the first call). */
int sk_last_device_status(void);

/* Limit, in SM clock cycles, of each wait of the attention kernel that can
 * give up (for a copy to land, a product to complete, another role to finish
 * its part of a tile).  It applies to the launches made after the call;
 * cycles < 0 restores the default of 4e9 (about two seconds).  Returns the
 * previous limit.  Waits for work a CTA has already issued -- its copies and
 * products in flight, before the CTA exits -- keep the default whatever this
 * limit is.  This is a test hook: a limit far below the memory latency makes
 * waits expire in an unchanged kernel, so the timeout path (SK_DEV_TIMEOUT,
 * then SK_ERR_TIMEOUT from sk_get_device_status) can be exercised without
 * faulting or hanging anything.  Process-wide; not for concurrent use with
 * other calls. */
long long sk_set_wait_limit(long long cycles);

/* Message for the last negative status returned on this thread. */
const char *sk_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SK_H_ */
