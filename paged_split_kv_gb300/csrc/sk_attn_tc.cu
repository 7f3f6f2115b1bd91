// Split-KV paged attention on the tcgen05 tensor cores (bf16 or fp8-e4m3 pages).
//
// One CTA per (sequence, segment, KV head) work item, as in SGLang PR 39172
// (Modifications, second item).  The GQA group's R = G * q_len query rows
// share every K/V byte, so the two products of a tile are dense contractions
// (per 128 tokens):
//     S^T [128 tokens x R] = K_half [128 x 128 dims] . Q^T
//     O^T [128 dims   x R] += V_tile^T [128 dims x tile tokens] . P^T
// Tokens and dimensions take the MMA's M = 128 and the query rows its N
// (16, 32 or 64 columns).  S^T (four buffers of a 128-token tile, or two of a
// 256-token one) and O^T live in tensor memory (TMEM lane = token for S, =
// dimension for O).  An item with more than 64
// rows is split into row blocks of 64, one CTA each, placed next to each other
// so that they stream the same pages at about the same time (L2 serves the
// repeats).
//
// Roles (352 threads; 608 for fp8 with 64 rows, with four softmax warpgroups):
//   warp 0   TMA producer: one 4-D copy per page (8 or 16 per tile) into
//            128-byte-swizzled atoms that are at once the K-major K operand
//            and the MN-major V^T operand (layout below).  Pages past the
//            segment end are out-of-bounds boxes: zero-filled, no HBM traffic.
//            It starts as soon as the mbarriers exist, with the block ids of
//            its first tiles already read; later it reads them a ring ahead.
//            On e4m3 pages with up to 32 rows each 128-token half of a tile
//            lands on its own barrier, so QK starts on the first half.
//   warp 1   allocates TMEM; issues the QK products.
//   warp 10 (18)  issues the PV products.  Both issuers run converged and issue
//            through one elected lane, so the descriptors stay warp-uniform.
//   warps 2-9 (2-17)  softmax, two (four) warpgroups: one thread per token of each 128-token
//            half of the tile (its TMEM lane); warps 2-5 take the first half of
//            the query rows, warps 6-9 the second, each group on its own.
//            The running max per query row is kept lazily: scores are
//            exponentiated against the current max unless one beats it by
//            2^8 (2^4 for fp8), which the group decides with one bar.red per
//            tile; only then is the tile max reduced across the 128 threads
//            and O rescaled (which waits for the previous PV).
//            Row sums are kept per thread and reduced once at the end.
//            On e4m3 pages the per-score work runs in packed f16 (d = s * c -
//            msub by FFMA, ex2.f16x2 on pairs, the rescale vote from a packed
//            max, the two e4m3 terms of P from a mask and a packed subtract).
//            P^T is written over the tile's own K area, which QK no longer
//            needs, so every stage carries its own P buffer.  At the end the
//            same warps move O^T from TMEM into the partials, 16 bytes a lane
//            after a transpose within lane quads.
// fp8 pages: both products run as kind::f8f6f4 on the e4m3 codes as they
// arrive, so a stage holds only codes: a 256-token tile (64 KB, three stages),
// whose single softmax pass covers as many bytes as a bf16 tile's.  With 64 rows
// the rows are split over four softmax warpgroups (608 threads) instead of two,
// so that a thread holds 16 rows of its two tokens.
// QK splits Q into two e4m3 terms (q * 2^e_r = hi + lo, a power-of-two scale
// per row), stacked as one operand of 2R rows, so one product per 32
// dimensions gives S_hi | S_lo (K read once), added by the softmax.  With 64
// rows one S buffer of a tile is 256 TMEM columns, so there is a single one
// (with O that is 384 of the 512 columns).  PV splits
// P the same way (p * 2^4 = hi + lo, about 8 significant bits), stacked as
// 2R columns of P^T, so O^T holds O_hi | O_lo, added at the end.  The scales
// k_scale and v_scale are folded into the score scale and the output.
//
// Every mbarrier wait is bounded (about two seconds unless sk_set_wait_limit
// says otherwise); on expiry the CTA sets SK_DEV_TIMEOUT in the device status
// word and every role gives up.  Before the CTA exits, the producer waits for
// every copy it issued to land and each issuer for its last commit (these waits
// keep the two-second bound whatever the limit), so no copy or product outlives
// the CTA's shared memory or TMEM.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <mutex>

#include "sk_internal.cuh"
#include "sk_sm100.cuh"

namespace sk {
namespace {

using namespace sm100;

constexpr int kTokTile = 128;                       // tokens per MMA (M)
constexpr int kSoftmaxWarp0 = 2;
constexpr long long kDrainLimit = 4000000000LL;     // cycles (~2 s): waits for work already issued
constexpr uint32_t kFull = 0xffffffffu;
constexpr int kMaxSmem = 232448;                    // 227 KB per CTA
// e4m3 path: the subtrahend of a row whose running max is still -inf.  Any visible score then
// gives d = s * c - msub far above the rescale threshold (f16 +inf), so the running max is set
// before any P of that row is formed; a masked score gives -inf - msub = -inf, p = 0.
constexpr float kMsubNone = -0x1p100f;

// Stage layout.  One TMA copy per page brings its 16 token rows as two 8-token
// groups, each group as its 128-byte chunks of the row, each chunk an 8 x 128 B
// swizzle atom: token t's chunk c sits at (t / 8) * kGroupBytes + c * 1 KB +
// (t % 8) * 128.  Every chunk is then a K-major (or MN-major) 128-byte-swizzled
// operand over 128 tokens whose 8-row groups are kGroupBytes apart.
//   bf16: 128-token tiles, 64 KB stages, groups of 4 KB: chunks K 0-63 (later P^T),
//         K 64-127, V 0-63, V 64-127
//   fp8:  groups of 2 KB: chunks K codes (later P^T), V codes.  A tile is 256 tokens
//         (64 KB, two 128-token halves 32 KB apart), so the softmax's fixed cost per tile
//         is spread over as many bytes as a bf16 tile.
template <int RP, bool FP8>
struct Cfg {
    static_assert(RP == 16 || RP == 32 || RP == 64, "rows per work item: 16, 32 or 64");
    static constexpr int kQBytes = 2 * RP * 128;            // bf16: two 64-column chunks; fp8: hi and lo terms
    static constexpr int kMiscBytes = 8192;
    // Softmax warpgroups splitting the query rows: two, or four for fp8 with 64 rows, so
    // that every softmax thread holds at most 16 rows of a 256-token fp8 tile's two tokens
    static constexpr int kGroups = (FP8 && RP == 64) ? 4 : 2;
    static constexpr int kSoftmaxWarps = 4 * kGroups;
    static constexpr int kPvWarp = kSoftmaxWarp0 + kSoftmaxWarps;   // issues the PV products
    static constexpr int kThreads = 32 * (kPvWarp + 1);      // 352, or 608
    static constexpr int kRH = RP / kGroups;                  // rows per softmax warpgroup
    static constexpr int kTile = FP8 ? 256 : 128;             // tokens per tile
    static constexpr int kHalves = kTile / kTokTile;          // 128-token MMAs per tile
    static constexpr int kPagesPerTile = kTile / kPage;       // TMA copies per tile (<= 32 lanes)
    static constexpr int kStageBytes = kTile * (FP8 ? 256 : 512);
    // S^T buffers in TMEM: QK may run this many tiles ahead of the softmax (fp8 with 64 rows:
    // one, since a stacked S buffer of a 256-token tile is 256 columns)
    static constexpr int kSBufs = kHalves == 2 ? (RP == 64 ? 1 : 2) : 4;
    static constexpr int kStagesFit = (kMaxSmem - kQBytes - kMiscBytes) / kStageBytes;
    static constexpr int kStages = kStagesFit < 6 ? kStagesFit : 6;
    static constexpr int kOffQ = kStages * kStageBytes;
    static constexpr int kOffMisc = kOffQ + kQBytes;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes;
    // fp8: Q's hi and lo terms are one operand of 2*RP rows, so one product per 32 dimensions
    // gives S_hi | S_lo side by side (K read once), summed by the softmax.  (With 64 rows as two
    // products into one S, each tile took 16 products reading K twice: 183.6 -> 175.1 us on a
    // 16 x 119k verify batch with the stacked operand.)
    static constexpr bool kStackQ = FP8;
    static constexpr int kSCols = kStackQ ? 2 * RP : RP;     // TMEM columns of one S buffer
    static constexpr int kOCols = FP8 ? 2 * RP : RP;         // O^T, or O_hi^T | O_lo^T
    static constexpr int kSBufCols = kHalves * kSCols;       // one S buffer: a tile's halves side by side
    static constexpr int kTmemNeed = kSBufs * kSBufCols + kOCols;
    static constexpr int kTmemCols = kTmemNeed <= 128 ? 128 : kTmemNeed <= 256 ? 256 : 512;
    static_assert(kTmemNeed <= 512, "TMEM columns");
    static constexpr uint32_t kTxBytes = kStageBytes;        // bytes the TMA brings per stage
    static constexpr int kGroupBytes = FP8 ? 2048 : 4096;     // one 8-token group of the raw rows
    static constexpr int kPageBytes = 2 * kGroupBytes;        // one page (one TMA copy)
    // V^T operand: bf16 chunks 2-3 (two 64-dimension atoms 1 KB apart), fp8 chunk 1 (one atom)
    static constexpr int kOffV = FP8 ? 1024 : 2048;
    // Lazy running max: scores are exponentiated against the running max unless one beats it
    // by 2^kThrLog2.  fp8 P is formed as p * 2^kPShift <= 2^8, which keeps the small
    // probabilities clear of the e4m3 subnormals; the shift cancels in o / l and is undone
    // in the partials.
    static constexpr float kThrLog2 = FP8 ? 4.0f : 8.0f;
    static constexpr int kPShift = FP8 ? 4 : 0;
    static_assert(kPShift >= 0 && kPShift < 8, "P * 2^kPShift stays inside the e4m3 range");
    // misc area
    // Landing barriers per stage: one per 128-token half for e4m3 with up to 32 rows, where QK runs
    // ahead of the softmax (two S buffers) and so waits for copies: the first half's products go
    // out while the second half lands (draft-extend workload 194.0 -> 192.8 us per step).  With
    // 64 rows QK waits for the single S buffer instead, and a second check only cost time
    // (179.5 -> 182.9 us).
    static constexpr int kLand = (FP8 && RP <= 32) ? kHalves : 1;
    static constexpr int kBarFull = 0;                       // [kStages][kLand]: (a half of) the tile landed
    static constexpr int kBarEmpty = 8 * kStages * kLand;    // [kStages]
    static constexpr int kBarSFull = kBarEmpty + 8 * kStages; // [kSBufs]
    static constexpr int kBarSFree = kBarSFull + 8 * kSBufs; // [kSBufs]
    static constexpr int kBarPFull = kBarSFree + 8 * kSBufs; // [kStages], by stage
    static constexpr int kBarODone = kBarPFull + 8 * kStages; // committed once, after the last PV
    static constexpr int kTmemSlot = kBarODone + 8;
    static constexpr int kAbort = kTmemSlot + 4;
    static constexpr int kRed = 320;                         // float[group][4][32]
    static constexpr int kMrun = kRed + kGroups * 4 * 32 * 4;   // float[64] running max (log2 units)
    static constexpr int kMthr = kMrun + 64 * 4;             // float[64] running max + rescale threshold
    static constexpr int kMsub = kMthr + 64 * 4;             // float[64] running max - kPShift, -inf -> 0
    static constexpr int kAlpha = kMsub + 64 * 4;            // float[64]; reused for the final l
    static constexpr int kCrow = kAlpha + 64 * 4;            // float[64] per-row score scale (log2 units)
    static constexpr int kSlot = kCrow + 64 * 4;             // long long[64]: partial slot of each row
    static_assert(kStages >= 2, "shared memory");
    static_assert(kAbort + 4 <= kRed, "misc area");
    static_assert(kSlot + 64 * 8 <= kMiscBytes, "misc area");
    static_assert(kSmemBytes <= kMaxSmem, "shared memory");
    static_assert((kOffQ % 1024) == 0 && (kMrun % 16) == 0 && (kMthr % 16) == 0 && (kMsub % 16) == 0 &&
                      (kCrow % 16) == 0,
                  "operand and vector alignment");
};

// Sum (or max) of each of the N values across the 32 lanes of the warp.
// Each step sends half of the live values to the partner lane `OFF` away and
// keeps the other half, so after the steps lane l holds the result for row
// reduce_row0<N>(l) in v[0] (N <= 32).  All indices are compile-time.
template <int N, int OFF, bool MAX>
struct TransposeReduce {
    static __device__ __forceinline__ void run(float *v, int lane)
    {
        if constexpr (N >= 2) {
            const bool upper = (lane & OFF) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float send = upper ? v[i] : v[i + N / 2];
                const float keep = upper ? v[i + N / 2] : v[i];
                const float got = __shfl_xor_sync(kFull, send, OFF);
                v[i] = MAX ? fmaxf(keep, got) : keep + got;
            }
            if constexpr (OFF > 1)
                TransposeReduce<N / 2, OFF / 2, MAX>::run(v, lane);
        } else {
            const float got = __shfl_xor_sync(kFull, v[0], OFF);
            v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
            if constexpr (OFF > 1)
                TransposeReduce<1, OFF / 2, MAX>::run(v, lane);
        }
    }
};

template <int N, bool MAX>
__device__ __forceinline__ void warp_transpose_reduce(float (&v)[N], int lane)
{
    static_assert(N >= 1 && N <= 32, "at most one value per lane remains");
    TransposeReduce<N, 16, MAX>::run(v, lane);
}

template <int N>
__device__ __forceinline__ int reduce_row0(int lane)
{
    return lane / (32 / N);
}

// 2^x on the special-function unit, flushing subnormal results to zero; 2^-inf = 0.
__device__ __forceinline__ float ex2_ftz(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two floats to a packed pair (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two floats to packed e4m3 codes (lo in the low byte), nearest even, saturated to +-448.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packed e4m3 pair (low 16 bits) -> packed f16 pair (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v)
{
    uint32_t r;
    const uint16_t h = (uint16_t)(v & 0xFFFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
    return r;
}

// Low half of a packed f16 pair as float.
__device__ __forceinline__ float f16lo_to_float(uint32_t v)
{
    float f;
    const uint16_t h = (uint16_t)(v & 0xFFFFu);
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Two floats to a packed f16 pair (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t hmax2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// lo += low half of v, hi += high half of v (f16 added into fp32, one rounding each).
__device__ __forceinline__ void add_f16x2_to_f32(uint32_t v, float &lo, float &hi)
{
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tadd.rn.f32.f16 %0, a, %0;\n\tadd.rn.f32.f16 %1, b, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(v));
}

// 2^x of both halves on the special-function unit (half precision).
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x)
{
    uint32_t r;
    asm("ex2.approx.f16x2 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

// Whether either half of a packed f16 pair exceeds `thr`.
__device__ __forceinline__ bool f16x2_any_gt(uint32_t v, float thr)
{
    float lo, hi;
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(v));
    return fmaxf(lo, hi) > thr;
}

// Two packed f16 pairs to four e4m3 codes (a's low half in the low byte, then a's high
// half, b's low, b's high), nearest even, saturated to +-448.
__device__ __forceinline__ uint32_t e4m3x4_from_f16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f16x2 lo, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f16x2 hi, %2;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "r"(a), "r"(b));
    return r;
}

template <int RP, bool FP8>
__global__ void __launch_bounds__(Cfg<RP, FP8>::kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap kv_map, const AttnParams p)
{
    using C = Cfg<RP, FP8>;
    extern __shared__ __align__(1024) uint8_t smem[];

    wait_prior_grid();    // the plan, Q and the pages may come from the kernels before this one
    // the fixed split has no plan kernel to check that cu_seqlens_q covers [0, num_tokens)
    if (p.plan == nullptr && blockIdx.x == 0 && threadIdx.x == 0 &&
        (__ldg(p.cu_q) != 0 || __ldg(p.cu_q + p.bs) != p.num_tokens))
        atomicOr(p.status, SK_DEV_BAD_SEQ);
    // CTA b: row block b % row_blocks (neighbouring CTAs share a work item's pages, so
    // the later reads of a page find it in L2) of work item / KV head b / row_blocks.
    const int ih = blockIdx.x / p.row_blocks;
    const int rb = blockIdx.x - ih * p.row_blocks;
    const int item = ih / p.H_kv;
    const int h = ih - item * p.H_kv;
    WorkItem w;
    if (item >= p.num_items || !decode_work_item(p, item, w))
        return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R_all = p.G * w.q_len;                  // the item's rows, r = j * G + i
    const int row0 = rb * RP;                         // this CTA's first row
    const int R = R_all - row0 < RP ? R_all - row0 : RP;
    const uint32_t sbase = smem_u32(smem);
    if (R_all > p.row_blocks * RP || (sbase & 1023u) != 0) {
        if (threadIdx.x == 0 && rb == 0)
            atomicOr(p.status, R_all > p.row_blocks * RP ? SK_DEV_BAD_SEQ : SK_DEV_INTERNAL);
        return;
    }
    if (R <= 0)
        return;                                       // a row block past this item's rows

    uint8_t *misc = smem + C::kOffMisc;
    const uint32_t mbase = sbase + C::kOffMisc;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + C::kAbort);
    float *red = reinterpret_cast<float *>(misc + C::kRed);
    float *m_run = reinterpret_cast<float *>(misc + C::kMrun);
    float *m_thr = reinterpret_cast<float *>(misc + C::kMthr);
    float *m_sub = reinterpret_cast<float *>(misc + C::kMsub);
    float *alpha_s = reinterpret_cast<float *>(misc + C::kAlpha);
    float *crow = reinterpret_cast<float *>(misc + C::kCrow);
    auto bar_full = [&](int s, int hf) { return mbase + C::kBarFull + 8 * (s * C::kLand + hf); };
    auto bar_empty = [&](int s) { return mbase + C::kBarEmpty + 8 * s; };
    auto bar_sfull = [&](int b) { return mbase + C::kBarSFull + 8 * b; };
    auto bar_sfree = [&](int b) { return mbase + C::kBarSFree + 8 * b; };
    auto bar_pfull = [&](int b) { return mbase + C::kBarPFull + 8 * b; };
    const uint32_t bar_odone = mbase + C::kBarODone;
    const uint32_t q_s = sbase + C::kOffQ;
    auto stage = [&](int s) { return sbase + (uint32_t)(s * C::kStageBytes); };

    const int k0 = w.k0, k1 = w.k1;
    const int ntiles = k1 > k0 ? (k1 - k0 + C::kTile - 1) / C::kTile : 0;

    // ---- set-up: barriers, TMEM, Q in shared memory (K-major, 128-byte swizzle)
    // Q is read into registers before the producer starts, so that its loads are not queued
    // behind every CTA's first copies.
    constexpr uint32_t kSetupBar = 8;          // ids 1..kGroups belong to the softmax groups
    constexpr int kSetupThreads = C::kThreads - 32;
    const int st_tid = threadIdx.x - 32;
    constexpr int kQUnits = FP8 ? (RP + kSetupThreads / 32 - 1) / (kSetupThreads / 32)   // rows per warp
                                : (RP * 16 + kSetupThreads - 1) / kSetupThreads;         // 16-byte units per thread
    uint4 qpre[FP8 ? 1 : kQUnits];
    uint2 qraw[FP8 ? kQUnits : 1];
    if (warp != 0) {
        if constexpr (!FP8) {
#pragma unroll
            for (int k = 0; k < kQUnits; ++k) {
                const int u = st_tid + k * kSetupThreads, r = u >> 4, unit = u & 15;
                qpre[k] = make_uint4(0u, 0u, 0u, 0u);
                if (u < RP * 16 && r < R) {
                    const int j = (row0 + r) / p.G, i = row0 + r - j * p.G;
                    const uint16_t *src = p.q + ((long long)(w.tok0 + j) * p.H_q + h * p.G + i) * kHeadDim + unit * 8;
                    qpre[k] = __ldg(reinterpret_cast<const uint4 *>(src));
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < kQUnits; ++k) {
                const int r = warp - 1 + k * (kSetupThreads / 32);
                qraw[k] = make_uint2(0u, 0u);
                if (r < R) {
                    const int j = (row0 + r) / p.G, i = row0 + r - j * p.G;
                    qraw[k] = __ldg(reinterpret_cast<const uint2 *>(
                        p.q + ((long long)(w.tok0 + j) * p.H_q + h * p.G + i) * kHeadDim + lane * 4));
                }
            }
        }
    }
    // The producer's block ids for the first kStages tiles (one page per lane), read before the
    // barriers are set up; later it keeps them a full ring of tiles ahead: q_blk[s] belongs to
    // tile j + s, so the first copies go out back to back.
    int q_blk[C::kStages];
    if (warp == 0) {
        const int pg0 = k0 / kPage, pge = (k1 + kPage - 1) / kPage;
        const int32_t *btr = p.block_table + (long long)w.s * p.bt_stride;
#pragma unroll
        for (int s2 = 0; s2 < C::kStages; ++s2) {
            const int pg = pg0 + s2 * C::kPagesPerTile + lane;
            q_blk[s2] = (lane < C::kPagesPerTile && s2 < ntiles && pg < pge) ? __ldg(btr + pg) : -1;
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            for (int hf = 0; hf < C::kLand; ++hf)
                mbar_init(bar_full(s, hf), 1);
            mbar_init(bar_empty(s), 1);
            mbar_init(bar_pfull(s), C::kSoftmaxWarps);
        }
        for (int b = 0; b < C::kSBufs; ++b) {
            mbar_init(bar_sfull(b), 1);
            mbar_init(bar_sfree(b), C::kSoftmaxWarps);
        }
        mbar_init(bar_odone, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();   // barriers initialised: the producer starts its copies now
    // The other warps set up TMEM and Q meanwhile, then meet at a barrier of their own.
    if (warp != 0) {
        if (warp == 1) {
            tmem_alloc(mbase + C::kTmemSlot, C::kTmemCols);
            tmem_relinquish();
        }
        if constexpr (!FP8) {
#pragma unroll
            for (int k = 0; k < kQUnits; ++k) {
                const int u = st_tid + k * kSetupThreads, r = u >> 4, unit = u & 15;
                const int chunk = unit >> 3, uu = unit & 7;
                if (u < RP * 16)
                    st_shared_v4(q_s + chunk * (RP * 128) + r * 128 + ((uu ^ (r & 7)) << 4), qpre[k].x, qpre[k].y,
                                 qpre[k].z, qpre[k].w);
            }
            for (int r = st_tid; r < RP; r += kSetupThreads)
                crow[r] = p.score_scale_log2;
        } else {
            // Row r of Q scaled by 2^e (max |q| lands in [128, 256)), as two e4m3 terms hi + lo.
            // One warp per row; lane l owns dimensions 4l..4l+3.
#pragma unroll
            for (int k = 0; k < kQUnits; ++k) {
                const int r = warp - 1 + k * (kSetupThreads / 32);
                if (r >= RP)
                    break;
                const uint2 raw = qraw[k];                   // zeros past the item's rows
                float qv[4];
                qv[0] = __uint_as_float(raw.x << 16);
                qv[1] = __uint_as_float(raw.x & 0xFFFF0000u);
                qv[2] = __uint_as_float(raw.y << 16);
                qv[3] = __uint_as_float(raw.y & 0xFFFF0000u);
                float amax = fmaxf(fmaxf(fabsf(qv[0]), fabsf(qv[1])), fmaxf(fabsf(qv[2]), fabsf(qv[3])));
                for (int o = 16; o > 0; o >>= 1)
                    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
                int e = 0;
                if (amax > 0.f && amax < CUDART_INF_F) {
                    int ex;
                    frexpf(amax, &ex);               // amax in [2^(ex-1), 2^ex)
                    e = 8 - ex;                      // amax * 2^e in [128, 256)
                    e = e > 100 ? 100 : (e < -100 ? -100 : e);
                }
                float lo[4];
                uint32_t hcodes = 0;
#pragma unroll
                for (int k = 0; k < 4; k += 2) {
                    const float x0 = ldexpf(qv[k], e), x1 = ldexpf(qv[k + 1], e);
                    const uint32_t hc = pack_e4m3x2(x0, x1);
                    const uint32_t hf = e4m3x2_to_f16x2(hc);              // the hi terms back, exactly
                    lo[k] = x0 - f16lo_to_float(hf);
                    lo[k + 1] = x1 - f16lo_to_float(hf >> 16);
                    hcodes |= (hc & 0xFFFFu) << (8 * k);
                }
                const uint32_t lcodes = (pack_e4m3x2(lo[0], lo[1]) & 0xFFFFu) | ((pack_e4m3x2(lo[2], lo[3]) & 0xFFFFu) << 16);
                // byte offset of dims 4l..4l+3 in the swizzled 128-byte row: 16-byte unit l/4, 4 bytes at (l%4)*4
                const uint32_t off = (uint32_t)(r * 128 + ((((lane >> 2) ^ (r & 7)) << 4) | ((lane & 3) << 2)));
                *reinterpret_cast<uint32_t *>(smem + C::kOffQ + off) = hcodes;
                *reinterpret_cast<uint32_t *>(smem + C::kOffQ + RP * 128 + off) = lcodes;
                if (lane == 0)
                    crow[r] = p.score_scale_log2 * ldexpf(1.f, -e);
            }
        }
        for (int r = st_tid; r < RP; r += kSetupThreads) {
            long long slot = -1;
            if (r < R) {
                const int jq = (row0 + r) / p.G, i = row0 + r - jq * p.G;
                slot = (long long)(w.tok0 + jq) * p.seg_max * p.H_q + (long long)w.g * p.H_q + h * p.G + i;
            }
            reinterpret_cast<long long *>(misc + C::kSlot)[r] = slot;
            m_run[r] = -CUDART_INF_F;
            m_thr[r] = -CUDART_INF_F;
            m_sub[r] = FP8 ? kMsubNone : 0.f;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(kSetupBar, kSetupThreads);
        tc_fence_after();
    }
    const uint32_t tmem = warp != 0 ? *reinterpret_cast<volatile uint32_t *>(misc + C::kTmemSlot) : 0u;
    const uint32_t tmem_s0 = tmem, tmem_o = tmem + C::kSBufs * C::kSBufCols;

    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0)
            prefetch_tensormap(&kv_map);
        const int page0 = k0 / kPage;
        const int page_end = (k1 + kPage - 1) / kPage;
        const int32_t *bt_row = p.block_table + (long long)w.s * p.bt_stride;
        int issued = 0;
        bool ok = true;
        for (int j = 0; j < ntiles && ok; ++j) {
            const int st = j % C::kStages;
            if (j >= C::kStages)
                ok = mbar_wait_bounded(bar_empty(st), ((j / C::kStages) - 1) & 1, abort_flag, p.wait_limit);
            ok = __all_sync(kFull, ok);
            if (!ok)
                break;
            const int blk = q_blk[0];
            const int pg = page0 + j * C::kPagesPerTile + lane;
            const int pg_far = pg + C::kStages * C::kPagesPerTile;     // tile j + kStages
#pragma unroll
            for (int s2 = 0; s2 + 1 < C::kStages; ++s2)
                q_blk[s2] = q_blk[s2 + 1];
            q_blk[C::kStages - 1] = (lane < C::kPagesPerTile && j + C::kStages < ntiles && pg_far < page_end)
                                        ? __ldg(bt_row + pg_far) : -1;
            if (lane == 0)
                for (int hf = 0; hf < C::kLand; ++hf)
                    mbar_arrive_expect_tx(bar_full(st, hf), C::kTxBytes / C::kLand);
            __syncwarp();
            if (lane < C::kPagesPerTile) {
                int grp = -2;                         // whole box out of bounds: zero fill
                if (pg < page_end) {
                    if (blk >= 0 && blk < p.num_blocks)
                        grp = (blk * p.H_kv + h) * 2;
                    else
                        atomicOr(p.status, SK_DEV_BAD_BLOCK);
                }
                tma_load_4d(stage(st) + lane * C::kPageBytes, &kv_map, 0, 0, 0, grp,
                            bar_full(st, lane / (C::kPagesPerTile / C::kLand)));
                // bf16: tile j + 1 goes to L2 now, so that its copy into a stage, which waits for a
                // stage to free, mostly hits L2 (one tile more in flight than the stages hold).
                // (fp8's 256-token tiles were measured slower with it: 198 -> 208 us on a 1.19 GB batch.)
                if constexpr (!FP8) {
                    const int pg1 = pg + C::kPagesPerTile;
                    const int blk1 = q_blk[0];                 // tile j + 1 (the ring has moved on)
                    if (j + 1 >= C::kStages && j + 1 < ntiles && pg1 < page_end && blk1 >= 0 && blk1 < p.num_blocks)
                        tma_prefetch_l2_4d(&kv_map, 0, 0, 0, (blk1 * p.H_kv + h) * 2);
                }
            }
            issued = j + 1;
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0)
                atomicOr(p.status, SK_DEV_TIMEOUT);
        }
        // Every copy issued lands before the CTA exits, even when a consumer gave up before
        // waiting for it.  Tiles before issued - kStages were consumed before their stage was
        // reused; each of the last kStages tiles is the last phase its barrier will see, so these
        // waits are unambiguous and return at once when the consumers already saw them land.
        for (int t = issued > C::kStages ? issued - C::kStages : 0; t < issued; ++t)
            for (int hf = 0; hf < C::kLand; ++hf)
                mbar_wait_bounded(bar_full(t % C::kStages, hf), (t / C::kStages) & 1, nullptr, kDrainLimit);
    } else if (warp == 1 || warp == C::kPvWarp) {
        // ================================================================ MMA issuers
        // Whole warps run these loops; one elected lane issues each MMA and commit.
        // QK: bf16 kind::f16, 8 steps of 16 dims; fp8 kind::f8f6f4, 4 steps of 32 dims, on the
        // stacked hi|lo Q (up to 32 rows) or once per Q term.
        // PV: V^T (MN-major) x P^T (MN-major): bf16 kind::f16, 8 steps of 16 tokens; fp8
        // kind::f8f6f4 on the V codes and the stacked hi|lo P, 4 steps of 32 tokens.
        // Descriptors are built once for stage 0 / Q; an operand elsewhere is the same descriptor
        // advanced by (byte offset >> 4) in its start-address field (shared addresses < 256 KB).
        constexpr uint32_t idesc_qk = FP8 ? idesc_e4m3_f32(kTokTile, C::kSCols, 0, 0) : idesc_bf16_f32(kTokTile, RP, 0, 0);
        constexpr uint32_t idesc_pv = FP8 ? idesc_e4m3_f32(kTokTile, C::kOCols, 1, 1) : idesc_bf16_f32(kTokTile, RP, 1, 1);
        const uint64_t d_kv0 = smem_desc_sw128(stage(0), 16, C::kGroupBytes);           // K-major K tile
        const uint64_t d_v0 = smem_desc_sw128(stage(0) + C::kOffV, 1024, C::kGroupBytes); // MN-major V^T
        const uint64_t d_p0 = smem_desc_sw128(stage(0), 1024, C::kGroupBytes);          // MN-major P^T
        const uint64_t d_q0 = smem_desc_sw128(q_s, 16, 1024);                          // K-major Q
        auto adv = [](uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); };
        bool ok = true;
        int last = -1;
        if (warp == 1) {
            // QK(j) once tile j has landed and its S buffer (j % kSBufs) is free.  The buffer's
            // condition is checked first, while tile j is still in flight, so that once it lands
            // only its own wait stands before the products (an mbarrier check can take hundreds
            // of cycles while the softmax warps keep shared memory busy).  P_full is indexed by
            // stage, so it cannot run ahead of its PV: tile j + kStages reuses the stage only after
            // PV(j) has completed.
            for (int j = 0; j < ntiles && ok; ++j) {
                const int st = j % C::kStages, b = j % C::kSBufs;
                if (j >= C::kSBufs)
                    ok = mbar_wait_bounded(bar_sfree(b), ((j / C::kSBufs) - 1) & 1, abort_flag, p.wait_limit);
                if constexpr (C::kLand == 1) {
                    if (ok)
                        ok = mbar_wait_bounded(bar_full(st, 0), (j / C::kStages) & 1, abort_flag, p.wait_limit);
                }
                ok = __all_sync(kFull, ok);
                if (!ok)
                    break;
                if constexpr (C::kLand == 1)
                    tc_fence_after();
#pragma unroll
                for (int hf = 0; hf < C::kHalves && ok; ++hf) {
                    // half hf: tokens [128 hf, 128 hf + 128) of the tile, 16 groups further on; with a
                    // landing barrier per half, its products go out as soon as its pages have landed
                    if constexpr (C::kLand > 1) {
                        ok = __all_sync(kFull, mbar_wait_bounded(bar_full(st, hf), (j / C::kStages) & 1, abort_flag,
                                                                 p.wait_limit));
                        if (!ok)
                            break;
                        tc_fence_after();
                    }
                    const uint32_t so = (uint32_t)(st * C::kStageBytes + hf * 16 * C::kGroupBytes);
                    const uint32_t sd = tmem_s0 + b * C::kSBufCols + hf * C::kSCols;
                    if constexpr (C::kStackQ) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_f8_ss_warp(sd, adv(d_kv0, so + k * 32), adv(d_q0, k * 32), idesc_qk, k > 0 ? 1u : 0u);
                    } else if constexpr (FP8) {
#pragma unroll
                        for (int t = 0; t < 2; ++t)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_f8_ss_warp(sd, adv(d_kv0, so + k * 32), adv(d_q0, t * (RP * 128) + k * 32), idesc_qk,
                                               (t > 0 || k > 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int k = 0; k < kHeadDim / 16; ++k) {
                            const uint32_t off = (uint32_t)((k >> 2) * 1024 + (k & 3) * 32);
                            const uint32_t qoff = (uint32_t)((k >> 2) * (RP * 128) + (k & 3) * 32);
                            mma_f16_ss_warp(sd, adv(d_kv0, so + off), adv(d_q0, qoff), idesc_qk, k > 0 ? 1u : 0u);
                        }
                    }
                }
                mma_commit_warp(bar_sfull(b));
                last = j;
            }
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    atomicOr(p.status, SK_DEV_TIMEOUT);
                }
            }
            // this warp's products finish before TMEM is freed, also when the softmax gave up
            // before consuming them (QK(last) is the last commit sfull[last % kSBufs] sees)
            if (last >= 0)
                mbar_wait_bounded(bar_sfull(last % C::kSBufs), (last / C::kSBufs) & 1, nullptr, kDrainLimit);
        } else {
            // PV(i) as soon as the softmax threads have written P(i).  Its completion frees the
            // stage (empty), which is also how the softmax learns that O holds tile i.
            for (int i = 0; i < ntiles && ok; ++i) {
                ok = mbar_wait_bounded(bar_pfull(i % C::kStages), (i / C::kStages) & 1, abort_flag, p.wait_limit);
                ok = __all_sync(kFull, ok);
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t so = (uint32_t)((i % C::kStages) * C::kStageBytes);    // P^T over the dead K area
                if constexpr (FP8) {
#pragma unroll
                    for (int k = 0; k < C::kTile / 32; ++k)
                        mma_f8_ss_warp(tmem_o, adv(d_v0, so + k * 4 * C::kGroupBytes), adv(d_p0, so + k * 4 * C::kGroupBytes),
                                       idesc_pv, (i > 0 || k > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_f16_ss_warp(tmem_o, adv(d_v0, so + k * 2 * C::kGroupBytes), adv(d_p0, so + k * 2 * C::kGroupBytes),
                                        idesc_pv, (i > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit_warp(bar_empty(i % C::kStages));
                last = i;
            }
            if (last >= 0)
                mma_commit_warp(bar_odone);   // completes once every PV issued has completed
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    atomicOr(p.status, SK_DEV_TIMEOUT);
                }
            }
            // every PV completes before TMEM is freed, also when the softmax gave up waiting
            if (last >= 0)
                mbar_wait_bounded(bar_odone, 0, nullptr, kDrainLimit);
        }
        __syncwarp();
    } else if constexpr (FP8) {
        // ================================================================ softmax warpgroups, e4m3 pages
        // Group g owns query rows [g*RH, (g+1)*RH) and each thread the two tokens tau and 128 + tau
        // of the tile (its TMEM lane in each half).  Per score the work is kept to a few
        // instructions, since with 64 rows this path is bound by instruction issue:
        //   d = s * c_r - msub_r      one FFMA (c_r: the row's score scale in log2 units, Q's
        //                             power-of-two row scale included; msub_r: its running max
        //                             less kPShift), packed in pairs to f16;
        //   rescale vote              one packed max per pair: the running max moves only when
        //                             some d exceeds kThrLog2 + kPShift (p would pass 2^8);
        //   p * 2^kPShift = 2^d       one ex2.approx.f16x2 per pair;
        //   hi, lo                    hi = p with 3 fraction bits (a mask), lo = p - hi (exact
        //                             in f16), each then one e4m3 code: p = hi + lo within 2^-8;
        //   row sums                  the two tokens' p of a row pair added in f16 (one packed
        //                             add per two pairs), then added into the fp32 sums by two
        //                             mixed-precision adds.
        // The f16 exponential's own error (about 2^-10) is below the split's.  (Row sums taken on
        // the tensor cores instead, as ones . P^T beside O, cost more than they saved: the
        // extra products lengthened every stage's life.)
        constexpr int RH = C::kRH;
        constexpr int NH = C::kHalves;
        constexpr int NP = RH / 2;                             // f16 pairs of rows per half
        constexpr int kLd = RH >= 32 ? 32 : RH;                // TMEM columns per load
        static_assert(kLd % 4 == 0 && RH % 8 == 0, "the epilogue transposes blocks of four rows");
        const int wg = (warp - kSoftmaxWarp0) >> 2;            // softmax group
        const int tw = (warp - kSoftmaxWarp0) & 3;             // warp within the group
        const int r0 = wg * RH;                                // first row of the group
        const uint32_t bar_id = 1 + wg;                        // named barrier of the group
        const int quarter = warp & 3;                          // TMEM lane quarter this warp may access
        const int tau = quarter * 32 + lane;                   // token row (S) / dimension (O) of this thread
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int tid = tw * 32 + lane;
        const int causal_base = w.L - w.q_len;
        const int last_page_end = (w.L + kPage - 1) / kPage * kPage;
        bool failed = false;
        float *gred = red + wg * (4 * 32);
        float lsum[RH];
#pragma unroll
        for (int r = 0; r < RH; ++r)
            lsum[r] = 0.f;

        // S of this thread's tokens (the stacked hi | lo Q terms summed)
        auto load_scores = [&](int sb, float (&x)[NH][RH]) {
#pragma unroll
            for (int hf = 0; hf < NH; ++hf) {
                const uint32_t s_col = tmem_s0 + sb * C::kSBufCols + hf * C::kSCols + r0 + lane_off;
#pragma unroll
                for (int c = 0; c < RH; c += kLd)
                    tmem_ld32<kLd>(s_col + c, x[hf] + c);
                if constexpr (C::kStackQ) {
                    // S_hi | S_lo side by side: one half's lo columns at a time keeps registers low
                    float y[RH];
#pragma unroll
                    for (int c = 0; c < RH; c += kLd)
                        tmem_ld32<kLd>(s_col + RP + c, y + c);
                    tmem_wait_ld();
#pragma unroll
                    for (int r = 0; r < RH; ++r)
                        x[hf][r] += y[r];
                }
            }
            if constexpr (!C::kStackQ)
                tmem_wait_ld();
        };
        // -inf where row r = j' * G + i does not see this thread's key of half hf (past the
        // segment end, or causally ahead of query token j'); whole tiles inside both limits
        // keep their scores (padding rows r >= R have zero Q: scores 0, never written out)
        auto mask_scores = [&](int j, bool ok, float (&x)[NH][RH]) {
#pragma unroll
            for (int hf = 0; hf < NH; ++hf) {
                const int tok = k0 + j * C::kTile + hf * kTokTile + tau;
                const int ahead = tok - causal_base;
                const int rmin = ((p.causal && ahead > 0) ? ahead * p.G : 0) - row0;
                if (!(ok && tok < k1 && rmin <= 0)) {
                    const bool tok_vis = ok && tok < k1;
#pragma unroll
                    for (int r = 0; r < RH; ++r) {
                        const int rg = r0 + r;
                        x[hf][r] = (tok_vis && rg >= rmin && rg < R) ? x[hf][r] : -CUDART_INF_F;
                    }
                }
            }
        };
        // d = s * c - msub in f16 pairs; returns whether some d passes the rescale threshold
        auto make_d = [&](const float (&x)[NH][RH], uint32_t (&dh)[NH][NP]) {
            uint32_t dmax = 0xFC00FC00u;                       // (-inf, -inf)
#pragma unroll
            for (int r = 0; r < RH; r += 4) {
                const float4 c = *reinterpret_cast<const float4 *>(crow + r0 + r);
                const float4 m = *reinterpret_cast<const float4 *>(m_sub + r0 + r);
#pragma unroll
                for (int hf = 0; hf < NH; ++hf) {
                    const uint32_t a = pack_f16x2(fmaf(x[hf][r], c.x, -m.x), fmaf(x[hf][r + 1], c.y, -m.y));
                    const uint32_t b = pack_f16x2(fmaf(x[hf][r + 2], c.z, -m.z), fmaf(x[hf][r + 3], c.w, -m.w));
                    dh[hf][r / 2] = a;
                    dh[hf][r / 2 + 1] = b;
                    dmax = hmax2(dmax, hmax2(a, b));
                }
            }
            return f16x2_any_gt(dmax, C::kThrLog2 + (float)C::kPShift);
        };

        for (int j = 0; j < ntiles; ++j) {
            const int sb = j % C::kSBufs;          // S buffer and its barriers
            const int st = j % C::kStages;
            float x[NH][RH];
            uint32_t dh[NH][NP];
            bool ok = !failed && mbar_wait_bounded(bar_sfull(sb), (j / C::kSBufs) & 1, abort_flag, p.wait_limit);
            ok = __all_sync(kFull, ok);          // tcgen05.ld is warp-collective
            if (ok) {
                tc_fence_after();
                load_scores(sb, x);
            }
            mask_scores(j, ok, x);
            const bool big = make_d(x, dh);
            // group decision, one reduction over the group's 128 threads: rescale needed or a wait
            // failed?  Only then a second one tells which (every thread gets the same answers).
            // The S buffer is released after it, so that the rare rescale can read S again.
            if (named_bar_or(bar_id, 128, big || !ok)) {
                if (named_bar_or(bar_id, 128, !ok)) {
                    if (tid == 0) {
                        *abort_flag = 1;
                        atomicOr(p.status, SK_DEV_TIMEOUT);
                    }
                    failed = true;
                    break;
                }
                tc_fence_after();
                load_scores(sb, x);                // S again: no score stayed live through make_d
                mask_scores(j, true, x);
                // exact tile max of s * c over the group's rows across its 128 threads (c > 0)
                constexpr int kRc = RH >= 32 ? 32 : RH;
#pragma unroll
                for (int c0 = 0; c0 < RH; c0 += kRc) {
                    float v[kRc];
#pragma unroll
                    for (int r = 0; r < kRc; ++r) {
                        float mx = x[0][c0 + r];
#pragma unroll
                        for (int hf = 1; hf < NH; ++hf)
                            mx = fmaxf(mx, x[hf][c0 + r]);
                        v[r] = mx * crow[r0 + c0 + r];
                    }
                    warp_transpose_reduce<kRc, true>(v, lane);
                    gred[tw * 32 + c0 + reduce_row0<kRc>(lane)] = v[0];
                }
                named_bar_sync(bar_id, 128);
                if (tid < RH) {
                    const int rg = r0 + tid;
                    const float mt = fmaxf(fmaxf(gred[tid], gred[32 + tid]), fmaxf(gred[64 + tid], gred[96 + tid]));
                    const float mo = m_run[rg];
                    const float mn = fmaxf(mo, mt);
                    alpha_s[rg] = (mo == -CUDART_INF_F) ? 0.f : exp2f(mo - mn);
                    m_run[rg] = mn;
                    m_sub[rg] = mn == -CUDART_INF_F ? kMsubNone : mn - (float)C::kPShift;
                }
                named_bar_sync(bar_id, 128);
#pragma unroll
                for (int r = 0; r < RH; ++r)
                    lsum[r] *= alpha_s[r0 + r];
                if (j > 0) {
                    // O holds tiles < j: wait for PV(j-1) (the same argument as for bf16 makes its
                    // phase of empty[(j-1) % kStages] unambiguous), then rescale this thread's
                    // dimension of O_hi and O_lo
                    const int jp = j - 1;
                    bool okp = mbar_wait_bounded(bar_empty(jp % C::kStages), (jp / C::kStages) & 1, abort_flag, p.wait_limit);
                    okp = __all_sync(kFull, okp);    // tcgen05.ld/st are warp-collective
                    if (okp) {
                        tc_fence_after();
#pragma unroll
                        for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
                            for (int c = 0; c < RH; c += kLd) {
                                float o[kLd];
                                const uint32_t col = tmem_o + blk * RP + r0 + c + lane_off;
                                tmem_ld32<kLd>(col, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int r = 0; r < kLd; ++r)
                                    o[r] *= alpha_s[r0 + c + r];
                                tmem_st32<kLd>(col, o);
                            }
                        }
                        tmem_wait_st();
                    } else {
                        failed = true;             // the next tile's vote takes the group out together
                    }
                }
                // against the new running max (every d <= kPShift); S is read once more, so that
                // no score stays live through the reductions and the O rescale above
                tc_fence_after();
                load_scores(sb, x);
                mask_scores(j, true, x);
                make_d(x, dh);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_sfree(sb));
            if (!failed) {
                // P^T over the tile's K codes, which QK(j) no longer needs: MN-major, 128-byte
                // swizzle, 16-byte unit u of token row t stored at u ^ (t % 8); row r's hi code at
                // byte r, its lo code at byte RP + r
#pragma unroll
                for (int hf = 0; hf < NH; ++hf) {
                    const int t = hf * kTokTile + tau;          // token of the tile
                    const uint32_t prow = stage(st) + (uint32_t)((t >> 3) * C::kGroupBytes + (t & 7) * 128);
#pragma unroll
                    for (int u0 = 0; u0 < RH / 8; u0 += 2) {
                        // 16 rows (8 when RH is 8): p, the row sums, the two terms' codes
                        constexpr int kU = RH >= 16 ? 2 : 1;
                        uint32_t hw[2 * kU], lw[2 * kU];
#pragma unroll
                        for (int v = 0; v < 2 * kU; ++v) {
                            const int k = 4 * u0 + 2 * v;              // first pair: rows 2k, 2k + 1
                            const uint32_t p0 = ex2_f16x2(dh[hf][k]), p1 = ex2_f16x2(dh[hf][k + 1]);
                            add_f16x2_to_f32(p0, lsum[2 * k], lsum[2 * k + 1]);
                            add_f16x2_to_f32(p1, lsum[2 * k + 2], lsum[2 * k + 3]);
                            const uint32_t h0 = p0 & 0xFF80FF80u, h1 = p1 & 0xFF80FF80u;
                            hw[v] = e4m3x4_from_f16x2(h0, h1);
                            lw[v] = e4m3x4_from_f16x2(hsub2(p0, h0), hsub2(p1, h1));
                        }
                        if constexpr (kU == 2) {
                            // 16 rows' codes leave as one 16-byte store per term
                            const int bh = r0 + 8 * u0, bl = RP + bh;      // multiples of 16
                            st_shared_v4(prow + (uint32_t)(((bh >> 4) ^ (t & 7)) << 4), hw[0], hw[1], hw[2], hw[3]);
                            st_shared_v4(prow + (uint32_t)(((bl >> 4) ^ (t & 7)) << 4), lw[0], lw[1], lw[2], lw[3]);
                        } else {
                            const int bh = r0 + 8 * u0, bl = RP + r0 + 8 * u0;   // byte of the first row
                            *reinterpret_cast<uint2 *>(smem + (prow - sbase) + (((bh >> 4) ^ (t & 7)) << 4) + (bh & 15)) =
                                make_uint2(hw[0], hw[1]);
                            *reinterpret_cast<uint2 *>(smem + (prow - sbase) + (((bl >> 4) ^ (t & 7)) << 4) + (bl & 15)) =
                                make_uint2(lw[0], lw[1]);
                        }
                    }
                }
#pragma unroll
                for (int hf = 0; hf < NH; ++hf) {
                    const int t = hf * kTokTile + tau;
                    const int tok = k0 + j * C::kTile + t;
                    if (tok >= w.L && tok < last_page_end) {
                        // past L in the last page the row holds anything (0 * NaN would reach O): this
                        // group's share of the token's 128 V code bytes becomes zeros
                        constexpr int kZeroBytes = 128 / C::kGroups;
                        uint8_t *vrow = smem + st * C::kStageBytes + C::kOffV + (t >> 3) * C::kGroupBytes + (t & 7) * 128 +
                                        wg * kZeroBytes;
#pragma unroll
                        for (int u = 0; u < kZeroBytes / 16; ++u)
                            *reinterpret_cast<uint4 *>(vrow + u * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_pfull(st));
            if (failed && lane == 0)
                *abort_flag = 1;                   // the next tile's vote propagates the failure
        }

        // ---- epilogue: row sums across the group's threads (they do not need the last PV, which
        // completes meanwhile), then O complete? and the partials
        {
            constexpr int kRc = RH >= 32 ? 32 : RH;
#pragma unroll
            for (int c0 = 0; c0 < RH; c0 += kRc) {
                float v[kRc];
#pragma unroll
                for (int r = 0; r < kRc; ++r)
                    v[r] = lsum[c0 + r];
                warp_transpose_reduce<kRc, false>(v, lane);
                gred[tw * 32 + c0 + reduce_row0<kRc>(lane)] = v[0];
            }
        }
        named_bar_sync(bar_id, 128);
        if (tid < RH)
            alpha_s[r0 + tid] = (gred[tid] + gred[32 + tid]) + (gred[64 + tid] + gred[96 + tid]);
        bool okf = !failed;
        if (okf && ntiles > 0)
            okf = mbar_wait_bounded(bar_odone, 0, abort_flag, p.wait_limit);
        // the group's verdict; the barrier also publishes the row sums written above
        const bool write = !named_bar_or(bar_id, 128, !okf);
        if (write) {
            if (ntiles > 0)
                tc_fence_after();
            const float o_scale = p.v_scale * (1.0f / (float)(1 << C::kPShift));
            const long long *slots = reinterpret_cast<const long long *>(misc + C::kSlot);
#pragma unroll
            for (int c = 0; c < RH; c += kLd) {
                float o[kLd];
                if (ntiles > 0) {
                    float o2[kLd];
                    tmem_ld32<kLd>(tmem_o + r0 + c + lane_off, o);
                    tmem_ld32<kLd>(tmem_o + RP + r0 + c + lane_off, o2);
                    tmem_wait_ld();
#pragma unroll
                    for (int r = 0; r < kLd; ++r)
                        o[r] += o2[r];
                } else {
#pragma unroll
                    for (int r = 0; r < kLd; ++r)
                        o[r] = 0.f;
                }
#pragma unroll
                for (int rr = 0; rr < kLd; ++rr)
                    o[rr] = alpha_s[r0 + c + rr] > 0.f ? o[rr] * o_scale : 0.f;
                // 4 x 4 transposes within lane quads: lane 4a + b ends with row 4k + b of each block of
                // four rows and dimensions 4a .. 4a + 3 of the warp's quarter, so a warp store writes
                // four rows of 128 contiguous bytes, 16 bytes a lane (part_o is 16-byte aligned)
                const int qb = lane & 3;
                const bool qb0 = (qb & 1) != 0, qb1 = (qb & 2) != 0;
                const int dim4 = quarter * 32 + (lane & ~3);
#pragma unroll
                for (int k = 0; k < kLd / 4; ++k) {
                    const float x0 = o[4 * k], x1 = o[4 * k + 1], x2 = o[4 * k + 2], x3 = o[4 * k + 3];
                    const float own0 = qb1 ? x2 : x0, own1 = qb1 ? x3 : x1;
                    const float rc0 = __shfl_xor_sync(kFull, qb1 ? x0 : x2, 2);
                    const float rc1 = __shfl_xor_sync(kFull, qb1 ? x1 : x3, 2);
                    const float zl0 = qb1 ? rc0 : own0, zl1 = qb1 ? rc1 : own1;
                    const float zh0 = qb1 ? own0 : rc0, zh1 = qb1 ? own1 : rc1;
                    const float rl = __shfl_xor_sync(kFull, qb0 ? zl0 : zl1, 1);
                    const float rh = __shfl_xor_sync(kFull, qb0 ? zh0 : zh1, 1);
                    const float kl = qb0 ? zl1 : zl0, kh = qb0 ? zh1 : zh0;
                    const float4 y = make_float4(qb0 ? rl : kl, qb0 ? kl : rl, qb0 ? rh : kh, qb0 ? kh : rh);
                    const int r = r0 + c + 4 * k + qb;
                    if (r < R)
                        *reinterpret_cast<float4 *>(p.part_o + slots[r] * kHeadDim + dim4) = y;
                }
            }
            const int r = r0 + tid;
            if (tid < RH && r < R) {
                const long long slot = slots[r];
                const float l = alpha_s[r] * (1.0f / (float)(1 << C::kPShift));
                p.part_m[slot] = l > 0.f ? m_run[r] * 0.69314718055994531f : -CUDART_INF_F;
                p.part_l[slot] = l;
            }
        }
    } else {
        // ================================================================ softmax warpgroups, bf16 pages
        // Group g owns query rows [g*RH, (g+1)*RH): their S and O columns, running max, row
        // sums and P entries, so the two groups never wait for each other.
        constexpr int RH = C::kRH;
        constexpr int kLd = RH >= 32 ? 32 : RH;                // TMEM columns per load
        static_assert(kLd % 4 == 0, "the epilogue transposes blocks of four rows");
        const int wg = (warp - kSoftmaxWarp0) >> 2;            // softmax group
        const int tw = (warp - kSoftmaxWarp0) & 3;             // warp within the group
        const int r0 = wg * RH;                                // first row of the group
        const uint32_t bar_id = 1 + wg;                        // named barrier of the group
        const int quarter = warp & 3;                          // TMEM lane quarter this warp may access
        const int tau = quarter * 32 + lane;                   // token row (S) / dimension (O) of this thread
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int tid = tw * 32 + lane;
        const int causal_base = w.L - w.q_len;
        const int last_page_end = (w.L + kPage - 1) / kPage * kPage;
        bool failed = false;
        float *gred = red + wg * (4 * 32);
        float lsum[RH];
#pragma unroll
        for (int r = 0; r < RH; ++r)
            lsum[r] = 0.f;

        for (int j = 0; j < ntiles; ++j) {
            const int sb = j % C::kSBufs;          // S buffer and its barriers
            const int st = j % C::kStages;
            constexpr int NH = C::kHalves;
            float x[NH][RH];                    // this thread's tokens: tau, 128 + tau
            bool ok = !failed && mbar_wait_bounded(bar_sfull(sb), (j / C::kSBufs) & 1, abort_flag, p.wait_limit);
            ok = __all_sync(kFull, ok);          // tcgen05.ld is warp-collective
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int hf = 0; hf < NH; ++hf) {
                    const uint32_t s_col = tmem_s0 + sb * C::kSBufCols + hf * C::kSCols + r0 + lane_off;
#pragma unroll
                    for (int c = 0; c < RH; c += kLd)
                        tmem_ld32<kLd>(s_col + c, x[hf] + c);
                }
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_sfree(sb));
            // mask and scale: this thread's key in half hf is `tok`; row r = j' * G + i sees it
            // when tok < segment end and (causal) j' >= tok - (L - q_len)
            bool need = false;
#pragma unroll
            for (int hf = 0; hf < NH; ++hf) {
                const int tok = k0 + j * C::kTile + hf * kTokTile + tau;
                const int ahead = tok - causal_base;       // > 0: only query tokens j' >= ahead see this key
                const int rmin = ((p.causal && ahead > 0) ? ahead * p.G : 0) - row0;   // first local row that sees it
                // (padding rows r >= R have zero Q, so their scores are 0: harmless, and never written out)
                if (ok && tok < k1 && rmin <= 0) {
#pragma unroll
                    for (int r = 0; r < RH; r += 4) {
                        const float4 t = *reinterpret_cast<const float4 *>(m_thr + r0 + r);
                        const float4 c = *reinterpret_cast<const float4 *>(crow + r0 + r);
                        x[hf][r] *= c.x;
                        x[hf][r + 1] *= c.y;
                        x[hf][r + 2] *= c.z;
                        x[hf][r + 3] *= c.w;
                        need |= (x[hf][r] > t.x) | (x[hf][r + 1] > t.y) | (x[hf][r + 2] > t.z) | (x[hf][r + 3] > t.w);
                    }
                } else {
                    const bool tok_vis = ok && tok < k1;
#pragma unroll
                    for (int r = 0; r < RH; ++r) {
                        const int rg = r0 + r;
                        x[hf][r] = (tok_vis && rg >= rmin && rg < R) ? x[hf][r] * crow[rg] : -CUDART_INF_F;
                        need |= x[hf][r] > m_thr[rg];
                    }
                }
            }
            // group decision, one reduction over the group's 128 threads: rescale needed or a wait
            // failed?  Only then a second one tells which (every thread gets the same answers).
            if (named_bar_or(bar_id, 128, need || !ok)) {
                if (named_bar_or(bar_id, 128, !ok)) {
                    failed = true;
                    break;
                }
                // exact tile max of the group's rows across its 128 threads
                constexpr int kRc = RH >= 32 ? 32 : RH;
#pragma unroll
                for (int c0 = 0; c0 < RH; c0 += kRc) {
                    float v[kRc];
#pragma unroll
                    for (int r = 0; r < kRc; ++r) {
                        v[r] = x[0][c0 + r];
#pragma unroll
                        for (int hf = 1; hf < NH; ++hf)
                            v[r] = fmaxf(v[r], x[hf][c0 + r]);
                    }
                    warp_transpose_reduce<kRc, true>(v, lane);
                    gred[tw * 32 + c0 + reduce_row0<kRc>(lane)] = v[0];
                }
                named_bar_sync(bar_id, 128);
                if (tid < RH) {
                    const int rg = r0 + tid;
                    const float mt = fmaxf(fmaxf(gred[tid], gred[32 + tid]), fmaxf(gred[64 + tid], gred[96 + tid]));
                    const float mo = m_run[rg];
                    const float mn = fmaxf(mo, mt);
                    alpha_s[rg] = (mo == -CUDART_INF_F) ? 0.f : exp2f(mo - mn);
                    m_run[rg] = mn;
                    m_thr[rg] = mn + C::kThrLog2;
                    m_sub[rg] = mn == -CUDART_INF_F ? 0.f : mn;
                }
                named_bar_sync(bar_id, 128);
#pragma unroll
                for (int r = 0; r < RH; ++r)
                    lsum[r] *= alpha_s[r0 + r];
                if (j > 0) {
                    // O holds tiles < j: wait for PV(j-1), then rescale this thread's dimension.
                    // PV(i) completes phase i / kStages of empty[i % kStages].  The phase before,
                    // PV(j-1-kStages), was seen by the producer before it loaded tile j-1, and the one
                    // after, PV(j-1+kStages), cannot start before P(j+1): PV(j-1)'s is unambiguous here.
                    const int jp = j - 1;
                    bool okp = mbar_wait_bounded(bar_empty(jp % C::kStages), (jp / C::kStages) & 1, abort_flag, p.wait_limit);
                    okp = __all_sync(kFull, okp);    // tcgen05.ld/st are warp-collective
                    if (okp) {
                        tc_fence_after();
#pragma unroll
                        for (int half = 0; half < C::kOCols / RP; ++half) {
#pragma unroll
                            for (int c = 0; c < RH; c += kLd) {
                                float o[kLd];
                                const uint32_t col = tmem_o + half * RP + r0 + c + lane_off;
                                tmem_ld32<kLd>(col, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int r = 0; r < kLd; ++r)
                                    o[r] *= alpha_s[r0 + c + r];
                                tmem_st32<kLd>(col, o);
                            }
                        }
                        tmem_wait_st();
                    } else {
                        failed = true;
                    }
                }
            }
            if (!failed) {
                // probabilities against the running max (masked entries are -inf -> 0), written as
                // this token's row of P^T over the tile's K area, which QK(j) no longer needs:
                // MN-major, 128-byte swizzle, 16-byte unit u of row t stored at u ^ (t % 8); row r
                // at bytes [2r, 2r + 2).
                // The group's running maxima are read before the first P store: the compiler cannot
                // tell the stores from these shared-memory words, so a read after a store would
                // wait for it (1-2 us per call on the large batches).
                float msub[RH];
#pragma unroll
                for (int r = 0; r < RH; r += 4) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(m_sub + r0 + r);
                    msub[r] = m4.x;
                    msub[r + 1] = m4.y;
                    msub[r + 2] = m4.z;
                    msub[r + 3] = m4.w;
                }
#pragma unroll
                for (int hf = 0; hf < NH; ++hf) {
                    const int t = hf * kTokTile + tau;          // token of the tile
                    uint8_t *prow = smem + st * C::kStageBytes + (t >> 3) * C::kGroupBytes + (t & 7) * 128;
#pragma unroll
                    for (int u = 0; u < RH / 8; ++u) {
                        const float *mm = msub + 8 * u;
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int r = 8 * u + 2 * e;
                            const float p0 = ex2_ftz(x[hf][r] - mm[2 * e]);
                            const float p1 = ex2_ftz(x[hf][r + 1] - mm[2 * e + 1]);
                            lsum[r] += p0;
                            lsum[r + 1] += p1;
                            pk[e] = pack_bf16x2(p0, p1);
                        }
                        const int ug = r0 / 8 + u;                     // unit of the row
                        *reinterpret_cast<uint4 *>(prow + ((ug ^ (t & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                    const int tok = k0 + j * C::kTile + t;
                    if (tok >= w.L && tok < last_page_end) {
                        // past L in the last page the row holds anything (0 * NaN would reach O): this
                        // group's share of the token's V row becomes zeros (chunk 2 + wg)
                        static_assert(C::kGroups == 2, "bf16 V rows are zeroed by chunk");
                        uint8_t *vrow = smem + st * C::kStageBytes + C::kOffV + (t >> 3) * C::kGroupBytes + (t & 7) * 128 +
                                        wg * 1024;
#pragma unroll
                        for (int u = 0; u < 128 / 16; ++u)
                            *reinterpret_cast<uint4 *>(vrow + u * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_pfull(st));
            if (failed) {
                // the next tile's group decision propagates the failure
                *abort_flag = 1;
            }
        }

        // ---- epilogue: row sums across the group's threads (they do not need the last PV, which
        // completes meanwhile), then O complete? and the partials.  (A stage barrier cannot tell
        // PV(last) from PV(last-1) here: both may still be running; bar_odone can.)
        {
            constexpr int kRc = RH >= 32 ? 32 : RH;
#pragma unroll
            for (int c0 = 0; c0 < RH; c0 += kRc) {
                float v[kRc];
#pragma unroll
                for (int r = 0; r < kRc; ++r)
                    v[r] = lsum[c0 + r];
                warp_transpose_reduce<kRc, false>(v, lane);
                gred[tw * 32 + c0 + reduce_row0<kRc>(lane)] = v[0];
            }
        }
        named_bar_sync(bar_id, 128);
        if (tid < RH)
            alpha_s[r0 + tid] = (gred[tid] + gred[32 + tid]) + (gred[64 + tid] + gred[96 + tid]);
        bool okf = !failed;
        if (okf && ntiles > 0)
            okf = mbar_wait_bounded(bar_odone, 0, abort_flag, p.wait_limit);
        // the group's verdict; the barrier also publishes the row sums written above
        const bool write = !named_bar_or(bar_id, 128, !okf);
        if (write) {
            // O^T of the group's rows straight from TMEM into the partials (a warp holds 32
            // dimensions of each row); the rows' slots were computed during the set-up
            if (ntiles > 0)
                tc_fence_after();
#pragma unroll
            for (int c = 0; c < RH; c += kLd) {
                float o[kLd];
                if (ntiles > 0) {
                    tmem_ld32<kLd>(tmem_o + r0 + c + lane_off, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int r = 0; r < kLd; ++r)
                        o[r] = 0.f;
                }
                const long long *slots = reinterpret_cast<const long long *>(misc + C::kSlot);
#pragma unroll
                for (int rr = 0; rr < kLd; ++rr)
                    o[rr] = alpha_s[r0 + c + rr] > 0.f ? o[rr] : 0.f;
                // 4 x 4 transposes within lane quads: lane 4a + b ends with row 4k + b of each block of
                // four rows and dimensions 4a .. 4a + 3 of the warp's quarter, so a warp store writes
                // four rows of 128 contiguous bytes, 16 bytes a lane (part_o is 16-byte aligned)
                const int qb = lane & 3;
                const bool qb0 = (qb & 1) != 0, qb1 = (qb & 2) != 0;
                const int dim4 = quarter * 32 + (lane & ~3);
#pragma unroll
                for (int k = 0; k < kLd / 4; ++k) {
                    const float x0 = o[4 * k], x1 = o[4 * k + 1], x2 = o[4 * k + 2], x3 = o[4 * k + 3];
                    const float own0 = qb1 ? x2 : x0, own1 = qb1 ? x3 : x1;
                    const float rc0 = __shfl_xor_sync(kFull, qb1 ? x0 : x2, 2);
                    const float rc1 = __shfl_xor_sync(kFull, qb1 ? x1 : x3, 2);
                    const float zl0 = qb1 ? rc0 : own0, zl1 = qb1 ? rc1 : own1;
                    const float zh0 = qb1 ? own0 : rc0, zh1 = qb1 ? own1 : rc1;
                    const float rl = __shfl_xor_sync(kFull, qb0 ? zl0 : zl1, 1);
                    const float rh = __shfl_xor_sync(kFull, qb0 ? zh0 : zh1, 1);
                    const float kl = qb0 ? zl1 : zl0, kh = qb0 ? zh1 : zh0;
                    const float4 y = make_float4(qb0 ? rl : kl, qb0 ? kl : rl, qb0 ? rh : kh, qb0 ? kh : rh);
                    const int r = r0 + c + 4 * k + qb;
                    if (r < R)
                        *reinterpret_cast<float4 *>(p.part_o + slots[r] * kHeadDim + dim4) = y;
                }
            }
            const int r = r0 + tid;
            if (tid < RH && r < R) {
                const long long slot = reinterpret_cast<const long long *>(misc + C::kSlot)[r];
                const float l = alpha_s[r];
                p.part_m[slot] = l > 0.f ? m_run[r] * 0.69314718055994531f : -CUDART_INF_F;
                p.part_l[slot] = l;
            }
        }
    }

    // ---- teardown: every role is done with TMEM and shared memory
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

template <int RP, bool FP8>
cudaError_t launch_rp(const CUtensorMap &map, const AttnParams &p, cudaStream_t stream)
{
    // per device and cheap: set on every launch
    const cudaError_t attr_err = cudaFuncSetAttribute(attn_tc_kernel<RP, FP8>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                      Cfg<RP, FP8>::kSmemBytes);
    if (attr_err != cudaSuccess)
        return attr_err;
    const dim3 grid((unsigned)p.num_items * (unsigned)p.H_kv * (unsigned)p.row_blocks);
    return launch_pdl(attn_tc_kernel<RP, FP8>, grid, dim3(Cfg<RP, FP8>::kThreads), Cfg<RP, FP8>::kSmemBytes, stream,
                      map, p);
}

}  // namespace

// Rows per CTA the kernel takes (16, 32 or 64; 0 when it cannot take the call);
// a work item with more rows than 64 is split into row blocks, one CTA each.
int attn_tc_rows(int kv_dtype, int rows_max, long long num_blocks, int H_kv)
{
    if ((kv_dtype != SK_KV_BF16 && kv_dtype != SK_KV_FP8_E4M3) || rows_max < 1 || rows_max > kMaxRowBlocks * 64)
        return 0;
    if (num_blocks * H_kv * 2 > 0x7FFFFFFFLL)
        return 0;
    return rows_max <= 16 ? 16 : rows_max <= 32 ? 32 : 64;     // above 64: row blocks of 64
}

cudaError_t launch_attn_tc(const AttnParams &p, int kv_dtype, int rp, cudaStream_t stream)
{
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr)
        return cudaErrorNotSupported;
    const bool fp8 = kv_dtype == SK_KV_FP8_E4M3;
    CUtensorMap map;
    // The pages [blocks][heads][16 tokens][K | V] seen as 4-D: (128 bytes of a row, token within an
    // 8-token group, 128-byte chunk of the row, 8-token group across all pages).  One box is a whole
    // page of one head and lands group by group, chunk by chunk, as 8 x 128 B swizzle atoms.
    const cuuint64_t row_bytes = (cuuint64_t)(2 * kHeadDim * (fp8 ? 1 : 2));
    const cuuint32_t nchunks = (cuuint32_t)(row_bytes / 128);
    const cuuint64_t dims[4] = {(cuuint64_t)(fp8 ? 128 : 64), 8, nchunks, (cuuint64_t)p.num_blocks * p.H_kv * 2};
    const cuuint64_t strides[3] = {row_bytes, 128, 8 * row_bytes};
    const cuuint32_t box[4] = {fp8 ? 128u : 64u, 8, nchunks, 2};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(&map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                     const_cast<void *>(p.kv), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    switch (rp * 2 + (fp8 ? 1 : 0)) {
    case 32:
        return launch_rp<16, false>(map, p, stream);
    case 64:
        return launch_rp<32, false>(map, p, stream);
    case 128:
        return launch_rp<64, false>(map, p, stream);
    case 33:
        return launch_rp<16, true>(map, p, stream);
    case 65:
        return launch_rp<32, true>(map, p, stream);
    case 129:
        return launch_rp<64, true>(map, p, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace sk
