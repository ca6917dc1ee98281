// fa_verify.cu — decode-shaped attention: a few query rows (1 <= Sq <= 16,
// e.g. the k+1 positions a speculative-decoding verify step scores in one
// target pass, "FlashAttention, speculative decoding, quantisation and
// parallelism", Speculative decoding) against a long KV cache.
//
// Plain tiled attention gives such a shape one CTA per (batch, head) and
// leaves most of the GPU idle; Flash-Decoding ("Lecture 06 — Making Decode
// Fast", section 5) splits the keys/values across SMs and finishes with a
// small combine. Here:
//   * K2 (fa_verify_split_kernel): one CTA per (key chunk, batch*head). A
//     producer warp streams 64-key K and V tiles of the chunk through a TMA
//     ring (128-byte swizzle); four consumer warps each take 16 keys of every
//     stage, form S = Q K^T with bf16 mma.sync (Q in registers, K via
//     ldmatrix), run the online softmax of "Warmup Guide — Inference
//     Optimization at Depth", Chapter 3 on their keys, and accumulate
//     O += P V (V via ldmatrix.trans). At the end the four warps' (m, l, O)
//     are combined in shared memory into the chunk's partial (O_s / l_s,
//     LSE_s); with a single chunk that partial is the answer.
//   * K3 (fa_verify_combine_kernel): per query row,
//       LSE = M + ln sum_s exp(LSE_s - M),  M = max_s LSE_s,
//       O   = sum_s exp(LSE_s - LSE) O_s,
//     the chunk-level form of Chapter 3's update (the pages give no formula
//     for the "final combine"; this is the one the update implies).
// Which keys a query row sees is a bitmask over the last Sq key positions
// (the draft positions; every key before them is visible): bits 0..i for the
// causal chain, every bit for non-causal, or a caller-given tree mask, where
// each candidate sees the cache and its own ancestors (tree-attention over a
// draft tree, "Lecture 06", section 3). K/V can come from a contiguous
// [B, H, Sk, d] tensor or from page pools through a block table with a
// length per sequence ("Warmup Guide", Chapter 8 and its Q&A: the kernel
// walks the block table once per tile); each 64-key stage is then one TMA box
// per page it spans.
// This shape moves ~5 flops per byte: it is bound by HBM, so the legacy
// warp-level MMA is ample; what matters is keeping enough bytes in flight.
#include <cmath>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace verify {

constexpr int kStageKeys = kVerifyStageKeys;  // keys per ring stage
constexpr int kConsumerWarps = 4;             // 16 keys of each stage per warp
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kMaxRows = 16;                  // mma M
constexpr int kBoxBytes = kStageKeys * 128;   // 64 keys x 64 columns bf16 (8 KB)

template <int D>
struct Cfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = kStageKeys * D * 2;  // K or V part of a stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = (D == 128) ? 3 : 6;    // 96 KB of ring: 2 CTAs per SM
    static constexpr int kOffBar = kStages * kStageBytes;
    static constexpr int kSmemBytes = kOffBar + 256 + 1024;
    // End-of-chunk combine scratch (reuses the ring): per warp m, l, O rows.
    static constexpr int kScratchBytes = kConsumerWarps * kMaxRows * (D + 2) * 4;
    static_assert(kScratchBytes <= kOffBar, "combine scratch must fit in the ring");
};

struct Params {
    int Sq, Sk, BH, H, n_split;
    int chunk;  // keys per split (multiple of kStageKeys)
    int mode;   // 0: every draft position, 1: causal chain, 2: tree_mask
    float scale, scale_log2;     // |scale|, |scale| * log2(e)
    uint32_t q_sign;             // 0x80008000 for a negative scale (Q enters as -Q), else 0
    uint32_t q_keep;             // 0 at scale 0 (every score is 0: Q enters as 0), else ~0
    const uint32_t *tree_mask;   // [B, Sq] (mode 2)
    const int32_t *seq_lens;     // [B] keys per sequence (paged); nullptr: Sk for all
    const int32_t *block_table;  // [B, max_pages] physical page of each logical page (paged)
    int page_size, max_pages, num_pages;
    const __nv_bfloat16 *q;
    __nv_bfloat16 *o;   // final output (used when n_split == 1)
    float *lse;         // final LSE (used when n_split == 1)
    float *ws_o;        // [n_split, BH, Sq, D] partial outputs
    float *ws_lse;      // [n_split, BH, Sq]
    unsigned int *status;
    uint64_t wait_ns;   // limit of every bounded wait (kWaitLimitNs unless a test lowers it)
    int stall_stage;    // test only: stage CTA (0, 0)'s producer skips (-1: none)
};

struct Bars {
    uint64_t full[8];
    uint64_t empty[8];
    int abort_flag;
};

// Bitmask over the Sq draft positions that row i sees.
__device__ __forceinline__ uint32_t draft_mask(const Params &p, int b, int i)
{
    if (i >= p.Sq)
        return 0u;
    const uint32_t all = p.Sq >= 32 ? ~0u : ((1u << p.Sq) - 1u);
    if (p.mode == 0)
        return all;
    if (p.mode == 1)
        return i >= 31 ? ~0u : ((2u << i) - 1u);
    if (!fa_check(b < p.BH / p.H, p.status))
        return 0u;
    return p.tree_mask[static_cast<size_t>(b) * p.Sq + i] & all;
}

// Key j (logical) is visible through mask `rm`: everything before the draft
// positions, and draft position j - prefix when its bit is set.
__device__ __forceinline__ bool key_visible(int j, int prefix, int Sk_b, uint32_t rm)
{
    return j < prefix || (j < Sk_b && ((rm >> (j - prefix)) & 1u));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t ld_bf16x2_or_zero(const __nv_bfloat16 *p, bool valid)
{
    return valid ? *reinterpret_cast<const uint32_t *>(p) : 0u;
}

// 5-D tiled load, coordinates innermost first.
__device__ __forceinline__ void tma_load_5d_hint(void *dst, const CUtensorMap *map, uint64_t *bar,
                                                 int32_t c0, int32_t c1, int32_t c2, int32_t c3,
                                                 int32_t c4, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3), "r"(c4), "l"(policy)
        : "memory");
}

// Where key row `key` (0-63 of a stage), 64-column half `half` and 16-byte
// chunk `chunk` of a K or V tile sit in the stage. Layout 0 (contiguous and
// pages of 64 keys or more, and d = 64): one 128-byte-swizzled box of 64 rows
// per half. Layout 1 (pages of 16 or 32 keys at d = 128): one box per page,
// its rows 256 bytes wide (both halves, so the page loads as one contiguous
// read), the 128-byte lines swizzled in order.
template <int kLayout>
__device__ __forceinline__ uint32_t kv_offset(int key, int half, uint32_t chunk, int page_shift)
{
    if constexpr (kLayout == 0) {
        return half * kBoxBytes + sw128_offset(static_cast<uint32_t>(key), chunk);
    } else {
        const uint32_t pg = static_cast<uint32_t>(key) >> page_shift;
        const uint32_t line = ((static_cast<uint32_t>(key) & ((1u << page_shift) - 1u)) << 1) + half;
        return (pg << (page_shift + 8)) + sw128_offset(line, chunk);
    }
}

// kKv: 0 contiguous K/V; 1 paged, layout 0; 2 paged, layout 1 (pages of 16
// or 32 keys at d = 128).
template <int D, int kKv>
__global__ void __launch_bounds__(kThreads, 2)
    fa_verify_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const Params p)
{
    constexpr bool kPaged = kKv != 0;
    constexpr int kLayout = kKv == 2 ? 1 : 0;
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    Bars *bars = reinterpret_cast<Bars *>(smem + C::kOffBar);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int split = blockIdx.x;
    const int bh = blockIdx.y;

    const int b = bh / p.H, h = bh % p.H;
    // Keys of this sequence; the draft positions are its last Sq keys.
    int Sk_b = p.Sk;
    if (kPaged && p.seq_lens && fa_check(b < p.BH / p.H, p.status)) {
        Sk_b = p.seq_lens[b];
        Sk_b = Sk_b < 0 ? 0 : min(Sk_b, p.max_pages * p.page_size);
    }
    const int prefix = Sk_b - p.Sq;
    // Keys this CTA covers: its chunk of the sequence.
    const int kv_begin = split * p.chunk;
    const int kv_end = min(kv_begin + p.chunk, Sk_b);
    const int n_st = kv_end > kv_begin ? (kv_end - kv_begin + kStageKeys - 1) / kStageKeys : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], kConsumerWarps);
        }
        bars->abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    int *abort_flag = &bars->abort_flag;

    if (warp == kProducerWarp) {
        // The whole warp walks the stages (it shares the block-table reads);
        // lane 0 issues the copies.
        const uint64_t pol = l2_policy_evict_first();  // K/V are streamed once
        const int P = p.page_size;
        const int n_pages_b = kPaged ? (Sk_b + P - 1) / P : 0;
        int cached = -1, my_page = 0;
        // Physical page of logical page lp (warp-collective): 32 entries of the
        // block table are read at a time, one per lane. Pages past the
        // sequence get an out-of-range index, which TMA fills with zeros.
        auto page_of = [&](int lp) {
            const int base = lp & ~31;
            if (base != cached) {
                cached = base;
                const int idx = base + lane;
                my_page = (idx < n_pages_b && fa_check(idx < p.max_pages, p.status))
                              ? p.block_table[static_cast<size_t>(b) * p.max_pages + idx]
                              : p.num_pages;
            }
            return __shfl_sync(0xffffffffu, my_page, lp & 31);
        };
        int st = 0;
        for (; st < n_st; ++st) {
            const int s = st % C::kStages;
            const uint32_t use = st / C::kStages;
            if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->empty[s], (use - 1) & 1,
                                                               abort_flag, p.status, p.wait_ns)))
                break;
            if (st == p.stall_stage && split == 0 && bh == 0)
                continue;  // test only: never issued, so the consumers' bounded wait runs out
            if (lane == 0)
                mbar_arrive_expect_tx(&bars->full[s], C::kStageBytes);
            uint8_t *dst = smem + s * C::kStageBytes;
            const int key = kv_begin + st * kStageKeys;
            if constexpr (!kPaged) {
                if (lane == 0)
                    fa_check(key < p.Sk && bh < p.BH, p.status);
                if (lane == 0)
                    for (int q = 0; q < C::kBoxes; ++q) {
                        tma_load_3d_hint(dst + q * kBoxBytes, &tm_k, &bars->full[s], q * 64, key,
                                         bh, pol);
                        tma_load_3d_hint(dst + C::kTileBytes + q * kBoxBytes, &tm_v,
                                         &bars->full[s], q * 64, key, bh, pol);
                    }
            } else if (kKv == 2) {
                // One box per page: all rows of the page, both halves (P * 256
                // contiguous bytes of K, and of V).
                for (int sub = 0; sub < kStageKeys / P; ++sub) {
                    const int pid = page_of(key / P + sub);
                    if (lane == 0) {
                        tma_load_5d_hint(dst + sub * P * 256, &tm_k, &bars->full[s], 0, 0, 0, h,
                                         pid, pol);
                        tma_load_5d_hint(dst + C::kTileBytes + sub * P * 256, &tm_v,
                                         &bars->full[s], 0, 0, 0, h, pid, pol);
                    }
                }
            } else if (P >= kStageKeys) {
                const int pid = page_of(key / P);
                if (lane == 0)
                    for (int q = 0; q < C::kBoxes; ++q) {
                        tma_load_4d_hint(dst + q * kBoxBytes, &tm_k, &bars->full[s], q * 64,
                                         key % P, h, pid, pol);
                        tma_load_4d_hint(dst + C::kTileBytes + q * kBoxBytes, &tm_v,
                                         &bars->full[s], q * 64, key % P, h, pid, pol);
                    }
            } else {
                // The stage spans kStageKeys / P pages: one box of P rows each,
                // placed at consecutive rows of the stage (P * 128 bytes is a
                // multiple of the 1024-byte swizzle atom).
                for (int sub = 0; sub < kStageKeys / P; ++sub) {
                    const int pid = page_of(key / P + sub);
                    if (lane == 0)
                        for (int q = 0; q < C::kBoxes; ++q) {
                            tma_load_4d_hint(dst + q * kBoxBytes + sub * P * 128, &tm_k,
                                             &bars->full[s], q * 64, 0, h, pid, pol);
                            tma_load_4d_hint(dst + C::kTileBytes + q * kBoxBytes + sub * P * 128,
                                             &tm_v, &bars->full[s], q * 64, 0, h, pid, pol);
                        }
                }
            }
        }
        if (lane == 0)
            for (int k = max(0, st - C::kStages); k < st; ++k)
                mbar_wait_drain(&bars->full[k % C::kStages], (k / C::kStages) & 1, p.status, p.wait_ns);
        // Match the consumers' two block barriers (ring -> scratch, scratch ready).
        __syncthreads();
        __syncthreads();
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane / 4;   // fragment row (and row + 8)
    const int tq = lane % 4;  // fragment column pair
    const float sl2 = p.scale_log2;
    const __nv_bfloat16 *qb = p.q + static_cast<size_t>(bh) * p.Sq * D;

    // Q as mma A fragments: rows g and g+8, columns kk*16 + 2*tq (+8).
    // A negative scale enters as -Q (an exact flip of each bf16 sign bit), so
    // scale * Q K^T = |scale| * (-Q) K^T and the softmax sees |scale| only; at
    // scale 0 Q enters as 0 and the softmax factor is 1 (every weight 1).
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const int c = kk * 16 + 2 * tq;
        qa[kk][0] = (ld_bf16x2_or_zero(qb + g * D + c, g < p.Sq) & p.q_keep) ^ p.q_sign;
        qa[kk][1] = (ld_bf16x2_or_zero(qb + (g + 8) * D + c, g + 8 < p.Sq) & p.q_keep) ^ p.q_sign;
        qa[kk][2] = (ld_bf16x2_or_zero(qb + g * D + c + 8, g < p.Sq) & p.q_keep) ^ p.q_sign;
        qa[kk][3] =
            (ld_bf16x2_or_zero(qb + (g + 8) * D + c + 8, g + 8 < p.Sq) & p.q_keep) ^ p.q_sign;
    }
    const uint32_t rm0 = draft_mask(p, b, g), rm1 = draft_mask(p, b, g + 8);

    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY;  // running max of raw scores, rows g, g+8
    float l0 = 0.0f, l1 = 0.0f;            // this thread's share of the running sums

    // ldmatrix row addresses (relative to a stage): matrix mi = lane / 8,
    // row lane % 8 of it.
    const int mi = lane / 8, mr = lane % 8;
    const int k_key = warp * 16 + ((mi >> 1) << 3) + mr;  // K: matrices (keys lo/hi) x (d lo/hi)
    const int k_half = mi & 1;
    const int v_key = warp * 16 + ((mi & 1) << 3) + mr;   // V: matrices (keys lo/hi) x (d lo/hi)
    const int v_half = mi >> 1;
    const uint32_t smem_a = smem_u32(smem);
    const int page_shift = kLayout == 1 ? (p.page_size == 16 ? 4 : 5) : 0;

    bool ok = true;
    for (int st = 0; st < n_st && ok; ++st) {
        const int s = st % C::kStages;
        // Warp-uniform outcome: the ldmatrix / mma.sync below need the whole
        // warp, and after a timeout elsewhere some lanes could give up while
        // others see the phase complete.
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[s], (st / C::kStages) & 1, abort_flag,
                                               p.status, p.wait_ns));
        if (!ok)
            break;
        const uint32_t sK = smem_a + s * C::kStageBytes;
        const uint32_t sV = sK + C::kTileBytes;

        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t chunk = 2 * (kk % 4) + k_half;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(sK + kv_offset<kLayout>(k_key, kk / 4, chunk, page_shift), b0, b1, b2, b3);
            mma_bf16_16816(sc[0], qa[kk], b0, b1);
            mma_bf16_16816(sc[1], qa[kk], b2, b3);
        }
        // Mask (only stages that reach the draft positions or past the end)
        // and online softmax over this warp's 16 keys.
        const int stage_key = kv_begin + st * kStageKeys;
        if (stage_key + kStageKeys > prefix) {
            const int key_base = stage_key + warp * 16 + 2 * tq;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = key_base + nt * 8 + e;
                    if (!key_visible(key, prefix, Sk_b, rm0))
                        sc[nt][e] = -INFINITY;
                    if (!key_visible(key, prefix, Sk_b, rm1))
                        sc[nt][2 + e] = -INFINITY;
                }
        }
        float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == -INFINITY ? 0.0f : mn0;
        const float mu1 = mn1 == -INFINITY ? 0.0f : mn1;
        // 0 while nothing was visible (tested on m itself: at scale 0 the
        // product (m - mu) * sl2 would be NaN).
        const float c0 = m0 == -INFINITY ? 0.0f : ex2_approx((m0 - mu0) * sl2);
        const float c1 = m1 == -INFINITY ? 0.0f : ex2_approx((m1 - mu1) * sl2);
        m0 = mn0;
        m1 = mn1;
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            pr[nt][0] = ex2_approx(fmaf(sc[nt][0], sl2, -mu0 * sl2));
            pr[nt][1] = ex2_approx(fmaf(sc[nt][1], sl2, -mu0 * sl2));
            pr[nt][2] = ex2_approx(fmaf(sc[nt][2], sl2, -mu1 * sl2));
            pr[nt][3] = ex2_approx(fmaf(sc[nt][3], sl2, -mu1 * sl2));
        }
        l0 = l0 * c0 + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
        l1 = l1 * c1 + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            o[n][0] *= c0;
            o[n][1] *= c0;
            o[n][2] *= c1;
            o[n][3] *= c1;
        }
        // P as the A fragment of the next MMA (the S accumulator layout maps
        // onto it directly): rows g / g+8, keys 2*tq (+8).
        const uint32_t pa[4] = {pack_bf16x2(pr[0][0], pr[0][1]), pack_bf16x2(pr[0][2], pr[0][3]),
                                pack_bf16x2(pr[1][0], pr[1][1]), pack_bf16x2(pr[1][2], pr[1][3])};
#pragma unroll
        for (int dd = 0; dd < D / 16; ++dd) {
            const uint32_t chunk = 2 * (dd % 4) + v_half;
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(sV + kv_offset<kLayout>(v_key, dd / 4, chunk, page_shift), b0, b1, b2,
                          b3);
            mma_bf16_16816(o[2 * dd], pa, b0, b1);
            mma_bf16_16816(o[2 * dd + 1], pa, b2, b3);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&bars->empty[s]);
    }

    // Quad-reduce the row sums (every lane of a quad holds the same max).
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    __syncthreads();  // all stages consumed and landed: the ring becomes scratch
    float *scr = reinterpret_cast<float *>(smem);
    constexpr int kRowStride = D + 2;  // per row: O[D], m, l
    float *mine = scr + warp * kMaxRows * kRowStride;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
        const int c = n * 8 + 2 * tq;
        mine[g * kRowStride + c] = o[n][0];
        mine[g * kRowStride + c + 1] = o[n][1];
        mine[(g + 8) * kRowStride + c] = o[n][2];
        mine[(g + 8) * kRowStride + c + 1] = o[n][3];
    }
    if (tq == 0) {
        mine[g * kRowStride + D] = m0;
        mine[g * kRowStride + D + 1] = l0;
        mine[(g + 8) * kRowStride + D] = m1;
        mine[(g + 8) * kRowStride + D + 1] = l1;
    }
    __syncthreads();

    const bool aborted = *reinterpret_cast<volatile int *>(abort_flag) != 0;
    const int tid = threadIdx.x;  // 0..127 (consumers)
    for (int idx = tid; idx < p.Sq * D && !aborted; idx += kConsumerWarps * 32) {
        const int row = idx / D, col = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
            M = fmaxf(M, scr[(w * kMaxRows + row) * kRowStride + D]);
        float L = 0.0f, acc = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float *rw = scr + (w * kMaxRows + row) * kRowStride;
                const float wt = rw[D] == -INFINITY ? 0.0f : ex2_approx((rw[D] - M) * sl2);
                L += rw[D + 1] * wt;
                acc += rw[col] * wt;
            }
        }
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
        const float lse = L > 0.0f ? M * p.scale + logf(L) : -INFINITY;
        const size_t row_g = static_cast<size_t>(bh) * p.Sq + row;
        if (!fa_check(row_g < static_cast<size_t>(p.BH) * p.Sq && split < p.n_split, p.status))
            continue;
        if (p.n_split == 1) {
            p.o[row_g * D + col] = __float2bfloat16_rn(acc * inv);
            if (col == 0)
                p.lse[row_g] = lse;
        } else {
            const size_t part = static_cast<size_t>(split) * p.BH * p.Sq + row_g;
            p.ws_o[part * D + col] = acc * inv;
            if (col == 0)
                p.ws_lse[part] = lse;
        }
    }
}

// One warp per query row: LSE-weighted combine of the n_split partials.
template <int D>
__global__ void __launch_bounds__(128)
    fa_verify_combine_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_lse,
                             __nv_bfloat16 *__restrict__ o, float *__restrict__ lse,
                             int n_rows, int n_split)
{
    const int row = blockIdx.x * 4 + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= n_rows)
        return;
    float M = -INFINITY;
    for (int s = 0; s < n_split; ++s)
        M = fmaxf(M, ws_lse[static_cast<size_t>(s) * n_rows + row]);
    constexpr int kPer = D / 32;
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e)
        acc[e] = 0.0f;
    float L = -INFINITY;
    if (M != -INFINITY) {
        float sum = 0.0f;
        for (int s = 0; s < n_split; ++s)
            sum += expf(ws_lse[static_cast<size_t>(s) * n_rows + row] - M);
        L = M + logf(sum);
        for (int s = 0; s < n_split; ++s) {
            const float w = expf(ws_lse[static_cast<size_t>(s) * n_rows + row] - L);
            const float *src = ws_o + (static_cast<size_t>(s) * n_rows + row) * D;
#pragma unroll
            for (int e = 0; e < kPer; ++e)
                acc[e] = fmaf(w, src[lane + 32 * e], acc[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < kPer; ++e)
        o[static_cast<size_t>(row) * D + lane + 32 * e] = __float2bfloat16_rn(acc[e]);
    if (lane == 0)
        lse[row] = L;
}

template <int D>
fa_status_t launch(const Problem &pr, int n_split, void *ws, size_t ws_bytes,
                   const VerifyOptions &opt)
{
    using C = Cfg<D>;
    const int64_t BH = pr.B * pr.H;
    const bool paged = opt.block_table != nullptr;
    const bool small_pages = paged && D == 128 && opt.page_size < kStageKeys;
    CUtensorMap tk, tv;
    if (!paged) {
        if (!encode_tmap_bf16_3d(&tk, pr.k, D, pr.Sk, BH, kStageKeys) ||
            !encode_tmap_bf16_3d(&tv, pr.v, D, pr.Sk, BH, kStageKeys))
            return FA_ERR_CUDA;
    } else if (small_pages) {
        if (!encode_tmap_bf16_pages_5d(&tk, pr.k, opt.page_size, pr.H, opt.num_pages) ||
            !encode_tmap_bf16_pages_5d(&tv, pr.v, opt.page_size, pr.H, opt.num_pages))
            return FA_ERR_CUDA;
    } else {
        const uint32_t box_rows =
            static_cast<uint32_t>(opt.page_size < kStageKeys ? opt.page_size : kStageKeys);
        if (!encode_tmap_bf16_4d(&tk, pr.k, D, opt.page_size, pr.H, opt.num_pages, box_rows) ||
            !encode_tmap_bf16_4d(&tv, pr.v, D, opt.page_size, pr.H, opt.num_pages, box_rows))
            return FA_ERR_CUDA;
    }
    Params p;
    p.Sq = static_cast<int>(pr.Sq);
    p.Sk = static_cast<int>(pr.Sk);
    p.BH = static_cast<int>(BH);
    p.H = static_cast<int>(pr.H);
    p.n_split = n_split;
    p.chunk = static_cast<int>(verify_chunk_keys(pr.Sk, n_split));
    p.mode = opt.tree_mask ? 2 : (pr.causal ? 1 : 0);
    p.scale = fabsf(pr.scale);
    p.q_keep = pr.scale == 0.0f ? 0u : ~0u;
    p.scale_log2 = pr.scale == 0.0f ? 1.0f : fabsf(pr.scale) * 1.4426950408889634f;
    p.q_sign = std::signbit(pr.scale) ? 0x80008000u : 0u;
    p.tree_mask = opt.tree_mask;
    p.seq_lens = opt.seq_lens;
    p.block_table = opt.block_table;
    p.page_size = static_cast<int>(opt.page_size);
    p.max_pages = static_cast<int>(opt.max_pages);
    p.num_pages = static_cast<int>(opt.num_pages);
    p.q = static_cast<const __nv_bfloat16 *>(pr.q);
    p.o = static_cast<__nv_bfloat16 *>(pr.o);
    p.lse = pr.lse;
    p.status = pr.status;
    p.wait_ns = kWaitLimitNs;
    p.stall_stage = -1;
    take_stall(kStallVerify, &p.stall_stage, &p.wait_ns);
    p.ws_o = nullptr;
    p.ws_lse = nullptr;
    if (n_split > 1) {
        const size_t need = verify_workspace_bytes(BH, pr.Sq, D, n_split);
        if (!ws || ws_bytes < need)
            return FA_ERR_WORKSPACE;
        const size_t o_bytes = (static_cast<size_t>(n_split) * BH * pr.Sq * D * 4 + 255) & ~size_t(255);
        p.ws_o = static_cast<float *>(ws);
        p.ws_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + o_bytes);
    }
    if (BH > 65535)
        return FA_ERR_UNSUPPORTED;
    auto kern = small_pages ? fa_verify_split_kernel<D, 2>
                            : (paged ? fa_verify_split_kernel<D, 1> : fa_verify_split_kernel<D, 0>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return FA_ERR_CUDA;
    dim3 grid(static_cast<unsigned>(n_split), static_cast<unsigned>(BH));
    kern<<<grid, kThreads, C::kSmemBytes, pr.stream>>>(tk, tv, p);
    if (cudaGetLastError() != cudaSuccess)
        return FA_ERR_CUDA;
    if (n_split > 1) {
        const int n_rows = static_cast<int>(BH * pr.Sq);
        fa_verify_combine_kernel<D><<<(n_rows + 3) / 4, 128, 0, pr.stream>>>(
            p.ws_o, p.ws_lse, p.o, p.lse, n_rows, n_split);
        if (cudaGetLastError() != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // namespace verify

int64_t verify_chunk_keys(int64_t Sk, int n_split)
{
    const int64_t per = (Sk + n_split - 1) / n_split;
    return (per + kVerifyStageKeys - 1) / kVerifyStageKeys * kVerifyStageKeys;
}

size_t verify_workspace_bytes(int64_t BH, int64_t Sq, int64_t d, int n_split)
{
    if (n_split <= 1)
        return 0;
    const size_t o_bytes = (static_cast<size_t>(n_split) * BH * Sq * d * 4 + 255) & ~size_t(255);
    const size_t l_bytes = (static_cast<size_t>(n_split) * BH * Sq * 4 + 255) & ~size_t(255);
    return o_bytes + l_bytes;
}

// Split count for a device with `num_sms` SMs running two split CTAs each:
// equal-cost CTAs run in waves, so pick the count whose (waves x chunk
// length, plus a fixed per-CTA start-up cost) is smallest.
int verify_auto_splits(int64_t BH, int64_t Sk, int num_sms)
{
    const int64_t slots = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 2;
    const int max_split = static_cast<int>((Sk + kVerifyStageKeys - 1) / kVerifyStageKeys);
    int best = 1;
    double best_cost = 1e300;
    for (int ns = 1; ns <= max_split && ns <= 256; ++ns) {
        const int64_t chunk = verify_chunk_keys(Sk, ns);
        if ((static_cast<int64_t>(ns) - 1) * chunk >= Sk)
            continue;  // an empty trailing chunk: same as fewer splits
        const int64_t ctas = BH * ns;
        const int64_t waves = (ctas + slots - 1) / slots;
        const double cost = static_cast<double>(waves) * static_cast<double>(chunk + 96);
        if (cost < best_cost * 0.999) {
            best_cost = cost;
            best = ns;
        }
    }
    return best;
}

fa_status_t launch_verify(const Problem &p, int n_split, void *workspace, size_t ws_bytes,
                          const VerifyOptions &opt)
{
    if (p.d == 128)
        return verify::launch<128>(p, n_split, workspace, ws_bytes, opt);
    if (p.d == 64)
        return verify::launch<64>(p, n_split, workspace, ws_bytes, opt);
    return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
