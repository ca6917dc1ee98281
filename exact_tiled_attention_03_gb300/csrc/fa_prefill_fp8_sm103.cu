// fa_prefill_fp8_sm103.cu — the attention forward with 8-bit float inputs on
// sm_103a tensor cores.
//
// The FP8 variant of the FlashAttention forward that "FlashAttention,
// speculative decoding, quantisation and parallelism" (The problem it solves)
// and "Lecture 06 — Making Decode Fast" (section 5, FlashAttention-3) name:
// Q, K and V arrive as E4M3 bytes with one fp32 descale per tensor, both
// products run on the FP8 tensor cores, and the rest is the tiled forward of
// "Warmup Guide — Inference Optimization at Depth", Chapter 4 (online
// softmax, causal tiles skipped or masked, O / l written once with the LSE).
//
// It keeps the bf16 kernel's structure (fa_prefill_sm103.cu): persistent CTAs
// take work items (two 128-row query tiles of one head, fa_schedule.cuh) from
// a per-launch counter and pass them to their warps through a shared-memory
// queue; warp 8 feeds a TMA ring of K/V tiles, warp 9 issues tcgen05.mma
// (here .kind::f8f6f4, 32 elements of K per instruction; both warps run their
// loops as a whole warp, one lane issuing), warps 0-3 and 4-7
// run the softmax of one tile each with S and O in tensor memory, and the MMA
// order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) overlaps each tile's softmax
// with the other's products. What differs:
//   * a 128 x 128 E4M3 tile is one 128-byte-swizzled TMA box (16 KB), so
//     the ring holds 8 tiles and Q two, and each tile has a whole 32 KB
//     staging buffer for its bf16 O tile;
//   * P is rounded to E4M3 before O += P V. The exponent is taken against an
//     integer reference M in log2 units, P = 2^(x - M + 4) with
//     x = s * scale * dq * dk * log2(e). M moves (to ceil of the tile max)
//     only when a tile's max exceeds it by more than tau = 4.8, so
//     P <= 2^(4 + 4.8) stays inside E4M3's range (448), and every rescale
//     factor 2^(M_old - M_new) is an exact power of two. As in the bf16
//     kernel the exponentials are computed against the current reference
//     while the tile's max is found, and redone only when the reference moves
//     (rare with tau = 4.8: in practice only on a row's first tile);
//   * relative to the row's final power-of-two max the effective scale of P
//     is 2^4 to 2^9, so every weight of at least 2^-10 of the row max rounds
//     to the same E4M3 value, up to an exact power of two, as with the scale
//     2^7 the reference rounding uses; smaller weights may fall on E4M3's
//     subnormal grid, a difference of at most 2^-12 of the row's largest
//     weight each (measured: 1.31 ms against 1.42 ms for a max-first form
//     whose scale 2^7 allows tau <= 1.8 only);
//   * P is packed four per 32-bit TMEM column (32 columns per 128 keys),
//     the A operand of the P V product read from tensor memory;
//   * the row sum l adds the fp32 P before rounding, so the LSE is that of
//     the unrounded weights; O is scaled by v_descale / l and written as bf16.
// Every wait is bounded as in the bf16 kernel.
#include <cmath>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_schedule.cuh"

namespace fa {
namespace prefill_fp8 {

constexpr int kD = 128;        // head dimension (bytes per E4M3 row)
constexpr int kBlockM = 128;   // query rows per tile = TMEM lanes
constexpr int kBlockN = 128;   // keys per K/V tile
constexpr int kTiles = 2;      // query tiles per item
constexpr int kThreads = 320;  // 2 softmax warpgroups + producer warp + MMA warp
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kChunk = 64;     // S columns per tcgen05.ld in the softmax
constexpr uint32_t kTmemCols = 512;
constexpr int kTileBytes = kBlockM * kD;   // one E4M3 tile = one TMA box (16 KB)
constexpr int kOutBoxBytes = kBlockM * 128;  // a 128-row x 64-column bf16 box
constexpr int kOutTileBytes = kBlockM * kD * 2;
constexpr int kStages = 8;
constexpr int kPShift = 4;       // P = 2^(x - M + kPShift)
constexpr float kTau = 4.8f;     // lazy-rescale threshold, log2 units: 2^(kPShift + kTau) <= 448
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kTiles * kTileBytes;
constexpr int kOffOut = kOffKV + kStages * kTileBytes;
constexpr int kOffBar = kOffOut + kTiles * kOutTileBytes;
constexpr int kSmemBytes = kOffBar + 512 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kTiles == sched::kTiles && kBlockM == sched::kTileRows && kBlockN == sched::kKeyTile,
              "the kernel's tiles are the schedule's items");
// S_t in TMEM columns [128 t, 128 t + 128); P_t (E4M3, four per column)
// over its first 32 columns; O_t in [256 + 128 t, 256 + 128 t + 128).
__device__ __forceinline__ uint32_t col_s(int t) { return 128u * static_cast<uint32_t>(t); }
__device__ __forceinline__ uint32_t col_o(int t) { return 256u + 128u * static_cast<uint32_t>(t); }

struct Params {
    sched::Schedule sc;  // items and their order (fa_schedule.cuh)
    float sl2;           // |scale| * q_descale * k_descale * log2(e)
    // kIdescNegateA for a negative scale, else 0: the S MMAs then form
    // -Q K^T, so the softmax sees the non-negative factor sl2.
    uint32_t idesc_qk_neg;
    // Scale 0: every score is 0 whatever Q holds, so Q tiles are read from
    // head index BH, outside the tensor (TMA fills zeros), and sl2 = 1.
    int zero_q;
    float v_descale;
    float *lse;
    unsigned int *status;
};

// Work-item queue slots, released when the consumers finish their item (at
// most one item beyond the running one per CTA).
constexpr int kQueue = 2;

struct Bars {
    uint64_t q_full[kTiles];   // Q_t of the current item landed (one phase per item with keys)
    uint64_t s_full[kTiles];   // S_t(j) in TMEM (one phase per key tile)
    uint64_t p_full[kTiles];   // P_t(j) in TMEM and O_t rescaled (one phase per key tile)
    uint64_t o_done[kTiles];   // last O_t += P_t V completed (one phase per item with keys)
    uint64_t item_full[kQueue];
    uint64_t item_empty[kQueue];
    uint64_t drain;
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    int items[kQueue];
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

using sched::Item;
using sched::visible_keys;

// 2^k for an integer k <= 0 given as a float (0 below the normal range or for -inf).
__device__ __forceinline__ float exp2_int(float k)
{
    if (!(k > -127.0f))
        return 0.0f;
    return __int_as_float((127 + static_cast<int>(k)) << 23);
}

__global__ void __launch_bounds__(kThreads, 1)
    fa_prefill_fp8_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_o, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *sQ = smem + kOffQ;
    uint8_t *sKV = smem + kOffKV;
    Bars *bars = reinterpret_cast<Bars *>(smem + kOffBar);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(&bars->q_full[t], 1);
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->p_full[t], 4);
            mbar_init(&bars->o_done[t], 1);
        }
        for (int s = 0; s < kQueue; ++s) {
            mbar_init(&bars->item_full[s], 1);
            mbar_init(&bars->item_empty[s], 1 + kSoftmaxWarps);  // MMA thread + softmax warps
        }
        mbar_init(&bars->drain, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->kv_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        bars->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    int *abort_flag = &bars->abort_flag;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        // Takes work items from the launch's counter, publishes each to the
        // other roles through the item queue, then loads its Q tiles and its
        // K_j, V_j through the ring, as the bf16 kernel does.
        // The whole warp runs the loop and polls each barrier together; lane 0
        // alone takes items and issues the copies and arrivals.
        {
            const uint64_t pol_stream = l2_policy_evict_first();  // Q: read once
            const uint64_t pol_keep = l2_policy_evict_last();     // K/V: re-read by other q-blocks
            int it = 0;                         // ring index, continuous across items
            // Q_t loads so far. Each is for an item with keys on tile t, which
            // also completes one o_done[t] phase when its last MMA is done.
            uint32_t q_loads[kTiles] = {0, 0};
            bool ok = true;
            // A bounded wait polled by the whole warp together, made warp-uniform.
            auto wwait = [&](uint64_t *bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.status));
            };
            auto load_kv = [&](int j, int which, int bh) {
                const int s = it % kStages;
                const uint32_t use = it / kStages;
                if (use > 0 && !wwait(&bars->kv_empty[s], (use - 1) & 1))
                    return false;
                if (lane == 0) {
                    fa_check(j * kBlockN < p.sc.Sk && bh < p.sc.BH, p.status);
                    mbar_arrive_expect_tx(&bars->kv_full[s], kTileBytes);
                    tma_load_3d_hint(sKV + s * kTileBytes, which == 0 ? &tm_k : &tm_v,
                                     &bars->kv_full[s], 0, j * kBlockN, bh, pol_keep);
                }
                __syncwarp();
                ++it;
                return true;
            };
            for (int n = 0; ok; ++n) {
                const int slot = n % kQueue;
                if (n >= kQueue && !wwait(&bars->item_empty[slot], ((n / kQueue) - 1) & 1))
                    break;
                int w = 0;
                if (lane == 0) {
                    w = sched::grab_item(p.sc);
                    bars->items[slot] = w;
                    mbar_arrive(&bars->item_full[slot]);  // release: the consumers read items[slot]
                }
                w = __shfl_sync(0xffffffffu, w, 0);
                if (w < 0)
                    break;
                const Item I = sched::decode_item(w, p.sc);
                if (I.n_kv_max == 0)
                    continue;
                // K_0 and V_0 first: they do not wait for the Q buffers.
                ok = load_kv(0, 0, I.bh) && load_kv(0, 1, I.bh);
                for (int t = 0; t < kTiles && ok; ++t) {
                    if (I.n_kv[t] == 0)
                        continue;
                    // Q_t's buffer is free once the previous item's last MMA on
                    // tile t has completed.
                    if (q_loads[t] > 0 && !wwait(&bars->o_done[t], (q_loads[t] - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        fa_check(I.q0[t] < p.sc.Sq && I.bh < p.sc.BH, p.status);
                        mbar_arrive_expect_tx(&bars->q_full[t], kTileBytes);
                        tma_load_3d_hint(sQ + t * kTileBytes, &tm_q, &bars->q_full[t], 0, I.q0[t],
                                         p.zero_q ? p.sc.BH : I.bh, pol_stream);
                    }
                    __syncwarp();
                    ++q_loads[t];
                }
                for (int j = 1; j < I.n_kv_max && ok; ++j)
                    ok = load_kv(j, 0, I.bh) && load_kv(j, 1, I.bh);
            }
            // Drain: every load issued must have landed before the CTA exits.
            if (lane == 0) {
                for (int t = 0; t < kTiles; ++t)
                    if (q_loads[t] > 0)
                        mbar_wait_drain(&bars->q_full[t], (q_loads[t] - 1) & 1, p.status);
                for (int k = max(0, it - kStages); k < it; ++k)
                    mbar_wait_drain(&bars->kv_full[k % kStages], (k / kStages) & 1, p.status);
            }
            __syncwarp();
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // Per item, ring order K_0, V_0, K_1, V_1, ...; issue order S_0(0),
        // S_1(0), then per j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), as in the
        // bf16 kernel, and like it run by the whole warp: the warp polls each
        // barrier together, and one elected lane issues each MMA and commit.
        {
            const uint32_t idesc_qk = idesc_e4m3_f32(kBlockM, kBlockN, false, false) | p.idesc_qk_neg;
            constexpr uint32_t idesc_pv = idesc_e4m3_f32(kBlockM, kD, false, true);
            const uint32_t sQ_a = smem_u32(sQ), sKV_a = smem_u32(sKV);
            // Q and K K-major (a k-step of 32 bytes within the swizzled row);
            // V MN-major: 8-key groups 1024 bytes apart, a k-step of 32 keys
            // = 4 KB; its 128-byte rows are exactly one swizzle atom wide.
            const uint64_t dq0 = smem_desc_sw128(sQ_a, 16, 1024);
            const uint64_t dk0 = smem_desc_sw128(sKV_a, 16, 1024);
            const uint64_t dv0 = smem_desc_sw128(sKV_a, kTileBytes, 1024);
            constexpr uint64_t kTileStep = kTileBytes >> 4;
            auto issue_s = [&](int t, int slot) {
                const uint64_t a0 = dq0 + kTileStep * t, b0 = dk0 + kTileStep * slot;
#pragma unroll
                for (int kk = 0; kk < kD / 32; ++kk)
                    umma_f8_ss_elect(tmem + col_s(t), a0 + 2 * kk, b0 + 2 * kk, idesc_qk, kk > 0 ? 1u : 0u);
            };
            auto issue_pv = [&](int t, int slot, int j) {
                const uint64_t b0 = dv0 + kTileStep * slot;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 32; ++kk)
                    umma_f8_ts_elect(tmem + col_o(t), tmem + col_s(t) + kk * 8,
                               b0 + static_cast<uint64_t>((kk * 32 * 128) >> 4), idesc_pv,
                               (j > 0 || kk > 0) ? 1u : 0u);
            };
            // A bounded wait polled by the whole warp together, made warp-uniform.
            auto wwait = [&](uint64_t *bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.status));
            };
            auto ring_wait = [&](int idx) {
                return wwait(&bars->kv_full[idx % kStages], (idx / kStages) & 1);
            };
            int it = 0;
            uint32_t q_waits[kTiles] = {0, 0}, p_waits[kTiles] = {0, 0};
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int slot = n % kQueue;
                if (!wwait(&bars->item_full[slot], (n / kQueue) & 1))
                    break;
                const int w = __shfl_sync(0xffffffffu, lane == 0 ? bars->items[slot] : 0, 0);
                if (w < 0)
                    break;
                const Item I = sched::decode_item(w, p.sc);
                if (I.n_kv_max == 0) {
                    if (lane == 0)
                        mbar_arrive(&bars->item_empty[slot]);
                    continue;
                }
                // S_t(0) as soon as Q_t is in.
                ok = ring_wait(it);  // K_0
                for (int t = 0; t < kTiles && ok; ++t) {
                    if (I.n_kv[t] == 0)
                        continue;
                    ok = wwait(&bars->q_full[t], (q_waits[t]++) & 1);
                    if (!ok)
                        break;
                    tc_fence_after_sync();
                    issue_s(t, it % kStages);
                    umma_commit_elect(&bars->s_full[t]);
                }
                if (!ok)
                    break;
                umma_commit_elect(&bars->kv_empty[it % kStages]);
                for (int j = 0; j < I.n_kv_max && ok; ++j) {
                    const int iv = it + 2 * j + 1, ik = it + 2 * j + 2;
                    ok = ring_wait(iv);  // V_j
                    if (!ok)
                        break;
                    tc_fence_after_sync();
                    bool k_ready = false;
                    for (int t = 0; t < kTiles && ok; ++t) {
                        if (j >= I.n_kv[t])
                            continue;
                        ok = wwait(&bars->p_full[t], (p_waits[t]++) & 1);
                        if (!ok)
                            break;
                        tc_fence_after_sync();
                        issue_pv(t, iv % kStages, j);
                        if (j + 1 < I.n_kv[t]) {
                            if (!k_ready) {
                                ok = ring_wait(ik);  // K_{j+1}
                                if (!ok)
                                    break;
                                tc_fence_after_sync();
                                k_ready = true;
                            }
                            issue_s(t, ik % kStages);
                            umma_commit_elect(&bars->s_full[t]);
                        } else {
                            umma_commit_elect(&bars->o_done[t]);  // this tile's last PV of the item
                        }
                    }
                    if (!ok)
                        break;
                    umma_commit_elect(&bars->kv_empty[iv % kStages]);
                    if (k_ready)
                        umma_commit_elect(&bars->kv_empty[ik % kStages]);
                }
                it += 2 * I.n_kv_max;
                if (lane == 0)
                    mbar_arrive(&bars->item_empty[slot]);  // every MMA of the item is issued
            }
            // Drain: all MMAs issued by the elected lane complete before TMEM is freed.
            umma_commit_elect(&bars->drain);
            if (lane == 0)
                mbar_wait_drain(&bars->drain, 0, p.status);
            __syncwarp();
        }
    } else if (warp < kSoftmaxWarps) {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = warp / 4;
        const int wq = warp % 4;
        const int r = wq * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_base + col_s(t);
        const uint32_t tO = tmem + lane_base + col_o(t);
        uint8_t *sOut = smem + kOffOut + t * kOutTileBytes;
        const uint32_t sOut_a = smem_u32(sOut);
        const float sl2 = p.sl2;
        const float2 sl2x2 = make_float2(sl2, sl2);
        uint32_t s_waits = 0, o_waits = 0;  // phases of s_full[t] and o_done[t] consumed
        bool ok = true;
        for (int n = 0; ok; ++n) {
            const int slot = n % kQueue;
            // Waits feed .sync.aligned TMEM instructions: keep their outcome
            // warp-uniform. The tile's 4 warps also leave the loop together
            // (their epilogue has named barriers), so the outcome is made
            // tile-uniform here.
            const bool got_item = __all_sync(
                0xffffffffu,
                mbar_wait(&bars->item_full[slot], (n / kQueue) & 1, abort_flag, p.status));
            if (named_bar_or(1 + t, 128, !got_item))
                break;
            const int w = *reinterpret_cast<volatile int *>(&bars->items[slot]);
            if (w < 0)
                break;
            // The item's slot is released when this warp has finished the item.
            auto release = [&]() {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars->item_empty[slot]);
            };
            const Item I = sched::decode_item(w, p.sc);
            const int q0 = I.q0[t], n_kv = I.n_kv[t], mask_from = I.mask_from[t];
            const int i = q0 + r;  // query row
            const int lim = visible_keys(i, p.sc.Sq, p.sc.Sk, p.sc.causal);

            // M: the integer reference (log2 units) of this row's exponentials,
            // -inf until a key is visible. O and l always share it.
            float M = -INFINITY;
            float l = 0.0f;
            for (int j = 0; j < n_kv && ok; ++j) {
                ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[t], (s_waits++) & 1,
                                                       abort_flag, p.status));
                if (!ok)
                    break;
                tc_fence_after_sync();
                const bool masked_tile = j >= mask_from;
                const int key0 = j * kBlockN;
                uint32_t pk[kBlockN / 4];
                float2 acc[4];
                // One pass over S_t: load, mask, and (with_exp) P = 2^(s sl2 + neg)
                // summed into acc and packed as E4M3 into pk. Returns the raw max.
                auto pass = [&](bool with_exp, float neg) {
                    const float2 negx2 = make_float2(neg, neg);
                    float mx = -INFINITY;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        acc[q] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int c0 = 0; c0 < kBlockN; c0 += kChunk) {
                        uint32_t raw[kChunk];
                        tmem_ld64_wait(tS + c0, raw);
                        float sv[kChunk];
#pragma unroll
                        for (int c = 0; c < kChunk; ++c)
                            sv[c] = __uint_as_float(raw[c]);
                        if (masked_tile) {
#pragma unroll
                            for (int c = 0; c < kChunk; ++c)
                                if (key0 + c0 + c >= lim)
                                    sv[c] = -INFINITY;
                        }
                        float part[kChunk / 16];
#pragma unroll
                        for (int k = 0; k < kChunk / 16; ++k) {
                            float x = fmax3(sv[16 * k], sv[16 * k + 1], sv[16 * k + 2]);
#pragma unroll
                            for (int e = 3; e < 15; e += 2)
                                x = fmax3(x, sv[16 * k + e], sv[16 * k + e + 1]);
                            part[k] = fmaxf(x, sv[16 * k + 15]);
                        }
#pragma unroll
                        for (int k = 0; k < kChunk / 16; ++k)
                            mx = fmaxf(mx, part[k]);
                        if (with_exp) {
#pragma unroll
                            for (int c = 0; c < kChunk / 4; ++c) {
                                const float2 xa =
                                    ffma2(make_float2(sv[4 * c], sv[4 * c + 1]), sl2x2, negx2);
                                const float2 xb =
                                    ffma2(make_float2(sv[4 * c + 2], sv[4 * c + 3]), sl2x2, negx2);
                                const float2 ea = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
                                const float2 eb = make_float2(ex2_approx(xb.x), ex2_approx(xb.y));
                                acc[c % 4] = fadd2(acc[c % 4], fadd2(ea, eb));
                                pk[c0 / 4 + c] = pack_e4m3x4(ea.x, ea.y, eb.x, eb.y);
                            }
                        }
                    }
                    return mx;
                };
                const bool spec = __all_sync(0xffffffffu, M != -INFINITY);
                const float mx = pass(spec, spec ? static_cast<float>(kPShift) - M : 0.0f);
                // x_max > M + tau moves the reference to ceil(x_max); NaN-free
                // since M = -inf with x_max = -inf compares false.
                const float xm = mx * sl2;
                const bool move = xm > M + kTau;
                const float M_use = move ? ceilf(xm) : M;
                const float corr = move ? exp2_int(M - M_use) : 1.0f;  // exact; 0 when M = -inf
                if (!spec || __any_sync(0xffffffffu, move)) {
                    pass(true, (M_use == -INFINITY) ? 0.0f : static_cast<float>(kPShift) - M_use);
                    // O_t *= corr (warp-uniform; lanes that did not move multiply
                    // by 1). PV_t(j-1) has completed: S_t(j), committed after it,
                    // is done.
                    if (j > 0 && __any_sync(0xffffffffu, move)) {
                        const float2 cx2 = make_float2(corr, corr);
#pragma unroll
                        for (int c0 = 0; c0 < kD; c0 += 32) {
                            uint32_t o[32];
                            tmem_ld32_wait(tO + c0, o);
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                const float2 v = fmul2(make_float2(__uint_as_float(o[2 * c]),
                                                                   __uint_as_float(o[2 * c + 1])),
                                                       cx2);
                                o[2 * c] = __float_as_uint(v.x);
                                o[2 * c + 1] = __float_as_uint(v.y);
                            }
                            tmem_st32(tO + c0, o);
                        }
                    }
                }
                tmem_st32(tS, pk);  // P (E4M3, four per column) over S_t's first 32 columns
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars->p_full[t]);
                const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
                const float2 a = fadd2(a01, a23);
                l = l * corr + (a.x + a.y);
                M = M_use;
            }

            // -------------------------------------------------------- epilogue
            // O * v_descale / l into this tile's staging buffer (swizzled like
            // the TMA boxes), two TMA stores, then the LSE. The next item's P_t
            // is published only after these TMEM reads, so its PV_t(0) cannot
            // overwrite O_t early.
            if (q0 >= p.sc.Sq) {
                release();
                continue;
            }
            // The previous item's stores may still be reading the staging
            // buffer: their issuer waits here, before the barrier below, so the
            // buffer is rewritten only after those reads (the wait is not taken
            // at the end of that epilogue, where it sat on the tile's critical path).
            if (r == 0)
                tma_store_wait_read_all();
            bool got = ok;
            if (got && n_kv > 0) {
                got = __all_sync(0xffffffffu, mbar_wait(&bars->o_done[t], (o_waits++) & 1,
                                                        abort_flag, p.status));
                if (got)
                    tc_fence_after_sync();
            }
            // The tile's 4 warps take the barriers below together or not at all.
            if (named_bar_or(1 + t, 128, !got)) {
                ok = false;
                break;
            }
            const float mul = (l > 0.0f) ? p.v_descale / l : 0.0f;
#pragma unroll
            for (int c0 = 0; c0 < kD; c0 += 32) {
                uint32_t o[32];
                if (n_kv > 0) {
                    tmem_ld32_wait(tO + c0, o);
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        o[c] = 0u;
                }
                uint32_t pkd[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2)
                    pkd[c / 2] = pack_bf16x2(__uint_as_float(o[c]) * mul,
                                             __uint_as_float(o[c + 1]) * mul);
                const int box = c0 / 64;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t chunk = ((c0 % 64) / 8) + q;
                    st_shared_v4(sOut_a + box * kOutBoxBytes +
                                     sw128_offset(static_cast<uint32_t>(r), chunk),
                                 pkd[q * 4], pkd[q * 4 + 1], pkd[q * 4 + 2], pkd[q * 4 + 3]);
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(1 + t, 128);
            if (r == 0) {
                fa_check(q0 < p.sc.Sq && I.bh < p.sc.BH, p.status);
                for (int b = 0; b < kD / 64; ++b)
                    tma_store_3d(&tm_o, sOut + b * kOutBoxBytes, b * 64, q0, I.bh);
                tma_store_commit();
                // The reads of the buffer are waited for at the next epilogue;
                // the writes to global memory finish on their own.
            }
            if (i < p.sc.Sq) {
                // lse = ln 2 * (M - kPShift + log2 l), in units of the scaled scores
                const float lse = (l > 0.0f)
                                      ? (M - static_cast<float>(kPShift)) * 0.69314718055994531f +
                                            logf(l)
                                      : -INFINITY;
                if (fa_check(I.bh < p.sc.BH, p.status))
                    p.lse[static_cast<size_t>(I.bh) * p.sc.Sq + i] = lse;
            }
            release();
        }
    }

    // Threads that issued TMA stores wait for their writes (not only for the
    // shared-memory reads) before the CTA exits, so that the next kernel in the
    // stream reads them.
    tma_store_wait_all();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == kMmaWarp)
        tmem_dealloc(tmem, kTmemCols);
    if (threadIdx.x == 0)
        sched::finish_cta(p.sc);
}

}  // namespace prefill_fp8

fa_status_t launch_prefill_fp8_sm103(const Problem &pr, float q_descale, float k_descale,
                                     float v_descale)
{
    using namespace prefill_fp8;
    if (pr.d != kD)
        return FA_ERR_UNSUPPORTED;
    CUtensorMap tq, tk, tv, to;
    const uint64_t BH = static_cast<uint64_t>(pr.B * pr.H);
    if (!encode_tmap_u8_3d(&tq, pr.q, kD, pr.Sq, BH, kBlockM) ||
        !encode_tmap_u8_3d(&tk, pr.k, kD, pr.Sk, BH, kBlockN) ||
        !encode_tmap_u8_3d(&tv, pr.v, kD, pr.Sk, BH, kBlockN) ||
        !encode_tmap_bf16_3d(&to, pr.o, kD, pr.Sq, BH, kBlockM))
        return FA_ERR_CUDA;
    Params p;
    // At scale 0 the scores are 0 (zero Q tiles), every weight is 2^kPShift
    // and the reference settles at 0 on the first visible key.
    p.zero_q = pr.scale == 0.0f ? 1 : 0;
    p.sl2 = p.zero_q ? 1.0f
                     : static_cast<float>(std::fabs(static_cast<double>(pr.scale)) * q_descale *
                                          k_descale * 1.4426950408889634);
    if (!std::isfinite(p.sl2))
        return FA_ERR_UNSUPPORTED;
    p.idesc_qk_neg = std::signbit(pr.scale) ? kIdescNegateA : 0u;
    unsigned grid = 0;
    const fa_status_t st =
        sched::make_schedule(pr, 2.0 * static_cast<double>(pr.Sk) * kD, &p.sc, &grid);
    if (st != FA_OK)
        return st;
    p.v_descale = v_descale;
    p.lse = pr.lse;
    p.status = pr.status;
    auto kern = fa_prefill_fp8_kernel;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
        return FA_ERR_CUDA;
    kern<<<grid, kThreads, kSmemBytes, pr.stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
