// fa_prefill_sm103.cu — tiled exact attention forward on sm_103a tensor cores.
//
// The method is the FlashAttention forward of "Warmup Guide — Inference
// Optimization at Depth", Chapter 4 and "FlashAttention, speculative
// decoding, quantisation and parallelism", Mechanics: each block of query
// rows stays on chip, K/V blocks stream through, S = Q K^T * scale is formed
// one tile at a time, the online softmax of Chapter 3 keeps a running max m
// and sum l and rescales the unnormalised accumulator by exp(m_old - m_new),
// key blocks above the causal diagonal are skipped and the diagonal ones
// masked, and O / l is written once together with the per-row statistics
// (LSE = m + ln l).
//
// The GB300 shape of it (not the pages' SRAM/Hopper design):
//   * one CTA per SM owns two 128-row query tiles of one (batch, head);
//     both share every K/V tile it loads;
//   * warp 8 (producer) moves Q once and then K_j, V_j through a ring of
//     shared-memory stages with TMA (128-byte swizzle), one mbarrier pair per
//     stage;
//   * warp 9 (one elected thread) issues tcgen05.mma: S_t = Q_t K_j^T into
//     tensor memory (TMEM), and O_t += P_t V_j with P_t read from TMEM and V
//     read MN-major straight from its row-major tile; completion is signalled
//     with tcgen05.commit. Issue order per key tile j: PV_0(j), S_0(j+1),
//     PV_1(j), S_1(j+1), so each tile's softmax overlaps the other tile's
//     two GEMMs (ping-pong);
//   * warps 0-3 and 4-7 are one softmax warpgroup per query tile; thread r
//     owns row r (TMEM lane r). It streams its S row out of TMEM in 64-column
//     chunks, masks, and computes exp2 of the log2(e)-scaled logits against
//     its current reference max while it finds the tile's max; only if that
//     max exceeds the reference by more than 2^8 (or on the row's first
//     tile) does it recompute the row against the new max and rescale its O
//     row in TMEM. It then writes P (bf16) over its S row in TMEM. At the end
//     it divides by l, writes the bf16 O row into shared memory for a TMA
//     store and writes its LSE.
// Every wait is bounded; on expiry the CTA stops, drains what it has in
// flight, frees its tensor memory and sets the device status word.
#include <cmath>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace prefill {

constexpr int kBlockM = 128;   // query rows per tile = TMEM lanes
constexpr int kBlockN = 128;   // keys per K/V tile
constexpr int kTiles = 2;      // query tiles per CTA
constexpr int kThreads = 320;  // 2 softmax warpgroups + producer warp + MMA warp
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;

// Columns of S a softmax thread pulls from TMEM at a time (64 measured faster
// on GB300 than 32, with or without double-buffered loads, and needs no
// register spills at 320 threads).
constexpr int kChunk = 64;
constexpr uint32_t kTmemCols = 512;
constexpr int kBoxBytes = kBlockM * 128;  // one 128-row x 64-column bf16 box (16 KB)
// Lazy rescale threshold, in log2 units of the exponent (factor 256).
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct Cfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = kBlockM * D * 2;  // Q, K, V or O tile
    static constexpr int kStages = (D == 128) ? 5 : 10;  // ~160 KB of K/V ring
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + kTiles * kTileBytes;
    static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
    static constexpr int kBarBytes = 512;
    static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + alignment slack
    // S_t in columns [128 t, 128 t + 128); P_t (bf16, two per column) is
    // written over the first 64 columns of S_t once S_t is in registers.
    static constexpr uint32_t kColS0 = 0, kColS1 = 128;
    static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
    static_assert(kColO1 + D <= kTmemCols, "TMEM budget");
};

struct Params {
    int Sq, Sk, BH, n_qblk;
    int causal;
    float scale;       // softmax scale
    float scale_log2;  // scale * log2(e)
    float *lse;
    unsigned int *status;
};

struct Bars {
    uint64_t q_full;
    uint64_t s_full[kTiles];   // S_t(j) in TMEM (one phase per key tile)
    uint64_t p_full[kTiles];   // P_t(j) in TMEM and O_t rescaled (one phase per key tile)
    uint64_t o_done[kTiles];   // last O_t += P_t V completed (one phase)
    uint64_t drain;
    uint64_t kv_full[16];
    uint64_t kv_empty[16];
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

// Number of keys visible to query row i (bottom-right causal alignment).
__device__ __forceinline__ int visible_keys(int i, int Sq, int Sk, int causal)
{
    if (!causal)
        return Sk;
    int n = i + (Sk - Sq) + 1;
    return n < 0 ? 0 : (n > Sk ? Sk : n);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, const Params p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms.
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sKV = smem + C::kOffKV;
    Bars *bars = reinterpret_cast<Bars *>(smem + C::kOffBar);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    // Head-major order, heaviest query block first within each head: the CTAs
    // running at the same time share a few heads' K/V in L2, and with the
    // causal mask the last query blocks (most keys) start first.
    const int bh = static_cast<int>(blockIdx.x / p.n_qblk);
    const int qblk = p.n_qblk - 1 - static_cast<int>(blockIdx.x % p.n_qblk);

    int q0[kTiles], n_kv[kTiles], mask_from[kTiles];
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
        q0[t] = qblk * (kTiles * kBlockM) + t * kBlockM;
        if (q0[t] < p.Sq) {
            const int last = min(q0[t] + kBlockM - 1, p.Sq - 1);
            n_kv[t] = (visible_keys(last, p.Sq, p.Sk, p.causal) + kBlockN - 1) / kBlockN;
            mask_from[t] = visible_keys(q0[t], p.Sq, p.Sk, p.causal) / kBlockN;
        } else {
            n_kv[t] = 0;
            mask_from[t] = 0;
        }
    }
    const int n_kv_max = max(n_kv[0], n_kv[1]);
    const bool any_tile = q0[0] < p.Sq;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->p_full[t], 4);
            mbar_init(&bars->o_done[t], 1);
        }
        mbar_init(&bars->drain, 1);
        for (int s = 0; s < C::kStages; ++s) {
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
        if (lane == 0 && any_tile) {
            const uint64_t pol_stream = l2_policy_evict_first();  // Q: read once
            const uint64_t pol_keep = l2_policy_evict_last();     // K/V: re-read by other q-blocks
            uint32_t q_bytes = 0;
            for (int t = 0; t < kTiles; ++t)
                if (q0[t] < p.Sq)
                    q_bytes += C::kTileBytes;
            mbar_arrive_expect_tx(&bars->q_full, q_bytes);
            for (int t = 0; t < kTiles; ++t)
                if (q0[t] < p.Sq)
                    for (int b = 0; b < C::kBoxes; ++b)
                        tma_load_3d_hint(sQ + t * C::kTileBytes + b * kBoxBytes, &tm_q,
                                         &bars->q_full, b * 64, q0[t], bh, pol_stream);
            int it = 0;
            bool ok = true;
            for (int j = 0; j < n_kv_max && ok; ++j) {
                for (int which = 0; which < 2 && ok; ++which, ++it) {
                    const int s = it % C::kStages;
                    const uint32_t use = it / C::kStages;
                    if (use > 0 &&
                        !mbar_wait(&bars->kv_empty[s], (use - 1) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars->kv_full[s], C::kTileBytes);
                    const CUtensorMap *tm = which == 0 ? &tm_k : &tm_v;
                    for (int b = 0; b < C::kBoxes; ++b)
                        tma_load_3d_hint(sKV + s * C::kTileBytes + b * kBoxBytes, tm,
                                         &bars->kv_full[s], b * 64, j * kBlockN, bh, pol_keep);
                }
            }
            // Drain: every load issued must have landed before the CTA exits.
            mbar_wait_drain(&bars->q_full, 0, p.status);
            for (int k = max(0, it - C::kStages); k < it; ++k)
                mbar_wait_drain(&bars->kv_full[k % C::kStages], (k / C::kStages) & 1, p.status);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // Ring order of the loads: K_0, V_0, K_1, V_1, ... (K_j at index 2j,
        // V_j at 2j+1), consumed in the same order. Issue order: S_0(0), S_1(0),
        // then per j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1). S_t(j+1) overwrites
        // the TMEM columns that held P_t(j); the tensor pipe executes one
        // thread's MMAs in order, so PV_t(j) has read P_t(j) by then.
        if (lane == 0 && any_tile && n_kv_max > 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kBlockM, kBlockN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kBlockM, D, false, true);
            const uint32_t colS[kTiles] = {C::kColS0, C::kColS1};
            const uint32_t colO[kTiles] = {C::kColO0, C::kColO1};
            const uint32_t sQ_a = smem_u32(sQ), sKV_a = smem_u32(sKV);
            // Descriptors are built once; a stage, tile or k-step only moves the
            // start address (bits 0-13, in 16-byte units) by a constant, which
            // never carries out of the field (shared memory is below 256 KB).
            const uint64_t dq0 = smem_desc_sw128(sQ_a, 16, 1024);
            const uint64_t dk0 = smem_desc_sw128(sKV_a, 16, 1024);
            const uint64_t dv0 = smem_desc_sw128(sKV_a, kBoxBytes, 1024);
            constexpr uint64_t kTileStep = C::kTileBytes >> 4;
            auto issue_s = [&](int t, int slot) {
                const uint64_t a0 = dq0 + kTileStep * t, b0 = dk0 + kTileStep * slot;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t koff = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
                    umma_bf16_ss(tmem + colS[t], a0 + koff, b0 + koff, idesc_qk, kk > 0 ? 1u : 0u);
                }
            };
            // One 64-key half of O_t += P_t V_j (k-steps 4h .. 4h+3).
            auto issue_pv_half = [&](int t, int slot, int j, int h) {
                const uint64_t b0 = dv0 + kTileStep * slot;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int kk = 4 * h + q;
                    umma_bf16_ts(tmem + colO[t], tmem + colS[t] + kk * 8,
                                 b0 + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_pv,
                                 (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            auto ring_wait = [&](int idx) {
                return mbar_wait(&bars->kv_full[idx % C::kStages], (idx / C::kStages) & 1,
                                 abort_flag, p.status);
            };
            bool ok = mbar_wait(&bars->q_full, 0, abort_flag, p.status) && ring_wait(0);  // K_0
            if (ok) {
                tc_fence_after_sync();
                for (int t = 0; t < kTiles; ++t)
                    if (n_kv[t] > 0) {
                        issue_s(t, 0);
                        umma_commit(&bars->s_full[t]);
                    }
                umma_commit(&bars->kv_empty[0]);
            }
            for (int j = 0; j < n_kv_max && ok; ++j) {
                const int iv = 2 * j + 1, ik = 2 * j + 2;
                ok = ring_wait(iv);  // V_j
                if (!ok)
                    break;
                tc_fence_after_sync();
                bool k_ready = false;
                for (int t = 0; t < kTiles && ok; ++t) {
                    if (j >= n_kv[t])
                        continue;
                    ok = mbar_wait(&bars->p_full[t], j & 1, abort_flag, p.status);
                    if (!ok)
                        break;
                    tc_fence_after_sync();
                    issue_pv_half(t, iv % C::kStages, j, 0);
                    issue_pv_half(t, iv % C::kStages, j, 1);
                    if (j + 1 < n_kv[t]) {
                        if (!k_ready) {
                            ok = ring_wait(ik);  // K_{j+1}
                            if (!ok)
                                break;
                            tc_fence_after_sync();
                            k_ready = true;
                        }
                        issue_s(t, ik % C::kStages);
                        umma_commit(&bars->s_full[t]);
                    } else {
                        umma_commit(&bars->o_done[t]);  // this tile's last PV
                    }
                }
                if (!ok)
                    break;
                umma_commit(&bars->kv_empty[iv % C::kStages]);
                if (k_ready)
                    umma_commit(&bars->kv_empty[ik % C::kStages]);
            }
            // Drain: all MMAs issued by this thread complete before TMEM is freed.
            umma_commit(&bars->drain);
            mbar_wait_drain(&bars->drain, 0, p.status);
        }
    } else if (warp < kSoftmaxWarps) {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = warp / 4;              // query tile of this warpgroup
        const int wq = warp % 4;             // TMEM lane quarter of this warp
        const int r = wq * 32 + lane;        // row within the tile
        const int i = q0[t] + r;             // query row
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_base + (t == 0 ? C::kColS0 : C::kColS1);
        const uint32_t tO = tmem + lane_base + (t == 0 ? C::kColO0 : C::kColO1);
        uint8_t *sOut = sQ + t * C::kTileBytes;  // Q_t's buffer, reused for the O tile
        const uint32_t sOut_a = smem_u32(sOut);
        const int lim = visible_keys(i, p.Sq, p.Sk, p.causal);
        const float sl2 = p.scale_log2;

        // m: the reference max of this row's exponentials (raw score units,
        // scale > 0). It is updated lazily: only when a tile's max exceeds it by
        // more than 2^kRescaleLog2 in the exponent (or on the first visible key).
        // O and l always share the same reference, so the result stays exact,
        // and P = 2^((s - m) * sl2) stays <= 2^kRescaleLog2.
        float m = -INFINITY;
        float l = 0.0f;       // running sum of 2^((s - m) * sl2)
        bool ok = true;
        if (q0[t] < p.Sq)
            ok = mbar_wait(&bars->q_full, 0, abort_flag, p.status);
        // Waits feed .sync.aligned TMEM instructions: keep their outcome warp-uniform.
        ok = __all_sync(0xffffffffu, ok);

        const float2 sl2x2 = make_float2(sl2, sl2);
        for (int j = 0; j < n_kv[t] && ok; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[t], j & 1, abort_flag, p.status));
            if (!ok)
                break;
            tc_fence_after_sync();
            const bool masked_tile = j >= mask_from[t];
            const int key0 = j * kBlockN;
            uint32_t pk[kBlockN / 2];
            float2 acc[4];
            // One pass over S_t in chunks of kChunk columns: load, mask, and (when
            // `with_exp`) p = 2^(s*sl2 + neg), accumulated into acc and packed
            // into pk. Returns the max of the raw scores it saw.
            auto pass = [&](bool with_exp, float neg) {
                const float2 negx2 = make_float2(neg, neg);
                float mx = -INFINITY;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[q] = make_float2(0.f, 0.f);
                // Process one chunk of kChunk scores starting at column c0.
                auto consume = [&](const uint32_t *raw, int c0) {
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
                        for (int c = 0; c < kChunk / 2; ++c) {
                            const float2 x = ffma2(make_float2(sv[2 * c], sv[2 * c + 1]), sl2x2, negx2);
                            const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                            acc[c % 4] = fadd2(acc[c % 4], e);
                            pk[c0 / 2 + c] = pack_bf16x2(e.x, e.y);
                        }
                    }
                };
#pragma unroll
                for (int c0 = 0; c0 < kBlockN; c0 += kChunk) {
                    uint32_t raw[kChunk];
                    tmem_ld64_wait(tS + c0, raw);
                    consume(raw, c0);
                }
                return mx;
            };
            // Speculative pass: when every lane already has a reference max, the
            // exponentials are computed against it while the tile's max is found.
            const bool spec = __all_sync(0xffffffffu, m != -INFINITY);
            const float mx = pass(spec, spec ? -m * sl2 : 0.0f);
            // The reference moves only when the tile's max exceeds it by more
            // than 2^kRescaleLog2 (or on the first visible key); O and l always
            // share it, so the result stays exact and P stays <= 2^kRescaleLog2.
            // NaN (both -inf) compares false: nothing visible yet, keep m.
            const float m_new = fmaxf(m, mx);
            const bool move = (m_new - m) * sl2 > kRescaleLog2;
            const float m_use = move ? m_new : m;
            const float corr = move ? ex2_approx((m - m_use) * sl2) : 1.0f;  // 0 when m = -inf
            if (!spec || __any_sync(0xffffffffu, move)) {
                // Second pass with the moved reference (lanes that did not move
                // recompute the same values). S_t is still intact: P has not
                // been written yet.
                pass(true, (m_use == -INFINITY) ? 0.0f : -m_use * sl2);
                // O_t *= corr (warp-uniform; lanes that did not move multiply by
                // 1). PV_t(j-1) has completed: S_t(j), committed after it, is done.
                if (j > 0 && __any_sync(0xffffffffu, move)) {
                    const float2 cx2 = make_float2(corr, corr);
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
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
            // P (bf16 pairs) over S_t's first 64 columns, then publish.
            {
                uint32_t lo[32], hi[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    lo[c] = pk[c];
                    hi[c] = pk[32 + c];
                }
                tmem_st32(tS, lo);
                tmem_st32(tS + 32, hi);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->p_full[t]);
            const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
            const float2 a = fadd2(a01, a23);
            l = l * corr + (a.x + a.y);
            m = m_use;
        }

        // ------------------------------------------------------------ epilogue
        if (ok && q0[t] < p.Sq) {
            if (n_kv[t] > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done[t], 0, abort_flag, p.status));
                tc_fence_after_sync();
            }
            if (ok) {
                const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    if (n_kv[t] > 0) {
                        tmem_ld32_wait(tO + c0, o);
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            o[c] = 0u;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 2)
                        pk[c / 2] = pack_bf16x2(__uint_as_float(o[c]) * inv_l,
                                                __uint_as_float(o[c + 1]) * inv_l);
                    const int box = c0 / 64;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t chunk = ((c0 % 64) / 8) + q;
                        st_shared_v4(sOut_a + box * kBoxBytes +
                                         sw128_offset(static_cast<uint32_t>(r), chunk),
                                     pk[q * 4], pk[q * 4 + 1], pk[q * 4 + 2], pk[q * 4 + 3]);
                    }
                }
                if (i < p.Sq) {
                    const float lse = (l > 0.0f) ? m * p.scale + logf(l) : -INFINITY;
                    p.lse[static_cast<size_t>(bh) * p.Sq + i] = lse;
                }
            }
        }
        tc_fence_before_sync();
        fence_proxy_async_smem();
        named_bar_sync(1 + t, 128);
        if (r == 0 && ok && q0[t] < p.Sq && !*reinterpret_cast<volatile int *>(abort_flag)) {
            for (int b = 0; b < C::kBoxes; ++b)
                tma_store_3d(&tm_o, sOut + b * kBoxBytes, b * 64, q0[t], bh);
            tma_store_commit();
            tma_store_wait_read_all();  // the staging buffer may go; the writes finish on their own
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == kMmaWarp)
        tmem_dealloc(tmem, kTmemCols);
}

template <int D>
fa_status_t launch(const Problem &pr)
{
    using C = Cfg<D>;
    CUtensorMap tq, tk, tv, to;
    const uint64_t BH = static_cast<uint64_t>(pr.B * pr.H);
    if (!encode_tmap_bf16_3d(&tq, pr.q, D, pr.Sq, BH, kBlockM) ||
        !encode_tmap_bf16_3d(&tk, pr.k, D, pr.Sk, BH, kBlockN) ||
        !encode_tmap_bf16_3d(&tv, pr.v, D, pr.Sk, BH, kBlockN) ||
        !encode_tmap_bf16_3d(&to, pr.o, D, pr.Sq, BH, kBlockM))
        return FA_ERR_CUDA;
    Params p;
    p.Sq = static_cast<int>(pr.Sq);
    p.Sk = static_cast<int>(pr.Sk);
    p.BH = static_cast<int>(BH);
    p.n_qblk = static_cast<int>((pr.Sq + kTiles * kBlockM - 1) / (kTiles * kBlockM));
    p.causal = pr.causal ? 1 : 0;
    p.scale = pr.scale;
    p.scale_log2 = pr.scale * 1.4426950408889634f;
    p.lse = pr.lse;
    p.status = pr.status;
    auto kern = fa_prefill_kernel<D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return FA_ERR_CUDA;

    const uint64_t grid = static_cast<uint64_t>(p.n_qblk) * BH;
    if (grid > 0x7FFFFFFFull)
        return FA_ERR_UNSUPPORTED;
    kern<<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, pr.stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace prefill

fa_status_t launch_prefill_sm103(const Problem &p)
{
    if (p.d == 128)
        return prefill::launch<128>(p);
    if (p.d == 64)
        return prefill::launch<64>(p);
    return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
