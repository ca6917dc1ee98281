// fa_backward_sm103.cu — gradients of the exact attention forward on sm_103a.
//
// The backward the pages describe ("Warmup Guide — Inference Optimization at
// Depth", Chapter 4): P is not stored; its tiles are recomputed from Q and K
// with the per-row statistics the forward kept (LSE = m + ln l), so
// P_ij = exp(scale * q_i . k_j - LSE_i) exactly. With dO the upstream
// gradient and D_i = dO_i . O_i:
//     dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),
//     dK = scale * dS^T Q,  dQ = scale * dS K.
// Three kernels:
//   * fa_bwd_prep_kernel: D_i and LSE in the exp2 domain (lse2 = LSE *
//     log2 e; +inf for rows with no visible key, so their P is 0), into
//     row-padded workspace rows;
//   * fa_bwd_dkdv_kernel: one CTA per 128-key tile of one (b, h). It keeps K
//     and V in shared memory, streams (Q_i, dO_i, lse2_i, D_i) for every
//     query tile that sees the key tile, forms S^T = K Q_i^T and
//     dP^T = V dO_i^T with tcgen05 MMAs into tensor memory, lets one thread
//     per key rebuild P^T and dS^T (bf16, written back over their own TMEM
//     columns), and accumulates dV += P^T dO_i and dK += dS^T Q_i with the A
//     operand read from TMEM;
//   * fa_bwd_dq_kernel: one CTA per 128-row query tile; for every key tile
//     it sees: S = Q K_j^T, dP = dO V_j^T, then one thread per query rebuilds
//     dS and dQ += dS K_j (A from TMEM).
// Both gradient kernels split each 128-column score tile into two halves of
// 64 columns with their own barriers: the MMA warp issues half 0's scores,
// then half 1's; warps 0-3 rebuild half 0 while the tensor core computes
// half 1, and half 0's gradient MMAs run while warps 4-7 rebuild half 1.
// The two warps of a sub-partition share TMEM lanes (lane quarter = warp
// mod 4) and split the columns. Each half packs its bf16 result into its own
// first 32 columns (0-31 and 64-95), so neither half overwrites columns the
// other has yet to read.
// The warp roles, TMA ring, mbarrier waits (bounded) and descriptor
// encodings are those of the forward kernel.
#include <cmath>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace bwd {

constexpr int kBlock = 128;             // keys or queries per tile = TMEM lanes
constexpr int kMathThreads = 256;       // warps 0-7: lane quarter warp % 4, column half warp / 4
constexpr int kThreads = kMathThreads + 64;  // + warp 8 producer, warp 9 MMA
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kHalf = kBlock / 2;        // score columns per half
constexpr uint32_t kTmemCols = 512;
constexpr int kBoxBytes = kBlock * 128;  // 128 rows x 64 columns bf16
constexpr int kChunk = 32;               // TMEM columns a math thread handles at a time

struct Params {
    int Sq, Sk, Sq_pad, BH, n_qtiles, n_ktiles;
    int causal;
    float scale, scale_log2;
    const float *lse2;  // [BH, Sq_pad], +inf padding
    const float *Dvec;  // [BH, Sq_pad], 0 padding
    unsigned int *status;
};

__device__ __forceinline__ int visible_keys(int i, int Sq, int Sk, int causal)
{
    if (!causal)
        return Sk;
    int n = i + (Sk - Sq) + 1;
    return n < 0 ? 0 : (n > Sk ? Sk : n);
}

// Untiled bulk copy global -> shared (16-byte aligned, multiple of 16 bytes).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- prep
// One warp per (bh, row of the padded row range).
template <int D>
__global__ void __launch_bounds__(256)
    fa_bwd_prep_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                       const float *__restrict__ lse, float *__restrict__ lse2,
                       float *__restrict__ Dvec, int BH, int Sq, int Sq_pad)
{
    const int row = blockIdx.x * 8 + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= BH * Sq_pad)
        return;
    const int bh = row / Sq_pad, i = row % Sq_pad;
    float acc = 0.0f;
    float l2 = INFINITY;
    if (i < Sq) {
        const size_t base = (static_cast<size_t>(bh) * Sq + i) * D;
#pragma unroll
        for (int t = lane; t < D; t += 32)
            acc = fmaf(__bfloat162float(o[base + t]), __bfloat162float(dout[base + t]), acc);
        const float L = lse[static_cast<size_t>(bh) * Sq + i];
        l2 = (L == -INFINITY) ? INFINITY : L * 1.4426950408889634f;
    }
#pragma unroll
    for (int off = 16; off > 0; off /= 2)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
        Dvec[row] = acc;
        lse2[row] = l2;
    }
}

// Pack two fp32 values as a bf16 pair (element 2c in the low half).
__device__ __forceinline__ uint32_t pk2(float a, float b) { return pack_bf16x2(a, b); }

// The epilogue of both gradient kernels: a 128 x D fp32 tile in TMEM (this
// thread's lane = row r; `taddr` addresses column 0 of that lane) times
// `mul`, to bf16, through shared memory (Q-tile sized staging at `stage`,
// swizzled like the TMA box), then TMA-stored. Column half `half` of the
// tile is this thread's; all math threads take part.
template <int D>
__device__ __forceinline__ void store_tile(uint32_t taddr, float mul, bool have, uint8_t *stage,
                                           const CUtensorMap *map, int row0, int bh, int r,
                                           int half, uint32_t bar_id)
{
    const uint32_t st_a = smem_u32(stage);
#pragma unroll
    for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
        uint32_t v[32];
        if (have) {
            tmem_ld32_wait(taddr + c0, v);
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c)
                v[c] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2)
            pk[c / 2] = pk2(__uint_as_float(v[c]) * mul, __uint_as_float(v[c + 1]) * mul);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t chunk = ((c0 % 64) / 8) + q;
            st_shared_v4(st_a + (c0 / 64) * kBoxBytes + sw128_offset(static_cast<uint32_t>(r), chunk),
                         pk[q * 4], pk[q * 4 + 1], pk[q * 4 + 2], pk[q * 4 + 3]);
        }
    }
    fence_proxy_async_smem();
    named_bar_sync(bar_id, kMathThreads);
    if (r == 0 && half == 0) {
        for (int b = 0; b < D / 64; ++b)
            tma_store_3d(map, stage + b * kBoxBytes, b * 64, row0, bh);
        tma_store_commit();
        tma_store_wait_read_all();
    }
    named_bar_sync(bar_id, kMathThreads);
}

// ---------------------------------------------------------------- dK, dV
template <int D>
struct KvCfg {
    static constexpr int kTile = kBlock * D * 2;
    static constexpr int kStages = (D == 128) ? 2 : 4;           // (Q_i, dO_i) pairs
    static constexpr int kOffK = 0, kOffV = kTile, kOffRing = 2 * kTile;
    static constexpr int kStageBytes = 2 * kTile;
    static constexpr int kOffVec = kOffRing + kStages * kStageBytes;  // lse2, D per stage
    static constexpr int kOffBar = kOffVec + kStages * 1024;
    static constexpr int kSmem = kOffBar + 512 + 1024;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
    static_assert(kColDK + D <= kTmemCols, "TMEM budget");
};

struct KvBars {
    uint64_t kv_full;
    uint64_t full[4], empty[4];
    uint64_t st_full[2];  // half h of S^T and dP^T of the current query tile in TMEM
    uint64_t p_full[2];   // half h of P^T and dS^T written back (4 warp arrivals)
    uint64_t o_done;   // last dV / dK MMAs completed
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dk,
                       const __grid_constant__ CUtensorMap tm_dv, const Params p)
{
    using C = KvCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    KvBars *bars = reinterpret_cast<KvBars *>(smem + C::kOffBar);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.x / p.n_ktiles;
    const int kt = p.n_ktiles - 1 - static_cast<int>(blockIdx.x % p.n_ktiles);  // long first
    const int kv0 = kt * kBlock;
    const int off = p.Sk - p.Sq;
    // Query tiles whose last row sees key kv0: [qt0, n_qtiles).
    int qt0 = 0;
    if (p.causal) {
        const int need = kv0 - off - (kBlock - 1);  // first row that can see kv0, rounded down
        qt0 = need <= 0 ? 0 : (need + kBlock - 1) / kBlock;
    }
    const int n_q = max(0, p.n_qtiles - qt0);

    if (threadIdx.x == 0) {
        mbar_init(&bars->kv_full, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bars->st_full[h], 1);
            mbar_init(&bars->p_full[h], 4);
        }
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    int *abort_flag = &bars->abort_flag;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars->kv_full, 2 * C::kTile);
            for (int b = 0; b < D / 64; ++b) {
                tma_load_3d(smem + C::kOffK + b * kBoxBytes, &tm_k, &bars->kv_full, b * 64, kv0, bh);
                tma_load_3d(smem + C::kOffV + b * kBoxBytes, &tm_v, &bars->kv_full, b * 64, kv0, bh);
            }
            int n = 0;
            for (; n < n_q; ++n) {
                const int s = n % C::kStages;
                const uint32_t use = n / C::kStages;
                if (use > 0 && !mbar_wait(&bars->empty[s], (use - 1) & 1, abort_flag, p.status))
                    break;
                const int q0 = (qt0 + n) * kBlock;
                uint8_t *st = smem + C::kOffRing + s * C::kStageBytes;
                mbar_arrive_expect_tx(&bars->full[s], C::kStageBytes + 1024);
                for (int b = 0; b < D / 64; ++b) {
                    tma_load_3d(st + b * kBoxBytes, &tm_q, &bars->full[s], b * 64, q0, bh);
                    tma_load_3d(st + C::kTile + b * kBoxBytes, &tm_do, &bars->full[s], b * 64, q0, bh);
                }
                const size_t vrow = static_cast<size_t>(bh) * p.Sq_pad + q0;
                bulk_load(smem + C::kOffVec + s * 1024, p.lse2 + vrow, 512, &bars->full[s]);
                bulk_load(smem + C::kOffVec + s * 1024 + 512, p.Dvec + vrow, 512, &bars->full[s]);
            }
            mbar_wait_drain(&bars->kv_full, 0, p.status);
            for (int k = max(0, n - C::kStages); k < n; ++k)
                mbar_wait_drain(&bars->full[k % C::kStages], (k / C::kStages) & 1, p.status);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0 && n_q > 0) {
            constexpr uint32_t idesc_h = idesc_bf16_f32(kBlock, kHalf, false, false);
            constexpr uint32_t idesc_g = idesc_bf16_f32(kBlock, D, false, true);
            const uint64_t dk0 = smem_desc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
            const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
            const uint32_t ring = smem_u32(smem + C::kOffRing);
            // Half h of S^T = K Q^T and dP^T = V dO^T: the query rows
            // [64h, 64h + 64) of the tile (both operands K-major).
            auto issue_scores = [&](int n, int h) {
                const uint32_t sq = ring + (n % C::kStages) * C::kStageBytes + h * kHalf * 128;
                const uint64_t dq0 = smem_desc_sw128(sq, 16, 1024);
                const uint64_t ddo0 = smem_desc_sw128(sq + C::kTile, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t koff = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
                    umma_bf16_ss(tmem + C::kColS + h * kHalf, dk0 + koff, dq0 + koff, idesc_h,
                                 kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t koff = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
                    umma_bf16_ss(tmem + C::kColDP + h * kHalf, dv0 + koff, ddo0 + koff, idesc_h,
                                 kk > 0);
                }
                umma_commit(&bars->st_full[h]);
            };
            // dV += P^T dO and dK += dS^T Q over the query rows of half h:
            // A (bf16 pairs) from the half's first 32 TMEM columns, B (dO, Q)
            // MN-major from shared memory.
            auto issue_grads = [&](int n, int h) {
                const uint32_t sq = ring + (n % C::kStages) * C::kStageBytes;
                const uint64_t bq = smem_desc_sw128(sq, kBoxBytes, 1024);
                const uint64_t bdo = smem_desc_sw128(sq + C::kTile, kBoxBytes, 1024);
#pragma unroll
                for (int k4 = 0; k4 < kHalf / 16; ++k4) {
                    const int kk = h * (kHalf / 16) + k4;
                    umma_bf16_ts(tmem + C::kColDV, tmem + C::kColS + h * kHalf + k4 * 8,
                                 bdo + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_g,
                                 (n > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int k4 = 0; k4 < kHalf / 16; ++k4) {
                    const int kk = h * (kHalf / 16) + k4;
                    umma_bf16_ts(tmem + C::kColDK, tmem + C::kColDP + h * kHalf + k4 * 8,
                                 bq + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_g,
                                 (n > 0 || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = mbar_wait(&bars->kv_full, 0, abort_flag, p.status) &&
                      mbar_wait(&bars->full[0], 0, abort_flag, p.status);
            if (ok) {
                tc_fence_after_sync();
                issue_scores(0, 0);
                issue_scores(0, 1);
            }
            // Tile n+1's half-0 scores are issued between tile n's two
            // gradient halves, so the tensor core has work while either
            // group of math warps is busy. MMAs from one thread run in
            // issue order, which orders each TMEM reuse after its reader.
            for (int n = 0; n < n_q && ok; ++n) {
                ok = mbar_wait(&bars->p_full[0], n & 1, abort_flag, p.status);
                if (!ok)
                    break;
                tc_fence_after_sync();
                issue_grads(n, 0);
                const bool next = n + 1 < n_q;
                if (next) {
                    ok = mbar_wait(&bars->full[(n + 1) % C::kStages], ((n + 1) / C::kStages) & 1,
                                   abort_flag, p.status);
                    if (!ok)
                        break;
                    tc_fence_after_sync();
                    issue_scores(n + 1, 0);
                }
                ok = mbar_wait(&bars->p_full[1], n & 1, abort_flag, p.status);
                if (!ok)
                    break;
                tc_fence_after_sync();
                issue_grads(n, 1);
                umma_commit(&bars->empty[n % C::kStages]);
                if (next)
                    issue_scores(n + 1, 1);
            }
            umma_commit(&bars->o_done);
            umma_commit(&bars->drain);
            mbar_wait_drain(&bars->drain, 0, p.status);
        }
    } else {
        // ------------------------------------------------------------ math warps
        const int quarter = warp & 3, half = warp >> 2;
        const int r = quarter * 32 + lane;  // key row within the tile = TMEM lane
        const int key = kv0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::kColS + half * kHalf;
        const uint32_t tDP = tmem + lane_base + C::kColDP + half * kHalf;
        const float sl2 = p.scale_log2;
        bool ok = true;
        for (int n = 0; n < n_q && ok; ++n) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bars->st_full[half], n & 1, abort_flag, p.status));
            if (!ok)
                break;
            tc_fence_after_sync();
            const int q0 = (qt0 + n) * kBlock + half * kHalf;  // first query of this half
            const float *vec = reinterpret_cast<const float *>(smem + C::kOffVec +
                                                               (n % C::kStages) * 1024) +
                               half * kHalf;
            // mask: key beyond Sk, or (causal) key after the query's last visible key
            const bool tile_masked = key >= p.Sk || (p.causal && kv0 + kBlock - 1 > q0 + off);
#pragma unroll
            for (int c0 = 0; c0 < kHalf; c0 += kChunk) {
                uint32_t sr[kChunk], dr[kChunk];
                tmem_ld32_wait(tS + c0, sr);
                tmem_ld32_wait(tDP + c0, dr);
                uint32_t pp[kChunk / 2], pd[kChunk / 2];
#pragma unroll
                for (int c = 0; c < kChunk; c += 2) {
                    float pv[2], dv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int qc = c0 + c + e;
                        float pr = ex2_approx(fmaf(__uint_as_float(sr[c + e]), sl2, -vec[qc]));
                        if (tile_masked &&
                            (key >= p.Sk || (p.causal && key > q0 + qc + off)))
                            pr = 0.0f;
                        pv[e] = pr;
                        dv[e] = pr * (__uint_as_float(dr[c + e]) - vec[128 + qc]);
                    }
                    pp[c / 2] = pk2(pv[0], pv[1]);
                    pd[c / 2] = pk2(dv[0], dv[1]);
                }
                // P^T and dS^T (bf16 pairs) over this half's own, already read columns
                tmem_st16(tS + c0 / 2, pp);
                tmem_st16(tDP + c0 / 2, pd);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->p_full[half]);
        }
        // ------------------------------------------------------------ epilogue
        if (ok && n_q > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done, 0, abort_flag, p.status));
            tc_fence_after_sync();
        }
        // All math threads take the epilogue (and its barriers) or none does.
        const bool skip =
            named_bar_or(1, kMathThreads, !ok || *reinterpret_cast<volatile int *>(abort_flag));
        if (!skip) {
            uint8_t *stage = smem + C::kOffRing;  // the ring is idle now
            store_tile<D>(tmem + lane_base + C::kColDV, 1.0f, n_q > 0, stage, &tm_dv, kv0, bh, r,
                          half, 2);
            store_tile<D>(tmem + lane_base + C::kColDK, p.scale, n_q > 0, stage, &tm_dk, kv0, bh,
                          r, half, 2);
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
}

// ---------------------------------------------------------------- dQ
template <int D>
struct QCfg {
    static constexpr int kTile = kBlock * D * 2;
    static constexpr int kStages = (D == 128) ? 2 : 4;  // (K_j, V_j) pairs
    static constexpr int kOffQ = 0, kOffDO = kTile, kOffRing = 2 * kTile;
    static constexpr int kStageBytes = 2 * kTile;
    static constexpr int kOffBar = kOffRing + kStages * kStageBytes;
    static constexpr int kSmem = kOffBar + 512 + 1024;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;
};

struct QBars {
    uint64_t q_full;
    uint64_t full[4], empty[4];
    uint64_t st_full[2], p_full[2];  // per column half, as in KvBars
    uint64_t o_done, drain;
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dq, const Params p)
{
    using C = QCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    QBars *bars = reinterpret_cast<QBars *>(smem + C::kOffBar);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.x / p.n_qtiles;
    const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x % p.n_qtiles);  // long first
    const int q0 = qt * kBlock;
    const int last = min(q0 + kBlock - 1, p.Sq - 1);
    const int n_kv = (visible_keys(last, p.Sq, p.Sk, p.causal) + kBlock - 1) / kBlock;
    const int mask_from = visible_keys(q0, p.Sq, p.Sk, p.causal) / kBlock;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bars->st_full[h], 1);
            mbar_init(&bars->p_full[h], 4);
        }
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    int *abort_flag = &bars->abort_flag;

    if (warp == kProducerWarp) {
        // A query tile that sees no key tile loads nothing: its epilogue
        // stages the zero dQ tile in Q's buffer, which a late load would
        // overwrite.
        if (lane == 0 && n_kv > 0) {
            mbar_arrive_expect_tx(&bars->q_full, 2 * C::kTile);
            for (int b = 0; b < D / 64; ++b) {
                tma_load_3d(smem + C::kOffQ + b * kBoxBytes, &tm_q, &bars->q_full, b * 64, q0, bh);
                tma_load_3d(smem + C::kOffDO + b * kBoxBytes, &tm_do, &bars->q_full, b * 64, q0, bh);
            }
            int j = 0;
            for (; j < n_kv; ++j) {
                const int s = j % C::kStages;
                const uint32_t use = j / C::kStages;
                if (use > 0 && !mbar_wait(&bars->empty[s], (use - 1) & 1, abort_flag, p.status))
                    break;
                uint8_t *st = smem + C::kOffRing + s * C::kStageBytes;
                mbar_arrive_expect_tx(&bars->full[s], C::kStageBytes);
                for (int b = 0; b < D / 64; ++b) {
                    tma_load_3d(st + b * kBoxBytes, &tm_k, &bars->full[s], b * 64, j * kBlock, bh);
                    tma_load_3d(st + C::kTile + b * kBoxBytes, &tm_v, &bars->full[s], b * 64,
                                j * kBlock, bh);
                }
            }
            mbar_wait_drain(&bars->q_full, 0, p.status);
            for (int k = max(0, j - C::kStages); k < j; ++k)
                mbar_wait_drain(&bars->full[k % C::kStages], (k / C::kStages) & 1, p.status);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0 && n_kv > 0) {
            constexpr uint32_t idesc_h = idesc_bf16_f32(kBlock, kHalf, false, false);
            constexpr uint32_t idesc_g = idesc_bf16_f32(kBlock, D, false, true);
            const uint64_t aq0 = smem_desc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
            const uint64_t ado0 = smem_desc_sw128(smem_u32(smem + C::kOffDO), 16, 1024);
            const uint32_t ring = smem_u32(smem + C::kOffRing);
            // Half h of S = Q K^T and dP = dO V^T: the keys [64h, 64h + 64)
            // of the tile (both operands K-major).
            auto issue_scores = [&](int j, int h) {
                const uint32_t sk = ring + (j % C::kStages) * C::kStageBytes + h * kHalf * 128;
                const uint64_t bk0 = smem_desc_sw128(sk, 16, 1024);
                const uint64_t bv0 = smem_desc_sw128(sk + C::kTile, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t koff = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
                    umma_bf16_ss(tmem + C::kColS + h * kHalf, aq0 + koff, bk0 + koff, idesc_h,
                                 kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t koff = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
                    umma_bf16_ss(tmem + C::kColDP + h * kHalf, ado0 + koff, bv0 + koff, idesc_h,
                                 kk > 0);
                }
                umma_commit(&bars->st_full[h]);
            };
            // dQ += dS K over the keys of half h: A = dS (bf16 pairs) from
            // the half's first 32 TMEM columns, B = K MN-major.
            auto issue_grad = [&](int j, int h) {
                const uint32_t sk = ring + (j % C::kStages) * C::kStageBytes;
                const uint64_t bkm = smem_desc_sw128(sk, kBoxBytes, 1024);
#pragma unroll
                for (int k4 = 0; k4 < kHalf / 16; ++k4) {
                    const int kk = h * (kHalf / 16) + k4;
                    umma_bf16_ts(tmem + C::kColDQ, tmem + C::kColS + h * kHalf + k4 * 8,
                                 bkm + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_g,
                                 (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = mbar_wait(&bars->q_full, 0, abort_flag, p.status) &&
                      mbar_wait(&bars->full[0], 0, abort_flag, p.status);
            if (ok) {
                tc_fence_after_sync();
                issue_scores(0, 0);
                issue_scores(0, 1);
            }
            // The same interleaving as the dK/dV kernel.
            for (int j = 0; j < n_kv && ok; ++j) {
                ok = mbar_wait(&bars->p_full[0], j & 1, abort_flag, p.status);
                if (!ok)
                    break;
                tc_fence_after_sync();
                issue_grad(j, 0);
                const bool next = j + 1 < n_kv;
                if (next) {
                    ok = mbar_wait(&bars->full[(j + 1) % C::kStages], ((j + 1) / C::kStages) & 1,
                                   abort_flag, p.status);
                    if (!ok)
                        break;
                    tc_fence_after_sync();
                    issue_scores(j + 1, 0);
                }
                ok = mbar_wait(&bars->p_full[1], j & 1, abort_flag, p.status);
                if (!ok)
                    break;
                tc_fence_after_sync();
                issue_grad(j, 1);
                umma_commit(&bars->empty[j % C::kStages]);
                if (next)
                    issue_scores(j + 1, 1);
            }
            umma_commit(&bars->o_done);
            umma_commit(&bars->drain);
            mbar_wait_drain(&bars->drain, 0, p.status);
        }
    } else {
        const int quarter = warp & 3, half = warp >> 2;
        const int r = quarter * 32 + lane;  // query row within the tile = TMEM lane
        const int i = q0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::kColS + half * kHalf;
        const uint32_t tDP = tmem + lane_base + C::kColDP + half * kHalf;
        const float sl2 = p.scale_log2;
        const size_t vrow = static_cast<size_t>(bh) * p.Sq_pad + i;
        const float l2 = p.lse2[vrow], Di = p.Dvec[vrow];  // padded rows: +inf, 0
        const int lim = visible_keys(i, p.Sq, p.Sk, p.causal);
        bool ok = true;
        for (int j = 0; j < n_kv && ok; ++j) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bars->st_full[half], j & 1, abort_flag, p.status));
            if (!ok)
                break;
            tc_fence_after_sync();
            const bool tile_masked = j >= mask_from;
            const int key0 = j * kBlock + half * kHalf;  // first key of this half
#pragma unroll
            for (int c0 = 0; c0 < kHalf; c0 += kChunk) {
                uint32_t sr[kChunk], dr[kChunk];
                tmem_ld32_wait(tS + c0, sr);
                tmem_ld32_wait(tDP + c0, dr);
                uint32_t pd[kChunk / 2];
#pragma unroll
                for (int c = 0; c < kChunk; c += 2) {
                    float ds[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float pr = ex2_approx(fmaf(__uint_as_float(sr[c + e]), sl2, -l2));
                        if (tile_masked && key0 + c0 + c + e >= lim)
                            pr = 0.0f;
                        ds[e] = pr * (__uint_as_float(dr[c + e]) - Di);
                    }
                    pd[c / 2] = pk2(ds[0], ds[1]);
                }
                tmem_st16(tS + c0 / 2, pd);  // dS (bf16 pairs) over this half's read columns
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->p_full[half]);
        }
        if (ok && n_kv > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done, 0, abort_flag, p.status));
            tc_fence_after_sync();
        }
        const bool skip =
            named_bar_or(1, kMathThreads, !ok || *reinterpret_cast<volatile int *>(abort_flag));
        if (!skip)
            store_tile<D>(tmem + lane_base + C::kColDQ, p.scale, n_kv > 0, smem + C::kOffQ,
                          &tm_dq, q0, bh, r, half, 2);
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
}

template <int D>
fa_status_t launch(const BackwardProblem &bp)
{
    const Problem &pr = bp.fwd;
    const int64_t BH = pr.B * pr.H;
    const int Sq_pad = static_cast<int>((pr.Sq + kBlock - 1) / kBlock * kBlock);
    float *lse2 = static_cast<float *>(bp.workspace);
    float *Dvec = lse2 + static_cast<size_t>(BH) * Sq_pad;
    {
        const int rows = static_cast<int>(BH * Sq_pad);
        fa_bwd_prep_kernel<D><<<(rows + 7) / 8, 256, 0, pr.stream>>>(
            static_cast<const __nv_bfloat16 *>(bp.o), static_cast<const __nv_bfloat16 *>(bp.dout),
            bp.lse, lse2, Dvec, static_cast<int>(BH), static_cast<int>(pr.Sq), Sq_pad);
        if (cudaGetLastError() != cudaSuccess)
            return FA_ERR_CUDA;
    }
    CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
    if (!encode_tmap_bf16_3d(&tq, pr.q, D, pr.Sq, BH, kBlock) ||
        !encode_tmap_bf16_3d(&tk, pr.k, D, pr.Sk, BH, kBlock) ||
        !encode_tmap_bf16_3d(&tv, pr.v, D, pr.Sk, BH, kBlock) ||
        !encode_tmap_bf16_3d(&tdo, bp.dout, D, pr.Sq, BH, kBlock) ||
        !encode_tmap_bf16_3d(&tdq, bp.dq, D, pr.Sq, BH, kBlock) ||
        !encode_tmap_bf16_3d(&tdk, bp.dk, D, pr.Sk, BH, kBlock) ||
        !encode_tmap_bf16_3d(&tdv, bp.dv, D, pr.Sk, BH, kBlock))
        return FA_ERR_CUDA;
    Params p;
    p.Sq = static_cast<int>(pr.Sq);
    p.Sk = static_cast<int>(pr.Sk);
    p.Sq_pad = Sq_pad;
    p.BH = static_cast<int>(BH);
    p.n_qtiles = static_cast<int>((pr.Sq + kBlock - 1) / kBlock);
    p.n_ktiles = static_cast<int>((pr.Sk + kBlock - 1) / kBlock);
    p.causal = pr.causal ? 1 : 0;
    p.scale = pr.scale;
    p.scale_log2 = pr.scale * 1.4426950408889634f;
    p.lse2 = lse2;
    p.Dvec = Dvec;
    p.status = pr.status;
    {
        auto kern = fa_bwd_dkdv_kernel<D>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 KvCfg<D>::kSmem) != cudaSuccess)
            return FA_ERR_CUDA;
        const uint64_t grid = static_cast<uint64_t>(p.n_ktiles) * BH;
        if (grid > 0x7FFFFFFFull)
            return FA_ERR_UNSUPPORTED;
        kern<<<static_cast<unsigned>(grid), kThreads, KvCfg<D>::kSmem, pr.stream>>>(tq, tk, tv, tdo,
                                                                                   tdk, tdv, p);
        if (cudaGetLastError() != cudaSuccess)
            return FA_ERR_CUDA;
    }
    {
        auto kern = fa_bwd_dq_kernel<D>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 QCfg<D>::kSmem) != cudaSuccess)
            return FA_ERR_CUDA;
        const uint64_t grid = static_cast<uint64_t>(p.n_qtiles) * BH;
        if (grid > 0x7FFFFFFFull)
            return FA_ERR_UNSUPPORTED;
        kern<<<static_cast<unsigned>(grid), kThreads, QCfg<D>::kSmem, pr.stream>>>(tq, tk, tv, tdo,
                                                                                 tdq, p);
        if (cudaGetLastError() != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // namespace bwd

size_t backward_workspace_bytes(int64_t BH, int64_t Sq)
{
    const int64_t Sq_pad = (Sq + bwd::kBlock - 1) / bwd::kBlock * bwd::kBlock;
    return static_cast<size_t>(2 * BH * Sq_pad) * sizeof(float);
}

fa_status_t launch_backward_sm103(const BackwardProblem &bp)
{
    if (bp.fwd.d == 128)
        return bwd::launch<128>(bp);
    if (bp.fwd.d == 64)
        return bwd::launch<64>(bp);
    return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
