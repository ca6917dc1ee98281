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
//   * fa_bwd_prep_kernel: -D_i and -LSE in the exp2 domain (lse2 = LSE *
//     log2 e; +inf for rows with no visible key, so their P is 0), into
//     row-padded workspace rows. They are stored negated because the
//     rebuilds add them (one packed f32x2 add or FMA per two entries);
//   * fa_bwd_dkdv_kernel: one CTA per 128-key tile of one (b, h). It keeps K
//     and V in shared memory, streams (Q_i, dO_i, lse2_i, D_i) for every
//     query tile that sees the key tile, forms S^T = K Q_i^T and
//     dP^T = V dO_i^T with 128-wide tcgen05 MMAs into tensor memory, lets
//     the math warps rebuild P^T (once S^T lands) and dS^T (once dP^T lands)
//     as bf16 written back over their own TMEM columns, and accumulates
//     dV += P^T dO_i and dK += dS^T Q_i with the A operand read from TMEM.
//     The MMAs are issued as dP(i) | dV(i) S(i+1) | dK(i) dP(i+1) | ..., so
//     each rebuild runs while two other MMAs of the tile pipeline execute;
//   * fa_bwd_dq_kernel: one CTA per 128-row query tile; for every key tile
//     it sees: S = Q K_j^T (two TMEM buffers), dP = dO V_j^T, then the math
//     warps rebuild P (fp32, in registers) once S lands and dS once dP
//     lands, written back as bf16 over dP's columns, and dQ += dS K_j (A
//     from TMEM). Issue order S(j+1) | dQ(j) dP(j+1) S(j+2) | ..., with K
//     in a 3-deep ring of its own (K_j is read by S(j) and again by dQ(j)).
// All score MMAs are 128 wide: an M = 128 MMA of N = 64 columns takes 45 to
// 54 cycles against 64 for N = 128 (K = 16, measured), so two 64-wide halves
// take 1.4x to 1.7x the tensor time of one 128-wide MMA.
// Math warps share TMEM lanes by sub-partition (lane quarter = warp mod 4)
// and split the columns: 16 warps of 32 columns in the dK/dV kernel, whose
// P^T rebuild is on the MMA chain, 8 warps of 64 in the dQ kernel. Each
// packs its bf16 result into the first half of its own columns, so no warp
// overwrites columns another has yet to read.
// The dQ kernel is launched with programmatic stream serialization: its CTAs
// start on the SMs the dK/dV kernel's last CTAs leave idle (it reads only
// what the prep kernel wrote), and wait for the dK/dV grid before exiting, so
// the launch as a whole still completes after both.
// The warp roles, TMA ring, mbarrier waits (bounded) and descriptor
// encodings are those of the forward kernel.
#include <cmath>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace bwd {

constexpr int kBlock = 128;             // keys or queries per tile = TMEM lanes
// dQ kernel: warps 0-7 do the math (lane quarter warp % 4, column half
// warp / 4), warp 8 loads, warp 9 issues the MMAs.
constexpr int kMathThreads = 256;
constexpr int kThreads = kMathThreads + 64;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// dK/dV kernel: warps 0-15 do the math (lane quarter warp % 4, column
// quarter warp / 4: 32 columns each), warp 16 loads, warp 17 issues.
constexpr int kKvGroups = 4;
constexpr int kKvMathThreads = kKvGroups * 128;
constexpr int kKvThreads = kKvMathThreads + 64;
constexpr int kKvProducerWarp = kKvMathThreads / 32;
constexpr int kKvMmaWarp = kKvProducerWarp + 1;
constexpr int kHalf = kBlock / 2;        // score columns per half
constexpr uint32_t kTmemCols = 512;
constexpr int kBoxBytes = kBlock * 128;  // 128 rows x 64 columns bf16
constexpr int kChunk = 32;               // TMEM columns a math thread handles at a time

struct Params {
    int Sq, Sk, Sq_pad, BH, n_qtiles, n_ktiles;
    int causal;
    float scale;       // the caller's scale (signed): dK, dQ = scale * ...
    float scale_log2;  // |scale| * log2(e), the factor of the P rebuild
    // kIdescNegateA for a negative scale, else 0: the score MMAs then form
    // -Q K^T (or -K Q^T), so P = 2^(scores * scale_log2 - lse2) as for scale > 0.
    uint32_t idesc_s_neg;
    const float *lse2;  // -lse2: [BH, Sq_pad], -inf padding
    const float *Dvec;  // -D: [BH, Sq_pad], -0 padding
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
// D / 8 threads per (bh, row of the padded row range), each reading 16 bytes
// of O and of dO.
template <int D>
__global__ void __launch_bounds__(256)
    fa_bwd_prep_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                       const float *__restrict__ lse, float *__restrict__ lse2,
                       float *__restrict__ Dvec, int BH, int Sq, int Sq_pad)
{
    constexpr int kLanes = D / 8;  // threads per row
    const int row = blockIdx.x * (256 / kLanes) + threadIdx.x / kLanes;
    const int part = threadIdx.x % kLanes;
    if (row >= BH * Sq_pad)  // whole row groups: the shuffles below stay within live lanes
        return;
    const int bh = row / Sq_pad, i = row % Sq_pad;
    float acc = 0.0f;
    float l2 = INFINITY;
    if (i < Sq) {
        const size_t base = (static_cast<size_t>(bh) * Sq + i) * D + part * 8;
        const uint4 ov = *reinterpret_cast<const uint4 *>(o + base);
        const uint4 dv = *reinterpret_cast<const uint4 *>(dout + base);
        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ow[e]));
            const float2 df = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&dw[e]));
            acc = fmaf(of.x, df.x, acc);
            acc = fmaf(of.y, df.y, acc);
        }
        const float L = lse[static_cast<size_t>(bh) * Sq + i];
        l2 = (L == -INFINITY) ? INFINITY : L * 1.4426950408889634f;
    }
    const unsigned mask = __activemask();
#pragma unroll
    for (int off = kLanes / 2; off > 0; off /= 2)
        acc += __shfl_xor_sync(mask, acc, off);
    if (part == 0) {  // stored negated: the rebuilds add them
        Dvec[row] = -acc;
        lse2[row] = -l2;
    }
}

// Pack two fp32 values as a bf16 pair (element 2c in the low half).
__device__ __forceinline__ uint32_t pk2(float a, float b) { return pack_bf16x2(a, b); }

__device__ __forceinline__ float2 f2(uint32_t a, uint32_t b)
{
    return make_float2(__uint_as_float(a), __uint_as_float(b));
}

// 32 columns at `a` into r, without the wait: r is valid only after
// tmem_ld_wait_regs32(r).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t a, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(a)
        : "memory");
}

// Wait for this thread's TMEM loads; r is an operand (read and written), so
// every use of the loaded registers stays after the wait.
__device__ __forceinline__ void tmem_ld_wait_regs32(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// P^T for one 32-column chunk of one key (this thread's TMEM lane):
// P^T = 2^(S^T sl2 + nl), nl = -lse2 of the query (nl: the chunk's 32
// queries, 16-byte aligned). The fp32 values go to pv, bf16 pairs to pp.
// kMask zeroes the entries where `keep` is false.
template <bool kMask, typename Keep>
__device__ __forceinline__ void rebuild_p(const uint32_t (&st)[32], float2 sl2, const float *nl,
                                          Keep keep, float *pv, uint32_t (&pp)[16])
{
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4 *>(nl + c);
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            const float2 x = ffma2(f2(st[c + e], st[c + e + 1]), sl2,
                                   e == 0 ? make_float2(l4.x, l4.y) : make_float2(l4.z, l4.w));
            float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
            if (kMask) {
                if (!keep(c + e))
                    p0 = 0.0f;
                if (!keep(c + e + 1))
                    p1 = 0.0f;
            }
            pv[c + e] = p0;
            pv[c + e + 1] = p1;
            pp[(c + e) / 2] = pk2(p0, p1);
        }
    }
}

// dS^T = P^T (dP^T + nd), nd = -D of the query, for one 32-column chunk, as
// bf16 pairs.
__device__ __forceinline__ void rebuild_ds(const uint32_t (&dt)[32], const float *pv,
                                           const float *nd, uint32_t (&pd)[16])
{
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
        const float4 d4 = *reinterpret_cast<const float4 *>(nd + c);
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            const float2 ds = fmul2(
                make_float2(pv[c + e], pv[c + e + 1]),
                fadd2(f2(dt[c + e], dt[c + e + 1]),
                      e == 0 ? make_float2(d4.x, d4.y) : make_float2(d4.z, d4.w)));
            pd[(c + e) / 2] = pk2(ds.x, ds.y);
        }
    }
}

// 16 TMEM columns of this thread's lane, with the wait.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// The epilogue of both gradient kernels: a 128 x D fp32 tile in TMEM (this
// thread's lane = row r; `taddr` addresses column 0 of that lane) times
// `mul`, to bf16, through shared memory (Q-tile sized staging at `stage`,
// swizzled like the TMA box), then TMA-stored. The tile's columns are split
// into kGroups groups; group `group` is this thread's. All kGroups * 128
// math threads take part.
template <int D, int kGroups>
__device__ __forceinline__ void store_tile(uint32_t taddr, float mul, bool have, uint8_t *stage,
                                           const CUtensorMap *map, int row0, int bh, int r,
                                           int group, uint32_t bar_id)
{
    constexpr int kCols = D / kGroups;
    constexpr int kStep = kCols < 32 ? kCols : 32;
    static_assert(kStep == 16 || kStep == 32, "16 or 32 columns per load");
    const uint32_t st_a = smem_u32(stage);
#pragma unroll
    for (int c0 = group * kCols; c0 < (group + 1) * kCols; c0 += kStep) {
        uint32_t v[kStep];
        if (have) {
            if constexpr (kStep == 32)
                tmem_ld32_wait(taddr + c0, v);
            else
                tmem_ld16_wait(taddr + c0, v);
        } else {
#pragma unroll
            for (int c = 0; c < kStep; ++c)
                v[c] = 0u;
        }
        uint32_t pk[kStep / 2];
#pragma unroll
        for (int c = 0; c < kStep; c += 2)
            pk[c / 2] = pk2(__uint_as_float(v[c]) * mul, __uint_as_float(v[c + 1]) * mul);
#pragma unroll
        for (int q = 0; q < kStep / 8; ++q) {
            const uint32_t chunk = ((c0 % 64) / 8) + q;
            st_shared_v4(st_a + (c0 / 64) * kBoxBytes + sw128_offset(static_cast<uint32_t>(r), chunk),
                         pk[q * 4], pk[q * 4 + 1], pk[q * 4 + 2], pk[q * 4 + 3]);
        }
    }
    fence_proxy_async_smem();
    named_bar_sync(bar_id, kGroups * 128);
    if (r == 0 && group == 0) {
        for (int b = 0; b < D / 64; ++b)
            tma_store_3d(map, stage + b * kBoxBytes, b * 64, row0, bh);
        tma_store_commit();
        tma_store_wait_read_all();
    }
    named_bar_sync(bar_id, kGroups * 128);
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
    uint64_t s_full, dp_full;  // S^T / dP^T of the current query tile in TMEM
    uint64_t p_full, ds_full;  // P^T / dS^T written back (8 warp arrivals each)
    uint64_t o_done;   // last dV / dK MMAs completed
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kKvThreads, 1)
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
    // The dQ grid may start on SMs this grid no longer needs.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.x / p.n_ktiles;
    const int kt = static_cast<int>(blockIdx.x % p.n_ktiles);  // long first
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
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->dp_full, 1);
        mbar_init(&bars->p_full, kKvMathThreads / 32);
        mbar_init(&bars->ds_full, kKvMathThreads / 32);
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kKvMmaWarp) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    int *abort_flag = &bars->abort_flag;

    if (warp == kKvProducerWarp) {
        {
            // The whole warp runs the loop and polls each barrier together;
            // lane 0 alone issues the copies.
            auto wwait = [&](uint64_t *bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.status));
            };
            if (lane == 0) {
                fa_check(kv0 < p.Sk && bh < p.BH, p.status);
                mbar_arrive_expect_tx(&bars->kv_full, 2 * C::kTile);
                for (int b = 0; b < D / 64; ++b) {
                    tma_load_3d(smem + C::kOffK + b * kBoxBytes, &tm_k, &bars->kv_full, b * 64, kv0, bh);
                    tma_load_3d(smem + C::kOffV + b * kBoxBytes, &tm_v, &bars->kv_full, b * 64, kv0, bh);
                }
            }
            __syncwarp();
            int n = 0;
            for (; n < n_q; ++n) {
                const int s = n % C::kStages;
                const uint32_t use = n / C::kStages;
                if (use > 0 && !wwait(&bars->empty[s], (use - 1) & 1))
                    break;
                if (lane == 0) {
                    const int q0 = (qt0 + n) * kBlock;
                    uint8_t *st = smem + C::kOffRing + s * C::kStageBytes;
                    mbar_arrive_expect_tx(&bars->full[s], C::kStageBytes + 1024);
                    for (int b = 0; b < D / 64; ++b) {
                        tma_load_3d(st + b * kBoxBytes, &tm_q, &bars->full[s], b * 64, q0, bh);
                        tma_load_3d(st + C::kTile + b * kBoxBytes, &tm_do, &bars->full[s], b * 64, q0,
                                    bh);
                    }
                    const size_t vrow = static_cast<size_t>(bh) * p.Sq_pad + q0;
                    fa_check(q0 < p.Sq && vrow + kBlock <= static_cast<size_t>(p.BH) * p.Sq_pad,
                             p.status);
                    bulk_load(smem + C::kOffVec + s * 1024, p.lse2 + vrow, 512, &bars->full[s]);
                    bulk_load(smem + C::kOffVec + s * 1024 + 512, p.Dvec + vrow, 512, &bars->full[s]);
                }
                __syncwarp();
            }
            if (lane == 0) {
                mbar_wait_drain(&bars->kv_full, 0, p.status);
                for (int k = max(0, n - C::kStages); k < n; ++k)
                    mbar_wait_drain(&bars->full[k % C::kStages], (k / C::kStages) & 1, p.status);
            }
            __syncwarp();
        }
    } else if (warp == kKvMmaWarp) {
        if (n_q > 0) {
            // The whole warp runs the issue loop (counters and descriptors stay
            // warp-uniform): it polls each barrier together, and one elected
            // lane issues each MMA and commit.
            auto wwait = [&](uint64_t *bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.status));
            };
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBlock, kBlock, false, false);
            constexpr uint32_t idesc_g = idesc_bf16_f32(kBlock, D, false, true);
            const uint64_t dk0 = smem_desc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
            const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
            const uint32_t ring = smem_u32(smem + C::kOffRing);
            // S^T = K Q^T (A = K, B = Q, both K-major), or dP^T = V dO^T,
            // over the tile's 128 queries.
            auto issue_scores = [&](int n, bool dp) {
                const uint32_t sq = ring + (n % C::kStages) * C::kStageBytes + (dp ? C::kTile : 0);
                const uint64_t b0 = smem_desc_sw128(sq, 16, 1024);
                const uint64_t a0 = dp ? dv0 : dk0;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t koff = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
                    umma_bf16_ss_elect(tmem + (dp ? C::kColDP : C::kColS), a0 + koff, b0 + koff,
                                 dp ? idesc_s : idesc_s | p.idesc_s_neg, kk > 0);
                }
                umma_commit_elect(dp ? &bars->dp_full : &bars->s_full);
            };
            // dV += P^T dO (A = P^T from the S columns) or dK += dS^T Q (A =
            // dS^T from the dP columns). A is bf16 pairs, each 32-query group
            // packed into its first 16 columns: K step kk (queries 16 kk ..
            // 16 kk + 15) at column (kk / 2) * 32 + (kk % 2) * 8. B (dO, Q)
            // MN-major from shared memory.
            auto issue_grad = [&](int n, bool dk) {
                const uint32_t sq = ring + (n % C::kStages) * C::kStageBytes + (dk ? 0 : C::kTile);
                const uint64_t b0 = smem_desc_sw128(sq, kBoxBytes, 1024);
                const uint32_t a0 = tmem + (dk ? C::kColDP : C::kColS);
#pragma unroll
                for (int kk = 0; kk < kBlock / 16; ++kk)
                    umma_bf16_ts_elect(tmem + (dk ? C::kColDK : C::kColDV),
                                 a0 + (kk / 2) * kChunk + (kk % 2) * 8,
                                 b0 + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_g,
                                 (n > 0 || kk > 0) ? 1u : 0u);
            };
            bool ok = wwait(&bars->kv_full, 0) &&
                      wwait(&bars->full[0], 0);
            if (ok) {
                tc_fence_after_sync();
                issue_scores(0, false);
                issue_scores(0, true);
            }
            // Issue order: ... dP(n) | dV(n) S(n+1) | dK(n) dP(n+1) | dV(n+1) ...
            // Each rebuild (P^T after S^T lands, dS^T after dP^T lands) has
            // two 128-wide MMAs ahead of the one that consumes it. MMAs from
            // one lane run in issue order, which orders each TMEM reuse
            // after its reader; the math warps read S^T (dP^T) before they
            // signal P^T (dS^T).
            for (int n = 0; n < n_q && ok; ++n) {
                ok = wwait(&bars->p_full, n & 1);
                if (!ok)
                    break;
                tc_fence_after_sync();
                issue_grad(n, false);
                const bool next = n + 1 < n_q;
                if (next) {
                    ok = wwait(&bars->full[(n + 1) % C::kStages], ((n + 1) / C::kStages) & 1);
                    if (!ok)
                        break;
                    tc_fence_after_sync();
                    issue_scores(n + 1, false);
                }
                ok = wwait(&bars->ds_full, n & 1);
                if (!ok)
                    break;
                tc_fence_after_sync();
                issue_grad(n, true);
                umma_commit_elect(&bars->empty[n % C::kStages]);
                if (next)
                    issue_scores(n + 1, true);
            }
            umma_commit_elect(&bars->o_done);
            umma_commit_elect(&bars->drain);
            if (lane == 0)
                mbar_wait_drain(&bars->drain, 0, p.status);
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ math warps
        // 16 warps: lane quarter warp % 4 (key rows), column quarter warp / 4
        // (queries 32 cq .. 32 cq + 31 of the tile); each packs its bf16
        // result into the first 16 of its own 32 columns.
        const int quarter = warp & 3, cq = warp >> 2;
        const int r = quarter * 32 + lane;  // key row within the tile = TMEM lane
        const int key = kv0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::kColS + cq * kChunk;
        const uint32_t tDP = tmem + lane_base + C::kColDP + cq * kChunk;
        const float2 sl2x2 = make_float2(p.scale_log2, p.scale_log2);
        const bool in_k = key < p.Sk;
        bool ok = true;
        for (int n = 0; n < n_q && ok; ++n) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full, n & 1, abort_flag, p.status));
            if (!ok)
                break;
            tc_fence_after_sync();
            const int q0 = (qt0 + n) * kBlock + cq * kChunk;  // first query of this thread's columns
            const float *vec = reinterpret_cast<const float *>(smem + C::kOffVec +
                                                               (n % C::kStages) * 1024) +
                               cq * kChunk;
            // mask: key beyond Sk, or (causal) key after the query's last visible key
            const bool masked = !in_k || (p.causal && kv0 + kBlock - 1 > q0 + off);
            // P^T = 2^(S^T sl2 - lse2), kept in fp32 for dS^T
            float pv[kChunk];
            {
                uint32_t sd[kChunk];
                tmem_ld32_wait(tS, sd);
                uint32_t pp[kChunk / 2];
                if (!masked) {
                    rebuild_p<false>(sd, sl2x2, vec, [](int) { return true; }, pv, pp);
                } else {
                    const int lim = q0 + off;  // the query of column c sees key <= lim + c
                    rebuild_p<true>(sd, sl2x2, vec,
                                    [&](int c) { return in_k && (!p.causal || key <= lim + c); },
                                    pv, pp);
                }
                tmem_st16(tS, pp);  // over this thread's own, already read columns
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->p_full);
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->dp_full, n & 1, abort_flag, p.status));
            if (!ok)
                break;
            tc_fence_after_sync();
            // dS^T = P^T (dP^T - D)
            {
                uint32_t sd[kChunk];
                tmem_ld32_wait(tDP, sd);
                uint32_t pd[kChunk / 2];
                rebuild_ds(sd, pv, vec + 128, pd);
                tmem_st16(tDP, pd);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->ds_full);
        }
        // ------------------------------------------------------------ epilogue
        if (ok && n_q > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done, 0, abort_flag, p.status));
            tc_fence_after_sync();
        }
        // All math threads take the epilogue (and its barriers) or none does.
        const uint32_t lane_tm = tmem + lane_base;
        const bool skip =
            named_bar_or(1, kKvMathThreads, !ok || *reinterpret_cast<volatile int *>(abort_flag));
        if (!skip) {
            uint8_t *stage = smem + C::kOffRing;  // the ring is idle now
            store_tile<D, kKvGroups>(lane_tm + C::kColDV, 1.0f, n_q > 0, stage, &tm_dv, kv0, bh, r,
                                     cq, 2);
            store_tile<D, kKvGroups>(lane_tm + C::kColDK, p.scale, n_q > 0, stage, &tm_dk, kv0,
                                     bh, r, cq, 2);
        }
    }
    // Threads that issued TMA stores wait for their writes (not only for the
    // shared-memory reads) before the CTA exits, so that the next kernel in the
    // stream reads them.
    tma_store_wait_all();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == kKvMmaWarp)
        tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- dQ
// P = 2^(S sl2 + nl) (nl = -lse2 of this thread's query) for one 32-column
// chunk, into pv. kMask zeroes the columns c >= n_vis.
template <bool kMask>
__device__ __forceinline__ void rebuild_q_p(const uint32_t (&st)[32], float2 sl2, float2 nl,
                                            int n_vis, float *pv)
{
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
        const float2 x = ffma2(f2(st[c], st[c + 1]), sl2, nl);
        float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
        if (kMask) {
            if (c >= n_vis)
                p0 = 0.0f;
            if (c + 1 >= n_vis)
                p1 = 0.0f;
        }
        pv[c] = p0;
        pv[c + 1] = p1;
    }
}

// dS = P (dP + nd) (nd = -D of this thread's query) for one 32-column chunk,
// as bf16 pairs.
__device__ __forceinline__ void rebuild_q_ds(const uint32_t (&dt)[32], const float *pv, float2 nd,
                                             uint32_t (&pd)[16])
{
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
        const float2 ds = fmul2(make_float2(pv[c], pv[c + 1]), fadd2(f2(dt[c], dt[c + 1]), nd));
        pd[c / 2] = pk2(ds.x, ds.y);
    }
}

// K and V tiles sit in rings of their own: K_j is read by S(j) and, later,
// by dQ(j); V_j only by dP(j), so K needs the deeper ring.
template <int D>
struct QCfg {
    static constexpr int kTile = kBlock * D * 2;
    static constexpr int kKStages = (D == 128) ? 3 : 4;
    static constexpr int kVStages = (D == 128) ? 2 : 4;
    static constexpr int kOffQ = 0, kOffDO = kTile, kOffK = 2 * kTile;
    static constexpr int kOffV = kOffK + kKStages * kTile;
    static constexpr int kOffBar = kOffV + kVStages * kTile;
    static constexpr int kSmem = kOffBar + 512 + 1024;
    // Two S buffers (S(j) in buffer j % 2), dP, dQ.
    static constexpr uint32_t kColS0 = 0, kColDP = 128, kColDQ = 256, kColS1 = 384;
    static_assert(kColDQ + D <= kColS1, "TMEM budget");
};

struct QBars {
    uint64_t q_full;
    uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
    uint64_t s_full[2];  // S(j) in buffer j % 2
    uint64_t dp_full;    // dP(j) in TMEM
    uint64_t ds_full;    // dS(j) written back (8 warp arrivals)
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
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        mbar_init(&bars->s_full[0], 1);
        mbar_init(&bars->s_full[1], 1);
        mbar_init(&bars->dp_full, 1);
        mbar_init(&bars->ds_full, kMathThreads / 32);
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
        if (n_kv > 0) {
            // The whole warp runs the loop and polls each barrier together;
            // lane 0 alone issues the copies.
            auto wwait = [&](uint64_t *bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.status));
            };
            if (lane == 0) {
                fa_check(q0 < p.Sq && bh < p.BH, p.status);
                mbar_arrive_expect_tx(&bars->q_full, 2 * C::kTile);
                for (int b = 0; b < D / 64; ++b) {
                    tma_load_3d(smem + C::kOffQ + b * kBoxBytes, &tm_q, &bars->q_full, b * 64, q0, bh);
                    tma_load_3d(smem + C::kOffDO + b * kBoxBytes, &tm_do, &bars->q_full, b * 64, q0, bh);
                }
            }
            __syncwarp();
            // K_j then V_j: V_j's slot frees (dP(j - kVStages) done) before
            // K_{j+1}'s (dQ(j + 1 - kKStages) done), so neither wait holds
            // up a copy that could already start.
            int j = 0;
            bool ok = true;
            for (; j < n_kv && ok; ++j) {
                const int sk = j % C::kKStages, sv = j % C::kVStages;
                const uint32_t uk = j / C::kKStages, uv = j / C::kVStages;
                if (uk > 0 && !wwait(&bars->k_empty[sk], (uk - 1) & 1))
                    break;
                if (lane == 0) {
                    fa_check(j * kBlock < p.Sk, p.status);
                    mbar_arrive_expect_tx(&bars->k_full[sk], C::kTile);
                    for (int b = 0; b < D / 64; ++b)
                        tma_load_3d(smem + C::kOffK + sk * C::kTile + b * kBoxBytes, &tm_k,
                                    &bars->k_full[sk], b * 64, j * kBlock, bh);
                }
                __syncwarp();
                if (uv > 0 && !wwait(&bars->v_empty[sv], (uv - 1) & 1)) {
                    ok = false;  // K_j is in flight: drain it below
                    ++j;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars->v_full[sv], C::kTile);
                    for (int b = 0; b < D / 64; ++b)
                        tma_load_3d(smem + C::kOffV + sv * C::kTile + b * kBoxBytes, &tm_v,
                                    &bars->v_full[sv], b * 64, j * kBlock, bh);
                }
                __syncwarp();
            }
            // Drain the copies in flight (at most the last ring's worth of each).
            if (lane == 0) {
                mbar_wait_drain(&bars->q_full, 0, p.status);
                const int nk = j, nv = ok ? j : j - 1;
                for (int k = max(0, nk - C::kKStages); k < nk; ++k)
                    mbar_wait_drain(&bars->k_full[k % C::kKStages], (k / C::kKStages) & 1, p.status);
                for (int k = max(0, nv - C::kVStages); k < nv; ++k)
                    mbar_wait_drain(&bars->v_full[k % C::kVStages], (k / C::kVStages) & 1, p.status);
            }
            __syncwarp();
        }
    } else if (warp == kMmaWarp) {
        if (n_kv > 0) {
            // The whole warp runs the issue loop (counters and descriptors stay
            // warp-uniform): it polls each barrier together, and one elected
            // lane issues each MMA and commit.
            auto wwait = [&](uint64_t *bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.status));
            };
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBlock, kBlock, false, false);
            constexpr uint32_t idesc_g = idesc_bf16_f32(kBlock, D, false, true);
            const uint64_t aq0 = smem_desc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
            const uint64_t ado0 = smem_desc_sw128(smem_u32(smem + C::kOffDO), 16, 1024);
            const uint32_t kring = smem_u32(smem + C::kOffK), vring = smem_u32(smem + C::kOffV);
            // S(j) = Q K_j^T into buffer j % 2, or dP(j) = dO V_j^T: 128 keys,
            // both operands K-major.
            auto issue_scores = [&](int j, bool dp) {
                const uint32_t sb = dp ? vring + (j % C::kVStages) * C::kTile
                                       : kring + (j % C::kKStages) * C::kTile;
                const uint64_t b0 = smem_desc_sw128(sb, 16, 1024);
                const uint64_t a0 = dp ? ado0 : aq0;
                const uint32_t col = dp ? C::kColDP : ((j & 1) ? C::kColS1 : C::kColS0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t koff = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
                    umma_bf16_ss_elect(tmem + col, a0 + koff, b0 + koff,
                                 dp ? idesc_s : idesc_s | p.idesc_s_neg, kk > 0);
                }
                if (dp) {
                    umma_commit_elect(&bars->dp_full);
                    umma_commit_elect(&bars->v_empty[j % C::kVStages]);
                } else {
                    umma_commit_elect(&bars->s_full[j & 1]);
                }
            };
            // dQ += dS K_j: A = dS (bf16 pairs: keys 0-63 in the dP region's
            // columns 0-31, keys 64-127 in 64-95), B = K_j MN-major.
            auto issue_grad = [&](int j) {
                const uint32_t sk = kring + (j % C::kKStages) * C::kTile;
                const uint64_t bkm = smem_desc_sw128(sk, kBoxBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < kBlock / 16; ++kk)
                    umma_bf16_ts_elect(tmem + C::kColDQ, tmem + C::kColDP + (kk / 4) * kHalf + (kk % 4) * 8,
                                 bkm + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_g,
                                 (j > 0 || kk > 0) ? 1u : 0u);
                umma_commit_elect(&bars->k_empty[j % C::kKStages]);
            };
            auto wait_k = [&](int j) {
                return wwait(&bars->k_full[j % C::kKStages], (j / C::kKStages) & 1);
            };
            auto wait_v = [&](int j) {
                return wwait(&bars->v_full[j % C::kVStages], (j / C::kVStages) & 1);
            };
            // Issue order: S(0) dP(0) S(1) | dQ(0) dP(1) S(2) | dQ(1) dP(2) S(3) | ...
            // dS(j) is rebuilt while dP(j)'s successors S(j+1) (and the
            // previous dQ) execute. dP(j+1) reuses dP's columns after dQ(j)
            // read dS(j) from them, and S(j+2) reuses S(j)'s buffer; MMAs
            // from one lane run in issue order, and the math warps read
            // S(j) and dP(j) before they signal dS(j).
            bool ok = wwait(&bars->q_full, 0) && wait_k(0);
            if (ok) {
                tc_fence_after_sync();
                issue_scores(0, false);
                ok = wait_v(0);
            }
            if (ok) {
                tc_fence_after_sync();
                issue_scores(0, true);
                if (n_kv > 1) {
                    ok = wait_k(1);
                    if (ok) {
                        tc_fence_after_sync();
                        issue_scores(1, false);
                    }
                }
            }
            for (int j = 0; j < n_kv && ok; ++j) {
                ok = wwait(&bars->ds_full, j & 1);
                if (!ok)
                    break;
                tc_fence_after_sync();
                issue_grad(j);
                if (j + 1 < n_kv) {
                    ok = wait_v(j + 1);
                    if (!ok)
                        break;
                    tc_fence_after_sync();
                    issue_scores(j + 1, true);
                }
                if (j + 2 < n_kv) {
                    ok = wait_k(j + 2);
                    if (!ok)
                        break;
                    tc_fence_after_sync();
                    issue_scores(j + 2, false);
                }
            }
            umma_commit_elect(&bars->o_done);
            umma_commit_elect(&bars->drain);
            if (lane == 0)
                mbar_wait_drain(&bars->drain, 0, p.status);
            __syncwarp();
        }
    } else {
        const int quarter = warp & 3, half = warp >> 2;
        const int r = quarter * 32 + lane;  // query row within the tile = TMEM lane
        const int i = q0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tDP = tmem + lane_base + C::kColDP + half * kHalf;
        const float2 sl2x2 = make_float2(p.scale_log2, p.scale_log2);
        const size_t vrow = static_cast<size_t>(bh) * p.Sq_pad + i;
        // -lse2 and -D of this query (padded rows: -inf, -0)
        const bool vrow_ok = fa_check(vrow < static_cast<size_t>(p.BH) * p.Sq_pad, p.status);
        const float nl = vrow_ok ? p.lse2[vrow] : -INFINITY, nd = vrow_ok ? p.Dvec[vrow] : -0.0f;
        const float2 nl2 = make_float2(nl, nl);
        const float2 nD = make_float2(nd, nd);
        const int lim = visible_keys(i, p.Sq, p.Sk, p.causal);
        bool ok = true;
        for (int j = 0; j < n_kv && ok; ++j) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bars->s_full[j & 1], (j >> 1) & 1, abort_flag, p.status));
            if (!ok)
                break;
            tc_fence_after_sync();
            const bool tile_masked = j >= mask_from;
            const int key0 = j * kBlock + half * kHalf;  // first key of this half
            const uint32_t tS = tmem + lane_base + ((j & 1) ? C::kColS1 : C::kColS0) + half * kHalf;
            // P for this thread's 64 keys, in fp32 (loads of the second
            // chunk in flight while the first is rebuilt)
            float pv[kHalf];
            {
                uint32_t sd[2][kChunk];
                tmem_ld32_wait(tS, sd[0]);
                tmem_ld32_nowait(tS + kChunk, sd[1]);
#pragma unroll
                for (int ch = 0; ch < kHalf / kChunk; ++ch) {
                    const int c0 = ch * kChunk;
                    if (ch > 0)
                        tmem_ld_wait_regs32(sd[ch]);
                    if (!tile_masked)
                        rebuild_q_p<false>(sd[ch], sl2x2, nl2, 0, pv + c0);
                    else
                        rebuild_q_p<true>(sd[ch], sl2x2, nl2, lim - (key0 + c0), pv + c0);
                }
            }
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->dp_full, j & 1, abort_flag, p.status));
            if (!ok)
                break;
            tc_fence_after_sync();
            // dS = P (dP - D), as bf16 pairs over this half's first 32 dP columns
            {
                uint32_t sd[2][kChunk];
                tmem_ld32_wait(tDP, sd[0]);
                tmem_ld32_nowait(tDP + kChunk, sd[1]);
#pragma unroll
                for (int ch = 0; ch < kHalf / kChunk; ++ch) {
                    const int c0 = ch * kChunk;
                    if (ch > 0)
                        tmem_ld_wait_regs32(sd[ch]);
                    uint32_t pd[kChunk / 2];
                    rebuild_q_ds(sd[ch], pv + c0, nD, pd);
                    tmem_st16(tDP + c0 / 2, pd);
                }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->ds_full);
        }
        if (ok && n_kv > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done, 0, abort_flag, p.status));
            tc_fence_after_sync();
        }
        const bool skip =
            named_bar_or(1, kMathThreads, !ok || *reinterpret_cast<volatile int *>(abort_flag));
        if (!skip)
            store_tile<D, 2>(tmem + lane_base + C::kColDQ, p.scale, n_kv > 0, smem + C::kOffQ,
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
    // Complete only after the dK/dV grid (this grid's programmatic
    // predecessor), so work queued after the backward sees dK and dV.
    asm volatile("griddepcontrol.wait;" ::: "memory");
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
        constexpr int kRowsPerBlock = 256 / (D / 8);
        fa_bwd_prep_kernel<D><<<(rows + kRowsPerBlock - 1) / kRowsPerBlock, 256, 0, pr.stream>>>(
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
    p.scale_log2 = fabsf(pr.scale) * 1.4426950408889634f;
    p.idesc_s_neg = std::signbit(pr.scale) ? kIdescNegateA : 0u;
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
        kern<<<static_cast<unsigned>(grid), kKvThreads, KvCfg<D>::kSmem, pr.stream>>>(tq, tk, tv, tdo,
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
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = QCfg<D>::kSmem;
        cfg.stream = pr.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, tdq, p) != cudaSuccess)
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
