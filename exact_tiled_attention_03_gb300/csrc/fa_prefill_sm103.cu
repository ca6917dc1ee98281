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
//   * persistent: one CTA per SM takes work items from a launch-wide counter
//     until none is left. An item is two 128-row query tiles of one
//     (batch, head); both share every K/V tile the CTA loads;
//   * warp 8 (producer; the whole warp runs its loop, lane 0 issues) takes
//     the items (in the order decode_item gives),
//     publishes each to the other warps
//     through a small shared-memory queue, and moves its Q tiles and then
//     K_j, V_j through a ring of shared-memory stages with TMA (128-byte
//     swizzle), one mbarrier pair per stage. The next item's first loads and
//     S MMAs run while the softmax warps finish the current item;
//   * warp 9 issues tcgen05.mma (the whole warp runs the issue loop, one
//     lane elected per MMA): S_t = Q_t K_j^T into
//     tensor memory (TMEM), and O_t += P_t V_j with P_t read from TMEM and V
//     read MN-major straight from its row-major tile; completion is signalled
//     with tcgen05.commit. Issue order per key tile j: PV_0(j), S_0(j+1),
//     PV_1(j), S_1(j+1), so each tile's softmax overlaps the other tile's
//     two GEMMs (ping-pong);
//   * warps 0-3 and 4-7 are one softmax warpgroup per query tile; thread r
//     owns row r (TMEM lane r). It streams its S row out of TMEM in 64-column
//     chunks, masks, and computes exp2 of the log2(e)-scaled logits against
//     its current reference max (at d = 64 while it finds the tile's max; at
//     d = 128 without it, the row sum of those exponentials showing whether
//     any exceeds 2^8). At d = 64 a tile whose max exceeds the reference by
//     more than 2^8 (or a row's first tile) is recomputed against the new max
//     and the O row rescaled in TMEM. At d = 128 a row sum above 2^8 adds the
//     tile's bf16 weights to O's divisor, and only a sum above 2^16 moves the
//     reference, by a power of two that scales P and O exactly; a row's first
//     tile, or a sum above 2^100, is recomputed against the max. It then
//     writes P (bf16) over its S row in TMEM. At the end
//     of an item it divides by l and writes its bf16 O row into the tile's
//     own staging box in shared memory, 64 columns at a time, each box sent
//     by one TMA store; then it writes its LSE. Q's buffers are reloaded for
//     the next item as soon as the item's MMAs are done.
// Every wait is bounded; on expiry the CTA stops, drains what it has in
// flight, frees its tensor memory and sets the device status word.
#include <cmath>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_schedule.cuh"

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
constexpr float kRescaleFactor = 256.0f;  // 2^kRescaleLog2
// d = 128: a row sum above 2^kRescaleLog2 but at most kMoveLimit leaves the
// reference where it is (every p of the tile is then at most 2^16, far inside
// bf16 and fp32 range). Up to kShiftLimit the reference moves by shifting the p
// already computed (below it no p can have overflowed); a larger sum
// recomputes against the exact max.
constexpr float kMoveLimit = 0x1p16f;
constexpr float kShiftLimit = 0x1p100f;

template <int D>
struct Cfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = kBlockM * D * 2;  // Q, K, V or O tile
    // K/V ring: 128-160 KB. At d = 128, 4 stages measured as fast as 5, and
    // the freed 32 KB hold the O staging boxes.
    static constexpr int kStages = (D == 128) ? 4 : 10;
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + kTiles * kTileBytes;
    // One 128-row x 64-column bf16 box per tile for staging O to its TMA store.
    static constexpr int kOffOut = kOffKV + kStages * kTileBytes;
    static constexpr int kOffBar = kOffOut + kTiles * kBoxBytes;
    static constexpr int kBarBytes = 512;
    static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    // S_t in columns [128 t, 128 t + 128); P_t (bf16, two per column) is
    // written over the first 64 columns of S_t once S_t is in registers.
    static constexpr uint32_t kColS0 = 0, kColS1 = 128;
    static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
    static_assert(kColO1 + D <= kTmemCols, "TMEM budget");
};

struct Params {
    sched::Schedule sc;  // items and their order (fa_schedule.cuh)
    float scale;         // |softmax scale|
    float scale_log2;    // |scale| * log2(e)
    // kIdescNegateA when the caller's scale is negative, else 0: the S MMAs
    // then form -Q K^T, so that scale * Q K^T = |scale| * (-Q K^T) and the
    // softmax below only ever sees a non-negative scale.
    uint32_t idesc_qk_neg;
    // Scale 0 makes every score 0 whatever Q holds: Q tiles are then read
    // from head index BH, outside the tensor, which TMA fills with zeros, and
    // the softmax runs with scale_log2 = 1.
    int zero_q;
    float *lse;
    unsigned int *status;
    uint64_t wait_ns;   // limit of every bounded wait (kWaitLimitNs unless a test lowers it)
    int stall_load;     // test only: ring load CTA 0's producer skips (-1: none)
    __device__ int q_head(int bh) const { return zero_q ? sc.BH : bh; }
};

// Work-item queue slots. The consumers release a slot when they have finished
// its item, so the producer holds at most one item beyond the running one
// (more would let a CTA hoard short items at the end of the launch).
constexpr int kQueue = 2;

struct Bars {
    uint64_t q_full[kTiles];   // Q_t of the current item landed (one phase per item with keys)
    uint64_t s_full[kTiles];   // S_t(j) in TMEM (one phase per key tile)
    uint64_t p_full[kTiles];   // P_t(j) in TMEM and O_t rescaled (one phase per key tile)
    uint64_t o_done[kTiles];   // last O_t += P_t V completed (one phase per item with keys)
    uint64_t item_full[kQueue];
    uint64_t item_empty[kQueue];
    uint64_t drain;
    uint64_t kv_full[16];
    uint64_t kv_empty[16];
    int items[kQueue];
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

using sched::Item;
using sched::visible_keys;
static_assert(kTiles == sched::kTiles && kBlockM == sched::kTileRows && kBlockN == sched::kKeyTile,
              "the kernel's tiles are the schedule's items");

// 64 TMEM columns of this thread's lane, without waiting: the registers are
// written when the load completes, which tmem_ld_wait_regs64 waits for.
__device__ __forceinline__ void tmem_ld64_nowait(uint32_t taddr, uint32_t (&r)[64])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]),
          "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
          "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
          "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]),
          "=r"(r[63])
        : "r"(taddr), "r"(taddr + 32u)
        : "memory");
}

// Wait for this thread's TMEM loads; r is an operand (read and written), so
// every use of the loaded registers stays after the wait.
__device__ __forceinline__ void tmem_ld_wait_regs64(uint32_t (&r)[64])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]),
                   "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]),
                   "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]),
                   "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]),
                   "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]),
                   "+r"(r[63])
                 :
                 : "memory");
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

    if (threadIdx.x == 0) {
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(&bars->q_full[t], 1);
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->p_full[t], 4);
            mbar_init(&bars->o_done[t], 1);
        }
        for (int s = 0; s < kQueue; ++s) {
            mbar_init(&bars->item_full[s], 1);
            mbar_init(&bars->item_empty[s], 1 + kSoftmaxWarps);  // MMA warp + softmax warps
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
        // Takes work items from the launch's counter, publishes each to the
        // other roles through the item queue, then loads its Q tiles and its
        // K_j, V_j through the ring. Items run back to back: the next item's
        // first K/V tiles and Q tiles load while the current one finishes.
        // The whole warp runs the loop and polls each barrier together; lane 0
        // alone takes items and issues the copies and arrivals.
        {
            const uint64_t pol_stream = l2_policy_evict_first();  // Q: read once
            const uint64_t pol_keep = l2_policy_evict_last();     // K/V: re-read by other q-blocks
            int it = 0;                       // ring index, continuous across items
            // Q_t loads so far. Each is for an item with keys on tile t, which
            // also completes one o_done[t] phase when its last MMA is done.
            uint32_t q_loads[kTiles] = {0, 0};
            bool ok = true;
            // A bounded wait polled by the whole warp together, made warp-uniform.
            auto wwait = [&](uint64_t *bar, uint32_t parity) {
                return __all_sync(0xffffffffu,
                                  mbar_wait(bar, parity, abort_flag, p.status, p.wait_ns));
            };
            auto load_kv = [&](int j, int which, int bh) {
                const int s = it % C::kStages;
                const uint32_t use = it / C::kStages;
                if (use > 0 && !wwait(&bars->kv_empty[s], (use - 1) & 1))
                    return false;
                if (it == p.stall_load && blockIdx.x == 0) {
                    // Test only: this load is never issued, so the MMA warp's
                    // bounded wait for it runs out and the CTA takes its abort path.
                    ++it;
                    return true;
                }
                if (lane == 0) {
                    fa_check(j * kBlockN < p.sc.Sk && bh < p.sc.BH, p.status);
                    mbar_arrive_expect_tx(&bars->kv_full[s], C::kTileBytes);
                    const CUtensorMap *tm = which == 0 ? &tm_k : &tm_v;
                    for (int b = 0; b < C::kBoxes; ++b)
                        tma_load_3d_hint(sKV + s * C::kTileBytes + b * kBoxBytes, tm,
                                         &bars->kv_full[s], b * 64, j * kBlockN, bh, pol_keep);
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
                        mbar_arrive_expect_tx(&bars->q_full[t], C::kTileBytes);
                        for (int b = 0; b < C::kBoxes; ++b)
                            tma_load_3d_hint(sQ + t * C::kTileBytes + b * kBoxBytes, &tm_q,
                                             &bars->q_full[t], b * 64, I.q0[t], p.q_head(I.bh),
                                             pol_stream);
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
                        mbar_wait_drain(&bars->q_full[t], (q_loads[t] - 1) & 1, p.status, p.wait_ns);
                for (int k = max(0, it - C::kStages); k < it; ++k)
                    mbar_wait_drain(&bars->kv_full[k % C::kStages], (k / C::kStages) & 1, p.status,
                                    p.wait_ns);
            }
            __syncwarp();
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // Per item, ring order of the loads: K_0, V_0, K_1, V_1, ... (K_j at
        // index 2j, V_j at 2j+1 from the item's first ring index), consumed in
        // the same order. Issue order: S_0(0), S_1(0), then per j: PV_0(j),
        // S_0(j+1), PV_1(j), S_1(j+1). S_t(j+1) overwrites the TMEM columns
        // that held P_t(j), and the next item's PV_t(0) overwrites O_t; the
        // tensor pipe executes one lane's MMAs in order, and the softmax
        // warps have read O_t (epilogue) before they publish the next P_t.
        // The whole warp runs the loop (its counters and descriptors stay
        // warp-uniform); the warp polls each barrier together, and one elected
        // lane issues each MMA and commit.
        {
            const uint32_t idesc_qk = idesc_bf16_f32(kBlockM, kBlockN, false, false) | p.idesc_qk_neg;
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
                    umma_bf16_ss_elect(tmem + colS[t], a0 + koff, b0 + koff, idesc_qk,
                                       kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int slot, int j) {
                const uint64_t b0 = dv0 + kTileStep * slot;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    umma_bf16_ts_elect(tmem + colO[t], tmem + colS[t] + kk * 8,
                                       b0 + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_pv,
                                       (j > 0 || kk > 0) ? 1u : 0u);
            };
            // A bounded wait polled by the whole warp together (each poll is one
            // warp instruction, and the warp sleeps in it), made warp-uniform.
            auto wwait = [&](uint64_t *bar, uint32_t parity) {
                return __all_sync(0xffffffffu,
                                  mbar_wait(bar, parity, abort_flag, p.status, p.wait_ns));
            };
            auto ring_wait = [&](int idx) {
                return wwait(&bars->kv_full[idx % C::kStages], (idx / C::kStages) & 1);
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
                // S_t(0) as soon as Q_t is in: tile 0's Q buffer frees a key
                // tile earlier than tile 1's at the end of a causal item.
                ok = ring_wait(it);  // K_0
                for (int t = 0; t < kTiles && ok; ++t) {
                    if (I.n_kv[t] == 0)
                        continue;
                    ok = wwait(&bars->q_full[t], (q_waits[t]++) & 1);
                    if (!ok)
                        break;
                    tc_fence_after_sync();
                    issue_s(t, it % C::kStages);
                    umma_commit_elect(&bars->s_full[t]);
                }
                if (!ok)
                    break;
                umma_commit_elect(&bars->kv_empty[it % C::kStages]);
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
                        issue_pv(t, iv % C::kStages, j);
                        if (j + 1 < I.n_kv[t]) {
                            if (!k_ready) {
                                ok = ring_wait(ik);  // K_{j+1}
                                if (!ok)
                                    break;
                                tc_fence_after_sync();
                                k_ready = true;
                            }
                            issue_s(t, ik % C::kStages);
                            umma_commit_elect(&bars->s_full[t]);
                        } else {
                            umma_commit_elect(&bars->o_done[t]);  // this tile's last PV of the item
                        }
                    }
                    if (!ok)
                        break;
                    umma_commit_elect(&bars->kv_empty[iv % C::kStages]);
                    if (k_ready)
                        umma_commit_elect(&bars->kv_empty[ik % C::kStages]);
                }
                it += 2 * I.n_kv_max;
                if (lane == 0)
                    mbar_arrive(&bars->item_empty[slot]);  // every MMA of the item is issued
            }
            // Drain: all MMAs issued by the elected lane complete before TMEM is freed.
            umma_commit_elect(&bars->drain);
            if (lane == 0)
                mbar_wait_drain(&bars->drain, 0, p.status, p.wait_ns);
            __syncwarp();
        }
    } else if (warp < kSoftmaxWarps) {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = warp / 4;              // query tile of this warpgroup
        const int wq = warp % 4;             // TMEM lane quarter of this warp
        const int r = wq * 32 + lane;        // row within the tile
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_base + (t == 0 ? C::kColS0 : C::kColS1);
        const uint32_t tO = tmem + lane_base + (t == 0 ? C::kColO0 : C::kColO1);
        const float sl2 = p.scale_log2;
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
                mbar_wait(&bars->item_full[slot], (n / kQueue) & 1, abort_flag, p.status, p.wait_ns));
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

            // ref: the reference of this row's exponentials, in log2 units of
            // the exponent (p = 2^(s * sl2 - ref), s the MMA's score). It is
            // set by the row's first visible tile to that tile's max. At d = 128
            // it moves only when a row sum of p against it exceeds kMoveLimit
            // (so P stays <= 2^16): by an integer k, multiplying the p already
            // computed (bf16) and O, l by 2^-k, all exact. At d = 64 it moves
            // when a tile's max lies more than 2^kRescaleLog2 above it (P stays
            // <= 2^kRescaleLog2). O and l always share the reference, so the
            // result stays exact.
            float ref = -INFINITY;
            float l = 0.0f;  // running sum of 2^(s * sl2 - ref), fp32 (for the LSE)
            // O's divisor: l, except that at d = 128 a tile with a row sum above
            // 2^kRescaleLog2 adds the sum of its bf16 weights (those P V used),
            // so that a row's dominant weight, rounded to bf16 there, cancels in
            // O / ln.
            float ln = 0.0f;
            for (int j = 0; j < n_kv && ok; ++j) {
                ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[t], (s_waits++) & 1,
                                                       abort_flag, p.status, p.wait_ns));
                if (!ok)
                    break;
                tc_fence_after_sync();
                const bool masked_tile = j >= mask_from;
                const int key0 = j * kBlockN;
                uint32_t pk[kBlockN / 2];
                float2 acc[4];
                // One pass over S_t in chunks of kChunk columns: load, mask, and
                // (when `with_exp`) p = 2^(s*sl2 + neg), accumulated into acc and
                // packed into pk. Returns the max of the raw scores (when
                // `with_max`; -inf otherwise).
                auto pass = [&](bool with_exp, bool with_max, float neg) {
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
                        if (with_max) {
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
                        }
                        if (with_exp) {
#pragma unroll
                            for (int c = 0; c < kChunk / 2; ++c) {
                                const float2 x = ffma2(make_float2(sv[2 * c], sv[2 * c + 1]), sl2x2,
                                                       negx2);
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
                // On the max-based path (d = 64, and d = 128's first tiles and
                // recomputations) the reference moves only when the tile's max
                // exceeds it by more than 2^kRescaleLog2 (or on the first visible
                // key), so that tile's P stays <= 2^kRescaleLog2; O and l always
                // share the reference, so the result stays exact. NaN (both -inf)
                // compares false: nothing visible yet, keep the reference. Until
                // P is written, S_t is intact and may be read again.
                float ref_use = ref, corr = 1.0f;
                bool any_move = false;  // some lane of the warp moved its reference
                float norm_sum = -1.0f;  // >= 0: this tile's contribution to ln (else the fp32 sum)
                // From the tile's max score mx: a row's first visible key sets the
                // reference to the max (tested on ref itself: at scale 0 a product
                // with sl2 would be NaN); later the reference moves to the max
                // when it lies more than 2^kRescaleLog2 above it.
                auto decide = [&](float mx) {
                    const float x_max = mx * sl2;
                    const bool first = ref == -INFINITY;
                    const bool move =
                        first ? (mx != -INFINITY) : (x_max - ref > kRescaleLog2);
                    ref_use = move ? x_max : ref;
                    corr = move ? (first ? 0.0f : ex2_approx(ref - ref_use)) : 1.0f;
                    any_move = __any_sync(0xffffffffu, move);
                };
                // Moves the reference up by the integer k >= 0 (per lane): the p
                // already in pk (bf16) and acc (fp32) are multiplied by 2^-k, and
                // corr = 2^-k takes O and l along. A product with a power of two
                // is exact; only weights below 2^-126 of the new reference round
                // (to a subnormal or 0). The same as recomputing p against
                // ref + k, without another pass over S.
                auto shift = [&](int k) {
                    const float f = __int_as_float((127 - k) << 23);
                    const uint32_t h = static_cast<uint32_t>(127 - k) << 7;
                    const uint32_t f2 = h | (h << 16);
#pragma unroll
                    for (int c = 0; c < kBlockN / 2; ++c)
                        pk[c] = mul_bf16x2(pk[c], f2);
                    const float2 fx2 = make_float2(f, f);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        acc[q] = fmul2(acc[q], fx2);
                    ref_use = ref + static_cast<float>(k);
                    corr = f;
                };
                // O_t *= corr after a move (warp-uniform; lanes that did not move
                // multiply by 1). PV_t(j-1) has completed: S_t(j), committed after
                // it, is done.
                auto rescale_o = [&]() {
                    if (j == 0 || !any_move)
                        return;
                    const float2 cx2 = make_float2(corr, corr);
                    // d = 128: 64 columns per TMEM round trip (0.98x the time on
                    // the 2K Q x 4 input against 32; at d = 64 that form measured
                    // 1.02x, so d = 64 keeps 32).
                    constexpr int kCols = (D == 128) ? 64 : 32;
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += kCols) {
                        uint32_t o[kCols];
                        if constexpr (kCols == 64)
                            tmem_ld64_wait(tO + c0, o);
                        else
                            tmem_ld32_wait(tO + c0, o);
#pragma unroll
                        for (int c = 0; c < kCols / 2; ++c) {
                            const float2 v = fmul2(make_float2(__uint_as_float(o[2 * c]),
                                                               __uint_as_float(o[2 * c + 1])),
                                                   cx2);
                            o[2 * c] = __float_as_uint(v.x);
                            o[2 * c + 1] = __float_as_uint(v.y);
                        }
                        if constexpr (kCols == 64)
                            tmem_st64(tO + c0, o);
                        else
                            tmem_st32(tO + c0, o);
                    }
                };
                if constexpr (D == 128) {
                    // Speculative pass without the max: when every lane has a
                    // reference, p is computed against it. Every p is >= 0, so a row
                    // sum of at most 2^kRescaleLog2 shows that no p exceeds
                    // 2^kRescaleLog2 and the reference stays. When every row sum
                    // is at most kMoveLimit the reference stays too, and O's
                    // divisor takes the tile's bf16 weights (those P V uses): a
                    // weight that dominates its row is then the same in O and in
                    // its divisor. A larger sum (up to kShiftLimit, so that no p
                    // can have overflowed) is settled from the packed p: their
                    // max, and a shift by its exponent when it exceeds
                    // 2^kRescaleLog2. Only a larger sum, or a row's first tile,
                    // runs the max pass and then the exponentials against the new
                    // reference. The passes run one per iteration of this loop,
                    // so the code holds one copy of the pass (three copies spilled
                    // at 168 registers). Stages: 0 speculative exponentials, 1 max,
                    // 2 exponentials.
                    int stage = __all_sync(0xffffffffu, ref != -INFINITY) ? 0 : 1;
#pragma unroll 1
                    while (true) {
                        const bool with_exp = stage != 1;
                        const float neg =
                            stage == 0 ? -ref : ((ref_use == -INFINITY) ? 0.0f : -ref_use);
                        const float mx = pass(with_exp, !with_exp, neg);
                        if (stage == 0) {
                            const float2 a = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
                            const float sum = a.x + a.y;
                            if (!__any_sync(0xffffffffu, sum > kRescaleFactor))
                                break;
                            if (__all_sync(0xffffffffu, sum <= kShiftLimit)) {
                                // Up to kMoveLimit the reference stays (0.84x the
                                // time of shifting by the max's exponent on the 2K
                                // Q x 4 input: no multiply of P, no TMEM round trip
                                // of O). A sum above it implies a p above 2^9, so
                                // some lane moves.
                                // O's divisor takes the bf16 weights (summed below
                                // the loop where norm_sum is set to 0): every lane's
                                // when the reference stays, the moved lanes' after a
                                // move.
                                norm_sum = 0.0f;
                                if (!__all_sync(0xffffffffu, sum <= kMoveLimit)) {
                                    const float pmax = max_bf16x2_row(pk);
                                    const int k =
                                        pmax > kRescaleFactor ? (__float_as_int(pmax) >> 23) - 127 : 0;
                                    norm_sum = k > 0 ? 0.0f : -1.0f;
                                    any_move = __any_sync(0xffffffffu, k > 0);
                                    if (any_move) {
                                        shift(k);
                                        rescale_o();
                                    }
                                }
                                break;
                            }
                            stage = 1;
                        } else if (stage == 1) {
                            decide(mx);
                            stage = 2;
                        } else {
                            rescale_o();
                            break;
                        }
                    }
                    if (norm_sum == 0.0f)
                        norm_sum = sum_bf16x2_row(pk);
                } else {
                    // d = 64: the speculative pass finds the tile's max while it
                    // computes p against the reference (the form above measured
                    // 1.01x to 1.07x slower at this head dim); a second pass
                    // follows when the reference moves (a shift in place of it
                    // measured 1.015x slower here).
                    const bool spec = __all_sync(0xffffffffu, ref != -INFINITY);
                    decide(pass(spec, true, spec ? -ref : 0.0f));
                    if (!spec || any_move) {
                        pass(true, true, (ref_use == -INFINITY) ? 0.0f : -ref_use);
                        rescale_o();
                    }
                }
                // P (bf16 pairs) over S_t's first 64 columns, then publish.
                tmem_st64(tS, pk);
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars->p_full[t]);
                const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
                const float2 a = fadd2(a01, a23);
                l = l * corr + (a.x + a.y);
                ln = ln * corr + (norm_sum >= 0.0f ? norm_sum : a.x + a.y);
                ref = ref_use;
            }

            // -------------------------------------------------------- epilogue
            // O / l into this tile's staging box (swizzled like the TMA box), one
            // 64-column box at a time, each sent by a TMA store, then the LSE.
            // The next item's P_t is published only after these TMEM reads, so
            // its PV_t(0) cannot overwrite O_t early.
            if (q0 >= p.sc.Sq) {
                release();
                continue;
            }
            // d = 128: the previous item's last store may still be reading the
            // staging box; its issuer waits here, before the barrier below, so
            // the box is rewritten only after that read. Waiting at the end of
            // that epilogue instead put the wait on the tile's critical path
            // (measured 1.002-1.014x the time); at d = 64, one box per tile,
            // the wait stays there (the deferred form measured 1.007x).
            constexpr bool kDeferLastRead = (D == 128);
            if (kDeferLastRead && r == 0)
                tma_store_wait_read_all();
            bool got = ok;
            if (got && n_kv > 0) {
                got = __all_sync(0xffffffffu, mbar_wait(&bars->o_done[t], (o_waits++) & 1,
                                                        abort_flag, p.status, p.wait_ns));
                if (got)
                    tc_fence_after_sync();
            }
            // The tile's 4 warps take the barriers below together or not at all.
            if (named_bar_or(1 + t, 128, !got)) {
                ok = false;
                break;
            }
            const float inv_l = (ln > 0.0f) ? 1.0f / ln : 0.0f;
            uint8_t *sOut = smem + C::kOffOut + t * kBoxBytes;
            const uint32_t sOut_a = smem_u32(sOut);
            // Box b (O's columns 64 b .. 64 b + 63) is in the staging box: send it.
            auto store_box = [&](int b) {
                fence_proxy_async_smem();
                named_bar_sync(1 + t, 128);
                if (r == 0) {
                    fa_check(q0 < p.sc.Sq && I.bh < p.sc.BH, p.status);
                    tma_store_3d(&tm_o, sOut, b * 64, q0, I.bh);
                    tma_store_commit();
                    // The next box is written only after this store has read the
                    // box (the barrier at the top of the next box); at d = 128
                    // the last box's read is waited for at the next epilogue.
                    // The writes to global memory finish on their own.
                    if (b + 1 < C::kBoxes || !kDeferLastRead)
                        tma_store_wait_read_all();
                }
            };
            if constexpr (D == 128) {
                // The second box's TMEM load is issued as soon as the first box
                // is in shared memory and waited for after the barrier, so its
                // latency overlaps the first box's store (0.99x the headline's
                // time against loading it after that barrier; at d = 64, one
                // box, a single 64-column load measured 1.017x, so d = 64 keeps
                // two 32-column loads below).
                uint32_t o[64];
                if (n_kv > 0) {
                    tmem_ld64_wait(tO, o);
                } else {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        o[c] = 0u;
                }
#pragma unroll
                for (int b = 0; b < C::kBoxes; ++b) {
                    if (b > 0) {
                        named_bar_sync(1 + t, 128);  // the previous box has been read out
                        if (n_kv > 0)
                            tmem_ld_wait_regs64(o);
                    }
                    uint32_t pko[32];
#pragma unroll
                    for (int c = 0; c < 64; c += 2)
                        pko[c / 2] = pack_bf16x2(__uint_as_float(o[c]) * inv_l,
                                                 __uint_as_float(o[c + 1]) * inv_l);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        st_shared_v4(sOut_a + sw128_offset(static_cast<uint32_t>(r), static_cast<uint32_t>(q)),
                                     pko[4 * q], pko[4 * q + 1], pko[4 * q + 2], pko[4 * q + 3]);
                    if (b + 1 < C::kBoxes && n_kv > 0)
                        tmem_ld64_nowait(tO + 64 * (b + 1), o);
                    store_box(b);
                }
            } else {
#pragma unroll
                for (int c1 = 0; c1 < 64; c1 += 32) {
                    uint32_t o[32];
                    if (n_kv > 0) {
                        tmem_ld32_wait(tO + c1, o);
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            o[c] = 0u;
                    }
                    uint32_t pko[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 2)
                        pko[c / 2] = pack_bf16x2(__uint_as_float(o[c]) * inv_l,
                                                 __uint_as_float(o[c + 1]) * inv_l);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t chunk = (c1 / 8) + q;
                        st_shared_v4(sOut_a + sw128_offset(static_cast<uint32_t>(r), chunk),
                                     pko[q * 4], pko[q * 4 + 1], pko[q * 4 + 2], pko[q * 4 + 3]);
                    }
                }
                store_box(0);
            }
            if (i < p.sc.Sq) {
                // ref is in log2 units: ref * ln 2 is the max in units of the
                // scaled scores
                const float lse = (l > 0.0f) ? ref * 0.69314718055994531f + logf(l) : -INFINITY;
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
    // The launch's last CTA to finish puts its work counters back to zero for
    // the next launch that takes this slot.
    if (threadIdx.x == 0)
        sched::finish_cta(p.sc);
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
    unsigned grid = 0;
    const fa_status_t st = sched::make_schedule(pr, 2.0 * static_cast<double>(pr.Sk) * D * 2.0,
                                                &p.sc, &grid);
    if (st != FA_OK)
        return st;
    p.scale = fabsf(pr.scale);
    p.zero_q = pr.scale == 0.0f ? 1 : 0;
    p.scale_log2 = p.zero_q ? 1.0f : fabsf(pr.scale) * 1.4426950408889634f;
    p.idesc_qk_neg = std::signbit(pr.scale) ? kIdescNegateA : 0u;
    p.lse = pr.lse;
    p.status = pr.status;
    p.wait_ns = kWaitLimitNs;
    p.stall_load = -1;
    take_stall(kStallPrefill, &p.stall_load, &p.wait_ns);
    auto kern = fa_prefill_kernel<D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return FA_ERR_CUDA;
    kern<<<grid, kThreads, C::kSmemBytes, pr.stream>>>(tq, tk, tv, to, p);
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
