// fa_schedule.cuh — work items of the persistent forward kernels (bf16 and
// FP8): what an item is, the order items are handed out in, and the
// per-launch counter CTAs take them from.
//
// An item is two consecutive 128-row query tiles of one (batch, head); its
// cost under the causal mask grows with its position. Heads are taken in
// groups of heads_per_group (the last group may be smaller) and, within a
// group, query blocks go heaviest first across all the group's heads. One
// head per group is head-major order, in which the items handed out together
// share a few heads' K/V in L2.
#pragma once

#include <algorithm>
#include <atomic>
#include <cmath>

#include "fa_internal.h"

namespace fa {
namespace sched {

constexpr int kTileRows = 128;  // query rows per tile
constexpr int kTiles = 2;       // query tiles per item
constexpr int kKeyTile = 128;   // keys per K/V tile

struct Schedule {
    int Sq, Sk, BH, n_qblk, n_items, heads_per_group, causal;
    unsigned long long *work;  // this launch's (next item, finished CTAs) pair
};

struct Item {
    int bh;
    int q0[kTiles], n_kv[kTiles], mask_from[kTiles];
    int n_kv_max;
};

// Number of keys visible to query row i (bottom-right causal alignment).
__device__ __forceinline__ int visible_keys(int i, int Sq, int Sk, int causal)
{
    if (!causal)
        return Sk;
    int n = i + (Sk - Sq) + 1;
    return n < 0 ? 0 : (n > Sk ? Sk : n);
}

__device__ __forceinline__ Item decode_item(int w, const Schedule &s)
{
    Item it;
    const int per_group = s.heads_per_group * s.n_qblk;
    const int g = w / per_group, rg = w % per_group;
    const int hg = min(s.heads_per_group, s.BH - g * s.heads_per_group);
    it.bh = g * s.heads_per_group + rg % hg;
    const int qblk = s.n_qblk - 1 - rg / hg;
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
        it.q0[t] = qblk * (kTiles * kTileRows) + t * kTileRows;
        if (it.q0[t] < s.Sq) {
            const int last = min(it.q0[t] + kTileRows - 1, s.Sq - 1);
            it.n_kv[t] = (visible_keys(last, s.Sq, s.Sk, s.causal) + kKeyTile - 1) / kKeyTile;
            it.mask_from[t] = visible_keys(it.q0[t], s.Sq, s.Sk, s.causal) / kKeyTile;
        } else {
            it.n_kv[t] = 0;
            it.mask_from[t] = 0;
        }
    }
    it.n_kv_max = max(it.n_kv[0], it.n_kv[1]);
    return it;
}

// The next work item of this launch, or -1 when none is left.
__device__ __forceinline__ int grab_item(const Schedule &s)
{
    const unsigned long long w = atomicAdd(s.work, 1ull);
    return w < static_cast<unsigned long long>(s.n_items) ? static_cast<int>(w) : -1;
}

// Called by one thread of each CTA as it exits: the launch's last CTA puts
// the counter pair back to zero for the next launch that takes the slot.
__device__ __forceinline__ void finish_cta(const Schedule &s)
{
    __threadfence();
    if (atomicAdd(s.work + 1, 1ull) == gridDim.x - 1) {
        atomicExch(s.work, 0ull);
        atomicExch(s.work + 1, 0ull);
    }
}

// Host side: the schedule of one launch and its grid (one CTA per SM, never
// more CTAs than items). kv_bytes_per_head is the size of one head's K and V.
//
// Item order. Causal items differ in cost, and when a CTA runs only a few of
// them the last ones decide the tail. Up to 2048 keys the heads are
// therefore taken in groups whose K/V share 48 MB of L2 and each group's
// query blocks go heaviest first across its heads; measured on the bf16
// kernel: 0.87x / 0.88x the time of head-major order at S = 1024 / 2048.
// Longer causal problems and non-causal ones (equal items) keep head-major
// order, which keeps each head's K/V reads together; grouping cost 1.02x at
// S = 4096.
//
// Launches take the counter slots in turn; a slot is back at zero when its
// launch ends, so only launches more than kWorkSlots apart that run at the
// same time could share one.
inline fa_status_t make_schedule(const Problem &pr, double kv_bytes_per_head, Schedule *s,
                                 unsigned *grid)
{
    if (!pr.work_slots || pr.num_sms <= 0)
        return FA_ERR_CUDA;
    const uint64_t BH = static_cast<uint64_t>(pr.B * pr.H);
    s->Sq = static_cast<int>(pr.Sq);
    s->Sk = static_cast<int>(pr.Sk);
    s->BH = static_cast<int>(BH);
    s->n_qblk = static_cast<int>((pr.Sq + kTiles * kTileRows - 1) / (kTiles * kTileRows));
    const uint64_t n_items = static_cast<uint64_t>(s->n_qblk) * BH;
    if (n_items > 0x7FFFFFFFull)
        return FA_ERR_UNSUPPORTED;
    s->n_items = static_cast<int>(n_items);
    s->causal = pr.causal ? 1 : 0;
    s->heads_per_group = 1;
    if (pr.causal && pr.Sk <= 2048) {
        const double budget = 48.0 * (1 << 20);
        s->heads_per_group = static_cast<int>(std::max(
            1.0, std::min(static_cast<double>(BH), std::floor(budget / kv_bytes_per_head))));
    }
    static std::atomic<unsigned int> next_slot{0};
    s->work = pr.work_slots +
              2 * (next_slot.fetch_add(1, std::memory_order_relaxed) % kWorkSlots);
    *grid = static_cast<unsigned>(std::min<uint64_t>(n_items, static_cast<uint64_t>(pr.num_sms)));
    return FA_OK;
}

}  // namespace sched
}  // namespace fa
