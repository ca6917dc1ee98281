// fa_internal.h — declarations shared by the library's translation units
// (argument bundle, launchers, tensor-map encoding). Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "fa.h"

namespace fa {

struct Problem {
    const void *q, *k, *v;
    void *o;
    float *lse;
    int64_t B, H, Sq, Sk, d;
    int causal;
    float scale;
    cudaStream_t stream;
    unsigned int *status;  // device status word (timeouts)
    int num_sms;           // SMs of the current device
    // Library-owned work counters of the persistent prefill kernel: kWorkSlots
    // pairs (next item, finished CTAs), all zero between launches.
    unsigned long long *work_slots;
};

constexpr int kWorkSlots = 1024;

// Row-major [depth, rows, inner] bf16 tensor as a 3-D TMA map with a
// (64 x box_rows x 1) box and 128-byte swizzle. Returns false on failure.
bool encode_tmap_bf16_3d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                         uint64_t depth, uint32_t box_rows);

// Row-major [depth, rows, inner] tensor of bytes (E4M3) as a 3-D TMA map with
// a (128 x box_rows x 1) box and 128-byte swizzle: one box spans a 128-byte
// row. Returns false on failure.
bool encode_tmap_u8_3d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                       uint64_t depth, uint32_t box_rows);

// Pages [num_pages, H, page_size, 128] bf16 as (64 columns, 2 column halves,
// page_size rows, H, num_pages), box = one page of one head (page_size * 256
// bytes), 128-byte swizzle.
bool encode_tmap_bf16_pages_5d(CUtensorMap *map, const void *base, uint64_t page_size, uint64_t H,
                               uint64_t num_pages);
// Row-major [outer, mid, rows, inner] bf16 tensor as a 4-D TMA map with a
// (64 x box_rows x 1 x 1) box and 128-byte swizzle (K/V page pools).
bool encode_tmap_bf16_4d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                         uint64_t mid, uint64_t outer, uint32_t box_rows);

// Options of the split-KV path beyond the contiguous causal/non-causal case.
struct VerifyOptions {
    const uint32_t *tree_mask = nullptr;  // [B, Sq] draft-position masks (replaces causal)
    // Paged K/V: Problem::k / v are page pools [num_pages, H, page_size, d],
    // Problem::Sk is the longest sequence.
    const int32_t *block_table = nullptr;  // [B, max_pages]
    const int32_t *seq_lens = nullptr;     // [B]
    int64_t page_size = 0, num_pages = 0, max_pages = 0;
};

// The backward pass: the forward's problem plus its O, LSE, the upstream
// gradient and the outputs.
struct BackwardProblem {
    Problem fwd;  // q, k, v, sizes, causal, scale, stream, status (o/lse unused)
    const void *o;
    const float *lse;
    const void *dout;
    void *dq, *dk, *dv;
    void *workspace;  // backward_workspace_bytes(B*H, Sq) bytes
};
size_t backward_workspace_bytes(int64_t BH, int64_t Sq);
fa_status_t launch_backward_sm103(const BackwardProblem &bp);

// Launchers. Each validates nothing (fa_abi.cu does) and returns FA_OK or
// FA_ERR_CUDA.
fa_status_t launch_prefill_sm103(const Problem &p);
// The FP8 forward: p.q/k/v hold E4M3 bytes, p.o bf16; d = 128 only.
fa_status_t launch_prefill_fp8_sm103(const Problem &p, float q_descale, float k_descale,
                                     float v_descale);
fa_status_t launch_selftest_umma_f8(const void *a, const void *b, float *c, int n, int b_mn_major,
                                    int a_tmem, cudaStream_t stream, unsigned int *status);
fa_status_t launch_verify(const Problem &p, int n_split, void *workspace, size_t ws_bytes,
                          const VerifyOptions &opt = VerifyOptions());
fa_status_t launch_reference_simt(const Problem &p);
fa_status_t launch_selftest_umma(const void *a, const void *b, float *c, int n, int k,
                                 int b_mn_major, cudaStream_t stream, unsigned int *status);
fa_status_t launch_selftest_umma_ts(const void *a, const void *b, float *c, int n, int k,
                                    int b_mn_major, cudaStream_t stream, unsigned int *status);
fa_status_t launch_selftest_wait(uint64_t timeout_ns, cudaStream_t stream, unsigned int *status);
fa_status_t launch_selftest_index_check(bool fail, cudaStream_t stream, unsigned int *status);
fa_status_t launch_selftest_elect(int *lanes, int trials, cudaStream_t stream);
fa_status_t launch_selftest_mufu(float *out, int blocks, int iters, cudaStream_t stream);
fa_status_t launch_selftest_mma_rate(long long *cycles, int mode, int blocks, int iters,
                                     cudaStream_t stream, unsigned int *status);

// The calling thread's current CUDA (driver) context, or nullptr if none is
// bound; device addresses looked up with cudaGetSymbolAddress are valid in
// this context only.
void *current_context();

// The argument checks of fa_verify_forward (shape, pointers, scale, Sq and
// B*H limits, split count range), in its order; touches no device.
fa_status_t verify_check_args(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                              int64_t d, float scale, int n_split);

// Test-only stall injection (fa_testing_stall_next_launch): the next launch
// of the named kernel takes the pending request, if any (one-shot), as the
// index of the load its first CTA's producer skips and the limit of its
// bounded waits; without a request both outputs are left unchanged.
constexpr int kStallPrefill = 1;
constexpr int kStallVerify = 2;
void take_stall(int kernel, int *skip_index, uint64_t *wait_ns);

// Split-KV geometry shared by the ABI (workspace sizing) and the launcher.
constexpr int kVerifyStageKeys = 64;
int verify_auto_splits(int64_t BH, int64_t Sk, int num_sms);
int64_t verify_chunk_keys(int64_t Sk, int n_split);
size_t verify_workspace_bytes(int64_t BH, int64_t Sq, int64_t d, int n_split);

}  // namespace fa
