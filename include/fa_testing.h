/*
 * fa_testing.h — test-only entry points of the attention library.
 *
 * None of these is on the product path; fa_forward never dispatches to them.
 * They exist so that the GPU test suite can check the pieces of the tensor-core
 * kernels in isolation and exercise the failure detection without faulting
 * or hanging a GPU. Conventions (pointers, stream, errors) are those of fa.h.
 */
#ifndef FA_TESTING_H
#define FA_TESTING_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Plain SIMT (CUDA-core, fp32) version of the tiled forward with the online
 * softmax of "Warmup Guide — Inference Optimization at Depth", Chapters 3-4:
 * one thread per query row, keys visited in order, running max / sum /
 * unnormalised O, one division at the end. Same arguments, layouts and
 * outputs as fa_forward; any d in [1, 128]; slow. A second, independent GPU
 * implementation for cross-checks.
 */
fa_status_t fa_reference_forward_simt(const void *q, const void *k, const void *v, void *o,
                                      float *lse, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                                      int64_t d, int causal, float scale, void *stream);

/*
 * One-CTA tcgen05 GEMM used to check the shared-memory/instruction
 * descriptor encodings and the TMA -> SMEM -> tcgen05.mma -> TMEM ->
 * tcgen05.ld path on their own:
 *     b_mn_major == 0 : C[128, N] = A[128, K] . B[N, K]^T   (B row-major N x K)
 *     b_mn_major == 1 : C[128, N] = A[128, K] . B[K, N]     (B row-major K x N)
 * A, B bf16 row-major device arrays, C fp32 row-major [128, N].
 * N in {64, 128}, K in {64, 128}.
 */
fa_status_t fa_selftest_umma(const void *a, const void *b, float *c, int n, int k,
                             int b_mn_major, void *stream);

/*
 * The same one-tile GEMM with A (128 x K) read by the MMA from tensor memory
 * instead of shared memory: row r of A goes to TMEM lane r, two bf16 per
 * 32-bit column (element 2c in the low half). Arguments as fa_selftest_umma.
 */
fa_status_t fa_selftest_umma_ts(const void *a, const void *b, float *c, int n, int k,
                                int b_mn_major, void *stream);

/*
 * The E4M3 products of fa_forward_fp8 on one tile, with .kind::f8f6f4 MMAs:
 *     C[128, N] = A[128, 128] . B,  B = b[N, 128]^T (b_mn_major 0, E4M3 bytes)
 *                                  or b[128, N]     (b_mn_major 1, N = 128).
 * a_tmem == 0: `a` is E4M3 bytes [128, 128], loaded by TMA into shared memory.
 * a_tmem == 1: `a` is fp32 [128, 128]; each row is rounded to E4M3 and packed
 * four per 32-bit TMEM column (element 4c + e in byte e), the MMA reading A
 * from tensor memory. C fp32 row-major [128, N]; N in {64, 128}.
 */
fa_status_t fa_selftest_umma_f8(const void *a, const void *b, float *c, int n, int b_mn_major,
                                int a_tmem, void *stream);

/*
 * exp2 (MUFU) throughput microbenchmark: `blocks` CTAs of 256 threads, each
 * thread running 8 independent chains of iters ex2.approx (with one FMA each to
 * keep the values in range), i.e. blocks * 256 * iters * 8 ex2 in all. `out`
 * receives one float per thread (blocks * 256, device memory). Time it with
 * events on `stream`; it gives the softmax's exponential rate bound.
 */
fa_status_t fa_selftest_mufu(float *out, int blocks, int iters, void *stream);

/*
 * tcgen05.mma rate microbenchmark (fp32 accumulator, M = 128): `blocks` CTAs
 * (one per SM at most is meaningful; each holds 97 KB of shared memory and all
 * 512 TMEM columns), one thread each issuing `iters` rounds of one
 * 128 x 128 x 128 product, in form `mode`:
 *   0  bf16, A and B from shared memory, N = 128 (8 instructions of K = 16)
 *   1  bf16, A and B from shared memory, two N = 64 halves (each 8
 *      back-to-back MMAs into its own accumulator)
 *   2  bf16, A from tensor memory, N = 128
 *   3  bf16, A from tensor memory, two N = 64 halves
 *   4  bf16, A and B from shared memory, N = 256 (a round is two products)
 *   5  E4M3 (.kind::f8f6f4), A and B from shared memory, N = 128
 *      (4 instructions of K = 32)
 *   6  E4M3, A from tensor memory, N = 128
 * cycles[b] (device memory, `blocks` entries) receives the SM clock cycles of
 * CTA b from its first issue to the completion of its last MMA, or -1 if the
 * bounded wait for completion gave up (the device status word then records
 * the timeout). Used to choose the MMA shapes of the gradient kernels.
 * Returns FA_ERR_UNSUPPORTED for another mode, FA_ERR_INVALID_ARG for a null
 * pointer or a non-positive count.
 */
fa_status_t fa_selftest_mma_rate(long long *cycles, int mode, int blocks, int iters, void *stream);

/*
 * Launches one CTA whose thread waits, with the same bounded wait the
 * attention kernels use, on an mbarrier that nothing ever completes. After
 * `timeout_ns` nanoseconds the wait gives up and sets the device status word
 * to FA_ERR_TIMEOUT; fa_device_status() then reports it. Nothing faults or
 * hangs: the kernel returns normally.
 */
fa_status_t fa_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

/*
 * Device-side index checks. A library compiled with FA_DEBUG defined (the
 * debug build, lib/libfa_gb300_debug.so, made by build.build_debug()) checks
 * the index arithmetic of its kernels before each plain global load or store
 * (skipping the access if the check fails) and the coordinates of each TMA
 * copy (reported only: the hardware bounds those itself). A failed check sets
 * a bit in the device status word, which fa_device_status() reports as
 * FA_ERR_BOUNDS. Nothing asserts or traps. Release builds compile the checks
 * away.
 * fa_testing_debug_checks: 1 in a debug build, 0 otherwise.
 * fa_selftest_index_check: launches one check that passes (fail == 0) or
 * fails (fail != 0); in a debug build a failing one makes the next
 * fa_device_status() return FA_ERR_BOUNDS.
 */
int fa_testing_debug_checks(void);
fa_status_t fa_selftest_index_check(int fail, void *stream);

/*
 * The lane that elect.sync picks in a converged warp. The MMA-issuing warps
 * of the prefill and backward kernels run their issue loops as a whole warp
 * and let elect.sync pick the lane that issues each tcgen05.mma and each
 * tcgen05.commit; a commit tracks only its own thread's MMAs, so every
 * election must pick the same lane. Launches one CTA of 4 warps; each warp
 * runs `trials` elections (after lane-dependent work and a reconvergence)
 * and writes the elected lane id of election i to lanes[warp * trials + i].
 *   lanes  : device int[4 * trials], caller-owned, written by the kernel
 *   trials : 1 .. 2^20
 * FA_ERR_INVALID_ARG for a null pointer or a count out of range;
 * asynchronous on `stream`.
 */
fa_status_t fa_selftest_elect(int *lanes, int trials, void *stream);

/*
 * Makes the next launch of one production kernel stall on purpose, so that
 * its bounded waits run out and its abort path runs (set the abort flag,
 * record FA_ERR_TIMEOUT in the device status word, drain the copies and MMAs
 * in flight, free tensor memory, put the work counter back) without faulting
 * or hanging the GPU:
 *   kernel 1  the bf16 prefill kernel (fa_prefill_forward, fa_forward for
 *             Sq > 16): the first CTA's producer skips its ring load number
 *             skip_index (K_0, V_0, K_1, V_1, ... counted across its items),
 *             so the MMA thread's wait for that load runs out;
 *   kernel 2  the split-KV verify kernel (fa_verify_forward and the entry
 *             points built on it): the producer of CTA (chunk 0, b*h 0) skips
 *             its 64-key stage number skip_index, so its consumers' wait runs
 *             out.
 * wait_limit_ns becomes the limit of every bounded wait of that launch
 * (including the drains), in place of the default 2 s. The request is taken
 * by the next launch of that kernel in this process and then cleared; if the
 * first CTA issues fewer loads than skip_index + 1, nothing is skipped. Call
 * fa_device_status() after the stalled launch: it reports FA_ERR_TIMEOUT and
 * clears the word, which the next launch needs (while the word records a
 * timeout every launch gives up at its first slow wait).
 * Returns FA_ERR_INVALID_ARG for another kernel, skip_index < 0, or
 * wait_limit_ns outside [1 ms, 10 s].
 */
fa_status_t fa_testing_stall_next_launch(int kernel, int skip_index, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* FA_TESTING_H */
