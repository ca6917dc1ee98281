// fa_selftest.cu — test-only kernels (declared in include/fa_testing.h).
//
//  * fa_selftest_umma_kernel: one CTA computes C[128, N] = A[128, K] . B^T
//    (or A . B) with the same TMA boxes, swizzle, shared-memory descriptors,
//    instruction descriptors and TMEM read-back as the attention kernel, so
//    the tests can check each encoding against a CPU matmul on its own.
//  * fa_selftest_umma_ts_kernel: the same GEMM with A read from tensor memory
//    (the operand form a P tile held in TMEM would use).
//  * fa_selftest_umma_f8_kernel: the E4M3 products of the FP8 forward (A from
//    shared or tensor memory, B K-major or MN-major).
//  * fa_selftest_mufu_kernel: exp2 (MUFU) throughput, the softmax's second bound.
//  * fa_selftest_mma_rate_kernel: cycles per tcgen05.mma product for the
//    operand shapes the kernels choose between (bf16 with N = 64 / 128 / 256,
//    A from shared or tensor memory; E4M3 with N = 128, A from shared or
//    tensor memory).
//  * fa_selftest_wait_kernel: the bounded mbarrier wait of the attention
//    kernels on a barrier that nothing completes; it must give up after the
//    limit, set the device status word and return.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace selftest {

constexpr int kThreads = 128;

struct UmmaBars {
    uint64_t tma;
    uint64_t mma;
    uint32_t tmem_base;
    int abort_flag;
};

// A: K-major, (K/64) boxes of [128 rows x 64 cols]. B: K-major (N rows x K)
// in (K/64) boxes of [N x 64], or MN-major (K rows x N) in (N/64) boxes of
// [K x 64].
__global__ void __launch_bounds__(kThreads, 1)
    fa_selftest_umma_kernel(const __grid_constant__ CUtensorMap tm_a,
                            const __grid_constant__ CUtensorMap tm_b, float *c, int N, int K,
                            int b_mn_major, unsigned int *status)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *sA = smem;                 // 128 x K bf16
    uint8_t *sB = smem + 128 * K * 2;   // N x K bf16
    UmmaBars *bars = reinterpret_cast<UmmaBars *>(smem + 128 * K * 2 + N * K * 2);
    const int warp = threadIdx.x / 32;

    if (threadIdx.x == 0) {
        mbar_init(&bars->tma, 1);
        mbar_init(&bars->mma, 1);
        bars->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem_base, 128);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;

    bool ok = true;
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bars->tma, static_cast<uint32_t>((128 + N) * K * 2));
        for (int b = 0; b < K / 64; ++b)
            tma_load_3d(sA + b * 128 * 128, &tm_a, &bars->tma, b * 64, 0, 0);
        if (!b_mn_major) {
            for (int b = 0; b < K / 64; ++b)
                tma_load_3d(sB + b * N * 128, &tm_b, &bars->tma, b * 64, 0, 0);
        } else {
            for (int b = 0; b < N / 64; ++b)
                tma_load_3d(sB + b * K * 128, &tm_b, &bars->tma, b * 64, 0, 0);
        }
        ok = mbar_wait_drain(&bars->tma, 0, status);
        tc_fence_after_sync();
        if (ok) {
            const uint32_t idesc = idesc_bf16_f32(128, N, false, b_mn_major != 0);
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
            for (int kk = 0; kk < K / 16; ++kk) {
                const uint32_t koff = (kk / 4) * 128 * 128 + (kk % 4) * 32;
                const uint64_t da = smem_desc_sw128(a0 + koff, 16, 1024);
                uint64_t db;
                if (!b_mn_major)
                    db = smem_desc_sw128(b0 + (kk / 4) * N * 128 + (kk % 4) * 32, 16, 1024);
                else
                    db = smem_desc_sw128(b0 + kk * 16 * 128, K * 128, 1024);
                umma_bf16_ss(tmem, da, db, idesc, kk > 0 ? 1u : 0u);
            }
        }
        umma_commit(&bars->mma);
    }
    __syncwarp();
    ok = mbar_wait_drain(&bars->mma, 0, status);
    tc_fence_after_sync();
    const int row = threadIdx.x;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t r[32];
        tmem_ld32_wait(taddr + c0, r);
        if (ok)
            for (int j = 0; j < 32; ++j)
                c[row * N + c0 + j] = __uint_as_float(r[j]);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0)
        tmem_dealloc(tmem, 128);
}

// Same GEMM with A taken from tensor memory: thread r writes row r of A into
// TMEM columns [128, 128 + K/2), two bf16 per 32-bit column (element 2c in
// the low half), then the MMA reads A from there (tcgen05.mma with [a_tmem]).
__global__ void __launch_bounds__(kThreads, 1)
    fa_selftest_umma_ts_kernel(const __grid_constant__ CUtensorMap tm_b, const uint32_t *a_pairs,
                               float *c, int N, int K, int b_mn_major, unsigned int *status)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *sB = smem;
    UmmaBars *bars = reinterpret_cast<UmmaBars *>(smem + N * K * 2);
    const int warp = threadIdx.x / 32;
    const int row = threadIdx.x;
    constexpr uint32_t kColA = 128;

    if (threadIdx.x == 0) {
        mbar_init(&bars->tma, 1);
        mbar_init(&bars->mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem_base, 256);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

    for (int c0 = 0; c0 < K / 2; c0 += 32) {
        uint32_t r[32];
        for (int j = 0; j < 32; ++j)
            r[j] = a_pairs[row * (K / 2) + c0 + j];
        tmem_st32(tmem + lane_base + kColA + c0, r);
    }
    tmem_st_wait();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    bool ok = true;
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bars->tma, static_cast<uint32_t>(N * K * 2));
        if (!b_mn_major) {
            for (int b = 0; b < K / 64; ++b)
                tma_load_3d(sB + b * N * 128, &tm_b, &bars->tma, b * 64, 0, 0);
        } else {
            for (int b = 0; b < N / 64; ++b)
                tma_load_3d(sB + b * K * 128, &tm_b, &bars->tma, b * 64, 0, 0);
        }
        ok = mbar_wait_drain(&bars->tma, 0, status);
        tc_fence_after_sync();
        if (ok) {
            const uint32_t idesc = idesc_bf16_f32(128, N, false, b_mn_major != 0);
            const uint32_t b0 = smem_u32(sB);
            for (int kk = 0; kk < K / 16; ++kk) {
                uint64_t db;
                if (!b_mn_major)
                    db = smem_desc_sw128(b0 + (kk / 4) * N * 128 + (kk % 4) * 32, 16, 1024);
                else
                    db = smem_desc_sw128(b0 + kk * 16 * 128, K * 128, 1024);
                umma_bf16_ts(tmem, tmem + kColA + kk * 8, db, idesc, kk > 0 ? 1u : 0u);
            }
        }
        umma_commit(&bars->mma);
    }
    __syncwarp();
    ok = mbar_wait_drain(&bars->mma, 0, status);
    tc_fence_after_sync();
    for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t r[32];
        tmem_ld32_wait(tmem + lane_base + c0, r);
        if (ok)
            for (int j = 0; j < 32; ++j)
                c[row * N + c0 + j] = __uint_as_float(r[j]);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0)
        tmem_dealloc(tmem, 256);
}

// The FP8 products of the E4M3 forward: C[128, N] = A[128, 128] . B with
// .kind::f8f6f4. B is E4M3 bytes, K-major (N rows of 128) or MN-major (128
// rows of N = 128), loaded by TMA as the attention kernel loads K and V. A is
// either E4M3 bytes loaded the same way (a_tmem = 0), or fp32 values that
// thread r rounds and packs with pack_e4m3x4 into TMEM columns [128, 160),
// four per column (a_tmem = 1), the form P takes in the attention kernel.
__global__ void __launch_bounds__(kThreads, 1)
    fa_selftest_umma_f8_kernel(const __grid_constant__ CUtensorMap tm_a,
                               const __grid_constant__ CUtensorMap tm_b, const float *a_f32,
                               float *c, int N, int b_mn_major, int a_tmem, unsigned int *status)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *sA = smem;
    uint8_t *sB = smem + 128 * 128;
    UmmaBars *bars = reinterpret_cast<UmmaBars *>(smem + 2 * 128 * 128);
    const int warp = threadIdx.x / 32;
    const int row = threadIdx.x;
    constexpr uint32_t kColA = 128;

    if (threadIdx.x == 0) {
        mbar_init(&bars->tma, 1);
        mbar_init(&bars->mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem_base, 256);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    if (a_tmem) {
        uint32_t r[32];
        for (int w = 0; w < 32; ++w) {
            const float *x = a_f32 + row * 128 + 4 * w;
            r[w] = pack_e4m3x4(x[0], x[1], x[2], x[3]);
        }
        tmem_st32(tmem + lane_base + kColA, r);
        tmem_st_wait();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    bool ok = true;
    if (threadIdx.x == 0) {
        const uint32_t b_bytes = b_mn_major ? 128u * 128u : static_cast<uint32_t>(N) * 128u;
        mbar_arrive_expect_tx(&bars->tma, b_bytes + (a_tmem ? 0u : 128u * 128u));
        if (!a_tmem)
            tma_load_3d(sA, &tm_a, &bars->tma, 0, 0, 0);
        tma_load_3d(sB, &tm_b, &bars->tma, 0, 0, 0);
        ok = mbar_wait_drain(&bars->tma, 0, status);
        tc_fence_after_sync();
        if (ok) {
            const uint32_t idesc = idesc_e4m3_f32(128, N, false, b_mn_major != 0);
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t db = b_mn_major ? smem_desc_sw128(b0 + kk * 32 * 128, 128 * 128, 1024)
                                               : smem_desc_sw128(b0 + kk * 32, 16, 1024);
                if (a_tmem)
                    umma_f8_ts(tmem, tmem + kColA + kk * 8, db, idesc, kk > 0 ? 1u : 0u);
                else
                    umma_f8_ss(tmem, smem_desc_sw128(a0 + kk * 32, 16, 1024), db, idesc,
                               kk > 0 ? 1u : 0u);
            }
        }
        umma_commit(&bars->mma);
    }
    __syncwarp();
    ok = mbar_wait_drain(&bars->mma, 0, status);
    tc_fence_after_sync();
    for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t r[32];
        tmem_ld32_wait(tmem + lane_base + c0, r);
        if (ok)
            for (int j = 0; j < 32; ++j)
                c[row * N + c0 + j] = __uint_as_float(r[j]);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0)
        tmem_dealloc(tmem, 256);
}

// Throughput of the exp2 unit (MUFU) that the softmax uses: every thread runs
// 8 independent chains of x <- ex2.approx(x) * c1 + c2 (the FMA keeps x in
// range and costs a quarter of the FMA pipe's rate), so the kernel is bound by
// ex2 issue. Each thread does iters * 8 ex2; the results are stored so that
// nothing is removed by the compiler.
__global__ void __launch_bounds__(256) fa_selftest_mufu_kernel(float *out, int iters)
{
    float x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        x[k] = -0.5f - 0.01f * static_cast<float>(k + (threadIdx.x & 7));
    for (int n = 0; n < iters; ++n) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            x[k] = fmaf(ex2_approx(x[k]), -0.5f, -0.25f);
    }
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        s += x[k];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// Cycles the tensor core takes per 128 x 128 x 128 bf16 product (8
// instructions of K = 16) in operand form `mode`:
//   0: A and B from shared memory, N = 128;   1: the same as two N = 64 halves;
//   2: A from tensor memory, N = 128;         3: the same as two N = 64 halves;
//   4: A and B from shared memory, N = 256 (two products per 8 instructions).
// A half is 8 back-to-back MMAs into one accumulator, as a kernel that splits
// its score tile into column halves issues them.
// One thread per CTA issues `iters` rounds back to back and records the
// clock64 difference from before the first issue to the completion of the
// last (one commit). Operand values are a constant bf16 pattern; the
// accumulator is overwritten at each round's first K step.
__global__ void __launch_bounds__(128, 1)
    fa_selftest_mma_rate_kernel(int mode, int iters, long long *cycles, unsigned int *status)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    constexpr int kOffA = 0, kOffB = 32768, kOffBar = 32768 + 65536;  // A 128 x 128, B 256 x 128
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *tmem_base = reinterpret_cast<uint32_t *>(smem + kOffBar + 64);
    for (int i = threadIdx.x; i < kOffBar / 4; i += blockDim.x)
        reinterpret_cast<uint32_t *>(smem)[i] = 0x3C003C00u;  // bf16 2^-7 pairs
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_base;
    if (threadIdx.x == 0) {
        const uint64_t a0 = smem_desc_sw128(smem_u32(smem + kOffA), 16, 1024);
        const uint64_t b0 = smem_desc_sw128(smem_u32(smem + kOffB), 16, 1024);
        constexpr uint32_t i128 = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t i64 = idesc_bf16_f32(128, 64, false, false);
        constexpr uint32_t i256 = idesc_bf16_f32(128, 256, false, false);
        // K-major boxes of 64 columns: 16 KB per box for 128 rows, 32 KB for 256
        auto koff = [](int kk, int box) -> uint64_t {
            return static_cast<uint64_t>(((kk / 4) * box + (kk % 4) * 32) >> 4);
        };
        // columns 0-63 of tensor memory hold the A operand of the TS forms
        for (int kk = 0; kk < 8; ++kk)
            umma_bf16_ss(tmem, a0 + koff(kk, 16384), b0 + koff(kk, 16384), i128, kk > 0);
        umma_commit(bar);
        bool ok = mbar_wait_drain(bar, 0, status);
        tc_fence_after_sync();
        // One loop per form, so that nothing but the MMAs sits in the issue loop.
        const long long t0 = clock64();
        if (ok && mode == 0) {
            for (int it = 0; it < iters; ++it)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_bf16_ss(tmem + 256, a0 + koff(kk, 16384), b0 + koff(kk, 16384), i128,
                                 kk > 0);
        } else if (ok && mode == 1) {
            for (int it = 0; it < iters; ++it)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_bf16_ss(tmem + 256 + 64 * h, a0 + koff(kk, 16384),
                                     b0 + koff(kk, 16384) + ((8192 * h) >> 4), i64, kk > 0);
        } else if (ok && mode == 2) {
            for (int it = 0; it < iters; ++it)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_bf16_ts(tmem + 256, tmem + kk * 8, b0 + koff(kk, 16384), i128, kk > 0);
        } else if (ok && mode == 3) {
            for (int it = 0; it < iters; ++it)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_bf16_ts(tmem + 256 + 64 * h, tmem + kk * 8,
                                     b0 + koff(kk, 16384) + ((8192 * h) >> 4), i64, kk > 0);
        } else if (ok && mode == 4) {
            for (int it = 0; it < iters; ++it)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_bf16_ss(tmem + 256, a0 + koff(kk, 16384), b0 + koff(kk, 32768), i256,
                                 kk > 0);
        } else if (ok && mode == 5) {
            // E4M3 A and B from shared memory: a 128-byte row holds all 128 K
            // elements, and a K = 32 step moves 32 bytes along it.
            constexpr uint32_t if8 = idesc_e4m3_f32(128, 128, false, false);
            for (int it = 0; it < iters; ++it)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_f8_ss(tmem + 256, a0 + 2 * kk, b0 + 2 * kk, if8, kk > 0);
        } else if (ok) {
            // E4M3 A from tensor memory (four per column: 8 columns per K = 32)
            constexpr uint32_t if8 = idesc_e4m3_f32(128, 128, false, false);
            for (int it = 0; it < iters; ++it)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_f8_ts(tmem + 256, tmem + kk * 8, b0 + 2 * kk, if8, kk > 0);
        }
        umma_commit(bar);
        ok = ok && mbar_wait_drain(bar, 1, status);
        cycles[blockIdx.x] = ok ? clock64() - t0 : -1;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (threadIdx.x < 32)
        tmem_dealloc(tmem, 512);
}

// One index check, passing or failing as asked (the debug build records a
// failure in the status word; a release build compiles the check away).
__global__ void fa_selftest_index_check_kernel(int fail, unsigned int *status)
{
    if (threadIdx.x == 0)
        fa_check(fail == 0, status);
}

// The lane elect.sync picks in a converged warp, `trials` times per warp (4
// warps), into lanes[warp * trials + i]. Before each election the lanes run
// loops of lane-dependent length and reconverge, so that the election does
// not follow a uniform history. The MMA issue loops rely on every election
// of the warp picking the same lane: a commit tracks only the MMAs its own
// thread issued.
__global__ void fa_selftest_elect_kernel(int *lanes, int trials)
{
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    volatile int sink = 0;
    for (int i = 0; i < trials; ++i) {
        for (int k = 0; k < ((lane * 7 + i) % 5); ++k)
            sink = sink + k;
        __syncwarp();
        uint32_t elected;
        asm volatile(
            "{\n\t.reg .pred e;\n\t"
            "elect.sync %0|e, 0xffffffff;\n\t}"
            : "=r"(elected));
        if (lane == 0)
            lanes[warp * trials + i] = static_cast<int>(elected);
    }
}

__global__ void fa_selftest_wait_kernel(uint64_t limit_ns, unsigned int *status)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait(&bar, 0, &abort_flag, status, limit_ns);  // nothing arrives
    __syncthreads();
}

}  // namespace selftest

fa_status_t launch_selftest_umma(const void *a, const void *b, float *c, int n, int k,
                                 int b_mn_major, cudaStream_t stream, unsigned int *status)
{
    CUtensorMap ta, tb;
    if (!encode_tmap_bf16_3d(&ta, a, k, 128, 1, 128))
        return FA_ERR_CUDA;
    const bool ok_b = b_mn_major ? encode_tmap_bf16_3d(&tb, b, n, k, 1, k)
                                 : encode_tmap_bf16_3d(&tb, b, k, n, 1, n);
    if (!ok_b)
        return FA_ERR_CUDA;
    const int smem = 128 * k * 2 + n * k * 2 + 64 + 1024;
    if (cudaFuncSetAttribute(selftest::fa_selftest_umma_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return FA_ERR_CUDA;
    selftest::fa_selftest_umma_kernel<<<1, selftest::kThreads, smem, stream>>>(ta, tb, c, n, k,
                                                                               b_mn_major, status);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t launch_selftest_umma_ts(const void *a, const void *b, float *c, int n, int k,
                                    int b_mn_major, cudaStream_t stream, unsigned int *status)
{
    CUtensorMap tb;
    const bool ok_b = b_mn_major ? encode_tmap_bf16_3d(&tb, b, n, k, 1, k)
                                 : encode_tmap_bf16_3d(&tb, b, k, n, 1, n);
    if (!ok_b)
        return FA_ERR_CUDA;
    const int smem = n * k * 2 + 64 + 1024;
    if (cudaFuncSetAttribute(selftest::fa_selftest_umma_ts_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return FA_ERR_CUDA;
    selftest::fa_selftest_umma_ts_kernel<<<1, selftest::kThreads, smem, stream>>>(
        tb, static_cast<const uint32_t *>(a), c, n, k, b_mn_major, status);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t launch_selftest_umma_f8(const void *a, const void *b, float *c, int n, int b_mn_major,
                                    int a_tmem, cudaStream_t stream, unsigned int *status)
{
    CUtensorMap ta, tb;
    const bool ok_b = b_mn_major ? encode_tmap_u8_3d(&tb, b, 128, 128, 1, 128)
                                 : encode_tmap_u8_3d(&tb, b, 128, n, 1, n);
    if (!ok_b)
        return FA_ERR_CUDA;
    // In the TMEM form `a` holds fp32 values and no A map is read; B's map
    // fills the parameter.
    if (a_tmem)
        ta = tb;
    else if (!encode_tmap_u8_3d(&ta, a, 128, 128, 1, 128))
        return FA_ERR_CUDA;
    const int smem = 2 * 128 * 128 + 64 + 1024;
    if (cudaFuncSetAttribute(selftest::fa_selftest_umma_f8_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return FA_ERR_CUDA;
    selftest::fa_selftest_umma_f8_kernel<<<1, selftest::kThreads, smem, stream>>>(
        ta, tb, static_cast<const float *>(a), c, n, b_mn_major, a_tmem, status);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t launch_selftest_mufu(float *out, int blocks, int iters, cudaStream_t stream)
{
    selftest::fa_selftest_mufu_kernel<<<blocks, 256, 0, stream>>>(out, iters);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t launch_selftest_mma_rate(long long *cycles, int mode, int blocks, int iters,
                                     cudaStream_t stream, unsigned int *status)
{
    const int smem = 32768 + 65536 + 128 + 1024;
    if (cudaFuncSetAttribute(selftest::fa_selftest_mma_rate_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return FA_ERR_CUDA;
    selftest::fa_selftest_mma_rate_kernel<<<blocks, 128, smem, stream>>>(mode, iters, cycles,
                                                                        status);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t launch_selftest_index_check(bool fail, cudaStream_t stream, unsigned int *status)
{
    selftest::fa_selftest_index_check_kernel<<<1, 32, 0, stream>>>(fail ? 1 : 0, status);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t launch_selftest_elect(int *lanes, int trials, cudaStream_t stream)
{
    selftest::fa_selftest_elect_kernel<<<1, 128, 0, stream>>>(lanes, trials);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t launch_selftest_wait(uint64_t timeout_ns, cudaStream_t stream, unsigned int *status)
{
    selftest::fa_selftest_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
