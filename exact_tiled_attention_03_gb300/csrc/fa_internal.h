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
};

// Row-major [depth, rows, inner] bf16 tensor as a 3-D TMA map with a
// (64 x box_rows x 1) box and 128-byte swizzle. Returns false on failure.
bool encode_tmap_bf16_3d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                         uint64_t depth, uint32_t box_rows);

// Launchers. Each validates nothing (fa_abi.cu does) and returns FA_OK or
// FA_ERR_CUDA.
fa_status_t launch_prefill_sm103(const Problem &p);
fa_status_t launch_verify(const Problem &p, int n_split, void *workspace, size_t ws_bytes);
fa_status_t launch_reference_simt(const Problem &p);
fa_status_t launch_selftest_umma(const void *a, const void *b, float *c, int n, int k,
                                 int b_mn_major, cudaStream_t stream, unsigned int *status);
fa_status_t launch_selftest_umma_ts(const void *a, const void *b, float *c, int n, int k,
                                    int b_mn_major, cudaStream_t stream, unsigned int *status);
fa_status_t launch_selftest_wait(uint64_t timeout_ns, cudaStream_t stream, unsigned int *status);

// Split-KV geometry shared by the ABI (workspace sizing) and the launcher.
constexpr int kVerifyStageKeys = 64;
int verify_auto_splits(int64_t BH, int64_t Sk, int num_sms);
int64_t verify_chunk_keys(int64_t Sk, int n_split);
size_t verify_workspace_bytes(int64_t BH, int64_t Sq, int64_t d, int n_split);

}  // namespace fa
