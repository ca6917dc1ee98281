// fa_simt.cu — plain CUDA-core (fp32) attention forward, a test tool.
//
// The online softmax of "Warmup Guide — Inference Optimization at Depth",
// Chapter 3, one key at a time: one thread per query row keeps the running
// max m, the running sum l and the unnormalised output row, rescales both by
// exp(m_old - m_new) when the max moves, and divides by l once at the end
// (Chapter 4). Keys are read straight from global memory. It is slow and
// exists only as a second GPU implementation for the test suite; fa_forward
// never dispatches to it.
#include <cuda_bf16.h>

#include <cmath>

#include "fa_internal.h"

namespace fa {
namespace simt {

constexpr int kMaxD = 128;
constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads)
    fa_reference_simt_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                             const __nv_bfloat16 *__restrict__ v, __nv_bfloat16 *__restrict__ o,
                             float *__restrict__ lse, int BH, int Sq, int Sk, int d, int causal,
                             float scale)
{
    const int bh = blockIdx.y;
    const int i = blockIdx.x * kThreads + threadIdx.x;
    if (bh >= BH || i >= Sq)
        return;
    const __nv_bfloat16 *qi = q + (static_cast<size_t>(bh) * Sq + i) * d;
    const __nv_bfloat16 *kb = k + static_cast<size_t>(bh) * Sk * d;
    const __nv_bfloat16 *vb = v + static_cast<size_t>(bh) * Sk * d;
    float qr[kMaxD], acc[kMaxD];
    for (int t = 0; t < d; ++t) {
        qr[t] = __bfloat162float(qi[t]);
        acc[t] = 0.0f;
    }
    int nv = Sk;
    if (causal) {
        nv = i + (Sk - Sq) + 1;
        nv = nv < 0 ? 0 : (nv > Sk ? Sk : nv);
    }
    float m = -INFINITY, l = 0.0f;
    for (int j = 0; j < nv; ++j) {
        const __nv_bfloat16 *kj = kb + static_cast<size_t>(j) * d;
        float dot = 0.0f;
        for (int t = 0; t < d; ++t)
            dot = fmaf(qr[t], __bfloat162float(kj[t]), dot);
        const float s = dot * scale;
        const float m_new = fmaxf(m, s);
        const float corr = expf(m - m_new);
        const float pj = expf(s - m_new);
        l = l * corr + pj;
        const __nv_bfloat16 *vj = vb + static_cast<size_t>(j) * d;
        for (int t = 0; t < d; ++t)
            acc[t] = fmaf(acc[t], corr, pj * __bfloat162float(vj[t]));
        m = m_new;
    }
    __nv_bfloat16 *oi = o + (static_cast<size_t>(bh) * Sq + i) * d;
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    for (int t = 0; t < d; ++t)
        oi[t] = __float2bfloat16_rn(acc[t] * inv);
    lse[static_cast<size_t>(bh) * Sq + i] = l > 0.0f ? m + logf(l) : -INFINITY;
}

}  // namespace simt

fa_status_t launch_reference_simt(const Problem &p)
{
    if (p.d > simt::kMaxD)
        return FA_ERR_UNSUPPORTED;
    const int64_t BH = p.B * p.H;
    if (BH > 65535)
        return FA_ERR_UNSUPPORTED;
    dim3 grid(static_cast<unsigned>((p.Sq + simt::kThreads - 1) / simt::kThreads),
              static_cast<unsigned>(BH));
    simt::fa_reference_simt_kernel<<<grid, simt::kThreads, 0, p.stream>>>(
        static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k),
        static_cast<const __nv_bfloat16 *>(p.v), static_cast<__nv_bfloat16 *>(p.o), p.lse,
        static_cast<int>(BH), static_cast<int>(p.Sq), static_cast<int>(p.Sk),
        static_cast<int>(p.d), p.causal, p.scale);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
