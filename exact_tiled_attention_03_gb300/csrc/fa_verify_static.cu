// fa_verify_static.cu — the split-KV (decode-shaped) path with library-owned
// scratch, for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: plugins loaded into a
// host runtime that owns all device memory and hands its plugins only their
// input and output buffers; serving loops that reserved nearly all of HBM for
// a KV-cache pool at start-up, where a late allocation can fail; and
// latency-critical loops that cannot accept the device-wide synchronisation
// an allocation may cause. fa_verify_forward_static serves them: its
// split-KV partials live in the file-scope device array below, so the call
// allocates nothing. The caller still passes Q, K, V, O and LSE.
//
// Properties callers must know:
//   * the array is FA_STATIC_SCRATCH_BYTES bytes on every GPU that loads the
//     library, held until the process exits;
//   * the first call on a device looks up the array's device address (with
//     that device current) and caches it; make that first call before any
//     stream capture;
//   * every call shares the one array, which keeps the last call's
//     contents, so calls that overlap on the GPU (other streams, other host
//     threads) race on it; nothing in it needs to start at zero, because the
//     split kernel of a call writes every partial its combine reads;
//   * shapes whose partials do not fit return FA_ERR_WORKSPACE.
#include <mutex>

#include "fa_internal.h"

// Split-KV partials of fa_verify_forward_static (host code must not use this
// name as an address: it is a host-side stand-in for the device array).
static __device__ __align__(256) unsigned char g_verify_scratch[FA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_verify_scratch on the current device, looked up once
// per device with that device current. nullptr on failure.
void *scratch_address()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr)
            return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" fa_status_t fa_verify_forward_static(const void *q, const void *k, const void *v,
                                                void *o, float *lse, int64_t B, int64_t H,
                                                int64_t Sq, int64_t Sk, int64_t d, int causal,
                                                float scale, int n_split, void *stream)
{
    if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || d <= 0 || n_split < 0)
        return FA_ERR_INVALID_ARG;
    // An explicit split count is checked against the limit before touching
    // the device; the automatic one needs the device's SM count.
    if (n_split > 0 &&
        fa::verify_workspace_bytes(B * H, Sq, d, n_split) > size_t(FA_STATIC_SCRATCH_BYTES))
        return FA_ERR_WORKSPACE;
    const int ns = n_split > 0 ? n_split : fa_verify_auto_splits(B, H, Sq, Sk, d);
    if (ns <= 0)
        return FA_ERR_CUDA;
    if (fa::verify_workspace_bytes(B * H, Sq, d, ns) > size_t(FA_STATIC_SCRATCH_BYTES))
        return FA_ERR_WORKSPACE;
    void *scratch = scratch_address();
    if (!scratch)
        return FA_ERR_CUDA;
    return fa_verify_forward(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, ns, scratch,
                             size_t(FA_STATIC_SCRATCH_BYTES), stream);
}
