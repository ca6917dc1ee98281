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
//     that device current) and caches it for the calling thread's CUDA
//     context; make that first call before any stream capture. A call made
//     in another context (after cudaDeviceReset, or under a driver context
//     the caller created) looks the address up again;
//   * every call shares the one array, which keeps the last call's
//     contents, so calls that overlap on the GPU (other streams, other host
//     threads) race on it; nothing in it needs to start at zero, because the
//     split kernel of a call writes every partial its combine reads;
//   * arguments are checked exactly as fa_verify_forward checks them, before
//     the scratch size; with n_split = 0 the automatic split count is
//     lowered, if need be, to the largest count whose partials fit (one split
//     needs no scratch at all); an explicit n_split whose partials do not fit
//     returns FA_ERR_WORKSPACE.
#include <mutex>

#include "fa_internal.h"

// Split-KV partials of fa_verify_forward_static (host code must not use this
// name as an address: it is a host-side stand-in for the device array).
static __device__ __align__(256) unsigned char g_verify_scratch[FA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
    void *ctx = nullptr;   // context the address was looked up in
    void *addr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];

// Device address of g_verify_scratch on the current device, looked up with
// that device current and cached per device for the context it belongs to.
// nullptr on failure.
void *scratch_address()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    void *ctx = fa::current_context();
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr &c = g_scratch[dev];
    if (!c.addr || ctx != c.ctx) {
        void *p = nullptr;
        c.addr = nullptr;
        if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr)
            return nullptr;
        c.addr = p;
        c.ctx = fa::current_context();  // bound by the lookup if it was not already
    }
    return c.addr;
}

bool fits(int64_t BH, int64_t Sq, int64_t d, int ns)
{
    return fa::verify_workspace_bytes(BH, Sq, d, ns) <= size_t(FA_STATIC_SCRATCH_BYTES);
}

}  // namespace

extern "C" fa_status_t fa_verify_forward_static(const void *q, const void *k, const void *v,
                                                void *o, float *lse, int64_t B, int64_t H,
                                                int64_t Sq, int64_t Sk, int64_t d, int causal,
                                                float scale, int n_split, void *stream)
{
    fa_status_t st = fa::verify_check_args(q, k, v, o, lse, B, H, Sq, Sk, d, scale, n_split);
    if (st != FA_OK)
        return st;
    int ns = n_split;
    if (ns > 0) {
        if (!fits(B * H, Sq, d, ns))
            return FA_ERR_WORKSPACE;
    } else {
        ns = fa_verify_auto_splits(B, H, Sq, Sk, d);
        if (ns <= 0)
            return FA_ERR_CUDA;
        while (ns > 1 && !fits(B * H, Sq, d, ns))
            --ns;
    }
    void *scratch = scratch_address();
    if (!scratch)
        return FA_ERR_CUDA;
    return fa_verify_forward(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, ns, scratch,
                             size_t(FA_STATIC_SCRATCH_BYTES), stream);
}
