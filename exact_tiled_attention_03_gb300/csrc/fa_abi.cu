// fa_abi.cu — the C ABI declared in include/fa.h and include/fa_testing.h:
// argument validation, shape dispatch (prefill vs split-KV), TMA descriptor
// encoding, the device status word, and the library's stream-ordered
// workspace pool. No compute happens here.
#include <cmath>
#include <cstring>
#include <mutex>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_testing.h"

// Library-owned status word (one per device): kernels OR in a bit when a
// bounded wait gives up; fa_device_status() reads and clears it.
__device__ unsigned int g_fa_status_word;

// Work counters of the persistent prefill kernel (see fa_prefill_sm103.cu):
// launches take slots in turn; each launch's last CTA puts its slot back to 0.
__device__ unsigned long long g_fa_work_slots[2 * fa::kWorkSlots];

namespace fa {

void *current_context()
{
    using CtxGetCurrentFn = CUresult (*)(CUcontext *);
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS)
        return nullptr;
    return ctx;
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    void *ctx = nullptr;  // the CUDA context the addresses below belong to
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    unsigned int *status = nullptr;
    unsigned long long *work = nullptr;
    cudaMemPool_t pool = nullptr;  // library pool for small workspaces (created on first use)
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Per-device facts and the device addresses of the status word and the work
// counters, looked up with the device current and kept while the calling
// thread's CUDA context stays the one they were looked up in (a device reset
// or a caller-made driver context triggers a fresh lookup).
const DeviceInfo *device_info()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    void *ctx = current_context();
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &di = g_dev[dev];
    if (!di.ready || ctx != di.ctx) {
        di.ready = false;
        if (cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return nullptr;
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_fa_status_word) != cudaSuccess)
            return nullptr;
        di.status = static_cast<unsigned int *>(addr);
        if (cudaGetSymbolAddress(&addr, g_fa_work_slots) != cudaSuccess)
            return nullptr;
        di.work = static_cast<unsigned long long *>(addr);
        di.ctx = current_context();  // the runtime has bound its context by now
        di.pool = nullptr;
        di.ready = true;
    }
    return &di;
}

// The library's stream-ordered memory pool on the current device, for the
// small workspaces fa_forward (split-KV partials) and fa_backward (per-row
// vectors) take when the caller passes none. Freed blocks stay in the pool
// (release threshold: never), so the next call's allocation is a
// suballocation, not a request to the driver at every synchronisation as
// with the device's default pool. nullptr on failure.
cudaMemPool_t library_pool(const DeviceInfo *cdi)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &di = g_dev[dev];
    if (&di != cdi || !di.ready)
        return nullptr;
    if (!di.pool) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess)
            return nullptr;
        uint64_t keep = UINT64_MAX;
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return nullptr;
        }
        di.pool = pool;
    }
    return di.pool;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape and argument checks shared by every attention entry point.
fa_status_t validate(const void *q, const void *k, const void *v, const void *o, const float *lse,
                     int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, float scale,
                     bool any_d)
{
    if (!q || !k || !v || !o || !lse)
        return FA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || d <= 0)
        return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale))
        return FA_ERR_INVALID_ARG;
    if (any_d ? (d > 128) : (d != 64 && d != 128))
        return FA_ERR_UNSUPPORTED;
    const int64_t lim31 = (int64_t(1) << 31) - 1;
    if (Sq > lim31 || Sk > lim31 || B > lim31 / H)
        return FA_ERR_UNSUPPORTED;
    const int64_t BH = B * H;
    const int64_t lim62 = int64_t(1) << 62;
    if (Sq > lim62 / (BH * d) || Sk > lim62 / (BH * d))
        return FA_ERR_UNSUPPORTED;
    if (!any_d && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)))
        return FA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
        return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

// The kernels are built for sm_103a only.
fa_status_t device_ok(const DeviceInfo **out)
{
    const DeviceInfo *di = device_info();
    if (!di)
        return FA_ERR_CUDA;
    if (di->cc_major != 10 || di->cc_minor != 3)
        return FA_ERR_UNSUPPORTED;
    *out = di;
    return FA_OK;
}

Problem make_problem(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                     int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal, float scale,
                     void *stream, unsigned int *status)
{
    Problem p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.Sq = Sq;
    p.Sk = Sk;
    p.d = d;
    p.causal = causal ? 1 : 0;
    p.scale = scale;
    p.stream = static_cast<cudaStream_t>(stream);
    p.status = status;
    const DeviceInfo *di = device_info();  // already looked up by the caller's device_ok()
    p.num_sms = di ? di->num_sms : 0;
    p.work_slots = di ? di->work : nullptr;
    return p;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Copy and compute streams (and events) fa_forward_host uses on a device,
// created on first use with the device current.
struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in[FA_HOST_CHUNKS] = {}, out[FA_HOST_CHUNKS] = {};
    std::mutex mu;  // one call enqueues at a time on these streams and events
};
HostPipe g_pipe[kMaxDevices];

HostPipe *host_pipe()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    HostPipe &hp = g_pipe[dev];
    std::lock_guard<std::mutex> lock(g_mu);
    if (!hp.ready) {
        const unsigned fl = cudaStreamNonBlocking;
        if (cudaStreamCreateWithFlags(&hp.h2d, fl) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.comp, fl) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.d2h, fl) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming) != cudaSuccess)
            return nullptr;
        for (int c = 0; c < FA_HOST_CHUNKS; ++c)
            if (cudaEventCreateWithFlags(&hp.in[c], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.out[c], cudaEventDisableTiming) != cudaSuccess)
                return nullptr;
        hp.ready = true;
    }
    return &hp;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// fa_forward_host's device-to-host copy of a group's O, made by a few CTAs
// that store straight into the caller's pinned buffer instead of by a copy
// engine. The copy engine moves each group's O in a burst at about 190 GB/s,
// and while it runs the host-to-device copies, which bound the call, slow
// down on the shared link; kHostWriteCtas CTAs return O at about the kernels'
// pace. Measured on the B4 H32 S8192 d128 causal problem (16 groups): 4.39 ms
// per call against 4.53 ms with the copy engine (4 or 8 CTAs fall behind and
// take longer; 16 to 64 measured the same).
constexpr int kHostWriteCtas = 16;

__global__ void __launch_bounds__(256) fa_host_write_kernel(const uint4 *__restrict__ src,
                                                            uint4 *__restrict__ dst, size_t n16)
{
    for (size_t i = static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x; i < n16;
         i += static_cast<size_t>(gridDim.x) * 256)
        dst[i] = src[i];
}

// True when the device can store to [p, p + bytes) through the same address:
// pinned host memory, mapped into the device's address space, at both ends of
// the range.
bool host_range_device_writable(void *p, size_t bytes)
{
    for (void *e : {p, static_cast<void *>(static_cast<uint8_t *>(p) + bytes - 1)}) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, e) != cudaSuccess) {
            cudaGetLastError();  // an unregistered pointer on older runtimes: not an error here
            return false;
        }
        if (a.type != cudaMemoryTypeHost || a.devicePointer != e)
            return false;
    }
    return true;
}

// Byte offsets of the staging buffers in fa_forward_host's workspace.
struct HostLayout {
    size_t q, k, v, o, lse, partials, total;
    int n_chunks, ns;  // groups, split count for a group (verify path)
};

HostLayout host_layout(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, int num_sms)
{
    HostLayout L;
    const int64_t BH = B * H;
    L.n_chunks = static_cast<int>(BH < FA_HOST_CHUNKS ? BH : FA_HOST_CHUNKS);
    const size_t qb = static_cast<size_t>(BH) * Sq * d * 2, kb = static_cast<size_t>(BH) * Sk * d * 2;
    L.q = 0;
    L.k = align256(L.q + qb);
    L.v = align256(L.k + kb);
    L.o = align256(L.v + kb);
    L.lse = align256(L.o + qb);
    L.partials = align256(L.lse + static_cast<size_t>(BH) * Sq * 4);
    L.ns = 0;
    size_t part = 0;
    if (Sq <= FA_VERIFY_MAX_SQ) {
        const int64_t group = (BH + L.n_chunks - 1) / L.n_chunks;
        L.ns = verify_auto_splits(group, Sk, num_sms);
        part = verify_workspace_bytes(group, Sq, d, L.ns);
    }
    L.total = L.partials + part;
    return L;
}

int verify_splits_or_auto(int n_split, int64_t BH, int64_t Sk, const DeviceInfo *di)
{
    return n_split > 0 ? n_split : verify_auto_splits(BH, Sk, di->num_sms);
}

}  // namespace

namespace {
struct StallRequest {
    int kernel = 0;  // 0: none pending
    int skip = -1;
    uint64_t wait_ns = 0;
};
std::mutex g_stall_mu;
StallRequest g_stall;
}  // namespace

void take_stall(int kernel, int *skip_index, uint64_t *wait_ns)
{
    std::lock_guard<std::mutex> lock(g_stall_mu);
    if (g_stall.kernel != kernel)
        return;
    *skip_index = g_stall.skip;
    *wait_ns = g_stall.wait_ns;
    g_stall = StallRequest();
}

fa_status_t verify_check_args(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                              int64_t d, float scale, int n_split)
{
    fa_status_t st = validate(q, k, v, o, lse, B, H, Sq, Sk, d, scale, false);
    if (st != FA_OK)
        return st;
    if (Sq > FA_VERIFY_MAX_SQ || B * H > 65535)
        return FA_ERR_UNSUPPORTED;
    const int64_t max_split = (Sk + kVerifyStageKeys - 1) / kVerifyStageKeys;
    if (n_split < 0 || n_split > max_split || n_split > 65535)
        return FA_ERR_INVALID_ARG;
    return FA_OK;
}

bool encode_tmap_bf16_3d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                         uint64_t depth, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {inner, rows, depth};
    const cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_u8_3d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                       uint64_t depth, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {inner, rows, depth};
    const cuuint64_t strides[2] = {inner, inner * rows};
    const cuuint32_t box[3] = {128, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_bf16_pages_5d(CUtensorMap *map, const void *base, uint64_t page_size, uint64_t H,
                               uint64_t num_pages)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[5] = {64, 2, page_size, H, num_pages};
    const cuuint64_t strides[4] = {128, 256, page_size * 256, H * page_size * 256};
    const cuuint32_t box[5] = {64, 2, static_cast<cuuint32_t>(page_size), 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_bf16_4d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                         uint64_t mid, uint64_t outer, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[4] = {inner, rows, mid, outer};
    const cuuint64_t strides[3] = {inner * 2, inner * rows * 2, inner * rows * mid * 2};
    const cuuint32_t box[4] = {64, box_rows, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fa

using namespace fa;

extern "C" {

const char *fa_status_string(fa_status_t s)
{
    switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported shape, alignment or device";
    case FA_ERR_CUDA: return "CUDA runtime or launch error";
    case FA_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_BOUNDS: return "a debug build's index check failed";
    }
    return "unknown status";
}

fa_status_t fa_prefill_forward(const void *q, const void *k, const void *v, void *o, float *lse,
                               int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d,
                               int causal, float scale, void *stream)
{
    fa_status_t st = validate(q, k, v, o, lse, B, H, Sq, Sk, d, scale, false);
    if (st != FA_OK)
        return st;
    const DeviceInfo *di = nullptr;
    if ((st = device_ok(&di)) != FA_OK)
        return st;
    return launch_prefill_sm103(
        make_problem(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, stream, di->status));
}

fa_status_t fa_forward_fp8(const void *q, const void *k, const void *v, void *o, float *lse,
                           int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal,
                           float scale, float q_descale, float k_descale, float v_descale,
                           void *stream)
{
    fa_status_t st = validate(q, k, v, o, lse, B, H, Sq, Sk, d, scale, false);
    if (st != FA_OK)
        return st;
    if (!std::isfinite(q_descale) || !std::isfinite(k_descale) || !std::isfinite(v_descale))
        return FA_ERR_INVALID_ARG;
    if (!(q_descale > 0.0f) || !(k_descale > 0.0f) || !(v_descale > 0.0f) || d != 128)
        return FA_ERR_UNSUPPORTED;
    const DeviceInfo *di = nullptr;
    if ((st = device_ok(&di)) != FA_OK)
        return st;
    return launch_prefill_fp8_sm103(
        make_problem(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, stream, di->status),
        q_descale, k_descale, v_descale);
}

size_t fa_verify_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d,
                                int n_split)
{
    if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || d <= 0 || n_split < 0)
        return 0;
    if (n_split == 0) {
        const DeviceInfo *di = device_info();
        if (!di)
            return 0;
        n_split = verify_auto_splits(B * H, Sk, di->num_sms);
    }
    return verify_workspace_bytes(B * H, Sq, d, n_split);
}

int fa_verify_auto_splits(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d)
{
    (void)Sq;
    (void)d;
    if (B <= 0 || H <= 0 || Sk <= 0)
        return 0;
    const DeviceInfo *di = device_info();
    if (!di)
        return 0;
    return verify_auto_splits(B * H, Sk, di->num_sms);
}

fa_status_t fa_verify_forward(const void *q, const void *k, const void *v, void *o, float *lse,
                              int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d,
                              int causal, float scale, int n_split, void *workspace,
                              size_t ws_bytes, void *stream)
{
    fa_status_t st = verify_check_args(q, k, v, o, lse, B, H, Sq, Sk, d, scale, n_split);
    if (st != FA_OK)
        return st;
    const DeviceInfo *di = nullptr;
    if ((st = device_ok(&di)) != FA_OK)
        return st;
    const int ns = verify_splits_or_auto(n_split, B * H, Sk, di);
    const size_t need = verify_workspace_bytes(B * H, Sq, d, ns);
    if (need > 0 && (!workspace || ws_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return FA_ERR_WORKSPACE;
    return launch_verify(
        make_problem(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, stream, di->status), ns,
        workspace, ws_bytes);
}

fa_status_t fa_verify_tree_forward(const void *q, const void *k, const void *v, void *o,
                                   float *lse, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                                   int64_t d, const uint32_t *tree_mask, float scale, int n_split,
                                   void *workspace, size_t ws_bytes, void *stream)
{
    if (!tree_mask || (reinterpret_cast<uintptr_t>(tree_mask) & 3u) != 0)
        return FA_ERR_INVALID_ARG;
    fa_status_t st = validate(q, k, v, o, lse, B, H, Sq, Sk, d, scale, false);
    if (st != FA_OK)
        return st;
    if (Sq > FA_VERIFY_MAX_SQ || B * H > 65535)
        return FA_ERR_UNSUPPORTED;
    const int64_t max_split = (Sk + kVerifyStageKeys - 1) / kVerifyStageKeys;
    if (n_split < 0 || n_split > max_split || n_split > 65535)
        return FA_ERR_INVALID_ARG;
    const DeviceInfo *di = nullptr;
    if ((st = device_ok(&di)) != FA_OK)
        return st;
    const int ns = verify_splits_or_auto(n_split, B * H, Sk, di);
    const size_t need = verify_workspace_bytes(B * H, Sq, d, ns);
    if (need > 0 && (!workspace || ws_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return FA_ERR_WORKSPACE;
    VerifyOptions opt;
    opt.tree_mask = tree_mask;
    return launch_verify(
        make_problem(q, k, v, o, lse, B, H, Sq, Sk, d, 1, scale, stream, di->status), ns,
        workspace, ws_bytes, opt);
}

fa_status_t fa_verify_paged_forward(const void *q, const void *k_pages, const void *v_pages,
                                    const int32_t *block_table, const int32_t *seq_lens, void *o,
                                    float *lse, int64_t B, int64_t H, int64_t Sq, int64_t d,
                                    int64_t num_pages, int64_t page_size,
                                    int64_t max_pages_per_seq, int64_t max_seq_len, int causal,
                                    const uint32_t *tree_mask, float scale, int n_split,
                                    void *workspace, size_t ws_bytes, void *stream)
{
    if (!block_table || !seq_lens)
        return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u) != 0 ||
        (tree_mask && (reinterpret_cast<uintptr_t>(tree_mask) & 3u) != 0))
        return FA_ERR_INVALID_ARG;
    if (num_pages < 1 || max_pages_per_seq < 1 || page_size < 1 || max_seq_len < 1)
        return FA_ERR_INVALID_ARG;
    const bool page_ok = page_size % 16 == 0 &&
                         (page_size < kVerifyStageKeys ? kVerifyStageKeys % page_size == 0
                                                       : page_size % kVerifyStageKeys == 0);
    if (!page_ok)
        return FA_ERR_UNSUPPORTED;
    const int64_t lim31 = (int64_t(1) << 31) - 1;
    if (num_pages > lim31 || max_pages_per_seq > lim31 / page_size ||
        max_seq_len > max_pages_per_seq * page_size)
        return FA_ERR_INVALID_ARG;
    // Validate shapes and pointers with the pool standing in for K/V.
    fa_status_t st = validate(q, k_pages, v_pages, o, lse, B, H, Sq, max_seq_len, d, scale, false);
    if (st != FA_OK)
        return st;
    if (Sq > FA_VERIFY_MAX_SQ || B * H > 65535)
        return FA_ERR_UNSUPPORTED;
    const int64_t max_split = (max_seq_len + kVerifyStageKeys - 1) / kVerifyStageKeys;
    if (n_split < 0 || n_split > max_split || n_split > 65535)
        return FA_ERR_INVALID_ARG;
    const DeviceInfo *di = nullptr;
    if ((st = device_ok(&di)) != FA_OK)
        return st;
    const int ns = verify_splits_or_auto(n_split, B * H, max_seq_len, di);
    const size_t need = verify_workspace_bytes(B * H, Sq, d, ns);
    if (need > 0 && (!workspace || ws_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return FA_ERR_WORKSPACE;
    VerifyOptions opt;
    opt.tree_mask = tree_mask;
    opt.block_table = block_table;
    opt.seq_lens = seq_lens;
    opt.page_size = page_size;
    opt.num_pages = num_pages;
    opt.max_pages = max_pages_per_seq;
    return launch_verify(make_problem(q, k_pages, v_pages, o, lse, B, H, Sq, max_seq_len, d,
                                      causal, scale, stream, di->status),
                         ns, workspace, ws_bytes, opt);
}

size_t fa_backward_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d)
{
    if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || d <= 0)
        return 0;
    return backward_workspace_bytes(B * H, Sq);
}

fa_status_t fa_backward(const void *q, const void *k, const void *v, const void *o,
                        const float *lse, const void *dout, void *dq, void *dk, void *dv,
                        int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal,
                        float scale, void *workspace, size_t ws_bytes, void *stream)
{
    if (!dout || !dq || !dk || !dv)
        return FA_ERR_INVALID_ARG;
    fa_status_t st = validate(q, k, v, o, lse, B, H, Sq, Sk, d, scale, false);
    if (st != FA_OK)
        return st;
    if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return FA_ERR_UNSUPPORTED;
    const DeviceInfo *di = nullptr;
    if ((st = device_ok(&di)) != FA_OK)
        return st;
    const size_t need = backward_workspace_bytes(B * H, Sq);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool owned = false;
    if (workspace) {
        if (ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return FA_ERR_WORKSPACE;
    } else {
        cudaMemPool_t pool = library_pool(di);
        if (!pool || cudaMallocFromPoolAsync(&workspace, need, pool, s) != cudaSuccess)
            return FA_ERR_CUDA;
        owned = true;
    }
    BackwardProblem bp;
    bp.fwd = make_problem(q, k, v, nullptr, nullptr, B, H, Sq, Sk, d, causal, scale, stream,
                          di->status);
    bp.o = o;
    bp.lse = lse;
    bp.dout = dout;
    bp.dq = dq;
    bp.dk = dk;
    bp.dv = dv;
    bp.workspace = workspace;
    st = launch_backward_sm103(bp);
    if (owned && cudaFreeAsync(workspace, s) != cudaSuccess && st == FA_OK)
        st = FA_ERR_CUDA;
    return st;
}

size_t fa_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d)
{
    if (Sq > FA_VERIFY_MAX_SQ)
        return 0;
    return fa_verify_workspace_size(B, H, Sq, Sk, d, 0);
}

fa_status_t fa_forward_ws(const void *q, const void *k, const void *v, void *o, float *lse,
                          int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal,
                          float scale, void *workspace, size_t ws_bytes, void *stream)
{
    if (Sq > 0 && Sq <= FA_VERIFY_MAX_SQ)
        return fa_verify_forward(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, 0, workspace,
                                 ws_bytes, stream);
    return fa_prefill_forward(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, stream);
}

fa_status_t fa_forward(const void *q, const void *k, const void *v, void *o, float *lse,
                       int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal,
                       float scale, void *stream)
{
    if (!(Sq > 0 && Sq <= FA_VERIFY_MAX_SQ))
        return fa_prefill_forward(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, stream);
    fa_status_t st = validate(q, k, v, o, lse, B, H, Sq, Sk, d, scale, false);
    if (st != FA_OK)
        return st;
    if (B * H > 65535)
        return FA_ERR_UNSUPPORTED;
    const DeviceInfo *di = nullptr;
    if ((st = device_ok(&di)) != FA_OK)
        return st;
    const int ns = verify_auto_splits(B * H, Sk, di->num_sms);
    const size_t need = verify_workspace_bytes(B * H, Sq, d, ns);
    void *ws = nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (need > 0) {
        cudaMemPool_t pool = library_pool(di);
        if (!pool || cudaMallocFromPoolAsync(&ws, need, pool, s) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    st = launch_verify(make_problem(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, stream,
                                    di->status),
                       ns, ws, need);
    if (ws && cudaFreeAsync(ws, s) != cudaSuccess && st == FA_OK)
        st = FA_ERR_CUDA;
    return st;
}

size_t fa_forward_host_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d)
{
    if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || d <= 0)
        return 0;
    const DeviceInfo *di = device_info();
    if (!di)
        return 0;
    return host_layout(B, H, Sq, Sk, d, di->num_sms).total;
}

fa_status_t fa_forward_host(const void *q, const void *k, const void *v, void *o, float *lse,
                            int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal,
                            float scale, void *workspace, size_t ws_bytes, void *stream)
{
    // Host pointers need no alignment for the copies; validate everything else
    // as for device pointers.
    if (!q || !k || !v || !o || !lse)
        return FA_ERR_INVALID_ARG;
    const void *aligned = reinterpret_cast<const void *>(uintptr_t(256));
    fa_status_t st = validate(aligned, aligned, aligned, aligned,
                              reinterpret_cast<const float *>(aligned), B, H, Sq, Sk, d, scale,
                              false);
    if (st != FA_OK)
        return st;
    if (Sq <= FA_VERIFY_MAX_SQ && B * H > 65535)
        return FA_ERR_UNSUPPORTED;
    const DeviceInfo *di = nullptr;
    if ((st = device_ok(&di)) != FA_OK)
        return st;
    const HostLayout L = host_layout(B, H, Sq, Sk, d, di->num_sms);
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    bool owned = false;
    if (workspace) {
        if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return FA_ERR_WORKSPACE;
    } else {
        if (cudaMallocAsync(&workspace, L.total, user) != cudaSuccess)
            return FA_ERR_CUDA;
        owned = true;
    }
    HostPipe *hp = host_pipe();
    if (!hp)
        return FA_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int64_t BH = B * H;
    const size_t q_row = static_cast<size_t>(Sq) * d * 2, k_row = static_cast<size_t>(Sk) * d * 2;
    const size_t l_row = static_cast<size_t>(Sq) * 4;
    const uint8_t *qh = static_cast<const uint8_t *>(q), *kh = static_cast<const uint8_t *>(k),
                  *vh = static_cast<const uint8_t *>(v);
    uint8_t *oh = static_cast<uint8_t *>(o), *lh = reinterpret_cast<uint8_t *>(lse);
    // O returns through CTA stores when the caller's buffer is pinned and
    // mapped (16-byte aligned rows); otherwise through cudaMemcpyAsync.
    const bool o_by_ctas = (reinterpret_cast<uintptr_t>(o) & 15u) == 0 && q_row % 16 == 0 &&
                           host_range_device_writable(o, static_cast<size_t>(BH) * q_row);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    {
        std::lock_guard<std::mutex> lock(hp->mu);
        bool good = ok(cudaEventRecord(hp->start, user)) &&
                    ok(cudaStreamWaitEvent(hp->h2d, hp->start, 0)) &&
                    ok(cudaStreamWaitEvent(hp->comp, hp->start, 0)) &&
                    ok(cudaStreamWaitEvent(hp->d2h, hp->start, 0));
        for (int c = 0; c < L.n_chunks && good; ++c) {
            const int64_t h0 = BH * c / L.n_chunks, h1 = BH * (c + 1) / L.n_chunks;
            const size_t nh = static_cast<size_t>(h1 - h0);
            // group c: host -> device
            good = ok(cudaMemcpyAsync(ws + L.q + h0 * q_row, qh + h0 * q_row, nh * q_row,
                                      cudaMemcpyHostToDevice, hp->h2d)) &&
                   ok(cudaMemcpyAsync(ws + L.k + h0 * k_row, kh + h0 * k_row, nh * k_row,
                                      cudaMemcpyHostToDevice, hp->h2d)) &&
                   ok(cudaMemcpyAsync(ws + L.v + h0 * k_row, vh + h0 * k_row, nh * k_row,
                                      cudaMemcpyHostToDevice, hp->h2d)) &&
                   ok(cudaEventRecord(hp->in[c], hp->h2d)) &&
                   ok(cudaStreamWaitEvent(hp->comp, hp->in[c], 0));
            if (!good)
                break;
            // group c: the kernels, as a problem of nh heads
            const Problem pr = make_problem(ws + L.q + h0 * q_row, ws + L.k + h0 * k_row,
                                            ws + L.v + h0 * k_row, ws + L.o + h0 * q_row,
                                            reinterpret_cast<float *>(ws + L.lse + h0 * l_row), 1,
                                            static_cast<int64_t>(nh), Sq, Sk, d, causal, scale,
                                            hp->comp, di->status);
            if (Sq <= FA_VERIFY_MAX_SQ) {
                const int ns = verify_auto_splits(static_cast<int64_t>(nh), Sk, di->num_sms);
                st = launch_verify(pr, ns, ws + L.partials, L.total - L.partials);
            } else {
                st = launch_prefill_sm103(pr);
            }
            if (st != FA_OK)
                break;
            // group c: device -> host
            good = ok(cudaEventRecord(hp->out[c], hp->comp)) &&
                   ok(cudaStreamWaitEvent(hp->d2h, hp->out[c], 0));
            if (good && o_by_ctas) {
                fa_host_write_kernel<<<kHostWriteCtas, 256, 0, hp->d2h>>>(
                    reinterpret_cast<const uint4 *>(ws + L.o + h0 * q_row),
                    reinterpret_cast<uint4 *>(oh + h0 * q_row), nh * q_row / 16);
                good = ok(cudaGetLastError());
            } else if (good) {
                good = ok(cudaMemcpyAsync(oh + h0 * q_row, ws + L.o + h0 * q_row, nh * q_row,
                                          cudaMemcpyDeviceToHost, hp->d2h));
            }
            good = good && ok(cudaMemcpyAsync(lh + h0 * l_row, ws + L.lse + h0 * l_row,
                                              nh * l_row, cudaMemcpyDeviceToHost, hp->d2h));
        }
        // the caller's stream resumes only after everything above
        good = good && st == FA_OK && ok(cudaEventRecord(hp->done, hp->d2h)) &&
               ok(cudaStreamWaitEvent(user, hp->done, 0));
        if (!good && st == FA_OK)
            st = FA_ERR_CUDA;
    }
    if (owned && cudaFreeAsync(workspace, user) != cudaSuccess && st == FA_OK)
        st = FA_ERR_CUDA;
    return st;
}

fa_status_t fa_device_status(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FA_ERR_CUDA;
    const DeviceInfo *di = device_info();
    if (!di)
        return FA_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, di->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return FA_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(di->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    if (word & kStatusBounds)
        return FA_ERR_BOUNDS;
    return (word & kStatusTimeout) ? FA_ERR_TIMEOUT : FA_OK;
}

fa_status_t fa_reference_forward_simt(const void *q, const void *k, const void *v, void *o,
                                      float *lse, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                                      int64_t d, int causal, float scale, void *stream)
{
    fa_status_t st = validate(q, k, v, o, lse, B, H, Sq, Sk, d, scale, true);
    if (st != FA_OK)
        return st;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) & 1u)
        return FA_ERR_UNSUPPORTED;
    const DeviceInfo *di = nullptr;
    if ((st = device_ok(&di)) != FA_OK)
        return st;
    return launch_reference_simt(
        make_problem(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, stream, di->status));
}

fa_status_t fa_selftest_umma(const void *a, const void *b, float *c, int n, int k, int b_mn_major,
                             void *stream)
{
    if (!a || !b || !c)
        return FA_ERR_INVALID_ARG;
    if ((n != 64 && n != 128) || (k != 64 && k != 128) || (b_mn_major != 0 && b_mn_major != 1))
        return FA_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(c))
        return FA_ERR_UNSUPPORTED;
    const DeviceInfo *di = nullptr;
    fa_status_t st = device_ok(&di);
    if (st != FA_OK)
        return st;
    return launch_selftest_umma(a, b, c, n, k, b_mn_major, static_cast<cudaStream_t>(stream),
                                di->status);
}

fa_status_t fa_selftest_umma_ts(const void *a, const void *b, float *c, int n, int k,
                                int b_mn_major, void *stream)
{
    if (!a || !b || !c)
        return FA_ERR_INVALID_ARG;
    if ((n != 64 && n != 128) || (k != 64 && k != 128) || (b_mn_major != 0 && b_mn_major != 1))
        return FA_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(c))
        return FA_ERR_UNSUPPORTED;
    const DeviceInfo *di = nullptr;
    fa_status_t st = device_ok(&di);
    if (st != FA_OK)
        return st;
    return launch_selftest_umma_ts(a, b, c, n, k, b_mn_major, static_cast<cudaStream_t>(stream),
                                   di->status);
}

fa_status_t fa_selftest_umma_f8(const void *a, const void *b, float *c, int n, int b_mn_major,
                                int a_tmem, void *stream)
{
    if (!a || !b || !c || (n != 64 && n != 128) || (b_mn_major != 0 && b_mn_major != 1) ||
        (a_tmem != 0 && a_tmem != 1) || (b_mn_major && n != 128))
        return FA_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(c))
        return FA_ERR_UNSUPPORTED;
    const DeviceInfo *di = nullptr;
    fa_status_t st = device_ok(&di);
    if (st != FA_OK)
        return st;
    return launch_selftest_umma_f8(a, b, c, n, b_mn_major, a_tmem,
                                   static_cast<cudaStream_t>(stream), di->status);
}

fa_status_t fa_selftest_mufu(float *out, int blocks, int iters, void *stream)
{
    if (!out || blocks <= 0 || iters <= 0)
        return FA_ERR_INVALID_ARG;
    const DeviceInfo *di = nullptr;
    fa_status_t st = device_ok(&di);
    if (st != FA_OK)
        return st;
    return launch_selftest_mufu(out, blocks, iters, static_cast<cudaStream_t>(stream));
}

fa_status_t fa_selftest_mma_rate(long long *cycles, int mode, int blocks, int iters, void *stream)
{
    if (!cycles || blocks <= 0 || iters <= 0)
        return FA_ERR_INVALID_ARG;
    if (mode < 0 || mode > 6)
        return FA_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(cycles) % alignof(long long) != 0)
        return FA_ERR_UNSUPPORTED;
    const DeviceInfo *di = nullptr;
    fa_status_t st = device_ok(&di);
    if (st != FA_OK)
        return st;
    return launch_selftest_mma_rate(cycles, mode, blocks, iters, static_cast<cudaStream_t>(stream),
                                    di->status);
}

int fa_testing_debug_checks(void)
{
#ifdef FA_DEBUG
    return 1;
#else
    return 0;
#endif
}

fa_status_t fa_selftest_index_check(int fail, void *stream)
{
    const DeviceInfo *di = nullptr;
    fa_status_t st = device_ok(&di);
    if (st != FA_OK)
        return st;
    return launch_selftest_index_check(fail != 0, static_cast<cudaStream_t>(stream), di->status);
}

fa_status_t fa_selftest_elect(int *lanes, int trials, void *stream)
{
    if (!lanes || trials <= 0 || trials > (1 << 20))
        return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(lanes) % alignof(int) != 0)
        return FA_ERR_UNSUPPORTED;
    const DeviceInfo *di = nullptr;
    fa_status_t st = device_ok(&di);
    if (st != FA_OK)
        return st;
    return launch_selftest_elect(lanes, trials, static_cast<cudaStream_t>(stream));
}

fa_status_t fa_testing_stall_next_launch(int kernel, int skip_index, uint64_t wait_limit_ns)
{
    if ((kernel != kStallPrefill && kernel != kStallVerify) || skip_index < 0 ||
        wait_limit_ns < 1000000ull || wait_limit_ns > 10000000000ull)
        return FA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_stall_mu);
    g_stall.kernel = kernel;
    g_stall.skip = skip_index;
    g_stall.wait_ns = wait_limit_ns;
    return FA_OK;
}

fa_status_t fa_selftest_wait_timeout(uint64_t timeout_ns, void *stream)
{
    if (timeout_ns == 0 || timeout_ns > 10000000000ull)
        return FA_ERR_INVALID_ARG;
    const DeviceInfo *di = nullptr;
    fa_status_t st = device_ok(&di);
    if (st != FA_OK)
        return st;
    return launch_selftest_wait(timeout_ns, static_cast<cudaStream_t>(stream), di->status);
}

}  // extern "C"
