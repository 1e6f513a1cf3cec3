// decode_noalloc.cu -- vq_decode_attend for callers that cannot allocate
// device memory.
//
// The regular entry point asks the caller for a workspace that holds the
// per-split partial results (m, l, o[D]) of the split-KV pass.  Some callers
// cannot obtain one: a plug-in running inside a host application that owns
// all device memory and forbids cudaMalloc, a runtime working from a fixed
// memory plan made before the model runs, or a latency-critical loop in
// which an allocation (and the device synchronisation it can cause) is not
// acceptable.  This variant keeps those partial results in a fixed array
// compiled into the library instead.
//
// Scratch: g_noalloc_scratch below, kNoAllocScratchBytes bytes of device
// memory that every GPU which loads the library holds until the process
// exits.  Every call shares it: two calls whose kernels overlap on the GPU
// (different streams, or different host threads) race on it and may return
// wrong results, so serialise them (one stream, or events between streams).
// Nothing in it has to start at zero: each call writes every partial record
// before the combine pass reads it; it keeps the last call's contents.
//
// Host code cannot pass the array's name to a kernel (on the host it only
// names a stand-in object, not device memory), so the first call on each
// device looks up the array's device address with cudaGetSymbolAddress while
// that device is current and keeps it; make that first call before any
// stream capture.  The address belongs to the device's context: it is kept
// together with the context's unique id (cuCtxGetId, reached through
// cudaGetDriverEntryPointByVersion, so the library needs no link to the
// driver library), and looked up again when a call finds another context
// current (after cudaDeviceReset, or when the host application released and
// re-created the primary context).  No allocation happens here at any time.
#include <cuda.h>

#include <mutex>

#include "vq_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = VQ_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchEntry {
    void *addr;
    unsigned long long ctx_id;   // 0: unknown
};
ScratchEntry g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
std::once_flag g_entry_once;

// Unique id of the current context (never reused within the process), or 0
// when there is no current context or the driver cannot tell.
unsigned long long current_context_id() {
    std::call_once(g_entry_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(fn);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!g_ctx_get_current || !g_ctx_get_id || g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        g_ctx_get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array in the current device's context
// (looked up once per context).  Returns VQ_OK or VQ_ERR_CUDA.
int scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return VQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    ScratchEntry &e = g_scratch[dev];
    const unsigned long long id = current_context_id();
    if (!e.addr || id == 0 || id != e.ctx_id) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return VQ_ERR_CUDA;
        e.addr = ptr;
        e.ctx_id = current_context_id();   // the lookup made the context current
    }
    *out = e.addr;
    return VQ_OK;
}

}  // namespace

extern "C" {

int vq_decode_attend_noalloc(const vq_attend_args *args, void *stream) {
    if (!args) return VQ_ERR_NULL;
    // the checks of vq_decode_attend, without the caller's workspace
    vq_attend_args a = vqkv::normalize_code_widths(*args);
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    int rc = vqkv::attend_validate(&a);
    if (rc != VQ_OK) return rc;
    if ((int64_t)a.B * a.H_q * a.S_q == 0) return VQ_OK;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return VQ_ERR_CUDA;
    const vqkv::AttendPlan plan =
        vqkv::plan_decode_capped(a, sms, kNoAllocScratchBytes);
    // even one key split needs more room than the built-in array has
    if (plan.n_split < 1) return VQ_ERR_WORKSPACE;
    void *scratch = nullptr;
    rc = scratch_for_current_device(&scratch);
    if (rc != VQ_OK) return rc;
    a.workspace = scratch;
    a.workspace_bytes = kNoAllocScratchBytes;
    return vqkv::launch_decode(a, plan, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? VQ_OK
               : VQ_ERR_CUDA;
}

}  // extern "C"
