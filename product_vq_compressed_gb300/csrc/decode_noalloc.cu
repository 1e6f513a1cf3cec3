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
// stream capture.  No allocation happens here at any time.
#include <mutex>

#include "vq_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = VQ_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device).  Returns VQ_OK or VQ_ERR_CUDA.
int scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return VQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return VQ_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return VQ_OK;
}

}  // namespace

extern "C" {

int vq_decode_attend_noalloc(const vq_attend_args *args, void *stream) {
    if (!args) return VQ_ERR_NULL;
    // same validation as vq_decode_attend, without the caller's workspace
    vq_attend_args a = vqkv::normalize_code_widths(*args);
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    if (a.B < 0 || a.H_q < 0 || a.H_kv < 0 || a.S_q < 0 || a.S_kv < 0 || a.D < 1 ||
        a.sliding_window < 0 || a.H_kv == 0 || a.H_q % a.H_kv != 0 ||
        a.k_sub_dim < 1 || a.v_sub_dim < 1 || a.D % a.k_sub_dim != 0 ||
        a.D % a.v_sub_dim != 0 || a.smooth_mode < 0 || a.smooth_mode > 2 ||
        ((a.causal || a.sliding_window > 0) && a.S_q > a.S_kv) ||
        (a.S_kv == 0 && a.S_q > 0 && a.B > 0 && a.H_q > 0) ||
        a.k_code_bytes < 0 || a.k_code_bytes > 2 || a.v_code_bytes < 0 || a.v_code_bytes > 2 ||
        a.kv_stride < 0 || (a.kv_stride > 0 && a.kv_stride < a.S_kv))
        return VQ_ERR_SHAPE;
    if (a.k_n_centroids < 1 || a.v_n_centroids < 1 ||
        a.k_n_centroids > (a.k_code_bytes == 1 ? 256 : 65536) ||
        a.v_n_centroids > (a.v_code_bytes == 1 ? 256 : 65536) ||
        (a.D & (a.D - 1)) != 0)
        return VQ_ERR_UNSUPPORTED;
    int rc = vqkv::decode_supported(a);
    if (rc != VQ_OK) return rc;
    if ((int64_t)a.B * a.H_q * a.S_q == 0) return VQ_OK;
    if (!a.q_f16 || !a.k_codes || !a.k_codebook || !a.v_codes || !a.v_codebook ||
        !a.out_f16 || (a.smooth_mode != 0 && !a.smooth))
        return VQ_ERR_NULL;
    const void *ptrs[] = {a.q_f16, a.k_codes, a.k_codebook, a.v_codes,
                          a.v_codebook, a.out_f16, a.smooth};
    for (const void *p : ptrs)
        if (p && (reinterpret_cast<uintptr_t>(p) & 15u)) return VQ_ERR_ALIGN;

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
