// prefill.cu -- tensor-core (tcgen05) attention over the coded cache for
// long query blocks.  Not built yet: every request is served by the split-KV
// path.
#include "vq_internal.cuh"

namespace vqkv {

int prefill_supported(const vq_attend_args &a) {
    (void)a;
    return VQ_ERR_UNSUPPORTED;
}

cudaError_t launch_prefill(const vq_attend_args &a, cudaStream_t stream) {
    (void)a;
    (void)stream;
    return cudaErrorNotSupported;
}

}  // namespace vqkv
