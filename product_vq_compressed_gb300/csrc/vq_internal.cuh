// vq_internal.cuh -- declarations shared by the CUDA translation units of
// libvqkv.so (kernel launchers and small device helpers).  Not installed.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vqkv.h"

namespace vqkv {

// ---------------------------------------------------------------- helpers
// Division by an invariant 32-bit divisor d >= 1 as a multiply-high, add and
// shift (Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994, the round-up method): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (mulhi(m, n) + n) >> l for every
// n < 2^31 (the sum stays below 2^32).
struct FastDiv {
    uint32_t d, m, l;
};
inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f{d, 0u, 0u};
    while ((1ull << f.l) < d) ++f.l;
    f.m = (uint32_t)((((1ull << f.l) - d) << 32) / d + 1);
    return f;
}
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv &f) {
    return (__umulhi(f.m, n) + n) >> f.l;
}

// ---------------------------------------------------------------- encode
struct EncodeParams {
    const __half *x;          // [n_vec, D]
    int64_t n_vec;
    int H, S, D, log2D;
    const float *codebook;    // [N, sub_dim]
    int N, sub_dim;
    const float *smooth;      // mode 1: [D], mode 2: [H, D], mode 0: null
    int smooth_mode;
    int rotate;               // 1 keys (smooth + Hadamard), 0 values
    void *codes;              // [n_vec, D/sub_dim], code_bytes each
    int code_bytes;
    __half *xhat;             // [n_vec, D] or null
    FastDiv div_S, div_H;     // by S and H (head of a token)
};

// Head of token v of a [B, H, S, D] tensor: (v / S) mod H.
__device__ __forceinline__ int token_head(const EncodeParams &p, int64_t v) {
    if (p.n_vec < (int64_t(1) << 31)) {
        const uint32_t q = fast_div((uint32_t)v, p.div_S);
        return (int)(q - fast_div(q, p.div_H) * (uint32_t)p.H);
    }
    return (int)((v / p.S) % p.H);
}
// Returns a cudaError_t of the launch.
cudaError_t launch_encode(const EncodeParams &p, cudaStream_t stream);
size_t encode_smem_bytes(int N, int sub_dim);
// Tensor-core screening variant (sub_dim 2, 4, 8 with the codebook's
// operands fitting in shared memory); launch_encode dispatches to it.
bool encode_mma_supported(int N, int sub_dim);
cudaError_t launch_encode_mma(const EncodeParams &p, cudaStream_t stream);

// ---------------------------------------------------------------- dequant
struct DequantParams {
    const void *codes;
    int code_bytes;
    int64_t n_vec;
    int n_sub;
    const float *codebook;
    int N, sub_dim;
    void *out;
    int out_is_f32;
};
cudaError_t launch_dequant(const DequantParams &p, cudaStream_t stream);

// ---------------------------------------------------------------- attend
struct AttendPlan {
    int n_split;        // 1 (0 when a capped plan cannot fit)
    int cols;           // query columns (head, row) pairs per column block
    int n_colblk;       // column blocks per (b, kv head)
    int tok_per_split;  // keys each unit scans
    int tile_lo, tiles; // every unit scans key tiles [tile_lo, tile_lo + tiles)
    int64_t total;      // units * tiles
    int64_t n_warps;    // warps sharing the flattened work
    int64_t share;      // tiles per warp (contiguous shares)
    int grid;           // CTAs
    int slots;          // partial records per warp
    size_t ws_bytes;    // partial records
};
AttendPlan plan_decode(const vq_attend_args &a, int num_sms);
// The same plan with at most max_ws_bytes of partial results (fewer key
// splits); n_split == 0 when even one split does not fit.
AttendPlan plan_decode_capped(const vq_attend_args &a, int num_sms,
                              size_t max_ws_bytes);
cudaError_t launch_decode(const vq_attend_args &a, const AttendPlan &plan,
                          cudaStream_t stream);
size_t decode_smem_bytes(const vq_attend_args &a);
int decode_supported(const vq_attend_args &a);   // VQ_OK or a status

int prefill_supported(const vq_attend_args &a);  // VQ_OK or a status
cudaError_t launch_prefill(const vq_attend_args &a, cudaStream_t stream);

}  // namespace vqkv
