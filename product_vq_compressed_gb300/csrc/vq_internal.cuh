// vq_internal.cuh -- declarations shared by the CUDA translation units of
// libvqkv.so (kernel launchers and small device helpers).  Not installed.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vqkv.h"

namespace vqkv {

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
};
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
