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

// ---------------------------------------------------------------- dependent launches
// A kernel launched with launch_dependent may start while the preceding
// kernel on the stream finishes, once every block of that kernel has called
// pdl_launch_dependents (or exited).  It must call pdl_wait before touching
// data the preceding kernel writes; pdl_wait returns when that kernel has
// completed and its memory operations are visible.  Both are no-ops for
// ordinary launches.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---------------------------------------------------------------- registers <-> memory
// E consecutive elements per lane (E a power of two; naturally aligned).

template <int E>
__device__ __forceinline__ void load_halves(const __half *src, float (&f)[E]) {
    if constexpr (E == 1) {
        f[0] = __half2float(src[0]);
    } else if constexpr (E == 2) {
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(src));
        f[0] = a.x; f[1] = a.y;
    } else {
#pragma unroll
        for (int j = 0; j < E; j += 4) {
            const uint2 raw = *reinterpret_cast<const uint2 *>(src + j);
            const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
            const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
            f[j] = lo.x; f[j + 1] = lo.y; f[j + 2] = hi.x; f[j + 3] = hi.y;
        }
    }
}

template <int E>
__device__ __forceinline__ void store_halves(__half *dst, const float (&f)[E]) {
    if constexpr (E == 1) {
        dst[0] = __float2half_rn(f[0]);
    } else if constexpr (E == 2) {
        *reinterpret_cast<__half2 *>(dst) = __floats2half2_rn(f[0], f[1]);
    } else {
#pragma unroll
        for (int j = 0; j < E; j += 4) {
            __half2 lo = __floats2half2_rn(f[j], f[j + 1]);
            __half2 hi = __floats2half2_rn(f[j + 2], f[j + 3]);
            uint2 raw;
            raw.x = *reinterpret_cast<uint32_t *>(&lo);
            raw.y = *reinterpret_cast<uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(dst + j) = raw;
        }
    }
}

template <int E>
__device__ __forceinline__ void load_floats(const float *src, float (&f)[E]) {
    if constexpr (E == 1) {
        f[0] = src[0];
    } else if constexpr (E == 2) {
        const float2 a = *reinterpret_cast<const float2 *>(src);
        f[0] = a.x; f[1] = a.y;
    } else {
#pragma unroll
        for (int j = 0; j < E; j += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(src + j);
            f[j] = a.x; f[j + 1] = a.y; f[j + 2] = a.z; f[j + 3] = a.w;
        }
    }
}

template <int E>
__device__ __forceinline__ void store_floats(float *dst, const float (&f)[E]) {
    if constexpr (E == 1) {
        dst[0] = f[0];
    } else if constexpr (E == 2) {
        *reinterpret_cast<float2 *>(dst) = make_float2(f[0], f[1]);
    } else {
#pragma unroll
        for (int j = 0; j < E; j += 4)
            *reinterpret_cast<float4 *>(dst + j) = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
    }
}

// Unnormalised Walsh-Hadamard transform (natural order) of the warp's D = 32 E
// elements, lane holding elements [E lane, E lane + E).  Stage h pairs i with
// i + h: a, b -> a + b, a - b.  Stages h < E are inside a lane; stage h >= E
// pairs lane with lane ^ (h / E), where the lower lane keeps own + other and
// the upper one other - own.
template <int E>
__device__ __forceinline__ void reg_fwht(float (&v)[E], int lane) {
#pragma unroll
    for (int h = 1; h < E; h <<= 1) {
#pragma unroll
        for (int i = 0; i < E; ++i) {
            if (i & h) continue;
            const float a = v[i], b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
        }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const float sg = (lane & m) ? -1.f : 1.f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
            v[i] = fmaf(sg, v[i], o);
        }
    }
}

// ---------------------------------------------------------------- packed codes
// Bit-packed codes (code_bytes == 0 at the boundary): b bits per code with
// 2^b >= n_centroids (b >= 1), the n_sub codes of a token as a little-endian
// bit stream (code m in bits [m b, m b + b)), every token row padded to whole
// 32-bit words.
inline int packed_code_bits(int n_centroids) {
    int b = 1;
    while ((1 << b) < n_centroids) ++b;
    return b;
}
__host__ __device__ inline int packed_row_words(int n_sub, int bits) {
    return (n_sub * bits + 31) / 32;
}
// OR code c into position m of a row of 32-bit words (shared memory).
__device__ __forceinline__ void packed_or(uint32_t *row, int m, int bits, uint32_t c) {
    const int bit = m * bits, w = bit >> 5, sh = bit & 31;
    atomicOr(row + w, c << sh);
    if (sh + bits > 32) atomicOr(row + w + 1, c >> (32 - sh));
}
// Code m of a packed row.
__device__ __forceinline__ uint32_t packed_get(const uint32_t *row, int m, int bits) {
    const int bit = m * bits, w = bit >> 5, sh = bit & 31;
    uint64_t x = row[w];
    if (sh + bits > 32) x |= (uint64_t)row[w + 1] << 32;
    return (uint32_t)(x >> sh) & ((1u << bits) - 1u);
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
    void *codes;              // [n_vec, D/sub_dim], code_bytes each (0: packed rows)
    int code_bytes;
    int code_bits, row_words; // packed codes: bits per code, words per token row
    __half *xhat;             // [n_vec, D] or null
    FastDiv div_S, div_H;     // by S and H (head of a token)
    int cap, off;             // code rows per (b, h) and the first row written
};

// Cache row of token v: token t of (b, h) goes to row off + t of that
// (b, h)'s cap rows.
__device__ __forceinline__ int64_t token_row(const EncodeParams &p, int64_t v) {
    if (p.cap == p.S && p.off == 0) return v;
    const int64_t bh = p.n_vec < (int64_t(1) << 31) ? (int64_t)fast_div((uint32_t)v, p.div_S)
                                                    : v / p.S;
    return (bh * p.cap + p.off) + (v - bh * p.S);
}
// Code index of sub-vector m of token v.
__device__ __forceinline__ int64_t code_index(const EncodeParams &p, int64_t v, int n_sub,
                                              int m) {
    return token_row(p, v) * n_sub + m;
}

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
    int code_bytes;           // 1, 2, or 0: packed rows
    int code_bits, row_words; // packed codes: bits per code, words per row of n_sub codes
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
// The same arguments with packed rows of 8- or 16-bit codes described as
// uint8 / uint16 codes (identical bytes), so that they take those paths.
vq_attend_args normalize_code_widths(const vq_attend_args &a);

int prefill_supported(const vq_attend_args &a);  // VQ_OK or a status
cudaError_t launch_prefill(const vq_attend_args &a, cudaStream_t stream);

}  // namespace vqkv
