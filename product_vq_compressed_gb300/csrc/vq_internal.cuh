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
// ---------------------------------------------------------------- certified codes
// The encode kernels decide in fp32.  A code is kept only when a rigorous
// bound shows that it is the exact nearest centroid of the exact rotated
// sub-vector y = Hn (s (.) x); otherwise it is decided again in float-float
// arithmetic (nearest_exact: about 44 significant bits), so that a code can
// differ from an exact (or float64) decision only where two squared
// distances agree to about 1e-10 relative.  Error model (u = 2^-24):
//   * the fp32 rotation: every element of y~ is within
//       delta = (log2 D + 3) u sum_i |x_i s_i| / sqrt D
//     of y (one rounding per butterfly stage, gamma_L <= (L + 3) u with the
//     smooth product and the 1/sqrt D factor; delta = 0 without rotation);
//     so | |y~ - c| - |y - c| | <= Delta = sqrt(sub_dim) delta for every c;
//   * an fp32 squared distance of y~ (subtract, multiply-add chain) is within
//     a relative (sub_dim + 4) u of the exact |y~ - c|^2.
// With b an upper bound on the chosen centroid's |y~ - c|^2 and lo a lower
// bound on every other centroid's, the choice is exact when
//   sqrt(lo) - Delta > sqrt(b) + Delta.
constexpr float kEncU = 5.9604645e-8f;   // 2^-24

// delta per unit of sum_i |fl(x_i s_i)| (slack 1.002 covers the fp32 sum of
// those terms, the rounding of 1/sqrt D and of the bound itself)
__device__ __forceinline__ float rotation_delta_coef(int log2D, float inv_sqrt_d) {
    return (float)(log2D + 3) * kEncU * 1.002f * inv_sqrt_d;
}

// sqrt(SUBD), rounded up
template <int SUBD>
struct SqrtSub {
    static constexpr float v = SUBD == 1 ? 1.f : SUBD == 2 ? 1.4142136f : SUBD == 4 ? 2.f
                             : SUBD == 8 ? 2.8284272f : 4.f;
};

// true when the fp32 decision is certified exact (see above): b and lo are
// the fp32-computed values bounding the winner and the others
template <int SUBD>
__device__ __forceinline__ bool code_certified(float b, float lo, float delta) {
    constexpr float gdir = (float)(SUBD + 4) * kEncU * 1.01f;
    if (!(lo < INFINITY)) return b < INFINITY;   // no other candidate
    const float ub = b * (1.f + gdir);
    const float lb = lo * (1.f - gdir);
    if (!(lb > 0.f) || !(ub >= 0.f)) return false;
    const float two_delta = 2.004f * SqrtSub<SUBD>::v * delta;   // 2 Delta with rounding slack
    // sqrt(lb) - sqrt(ub) >= (lb - ub) / (2 sqrt(lb)) >= (lb - ub) / (lb + 1):
    // a sufficient test without square roots, then the exact one
    if ((lb - ub) * (1.f - 4.f * kEncU) > two_delta * (lb + 1.f) * (1.f + 4.f * kEncU))
        return true;
    return sqrtf(lb) * (1.f - 4.f * kEncU) - sqrtf(ub) * (1.f + 4.f * kEncU) > two_delta;
}

// Float-float numbers hi + lo (|lo| <= ulp(hi) / 2 after normalisation),
// from the error-free transformations TwoSum (Knuth, "The Art of Computer
// Programming" vol. 2, 4.2.2) and the FMA form of TwoProduct.  Each
// operation keeps about 44 significant bits.
struct FF {
    float hi, lo;
};
__device__ __forceinline__ FF ff_two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    return {s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ FF ff_fast_two_sum(float a, float b) {   // |a| >= |b| or a == 0
    const float s = a + b;
    return {s, b - (s - a)};
}
__device__ __forceinline__ FF ff_two_prod(float a, float b) {
    const float p = a * b;
    return {p, fmaf(a, b, -p)};
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
    const FF s = ff_two_sum(a.hi, b.hi);
    return ff_fast_two_sum(s.hi, s.lo + (a.lo + b.lo));
}
__device__ __forceinline__ FF ff_mul(FF a, FF c) {
    const FF p = ff_two_prod(a.hi, c.hi);
    return ff_fast_two_sum(p.hi, fmaf(a.hi, c.lo, fmaf(a.lo, c.hi, p.lo)));
}
__device__ __forceinline__ bool ff_less(FF a, FF b) {
    return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}

// 1/sqrt(32 E) as a float-float constant (from the decimal value of the
// mathematical constant; exact for E = 2, 8)
template <int E>
struct InvSqrtD {
    static constexpr double v = E == 1 ? 0.17677669529663688110 : E == 2 ? 0.125
                              : E == 4 ? 0.08838834764831844055 : E == 8 ? 0.0625
                                       : 0.04419417382415922028;
    static constexpr float hi = (float)v;
    static constexpr float lo = (float)(v - (double)hi);
};

// Nearest centroid of sub-vector m of one token in float-float arithmetic,
// by the whole warp (every lane returns it).  xv: the token's D = 32 E fp16
// inputs; sm: its smooth factors or null; cent(c, t): coordinate t of
// centroid c (fp32); delta: the token's fp32 rotation bound (above).  y is
// recomputed from the fp16 input: each element is the signed sum over the
// token of x_i s_i ((-1)^popc(r & i), the natural-order Sylvester sign) times
// 1/sqrt D; without rotation y = x.  Distances in the direct form
// sum_t (y_t - c_t)^2, the lowest index on ties (non-finite inputs: code 0).
template <int SUBD, int E, typename Cent>
__device__ __forceinline__ int nearest_exact_e(const __half *xv, const float *sm, int rotate,
                                               Cent cent, int N, int m, float delta, int lane) {
    FF y[SUBD];
    if (rotate) {
        // lane holds elements [E lane, E lane + E): all loads issued together
        float xf[E], sf[E];
        load_halves<E>(xv + lane * E, xf);
        if (sm) {
            load_floats<E>(sm + lane * E, sf);
        } else {
#pragma unroll
            for (int j = 0; j < E; ++j) sf[j] = 1.f;
        }
#pragma unroll
        for (int t = 0; t < SUBD; ++t) y[t] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < E; ++j) {
            const int i = lane * E + j;
            const FF xs = ff_two_prod(xf[j], sf[j]);   // x_i s_i exactly
#pragma unroll
            for (int t = 0; t < SUBD; ++t) {
                const bool neg = __popc((m * SUBD + t) & i) & 1;
                y[t] = ff_add(y[t], neg ? FF{-xs.hi, -xs.lo} : xs);
            }
        }
#pragma unroll
        for (int t = 0; t < SUBD; ++t) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                y[t] = ff_add(y[t], FF{__shfl_xor_sync(0xffffffffu, y[t].hi, off),
                                       __shfl_xor_sync(0xffffffffu, y[t].lo, off)});
            // one value for every lane (the butterfly sums may differ in the last bit)
            y[t] = ff_mul(FF{__shfl_sync(0xffffffffu, y[t].hi, 0), __shfl_sync(0xffffffffu, y[t].lo, 0)},
                          FF{InvSqrtD<E>::hi, InvSqrtD<E>::lo});
        }
    } else {
#pragma unroll
        for (int t = 0; t < SUBD; ++t) y[t] = {__half2float(xv[m * SUBD + t]), 0.f};
    }
    // Candidates that can win: a screen in fp32 from yr = y.hi, within
    // Delta_r = sqrt(SUBD) (u max|y| + delta) of y in the Euclidean norm
    // (delta bounds the float-float sum's error many times over); fp32
    // distances are within a relative (SUBD + 4) u.  Only candidates whose
    // lower bound reaches the smallest upper bound are evaluated exactly.
    float yr[SUBD];
    float ymax = 0.f;
#pragma unroll
    for (int t = 0; t < SUBD; ++t) {
        yr[t] = y[t].hi;
        ymax = fmaxf(ymax, fabsf(yr[t]));
    }
    constexpr float g = (float)(SUBD + 4) * kEncU * 1.01f;
    const float dr = SqrtSub<SUBD>::v * (ymax * kEncU + delta) * 1.01f;
    auto d32 = [&](int c) {
        float d = 0.f;
#pragma unroll
        for (int t = 0; t < SUBD; ++t) {
            const float e = yr[t] - cent(c, t);
            d = fmaf(e, e, d);
        }
        return d;
    };
    float dmin = INFINITY;
    for (int c = lane; c < N; c += 32) dmin = fminf(dmin, d32(c));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dmin = fminf(dmin, __shfl_xor_sync(0xffffffffu, dmin, off));
    // candidate c survives when sqrt(d32 (1 - g)) - dr <= sqrt(dmin (1 + g)) + dr
    const float reach = (sqrtf(dmin * (1.f + g)) + 2.f * dr) * (1.f + 4.f * kEncU);
    const float reach2 = reach * reach * (1.f + 4.f * kEncU);
    FF best = {INFINITY, 0.f};
    int bi = 0x7fffffff;
    for (int c = lane; c < N; c += 32) {
        if (!(d32(c) * (1.f - g) <= reach2)) continue;   // cannot be the nearest
        FF acc = {0.f, 0.f};
#pragma unroll
        for (int t = 0; t < SUBD; ++t) {
            const FF s = ff_two_sum(y[t].hi, -cent(c, t));
            const FF e = ff_fast_two_sum(s.hi, s.lo + y[t].lo);
            const FF q = ff_two_prod(e.hi, e.hi);
            acc = ff_add(acc, ff_fast_two_sum(q.hi, fmaf(2.f * e.hi, e.lo, q.lo)));
        }
        if (ff_less(acc, best)) { best = acc; bi = c; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const FF ob = {__shfl_xor_sync(0xffffffffu, best.hi, off),
                       __shfl_xor_sync(0xffffffffu, best.lo, off)};
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ff_less(ob, best) || (ob.hi == best.hi && ob.lo == best.lo && oi < bi)) {
            best = ob;
            bi = oi;
        }
    }
    return bi == 0x7fffffff ? 0 : bi;
}

// nearest_exact_e for sub-vector m of token v of an encode call.
template <int SUBD, typename Cent>
__device__ __forceinline__ int nearest_exact_token(const EncodeParams &p, int64_t v, int m,
                                                   Cent cent, float delta, int lane) {
    const float *sm = !p.rotate || p.smooth_mode == 0 ? nullptr
                      : p.smooth_mode == 2 ? p.smooth + (size_t)token_head(p, v) * p.D
                                           : p.smooth;
    const __half *xv = p.x + v * p.D;
    switch (p.D) {
        case 32: return nearest_exact_e<SUBD, 1>(xv, sm, p.rotate, cent, p.N, m, delta, lane);
        case 64: return nearest_exact_e<SUBD, 2>(xv, sm, p.rotate, cent, p.N, m, delta, lane);
        case 128: return nearest_exact_e<SUBD, 4>(xv, sm, p.rotate, cent, p.N, m, delta, lane);
        case 256: return nearest_exact_e<SUBD, 8>(xv, sm, p.rotate, cent, p.N, m, delta, lane);
        default: return nearest_exact_e<SUBD, 16>(xv, sm, p.rotate, cent, p.N, m, delta, lane);
    }
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
// Argument checks of the attention entry points (sizes, limits, pointers,
// alignment; in the order include/vqkv.h states), VQ_OK or a status.  The
// workspace size is checked by each entry point against its own plan.
int attend_validate(const vq_attend_args *a);

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
// reserved_warps: warps of every CTA that take no share (a decode step's
// encoding warps, kStepEncodeWarps)
constexpr int kStepEncodeWarps = 4;
AttendPlan plan_decode(const vq_attend_args &a, int num_sms, int reserved_warps = 0);
// A decode step's flags for its new rows: their offset in the workspace
// (after the plan's partial records) and size.
size_t step_flags_offset(const AttendPlan &plan);
size_t step_flags_bytes(const vq_attend_args &a);
// The same plan with at most max_ws_bytes of partial results (fewer key
// splits); n_split == 0 when even one split does not fit.
AttendPlan plan_decode_capped(const vq_attend_args &a, int num_sms,
                              size_t max_ws_bytes);
// k_new / v_new (both or neither): one decode step in one cooperative
// launch -- the new tokens [B, H_kv, S_q, D] are encoded into cache rows
// S_kv - S_q .. S_kv - 1 first, and the key splits are merged in the launch.
cudaError_t launch_decode(const vq_attend_args &a, const AttendPlan &plan,
                          cudaStream_t stream, const void *k_new = nullptr,
                          const void *v_new = nullptr);
int decode_step_supported(const vq_attend_args &a);   // VQ_OK or a status
size_t decode_smem_bytes(const vq_attend_args &a);
int decode_supported(const vq_attend_args &a);   // VQ_OK or a status
// The same arguments with packed rows of 8- or 16-bit codes described as
// uint8 / uint16 codes (identical bytes), so that they take those paths.
vq_attend_args normalize_code_widths(const vq_attend_args &a);

int prefill_supported(const vq_attend_args &a);  // VQ_OK or a status
cudaError_t launch_prefill(const vq_attend_args &a, cudaStream_t stream);

}  // namespace vqkv
