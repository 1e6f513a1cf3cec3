// encode.cu -- key / value encode (smooth, Walsh-Hadamard rotation, nearest
// centroid per sub-vector) and the codebook gather.
//
// Pages: "Metal Kernels API", section "VecInfer kernels":
//   vecinfer_encode_decode_metal  smooth -> WHT -> VQ encode -> dequant ->
//                                 inverse WHT -> inverse smooth (keys);
//   vecinfer_encode_decode_simple_metal  the same without smooth and WHT
//                                 (values);
//   vecinfer_quantize_metal       squared distances to every centroid kept in
//                                 registers, one index per sub-vector;
//   vecinfer_dequant_metal        codebook gather.
//
// GB300 layout.  A block of 128 threads stages the whole codebook (fp32) in
// shared memory once and then walks a persistent loop over tiles of 512
// sub-vectors (512 / n_sub tokens):
//   1. one warp per token: fp16 load (8-byte vectors, coalesced), smooth and
//      1/sqrt(D) folded into the load, in-place FWHT in shared memory;
//   2. every thread owns four sub-vectors and scans the codebook; all threads
//      read the same centroid at the same time, so each shared-memory read
//      is a broadcast, and one centroid load serves all four.  The
//      scan screens with f_c = |c|^2 - 2 y.c (one fused multiply-add per
//      dimension; -2c and |c|^2 are staged once), tracking the best and the
//      second-best value with min/max only; the group of 8 candidates where
//      the best last improved is noted and its index found by recomputing
//      that group (lowest index on ties).  If
//      the two are closer than twice a rigorous bound on the fp32 error of
//      that form, the sub-vector is rescanned with the direct form
//      sum_t (y_t - c_t)^2, so every decision is the one the direct form
//      makes.  The decision is then certified against the rounding of the
//      fp32 rotation and distances (code_certified); the few sub-vectors
//      that are not certified are decided again in float-float arithmetic
//      by the whole warp (nearest_exact).  Codes are written in sub-vector order (coalesced
//      stores);
//   3. optional reconstruction: the chosen centroids replace the sub-vectors
//      in shared memory, one warp per token runs the FWHT again (Hn is
//      symmetric and its own inverse), divides by the smooth factors and
//      stores fp16 (round to nearest even).
// The scan of phase 2 is the cost: N * sub_dim fused multiply-adds plus a
// compare/select per candidate.
#include <math.h>

#include <type_traits>

#include "vq_internal.cuh"

namespace vqkv {
namespace {

constexpr int kEncThreads = 128;
constexpr int kSlots = 512;  // sub-vectors per tile
constexpr int kR = kSlots / kEncThreads;  // sub-vectors per thread

// Unnormalised in-place Walsh-Hadamard transform (natural order) of the D
// floats at v, by one warp.  Butterfly at stride h pairs i and i + h.
__device__ __forceinline__ void warp_fwht(float *v, int D, int lane) {
    for (int h = 1; h < D; h <<= 1) {
        for (int p = lane; p < (D >> 1); p += 32) {
            const int i = ((p & ~(h - 1)) << 1) | (p & (h - 1));
            const float a = v[i], b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
        }
        __syncwarp();
    }
}

template <int SUBD>
__device__ __forceinline__ void load_sub(const float *src, float (&dst)[SUBD]) {
    if constexpr (SUBD % 4 == 0) {
#pragma unroll
        for (int t = 0; t < SUBD; t += 4) {
            const float4 q = *reinterpret_cast<const float4 *>(src + t);
            dst[t] = q.x; dst[t + 1] = q.y; dst[t + 2] = q.z; dst[t + 3] = q.w;
        }
    } else if constexpr (SUBD == 2) {
        const float2 q = *reinterpret_cast<const float2 *>(src);
        dst[0] = q.x; dst[1] = q.y;
    } else {
        dst[0] = src[0];
    }
}

template <int SUBD, typename CodeT>
__global__ void __launch_bounds__(kEncThreads)
encode_kernel(EncodeParams p, float inv_sqrt_d) {
    extern __shared__ __align__(16) float smem[];
    const int N = p.N, D = p.D;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // a dependent attention launch may be scheduled now (it waits for this grid)
    pdl_launch_dependents();
    // shared memory: -2c [N][SUBD], |c|^2 [N], max |c|^2, sub-vectors [512][SUBD]
    float *cb_s = smem;
    float *nrm_s = cb_s + ((N * SUBD + 3) & ~3);
    float *maxn2_s = nrm_s + ((N + 3) & ~3);
    float *y_s = maxn2_s + 4;
    // packed codes (CodeT = uint32_t): the tile's token rows, assembled here
    constexpr bool kPacked = std::is_same<CodeT, uint32_t>::value;
    uint32_t *ptile = reinterpret_cast<uint32_t *>(y_s + kSlots * SUBD);
    // rotation error bound of every token of the tile (<= 256 tokens)
    float *delta_s = reinterpret_cast<float *>(ptile + 768);
    const float dcoef = rotation_delta_coef(p.log2D, inv_sqrt_d);

    if (tid == 0) *maxn2_s = 0.f;
    for (int i = tid; i < N * SUBD; i += kEncThreads) cb_s[i] = -2.0f * p.codebook[i];
    __syncthreads();
    for (int c = tid; c < N; c += kEncThreads) {
        float n2 = 0.f;
        for (int t = 0; t < SUBD; ++t) {
            const float v = p.codebook[c * SUBD + t];
            n2 = fmaf(v, v, n2);
        }
        nrm_s[c] = n2;
        // non-negative floats order like their bit patterns
        atomicMax(reinterpret_cast<int *>(maxn2_s), __float_as_int(n2));
    }
    __syncthreads();

    const int n_sub = D / SUBD;
    const int lsub = p.log2D - (SUBD == 1 ? 0 : SUBD == 2 ? 1 : SUBD == 4 ? 2 : SUBD == 8 ? 3 : 4);
    const int tok = kSlots / n_sub;  // tokens per tile (n_sub divides 512)
    const int64_t n_tiles = (p.n_vec + tok - 1) / tok;
    CodeT *codes = reinterpret_cast<CodeT *>(p.codes);

    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int64_t v0 = tile * tok;
        // ---- 1. load, smooth, rotate
        for (int t = warp; t < tok; t += kEncThreads / 32) {
            const int64_t v = v0 + t;
            float *yv = y_s + t * D;
            if (v < p.n_vec) {
                const __half *xv = p.x + v * D;
                const int h = token_head(p, v);
                const float *sm = p.smooth_mode == 2 ? p.smooth + (size_t)h * D
                                                     : p.smooth;
                float asum = 0.f;   // sum |fl(x s)|: size of the rotation's rounding error
                for (int e = lane * 4; e < D; e += 128) {
                    const uint2 raw = *reinterpret_cast<const uint2 *>(xv + e);
                    const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
                    const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
                    float4 f = make_float4(lo.x, lo.y, hi.x, hi.y);
                    if (p.rotate) {
                        if (p.smooth_mode != 0) {
                            const float4 s = *reinterpret_cast<const float4 *>(sm + e);
                            f.x *= s.x; f.y *= s.y; f.z *= s.z; f.w *= s.w;
                        }
                        asum += fabsf(f.x) + fabsf(f.y) + fabsf(f.z) + fabsf(f.w);
                        f.x *= inv_sqrt_d; f.y *= inv_sqrt_d;
                        f.z *= inv_sqrt_d; f.w *= inv_sqrt_d;
                    }
                    *reinterpret_cast<float4 *>(yv + e) = f;
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) asum += __shfl_xor_sync(0xffffffffu, asum, off);
                if (lane == 0) delta_s[t] = asum * dcoef;
                __syncwarp();
                if (p.rotate) warp_fwht(yv, D, lane);
            } else {
                for (int e = lane; e < D; e += 32) yv[e] = 0.f;
                if (lane == 0) delta_s[t] = 0.f;
            }
        }
        if constexpr (kPacked) {
            for (int i = tid; i < tok * p.row_words; i += kEncThreads) ptile[i] = 0u;
        }
        __syncthreads();

        // ---- 2. nearest centroid of kR sub-vectors per thread
        {
            float y[kR][SUBD];
#pragma unroll
            for (int r = 0; r < kR; ++r) load_sub<SUBD>(y_s + (tid + r * kEncThreads) * SUBD, y[r]);
            // screening in the expanded form f_c = |c|^2 - 2 y.c (one fused
            // multiply-add per dimension), keeping the best and second-best
            // value; the best's index is located afterwards: only the group
            // of kGroup candidates in which the best last improved is noted
            // (strict '<', so the earliest group wins ties)
            constexpr int kGroup = 8;
            float f1[kR], f2[kR];
            int grp[kR], i1[kR];
#pragma unroll
            for (int r = 0; r < kR; ++r) { f1[r] = INFINITY; f2[r] = INFINITY; grp[r] = 0; i1[r] = 0; }
            const int n_full = N & ~(kGroup - 1);
            for (int g0 = 0; g0 < n_full; g0 += kGroup) {
                float fb[kR];
#pragma unroll
                for (int r = 0; r < kR; ++r) fb[r] = f1[r];
#pragma unroll
                for (int k = 0; k < kGroup; k += 2) {   // two candidates per round
                    float ca[SUBD], cb[SUBD];
                    load_sub<SUBD>(cb_s + (g0 + k) * SUBD, ca);
                    load_sub<SUBD>(cb_s + (g0 + k + 1) * SUBD, cb);
                    const float na = nrm_s[g0 + k], nb = nrm_s[g0 + k + 1];
#pragma unroll
                    for (int r = 0; r < kR; ++r) {
                        float fa = na, fb = nb;
#pragma unroll
                        for (int t = 0; t < SUBD; ++t) {
                            fa = fmaf(ca[t], y[r][t], fa);
                            fb = fmaf(cb[t], y[r][t], fb);
                        }
                        // second smallest of {f1 <= f2, fa, fb}:
                        // min(f2, max(f1, min(fa, fb)), max(fa, fb))
                        const float lo = fminf(fa, fb), hi = fmaxf(fa, fb);
                        f2[r] = fminf(fminf(f2[r], fmaxf(f1[r], lo)), hi);
                        f1[r] = fminf(f1[r], lo);
                    }
                }
#pragma unroll
                for (int r = 0; r < kR; ++r) grp[r] = f1[r] < fb[r] ? g0 : grp[r];
            }
            // index of the best inside its group: recompute that group (the
            // same arithmetic, so the best value reappears bit for bit)
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                int found = -1;
#pragma unroll
                for (int k = 0; k < kGroup; ++k) {
                    const int c = grp[r] + k;
                    if (c >= n_full) break;
                    float f = nrm_s[c];
#pragma unroll
                    for (int t = 0; t < SUBD; ++t) f = fmaf(cb_s[c * SUBD + t], y[r][t], f);
                    if (found < 0 && f == f1[r]) found = c;
                }
                i1[r] = found < 0 ? 0 : found;
            }
            // candidates past the last full group (N not a multiple of kGroup)
            for (int c = n_full; c < N; ++c) {
                float cv[SUBD];
                load_sub<SUBD>(cb_s + c * SUBD, cv);
                const float nc = nrm_s[c];
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    float f = nc;
#pragma unroll
                    for (int t = 0; t < SUBD; ++t) f = fmaf(cv[t], y[r][t], f);
                    f2[r] = fminf(f2[r], fmaxf(f1[r], f));
                    const bool lt = f < f1[r];
                    i1[r] = lt ? c : i1[r];
                    f1[r] = lt ? f : f1[r];
                }
            }
            // When the two best screened values are closer than twice the
            // fp32 error bound of the expanded form, or the screen cannot
            // certify the decision, rescan with the direct form
            // sum_t (y_t - c_t)^2 (c = -cb/2).
            // The decision is then certified (code_certified) from a lower
            // bound on the other candidates' distances and an upper bound on
            // the winner's, both to the fp32 sub-vector y~.
            const float maxn2 = *maxn2_s;
            const int64_t lim = p.n_vec * n_sub;
            bool cert[kR];
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const int sl = tid + r * kEncThreads;
                const float delta = delta_s[sl >> lsub];
                float ny2 = 0.f;
#pragma unroll
                for (int t = 0; t < SUBD; ++t) ny2 = fmaf(y[r][t], y[r][t], ny2);
                const float bound = (4.0f * SUBD + 8.0f) * 5.9604645e-8f *
                                    (maxn2 + 2.0f * sqrtf(maxn2 * ny2) + 1e-30f);
                // screened values are within `bound` of the exact f_c; |y~|^2
                // within (SUBD + 8) u of ny2 with the sums' rounding
                const float slack = (float)(SUBD + 8) * 5.9604645e-8f;
                const float hi = (f1[r] + ny2) + (bound + slack * (fabsf(f1[r]) + ny2));
                const float lo = f2[r] < INFINITY
                                     ? (f2[r] + ny2) - (bound + slack * (fabsf(f2[r]) + ny2))
                                     : INFINITY;
                cert[r] = f2[r] - f1[r] > 2.0f * bound && code_certified<SUBD>(hi, lo, delta);
                if (!cert[r]) {
                    // rescan in the direct form: the order of the direct form,
                    // and every candidate's distance for the certificate
                    float best = INFINITY, second = INFINITY;
                    int bi = 0;
                    for (int c = 0; c < N; ++c) {
                        float d = 0.f;
#pragma unroll
                        for (int t = 0; t < SUBD; ++t) {
                            const float e = y[r][t] + 0.5f * cb_s[c * SUBD + t];
                            d = fmaf(e, e, d);
                        }
                        second = fminf(second, fmaxf(best, d));
                        if (d < best) { best = d; bi = c; }
                    }
                    i1[r] = bi;
                    cert[r] = code_certified<SUBD>(best, second, delta);
                }
                cert[r] = cert[r] || v0 * n_sub + sl >= lim;
            }
            // sub-vectors the fp32 arithmetic cannot certify: float-float, whole warp
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                unsigned m = __ballot_sync(0xffffffffu, !cert[r]);
                while (m) {
                    const int src = __ffs(m) - 1;
                    m &= m - 1;
                    const int sl = warp * 32 + src + r * kEncThreads;
                    // cb_s holds -2 c (exact), so -0.5 cb_s is the centroid
                    const int cx = nearest_exact_token<SUBD>(
                        p, v0 + (sl >> lsub), sl & (n_sub - 1),
                        [cb_s](int c, int t) { return -0.5f * cb_s[c * SUBD + t]; },
                        delta_s[sl >> lsub], lane);
                    if (lane == src) i1[r] = cx;
                }
            }
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const int sl = tid + r * kEncThreads;
                const int64_t gi = v0 * n_sub + sl;
                if (gi < lim) {
                    if constexpr (kPacked)
                        packed_or(ptile + (sl >> lsub) * p.row_words, sl & (n_sub - 1),
                                  p.code_bits, (uint32_t)i1[r]);
                    else
                        codes[code_index(p, gi >> lsub, n_sub, (int)(gi & (n_sub - 1)))] = (CodeT)i1[r];
                }
                if (p.xhat) {
#pragma unroll
                    for (int t = 0; t < SUBD; ++t)
                        y_s[sl * SUBD + t] = -0.5f * cb_s[i1[r] * SUBD + t];
                }
            }
        }
        __syncthreads();
        if constexpr (kPacked) {   // the tile's packed token rows -> the cache
            uint32_t *cw = reinterpret_cast<uint32_t *>(p.codes);
            for (int i = tid; i < tok * p.row_words; i += kEncThreads) {
                const int t = i / p.row_words, w = i - t * p.row_words;
                if (v0 + t < p.n_vec) cw[token_row(p, v0 + t) * p.row_words + w] = ptile[i];
            }
            __syncthreads();   // before the next tile clears the rows
        }

        // ---- 3. optional reconstruction s^-1 (.) Hn y_hat -> fp16
        if (p.xhat) {
            for (int t = warp; t < tok; t += kEncThreads / 32) {
                const int64_t v = v0 + t;
                if (v >= p.n_vec) continue;
                float *yv = y_s + t * D;
                if (p.rotate) warp_fwht(yv, D, lane);
                const int h = token_head(p, v);
                const float *sm = p.smooth_mode == 2 ? p.smooth + (size_t)h * D
                                                     : p.smooth;
                __half *ov = p.xhat + v * D;
                for (int e = lane * 4; e < D; e += 128) {
                    float4 f = *reinterpret_cast<const float4 *>(yv + e);
                    if (p.rotate) {
                        f.x *= inv_sqrt_d; f.y *= inv_sqrt_d;
                        f.z *= inv_sqrt_d; f.w *= inv_sqrt_d;
                        if (p.smooth_mode != 0) {
                            const float4 s = *reinterpret_cast<const float4 *>(sm + e);
                            f.x /= s.x; f.y /= s.y; f.z /= s.z; f.w /= s.w;
                        }
                    }
                    __half2 lo = __floats2half2_rn(f.x, f.y);
                    __half2 hi = __floats2half2_rn(f.z, f.w);
                    uint2 raw;
                    raw.x = *reinterpret_cast<uint32_t *>(&lo);
                    raw.y = *reinterpret_cast<uint32_t *>(&hi);
                    *reinterpret_cast<uint2 *>(ov + e) = raw;
                }
            }
            __syncthreads();
        }
    }
}

template <typename CodeT>
__global__ void dequant_kernel(DequantParams p) {
    constexpr bool kPacked = std::is_same<CodeT, uint32_t>::value;
    const CodeT *codes = reinterpret_cast<const CodeT *>(p.codes);
    const int64_t total = p.n_vec * p.n_sub;
    const int d = p.sub_dim;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int c;
        if constexpr (kPacked) {
            const int64_t v = i / p.n_sub;
            c = (int)packed_get(reinterpret_cast<const uint32_t *>(p.codes) + v * p.row_words,
                                (int)(i - v * p.n_sub), p.code_bits);
        } else {
            c = (int)codes[i];
        }
        c = c < p.N ? c : p.N - 1;
        const float *src = p.codebook + (size_t)c * d;
        if (p.out_is_f32) {
            float *dst = reinterpret_cast<float *>(p.out) + i * d;
            for (int t = 0; t < d; ++t) dst[t] = src[t];
        } else {
            __half *dst = reinterpret_cast<__half *>(p.out) + i * d;
            for (int t = 0; t < d; ++t) dst[t] = __float2half_rn(src[t]);
        }
    }
}

template <int SUBD, typename CodeT>
cudaError_t launch_encode_t(const EncodeParams &p, cudaStream_t stream) {
    const size_t smem = encode_smem_bytes(p.N, SUBD);
    auto kern = encode_kernel<SUBD, CodeT>;
    cudaError_t err = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int dev = 0, sms = 0, per_sm = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount,
                                      dev)) != cudaSuccess)
        return err;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
             &per_sm, kern, kEncThreads, smem)) != cudaSuccess)
        return err;
    if (per_sm < 1) per_sm = 1;
    const int n_sub = p.D / SUBD;
    const int64_t tok = kSlots / n_sub;
    const int64_t n_tiles = (p.n_vec + tok - 1) / tok;
    int64_t grid = (int64_t)sms * per_sm;
    if (grid > n_tiles) grid = n_tiles;
    const float inv_sqrt_d = (float)(1.0 / sqrt((double)p.D));
    kern<<<(unsigned)grid, kEncThreads, smem, stream>>>(p, inv_sqrt_d);
    return cudaGetLastError();
}

template <int SUBD>
cudaError_t launch_encode_c(const EncodeParams &p, cudaStream_t s) {
    if (p.code_bytes == 0) return launch_encode_t<SUBD, uint32_t>(p, s);   // packed rows
    return p.code_bytes == 1 ? launch_encode_t<SUBD, uint8_t>(p, s)
                             : launch_encode_t<SUBD, uint16_t>(p, s);
}

}  // namespace

size_t encode_smem_bytes(int N, int sub_dim) {
    return sizeof(float) * ((((size_t)N * sub_dim + 3) & ~(size_t)3) +
                            (((size_t)N + 3) & ~(size_t)3) + 4 +
                            (size_t)kSlots * sub_dim) +
           sizeof(uint32_t) * 768 +  // packed token rows of a tile (<= 512 / n_sub x words)
           sizeof(float) * 256;      // rotation error bound per token (<= 512 / n_sub tokens)
}

cudaError_t launch_encode(const EncodeParams &p, cudaStream_t stream) {
    if (encode_mma_supported(p.N, p.sub_dim)) return launch_encode_mma(p, stream);
    switch (p.sub_dim) {
        case 1: return launch_encode_c<1>(p, stream);
        case 2: return launch_encode_c<2>(p, stream);
        case 4: return launch_encode_c<4>(p, stream);
        case 8: return launch_encode_c<8>(p, stream);
        case 16: return launch_encode_c<16>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_dequant(const DequantParams &p, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t err;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount,
                                      dev)) != cudaSuccess)
        return err;
    const int threads = 256;
    int64_t blocks = (p.n_vec * p.n_sub + threads - 1) / threads;
    if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
    if (blocks < 1) blocks = 1;
    if (p.code_bytes == 0)
        dequant_kernel<uint32_t><<<(unsigned)blocks, threads, 0, stream>>>(p);
    else if (p.code_bytes == 1)
        dequant_kernel<uint8_t><<<(unsigned)blocks, threads, 0, stream>>>(p);
    else
        dequant_kernel<uint16_t><<<(unsigned)blocks, threads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace vqkv
