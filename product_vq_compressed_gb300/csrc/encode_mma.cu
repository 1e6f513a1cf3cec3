// encode_mma.cu -- key / value encode with the candidate screening on the
// tensor cores (warp-level mma.sync m16n8k16, fp16 operands, fp32 sums).
//
// Same operation as encode.cu (page "Metal Kernels API", section "VecInfer
// kernels": vecinfer_encode_decode_metal, its value-side sibling and
// vecinfer_quantize_metal): y = Hn (s (.) x), code = nearest centroid of
// every sub-vector by squared distance, lowest index on ties, optional
// reconstruction.  The rotation and the search are organised differently.
//
// Rotation.  One warp per token holds the token in registers (D/32
// consecutive elements per lane), applies the butterflies below the lane
// stride locally and the rest with xor-shuffles, in the same stage order as
// the shared-memory transform of encode.cu, so y is bit-identical.
//
// Screening.  For sub-vector y and centroid c, f_c = |c|^2 - 2 y.c orders
// the candidates like |y - c|^2.  It is one matrix product: rows
// [y_hi, y_lo, y_hi, 1, 1] times columns [-2c_hi, -2c_hi, -2c_lo, |c|^2_hi,
// |c|^2_lo], with x_hi = fp16(x) and x_lo = fp16(x - x_hi).  The split keeps
// about 22 bits of each operand; `screen_bound` is a rigorous bound E on
// the difference to the exact f_c.
//
// Selection.  Per row, the four lanes of a quad see disjoint candidates (two
// columns of every 8-centroid n-tile).  A lane keeps only the minimum of
// each block of 64 centroids (its 16 of them, by 3-input min), writes the
// block and its quad position into the low mantissa bits of that minimum
// (moving it by less than 2^tbits ulp, accounted for below), and keeps the
// best and second-best tagged minimum over blocks.  A reduce-scatter over
// the quad leaves each lane the merged pair of one row.
//
// Exact decision.  The lane evaluates the 16 candidates of the winning
// (block, lane) in fp32 in the direct form sum_t (y_t - c_t)^2, in index
// order with strict '<' (lowest index on ties).  Every other candidate has
// exact distance >= (second best, untagged) + |y|^2 - E; unless that bound
// clears the best direct value by the fp32 error margins, the warp rescans
// the whole row in the direct form.  The winner is then certified against
// the rounding of the fp32 rotation and distances (code_certified); a row
// that is not certified is decided again in float-float arithmetic by the
// whole warp (nearest_exact, one or two in 10^4 rows), so a code can differ
// from the exact nearest centroid only where two squared distances agree to
// about 1e-10 relative.
#include <math.h>

#include <type_traits>

#include "vq_internal.cuh"

namespace vqkv {
namespace {

constexpr int kThr = 256;           // 8 warps
constexpr int kSlots = 512;         // sub-vectors per tile (64 per warp)
constexpr int kPassRows = 32;       // rows per warp pass (two 16-row m-tiles)
constexpr int kBlockCols = 64;      // centroids per screening block (8 n-tiles)
constexpr float kU = 5.9604645e-8f;    // 2^-24
constexpr float kU22 = 2.3841858e-7f;  // 2^-22
constexpr float kBigNorm = 30000.f; // screened |c|^2 of padding centroids
constexpr float kFarCoord = 1e18f;  // exact-step coordinates of padding centroids
constexpr float kFarDist = 1e30f;   // direct distances at or above this: padding
constexpr float kRange = 16384.f;   // |value| above which the fp16 split is not used

template <int SUBD>
struct Cfg {
    static constexpr int KCOLS = 3 * SUBD + 2;
    static constexpr int KS = (KCOLS + 15) / 16;   // k-steps of 16
    static constexpr int KW = KS * 8;              // 32-bit words per A row
    static constexpr int AST = KW + 1;             // A row stride in words (odd)
};

// Shared-memory row of centroid n: its low three bits are xor-ed with the
// screening block, so that lanes reading the winners of different blocks in
// the exact step spread over the banks.  A permutation within groups of 8.
__device__ __forceinline__ int cslot(int n) { return n ^ ((n / kBlockCols) & 7); }

__device__ __forceinline__ const float *smooth_row(const EncodeParams &p, int64_t v) {
    const int h = token_head(p, v);
    return p.smooth_mode == 2 ? p.smooth + (size_t)h * p.D : p.smooth;
}

// Token v -> y = (1/sqrt D) H (s (.) x) (keys) or y = x (values), into yv.
// Returns this lane's part of sum_i |fl(x_i s_i)| (keys; 0 for values), the
// size of the rotation's rounding error.
template <int E>
__device__ __forceinline__ float forward_token(const EncodeParams &p, int64_t v, float inv_sqrt_d,
                                               int lane, float *yv) {
    float f[E];
    float asum = 0.f;
    if (v < p.n_vec) {
        load_halves<E>(p.x + v * p.D + lane * E, f);
        if (p.rotate) {
            if (p.smooth_mode != 0) {
                float s[E];
                load_floats<E>(smooth_row(p, v) + lane * E, s);
#pragma unroll
                for (int j = 0; j < E; ++j) f[j] *= s[j];
            }
#pragma unroll
            for (int j = 0; j < E; ++j) {
                asum += fabsf(f[j]);
                f[j] *= inv_sqrt_d;
            }
            reg_fwht<E>(f, lane);
        }
    } else {
#pragma unroll
        for (int j = 0; j < E; ++j) f[j] = 0.f;
    }
    store_floats<E>(yv + lane * E, f);
    return asum;
}

// Chosen centroids in yv -> s^-1 (.) Hn y_hat (keys) or y_hat (values), fp16.
template <int E>
__device__ __forceinline__ void inverse_token(const EncodeParams &p, int64_t v, float inv_sqrt_d,
                                              int lane, const float *yv) {
    float f[E];
    load_floats<E>(yv + lane * E, f);
    if (p.rotate) {
        reg_fwht<E>(f, lane);
#pragma unroll
        for (int j = 0; j < E; ++j) f[j] *= inv_sqrt_d;
        if (p.smooth_mode != 0) {
            float s[E];
            load_floats<E>(smooth_row(p, v) + lane * E, s);
#pragma unroll
            for (int j = 0; j < E; ++j) f[j] /= s[j];
        }
    }
    store_halves<E>(p.xhat + v * p.D + lane * E, f);
}

// ------------------------------------------------------------ screening operands

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint2 b) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y));
}

__device__ __forceinline__ uint32_t pack2(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

__device__ __forceinline__ __half hi_part(float x) { return __float2half_rn(x); }
__device__ __forceinline__ __half lo_part(float x) {
    return __float2half_rn(x - __half2float(__float2half_rn(x)));
}

// Element k of the screening row of sub-vector y (A operand).
template <int SUBD>
__device__ __forceinline__ __half a_val(const float (&y)[SUBD], int k) {
    if (k < SUBD) return hi_part(y[k]);
    if (k < 2 * SUBD) return lo_part(y[k - SUBD]);
    if (k < 3 * SUBD) return hi_part(y[k - 2 * SUBD]);
    if (k < 3 * SUBD + 2) return __float2half_rn(1.f);
    return __float2half_rn(0.f);
}

// Element k of the screening column of centroid c with |c|^2 = n2 (B operand).
template <int SUBD>
__device__ __forceinline__ __half b_val(const float *c, float n2, int k) {
    if (k < SUBD) return __float2half_rn(-2.f * __half2float(hi_part(c[k])));
    if (k < 2 * SUBD) return __float2half_rn(-2.f * __half2float(hi_part(c[k - SUBD])));
    if (k < 3 * SUBD) return __float2half_rn(-2.f * __half2float(lo_part(c[k - 2 * SUBD])));
    if (k == 3 * SUBD) return hi_part(n2);
    if (k == 3 * SUBD + 1) return lo_part(n2);
    return __float2half_rn(0.f);
}

__device__ __forceinline__ float min3f(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ unsigned long long pack_f2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

// sum_t (y_t - c_t)^2 in fp32 with packed two-wide operations: the even and
// the odd dimensions are accumulated separately and added at the end.
// y holds the sub-vector as (y0, y1), (y2, y3), ...
template <int SUBD>
__device__ __forceinline__ float pair_dist(const unsigned long long (&y)[SUBD / 2], const float *cp) {
    float c[SUBD];
    load_floats<SUBD>(cp, c);
    unsigned long long acc = 0ull;
#pragma unroll
    for (int i = 0; i < SUBD / 2; ++i) {
        unsigned long long e;
        asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(e) : "l"(y[i]), "l"(pack_f2(c[2 * i], c[2 * i + 1])));
        if (i == 0)
            asm("mul.rn.f32x2 %0, %1, %1;" : "=l"(acc) : "l"(e));
        else
            asm("fma.rn.f32x2 %0, %1, %1, %2;" : "=l"(acc) : "l"(e), "l"(acc));
    }
    float a0, a1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc));
    return a0 + a1;
}

// (a1 <= a2) and (o1 <= o2), two smallest of disjoint sets -> the two
// smallest of the union (values are distinct: their tags differ)
__device__ __forceinline__ void merge_best2(float &a1, float &a2, float o1, float o2) {
    const float hi = fmaxf(a1, o1);
    a1 = fminf(a1, o1);
    a2 = min3f(hi, a2, o2);
}

// Upper bound on sqrt(x) from the approximate square root (relative error
// far below the 1e-4 added).
__device__ __forceinline__ float sqrt_up(float x) {
    float r;
    asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r * 1.0001f;
}

// Bound on |f~_c - f_c| for every centroid, |y|^2 = ny2, |c|^2 <= maxn2.
// Relative part: split residuals and the dropped y_lo c_lo product (each
// <= 2^-22 of its operand, counted 8 times), fp32 sums of K products
// allowing truncation (2 K u), both over a generous bound on the sum of
// term magnitudes (6 |y||c| + 2 |c|^2).  Absolute part: fp16 subnormal
// spacing (2^-24) in every split, over sum_t |c_t| + |y_t| <= sqrt(SUBD)
// (|y| + |c|), plus the same for the two norm parts.
template <int SUBD>
__device__ __forceinline__ float screen_bound(float ny2, float maxn2, float nc) {
    constexpr int K = Cfg<SUBD>::KS * 16;
    const float ny = sqrt_up(ny2);
    return (2.f * K * kU + 8.f * kU22) * (6.f * ny * nc + 2.f * maxn2) +
           kU22 * (4.f * sqrtf((float)SUBD) * (ny + nc) + 1.f);
}

template <int SUBD>
__device__ __forceinline__ float direct_dist(const float *y, const float *c) {
    float d = 0.f;
#pragma unroll
    for (int t = 0; t < SUBD; ++t) {
        const float e = y[t] - c[t];
        d = fmaf(e, e, d);
    }
    return d;
}

template <int SUBD, typename CodeT>
__global__ void __launch_bounds__(kThr, 3)
encode_mma_kernel(EncodeParams p, float inv_sqrt_d, int npad) {
    using C = Cfg<SUBD>;
    extern __shared__ __align__(16) float smem[];
    const int N = p.N, D = p.D;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // a dependent attention launch may be scheduled now (it waits for this grid)
    pdl_launch_dependents();
    const int g = lane >> 2, c4 = lane & 3;
    // shared memory: fp32 codebook [npad][SUBD] (row cslot(n)) | B fragments [n-tile][k-step]
    // [lane] | sub-vectors [512][SUBD] | per-warp A rows [32][AST] | max |c|^2,
    // codebook-range flag
    const int n_tiles8 = npad / 8;
    float *cb_s = smem;
    uint2 *bfrag = reinterpret_cast<uint2 *>(cb_s + npad * SUBD);
    float *y_s = reinterpret_cast<float *>(bfrag + (size_t)n_tiles8 * C::KS * 32);
    uint32_t *ascr = reinterpret_cast<uint32_t *>(y_s + kSlots * SUBD);
    float *misc = reinterpret_cast<float *>(ascr + (kThr / 32) * kPassRows * C::AST);
    int *bad_cb = reinterpret_cast<int *>(misc + 1);
    // packed codes (CodeT = uint32_t): the tile's token rows, assembled here
    constexpr bool kPacked = std::is_same<CodeT, uint32_t>::value;
    uint32_t *ptile = reinterpret_cast<uint32_t *>(misc + 4);
    // rotation error bound of every token of the tile (<= 128 tokens)
    float *delta_s = reinterpret_cast<float *>(ptile + 768);
    const float dcoef = rotation_delta_coef(p.log2D, inv_sqrt_d);

    if (tid == 0) { misc[0] = 0.f; *bad_cb = 0; }
    for (int i = tid; i < npad * SUBD; i += kThr)
        cb_s[cslot(i / SUBD) * SUBD + i % SUBD] = i < N * SUBD ? p.codebook[i] : kFarCoord;
    __syncthreads();
    for (int n = tid; n < N; n += kThr) {
        float n2 = 0.f;
        bool bad = false;
#pragma unroll
        for (int t = 0; t < SUBD; ++t) {
            const float v = cb_s[cslot(n) * SUBD + t];
            n2 = fmaf(v, v, n2);
            bad |= !(fabsf(v) <= kRange);
        }
        bad |= !(n2 <= kRange);
        // non-negative floats order like their bit patterns
        atomicMax(reinterpret_cast<int *>(&misc[0]), __float_as_int(n2));
        if (bad) atomicOr(bad_cb, 1);
    }
    // B fragments in the order the lanes load them: lane l of n-tile nt holds
    // centroid nt*8 + l/4 at k = 2(l%4) + {0, 1, 8, 9} of each k-step
    for (int i = tid; i < n_tiles8 * C::KS * 32; i += kThr) {
        const int nt = i / (C::KS * 32), rem = i % (C::KS * 32);
        const int ks = rem / 32, l = rem % 32;
        const int n = nt * 8 + (l >> 2), k0 = ks * 16 + 2 * (l & 3);
        const int kk[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
        __half v[4];
        if (n < N) {
            const float *c = cb_s + cslot(n) * SUBD;
            float n2 = 0.f;
#pragma unroll
            for (int t = 0; t < SUBD; ++t) n2 = fmaf(c[t], c[t], n2);
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = b_val<SUBD>(c, n2, kk[j]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = __float2half_rn(kk[j] == 3 * SUBD ? kBigNorm : 0.f);
        }
        bfrag[i] = make_uint2(pack2(v[0], v[1]), pack2(v[2], v[3]));
    }
    __syncthreads();
    const float maxn2 = misc[0];
    const float nc = sqrtf(maxn2) * 1.0001f;
    const bool cb_bad = *bad_cb != 0;
    // tag bits: 2 for the quad lane, the rest for the block index; a tagged
    // value moves by less than 2^tbits ulp, i.e. 2^(tbits - 23) relative
    const int nblk = npad / kBlockCols;
    const int tbits = 2 + (nblk > 1 ? 32 - __clz(nblk - 1) : 0);
    const uint32_t tmask = (1u << tbits) - 1u;
    const float tag_rel = ldexpf(1.f, tbits - 23);

    const int n_sub = D / SUBD;
    const int lsub = p.log2D - (SUBD == 1 ? 0 : SUBD == 2 ? 1 : SUBD == 4 ? 2 : SUBD == 8 ? 3 : 4);
    const int tok = kSlots / n_sub;   // n_sub divides 512
    const int64_t n_tiles = (p.n_vec + tok - 1) / tok;
    CodeT *codes = reinterpret_cast<CodeT *>(p.codes);
    const int64_t lim = p.n_vec * n_sub;
    uint32_t *arow = ascr + warp * kPassRows * C::AST;

    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int64_t v0 = tile * tok;
        // ---- 1. load, smooth, rotate: one warp per token, in registers
        for (int t = warp; t < tok; t += kThr / 32) {
            float *yv = y_s + t * D;
            float asum;
            switch (D) {
                case 32: asum = forward_token<1>(p, v0 + t, inv_sqrt_d, lane, yv); break;
                case 64: asum = forward_token<2>(p, v0 + t, inv_sqrt_d, lane, yv); break;
                case 128: asum = forward_token<4>(p, v0 + t, inv_sqrt_d, lane, yv); break;
                case 256: asum = forward_token<8>(p, v0 + t, inv_sqrt_d, lane, yv); break;
                default: asum = forward_token<16>(p, v0 + t, inv_sqrt_d, lane, yv); break;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) asum += __shfl_xor_sync(0xffffffffu, asum, off);
            if (lane == 0) delta_s[t] = asum * dcoef;
        }
        if constexpr (kPacked) {
            for (int i = tid; i < tok * p.row_words; i += kThr) ptile[i] = 0u;
        }
        __syncthreads();

        // ---- 2. nearest centroids, 64 sub-vectors per warp in two passes
        for (int pass = 0; pass < 2; ++pass) {
            const int R0 = warp * 64 + pass * kPassRows;
            // (a) lane l writes the screening row of sub-vector R0 + l
            {
                float y[SUBD];
#pragma unroll
                for (int t = 0; t < SUBD; ++t) y[t] = y_s[(R0 + lane) * SUBD + t];
#pragma unroll
                for (int w = 0; w < C::KW; ++w)
                    arow[lane * C::AST + w] = pack2(a_val<SUBD>(y, 2 * w), a_val<SUBD>(y, 2 * w + 1));
            }
            __syncwarp();
            uint32_t af[2][C::KS][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) {
                    const uint32_t *r0 = arow + (mt * 16 + g) * C::AST + ks * 8;
                    const uint32_t *r1 = r0 + 8 * C::AST;
                    af[mt][ks][0] = r0[c4];
                    af[mt][ks][1] = r1[c4];
                    af[mt][ks][2] = r0[c4 + 4];
                    af[mt][ks][3] = r1[c4 + 4];
                }
            __syncwarp();
            // (b) screening.  Row q of this lane: m-tile q/2, row g + 8 (q%2).
            //     Block minima carry their (block, lane) tag in the low bits.
            float f1[4], f2[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) { f1[q] = INFINITY; f2[q] = INFINITY; }
            for (int blk = 0; blk < npad / kBlockCols; ++blk) {
                float bm[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
                // software pipeline over the block's n-tiles: B fragments one
                // n-tile ahead, minima of n-tile j taken after n-tile j + 1's MMAs
                constexpr int NTB = kBlockCols / 8;
                const uint2 *bp = bfrag + (size_t)blk * NTB * C::KS * 32 + lane;
                uint2 bf[2][C::KS];
                float acc[2][2][4];
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) bf[0][ks] = bp[ks * 32];
#pragma unroll
                for (int j = 0; j <= NTB; ++j) {
                    if (j < NTB) {
                        if (j + 1 < NTB) {
#pragma unroll
                            for (int ks = 0; ks < C::KS; ++ks)
                                bf[(j + 1) & 1][ks] = bp[((j + 1) * C::KS + ks) * 32];
                        }
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc[j & 1][mt][e] = 0.f;
#pragma unroll
                            for (int ks = 0; ks < C::KS; ++ks)
                                mma16816(acc[j & 1][mt], af[mt][ks], bf[j & 1][ks]);
                        }
                    }
                    if (j > 0) {
                        const int pb = (j - 1) & 1;
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) {
                            bm[2 * mt] = min3f(bm[2 * mt], acc[pb][mt][0], acc[pb][mt][1]);
                            bm[2 * mt + 1] = min3f(bm[2 * mt + 1], acc[pb][mt][2], acc[pb][mt][3]);
                        }
                    }
                }
                const uint32_t tagv = ((uint32_t)blk << 2) | (uint32_t)c4;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float t = __uint_as_float((__float_as_uint(bm[q]) & ~tmask) | tagv);
                    f2[q] = fminf(f2[q], fmaxf(f1[q], t));
                    f1[q] = fminf(f1[q], t);
                }
            }
            // (c) reduce-scatter over the quad: afterwards quad lane c4 holds the
            //     merged best and second best of its row q = c4
            float r1, r2;
            {
                const bool b0 = c4 & 1, b1 = (c4 >> 1) & 1;
                float ka1 = b0 ? f1[1] : f1[0], ka2 = b0 ? f2[1] : f2[0];   // row b0
                float kb1 = b0 ? f1[3] : f1[2], kb2 = b0 ? f2[3] : f2[2];   // row 2 + b0
                const float sa1 = b0 ? f1[0] : f1[1], sa2 = b0 ? f2[0] : f2[1];
                const float sb1 = b0 ? f1[2] : f1[3], sb2 = b0 ? f2[2] : f2[3];
                merge_best2(ka1, ka2, __shfl_xor_sync(0xffffffffu, sa1, 1),
                            __shfl_xor_sync(0xffffffffu, sa2, 1));
                merge_best2(kb1, kb2, __shfl_xor_sync(0xffffffffu, sb1, 1),
                            __shfl_xor_sync(0xffffffffu, sb2, 1));
                r1 = b1 ? kb1 : ka1;
                r2 = b1 ? kb2 : ka2;
                const float t1 = b1 ? ka1 : kb1, t2 = b1 ? ka2 : kb2;
                merge_best2(r1, r2, __shfl_xor_sync(0xffffffffu, t1, 2),
                            __shfl_xor_sync(0xffffffffu, t2, 2));
            }
            // (d) direct-form distances of the winner's kBlockCols / 4 candidates
            //     (its lane's two columns of every n-tile of its block), in
            //     increasing index order, strict '<': lowest index on ties
            const int pr = (c4 >> 1) * 16 + g + (c4 & 1) * 8;   // this lane's row
            const float delta = delta_s[(R0 + pr) >> lsub];
            int code;
            bool amb, cert;
            {
                float y[SUBD];
                load_floats<SUBD>(y_s + (R0 + pr) * SUBD, y);
                unsigned long long y2[SUBD / 2];
#pragma unroll
                for (int i = 0; i < SUBD / 2; ++i) y2[i] = pack_f2(y[2 * i], y[2 * i + 1]);
                const uint32_t tg = __float_as_uint(r1) & tmask;
                const int nb = (int)(tg >> 2) * kBlockCols + 2 * (int)(tg & 3);
                const int sb = cslot(nb);   // slots of nb + 8 j + col: (sb + 8 j) ^ col
                // padding candidates (index >= N) sit at kFarCoord: d >= kFarDist
                float b = INFINITY, b2 = INFINITY;   // best and second best of the group
                int bj = 0;
#pragma unroll
                for (int j = 0; j < kBlockCols / 8; ++j) {
#pragma unroll
                    for (int col = 0; col < 2; ++col) {
                        const float d = pair_dist<SUBD>(y2, cb_s + ((sb + j * 8) ^ col) * SUBD);
                        b2 = fminf(b2, fmaxf(b, d));
                        if (d < b) { b = d; bj = 8 * j + col; }
                    }
                }
                const int bi = nb + bj;
                float ny2 = 0.f;
#pragma unroll
                for (int t = 0; t < SUBD; ++t) ny2 = fmaf(y[t], y[t], ny2);
                // every other candidate: screened value >= untagged r2, exact
                // distance >= that + |y|^2 - E, and its direct form within
                // (SUBD + 3) u of the exact one (ny2 within SUBD u)
                const float E = screen_bound<SUBD>(ny2, maxn2, nc);
                const float outside = r2 + ny2;
                const float margin = E + tag_rel * fabsf(r2) +
                                     (4.f * SUBD + 8.f) * kU * (fabsf(outside) + b + ny2 + maxn2);
                const bool live = v0 * n_sub + R0 + pr < lim;
                amb = live && (cb_bad || !(ny2 <= kRange * kRange) || !(b < kFarDist) ||
                               !(outside - b > margin));
                code = bi;
                // lower bound on every other candidate's exact distance to y~:
                // the group's second best, and the screen's bound for the
                // other groups (its own rounding and that of |y|^2 included)
                const float out_lb = outside - (E + tag_rel * fabsf(r2) +
                                                 (float)(SUBD + 8) * kU * (fabsf(r2) + ny2));
                cert = !live || amb || code_certified<SUBD>(b, fminf(b2, out_lb), delta);
                // only the screen's bound is too loose: the direct rescan below
                // gives every candidate's fp32 distance, then certify again
                if (!cert && code_certified<SUBD>(b, b2, delta)) {
                    amb = true;
                    cert = true;
                }
            }
            // (e) ambiguous rows: the whole warp rescans the row in the direct form
            {
                unsigned m = __ballot_sync(0xffffffffu, amb);
                while (m) {
                    const int src = __ffs(m) - 1;
                    m &= m - 1;
                    const int sc = src & 3;
                    const int spr = (sc >> 1) * 16 + (src >> 2) + (sc & 1) * 8;
                    const float *yr = y_s + (R0 + spr) * SUBD;
                    float best = INFINITY, second = INFINITY;
                    int bi = 0x7fffffff;
                    for (int n = lane; n < N; n += 32) {
                        const float d = direct_dist<SUBD>(yr, cb_s + cslot(n) * SUBD);
                        second = fminf(second, fmaxf(best, d));
                        if (d < best) { best = d; bi = n; }
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const float ob = __shfl_xor_sync(0xffffffffu, best, off);
                        const float os = __shfl_xor_sync(0xffffffffu, second, off);
                        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                        second = fminf(fminf(second, os), fmaxf(best, ob));
                        if (ob < best || (ob == best && oi < bi)) { best = ob; bi = oi; }
                    }
                    if (lane == src) {
                        code = bi == 0x7fffffff ? 0 : bi;
                        cert = code_certified<SUBD>(best, second, delta);
                    }
                }
            }
            // (e') rows the fp32 arithmetic cannot certify: float-float, whole warp
            {
                unsigned m = __ballot_sync(0xffffffffu, !cert);
                while (m) {
                    const int src = __ffs(m) - 1;
                    m &= m - 1;
                    const int sc = src & 3;
                    const int sl = R0 + (sc >> 1) * 16 + (src >> 2) + (sc & 1) * 8;
                    const int cx = nearest_exact_token<SUBD>(
                        p, v0 + (sl >> lsub), sl & (n_sub - 1),
                        [cb_s](int c, int t) { return cb_s[cslot(c) * SUBD + t]; },
                        delta_s[sl >> lsub], lane);
                    if (lane == src) code = cx;
                }
            }
            // (f) lane l takes the code of row l (held by quad lane q of quad
            //     l % 8): coalesced store; the chosen centroid replaces the
            //     sub-vector for the reconstruction
            const int mine = __shfl_sync(0xffffffffu, code,
                                         (lane & 7) * 4 + (((lane >> 4) << 1) | ((lane >> 3) & 1)));
            const int64_t gi = v0 * n_sub + R0 + lane;
            if (gi < lim) {
                if constexpr (kPacked)
                    packed_or(ptile + ((R0 + lane) >> lsub) * p.row_words, (R0 + lane) & (n_sub - 1),
                              p.code_bits, (uint32_t)mine);
                else
                    codes[code_index(p, gi >> lsub, n_sub, (int)(gi & (n_sub - 1)))] = (CodeT)mine;
            }
            __syncwarp();
            if (p.xhat) {
#pragma unroll
                for (int t = 0; t < SUBD; ++t)
                    y_s[(R0 + lane) * SUBD + t] = cb_s[cslot(mine) * SUBD + t];
            }
        }
        __syncthreads();
        if constexpr (kPacked) {   // the tile's packed token rows -> the cache
            uint32_t *cw = reinterpret_cast<uint32_t *>(p.codes);
            for (int i = tid; i < tok * p.row_words; i += kThr) {
                const int t = i / p.row_words, w = i - t * p.row_words;
                if (v0 + t < p.n_vec) cw[token_row(p, v0 + t) * p.row_words + w] = ptile[i];
            }
        }

        // ---- 3. optional reconstruction -> fp16
        if (p.xhat) {
            for (int t = warp; t < tok; t += kThr / 32) {
                const int64_t v = v0 + t;
                if (v >= p.n_vec) continue;   // warp-uniform
                const float *yv = y_s + t * D;
                switch (D) {
                    case 32: inverse_token<1>(p, v, inv_sqrt_d, lane, yv); break;
                    case 64: inverse_token<2>(p, v, inv_sqrt_d, lane, yv); break;
                    case 128: inverse_token<4>(p, v, inv_sqrt_d, lane, yv); break;
                    case 256: inverse_token<8>(p, v, inv_sqrt_d, lane, yv); break;
                    default: inverse_token<16>(p, v, inv_sqrt_d, lane, yv); break;
                }
            }
        }
        __syncthreads();
    }
}

template <int SUBD>
size_t mma_smem_bytes(int npad) {
    using C = Cfg<SUBD>;
    return sizeof(float) * (size_t)npad * SUBD + sizeof(uint2) * (size_t)(npad / 8) * C::KS * 32 +
           sizeof(float) * (size_t)kSlots * SUBD +
           sizeof(uint32_t) * (size_t)(kThr / 32) * kPassRows * C::AST + 16 +
           sizeof(uint32_t) * 768 +  // packed token rows of a tile (<= 512 / n_sub x words)
           sizeof(float) * 128;      // rotation error bound per token (<= 512 / n_sub tokens)
}

template <int SUBD, typename CodeT>
cudaError_t launch_t(const EncodeParams &p, cudaStream_t stream) {
    const int npad = (p.N + kBlockCols - 1) & ~(kBlockCols - 1);
    const size_t smem = mma_smem_bytes<SUBD>(npad);
    auto kern = encode_mma_kernel<SUBD, CodeT>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int dev = 0, sms = 0, per_sm = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return err;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThr, smem)) !=
        cudaSuccess)
        return err;
    if (per_sm < 1) per_sm = 1;
    const int n_sub = p.D / SUBD;
    const int64_t tok = kSlots / n_sub;
    const int64_t n_tiles = (p.n_vec + tok - 1) / tok;
    int64_t grid = (int64_t)sms * per_sm;
    if (grid > n_tiles) grid = n_tiles;
    const float inv_sqrt_d = (float)(1.0 / sqrt((double)p.D));
    kern<<<(unsigned)grid, kThr, smem, stream>>>(p, inv_sqrt_d, npad);
    return cudaGetLastError();
}

template <int SUBD>
cudaError_t launch_c(const EncodeParams &p, cudaStream_t s) {
    if (p.code_bytes == 0) return launch_t<SUBD, uint32_t>(p, s);   // packed rows
    return p.code_bytes == 1 ? launch_t<SUBD, uint8_t>(p, s) : launch_t<SUBD, uint16_t>(p, s);
}

}  // namespace

bool encode_mma_supported(int N, int sub_dim) {
    const int npad = (N + kBlockCols - 1) & ~(kBlockCols - 1);
    size_t bytes = 0;
    switch (sub_dim) {
        case 2: bytes = mma_smem_bytes<2>(npad); break;
        case 4: bytes = mma_smem_bytes<4>(npad); break;
        case 8: bytes = mma_smem_bytes<8>(npad); break;
        default: return false;
    }
    return bytes <= 200u * 1024u;
}

cudaError_t launch_encode_mma(const EncodeParams &p, cudaStream_t stream) {
    switch (p.sub_dim) {
        case 2: return launch_c<2>(p, stream);
        case 4: return launch_c<4>(p, stream);
        case 8: return launch_c<8>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace vqkv
