// decode.cu -- attention over the coded cache, split along the key axis
// (flash-decoding) with a combine pass.
//
// Page: "Metal Kernels API", section "Fused SDPA", metal_fused_sdpa (key
// dequant + scaled QK^T + softmax + weighted value sum in one pass, equal to
// SDPA on the dequantised K_hat; causal alignment to the tail of the cache;
// sliding window; H_q a multiple of H_kv), with the raw-query semantics of
// VecInferKVCache.fused_sdpa ("veloxquant_mlx.cache.vecinfer_cache module"):
// the dual transform q~ = Hn (q (.) s^-1) happens here, so q~ . K~^T =
// q . K_hat^T with K~ = dequant(codes) in the rotated domain.
//
// GB300 design
//   * Work item = (b, kv head g, column block, key split).  A column is one
//     (query head of the GQA group, query row) pair; up to 8 columns share
//     one pass over the codes, so one code fetch serves every query head of
//     the group.  The kernel is persistent: each CTA stages the codebooks
//     once and loops over items.
//   * Both codebooks live in shared memory as fp16, replicated so that every
//     copy sits in its own bank group (128 bytes per centroid row, lane l
//     reads copy l mod C): the random per-lane gathers are conflict-free.
//   * Scores and the value sum run on warp-level tensor-core MMA
//     (m16n8k16, fp16 x fp16 -> fp32) in "swap-AB" form: S^T[16 keys x 8
//     cols] = K~[16 x D] . Q~^T and O^T[D x 8] += V_hat^T[D x 16] . P^T.
//     The fragment registers are filled straight from the gathers; head
//     dimensions are permuted (consistently on both operands) so that one
//     gather of a whole sub-vector lands in one lane's fragment.  P moves
//     from accumulator to operand layout with movmatrix.trans.
//   * Online softmax in base 2 (scale * log2 e applied to the fp32 scores),
//     per column; masks only on tiles that need them; fully masked tiles are
//     skipped by clipping each item's key range.
//   * Each CTA merges its warps and writes one partial (m, l, o[D]) per
//     column; the combine kernel merges the splits and writes fp16.
#include <climits>
#include <math.h>

#include "vq_internal.cuh"

namespace vqkv {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kCols = 8;        // columns per item (MMA N)
constexpr int kTile = 16;       // keys per MMA tile
constexpr int kStepTiles = 2;   // tiles per softmax step
constexpr int kStep = kTile * kStepTiles;
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------ primitives

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n"
                 : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Streaming read-only loads of NB bytes (NB a power of two, naturally
// aligned) into 32-bit words.
template <int NB>
__device__ __forceinline__ void load_bytes(const uint8_t *p, uint32_t *w) {
    if constexpr (NB >= 16) {
#pragma unroll
        for (int i = 0; i < NB / 16; ++i) {
            uint4 v;
            asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "l"(p + 16 * i));
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
    } else if constexpr (NB == 8) {
        uint2 v;
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];\n"
                     : "=r"(v.x), "=r"(v.y) : "l"(p));
        w[0] = v.x; w[1] = v.y;
    } else if constexpr (NB == 4) {
        uint32_t v;
        asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];\n" : "=r"(v) : "l"(p));
        w[0] = v;
    } else if constexpr (NB == 2) {
        unsigned short v;
        asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];\n" : "=h"(v) : "l"(p));
        w[0] = v;
    } else {
        unsigned short v;
        asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];\n" : "=h"(v) : "l"(p));
        w[0] = v & 0xFFu;
    }
}

// n codes of `cb` bytes each starting at p, as 32-bit words (room for 2 bytes
// per code).
template <int NC>
__device__ __forceinline__ void load_codes(const uint8_t *p, int cb, uint32_t *w) {
    if (cb == 1) load_bytes<NC>(p, w);
    else load_bytes<NC * 2>(p, w);
}

template <int NC>
__device__ __forceinline__ uint32_t code_at(const uint32_t *w, int cb, int i) {
    // i is a compile-time constant after unrolling
    return cb == 1 ? ((w[i >> 2] >> ((i & 3) * 8)) & 0xFFu)
                   : ((w[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu);
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Gather one fp16 centroid of SUB dims (2*SUB bytes) into words.
template <int SUB>
__device__ __forceinline__ void gather(uint32_t addr, uint32_t *w) {
    if constexpr (SUB == 2) {
        w[0] = lds32(addr);
    } else if constexpr (SUB == 4) {
        const uint2 v = lds64(addr);
        w[0] = v.x; w[1] = v.y;
    } else {
        const uint4 v = lds128(addr);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    }
}

// ------------------------------------------------------------- the kernel

struct DecArgs {
    int B, H_q, H_kv, S_q, S_kv, G;
    const __half *q;
    const uint8_t *kc;
    int kcb;
    const float *kcbk;
    int Nk;
    const uint8_t *vc;
    int vcb;
    const float *vcbk;
    int Nv;
    const float *smooth;
    int smooth_mode;
    float sl;          // scale * log2(e)
    float inv_sqrt_d;
    int causal, window;
    float *ws;         // partials [item][kCols][D + 4]
    int n_split, n_colblk, tiles_per_split;
    int64_t n_items;
    int k_copies, v_copies;   // replicas per codebook row
};

template <int D>
struct Smem {
    // codebook tables follow this struct in dynamic shared memory
    float qt[kCols][D];                 // transformed queries (fp32)
    float o[kWarps][kCols][D];          // per-warp partial outputs
    float m[kWarps][kCols];
    float l[kWarps][kCols];
    int lo[kCols], hi[kCols];           // visible key range per column
};

template <int D, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
decode_kernel(DecArgs a) {
    constexpr int KSTEPS = D / 16;      // k-steps of the QK MMA
    constexpr int MT = D / 16;          // M tiles of the PV MMA
    constexpr int NKL = D / (4 * DK);   // key codes per lane and key
    constexpr int NVL = D / (8 * DV);   // value codes per lane and key
    constexpr int EK = 2 * DK, EV = 2 * DV;
    constexpr int KW = (NKL * 2 + 3) / 4;   // words for NKL codes (<= 2 bytes)
    constexpr int VW = (NVL * 2 + 3) / 4;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem<D> &sm = *reinterpret_cast<Smem<D> *>(smem_raw);
    unsigned char *ktab = smem_raw + sizeof(Smem<D>);
    const int krow = a.k_copies * EK;               // bytes per centroid row
    unsigned char *vtab = ktab + (size_t)a.Nk * krow;
    const int vrow = a.v_copies * EV;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, c4 = lane & 3;

    // ---- stage both codebooks as fp16, replicated per bank group
    for (int i = tid; i < a.Nk * (krow / 4); i += kThreads) {
        const int c = i / (krow / 4), wi = i % (krow / 4);
        const int t = ((wi * 4) % EK) / 2;
        reinterpret_cast<uint32_t *>(ktab)[i] =
            pack_h2(a.kcbk[c * DK + t], a.kcbk[c * DK + t + 1]);
    }
    for (int i = tid; i < a.Nv * (vrow / 4); i += kThreads) {
        const int c = i / (vrow / 4), wi = i % (vrow / 4);
        const int t = ((wi * 4) % EV) / 2;
        reinterpret_cast<uint32_t *>(vtab)[i] =
            pack_h2(a.vcbk[c * DV + t], a.vcbk[c * DV + t + 1]);
    }
    const uint32_t kbase = (uint32_t)__cvta_generic_to_shared(ktab) +
                           (uint32_t)((lane % a.k_copies) * EK);
    const uint32_t vbase = (uint32_t)__cvta_generic_to_shared(vtab) +
                           (uint32_t)((lane % a.v_copies) * EV);
    const int64_t k_tok_bytes = (int64_t)(D / DK) * a.kcb;
    const int64_t v_tok_bytes = (int64_t)(D / DV) * a.vcb;
    const int n_cols_total = a.G * a.S_q;

    for (int64_t item = blockIdx.x; item < a.n_items; item += gridDim.x) {
        const int split = (int)(item % a.n_split);
        const int64_t rest = item / a.n_split;
        const int cblk = (int)(rest % a.n_colblk);
        const int64_t bg = rest / a.n_colblk;
        const int b = (int)(bg / a.H_kv), g = (int)(bg % a.H_kv);

        __syncthreads();  // previous item finished with the smem scratch
        // ---- transformed queries: q~ = Hn (q (.) s_g^-1), one warp per column
        for (int col = warp; col < kCols; col += kWarps) {
            const int cg = cblk * kCols + col;
            float *qv = sm.qt[col];
            if (cg < n_cols_total) {
                const int i = cg / a.G, gam = cg % a.G;
                const int hq = g * a.G + gam;
                const __half *qp = a.q + (((int64_t)b * a.H_q + hq) * a.S_q + i) * D;
                const float *sp = a.smooth_mode == 2 ? a.smooth + (size_t)g * D : a.smooth;
                for (int e = lane; e < D; e += 32) {
                    float v = __half2float(qp[e]);
                    if (a.smooth_mode != 0) v = v / sp[e];
                    qv[e] = v * a.inv_sqrt_d;
                }
                __syncwarp();
                for (int h = 1; h < D; h <<= 1) {
                    for (int p = lane; p < D / 2; p += 32) {
                        const int x = ((p & ~(h - 1)) << 1) | (p & (h - 1));
                        const float u = qv[x], w = qv[x + h];
                        qv[x] = u + w;
                        qv[x + h] = u - w;
                    }
                    __syncwarp();
                }
                if (lane == 0) {
                    const int q_abs = a.S_kv - a.S_q + i;
                    int hi = a.causal ? q_abs : a.S_kv - 1;
                    if (hi > a.S_kv - 1) hi = a.S_kv - 1;
                    int lo = a.window > 0 ? q_abs - a.window + 1 : 0;
                    if (lo < 0) lo = 0;
                    sm.lo[col] = lo;
                    sm.hi[col] = hi;
                }
            } else {
                for (int e = lane; e < D; e += 32) qv[e] = 0.f;
                if (lane == 0) { sm.lo[col] = 1; sm.hi[col] = 0; }  // empty
            }
        }
        __syncthreads();

        // ---- query B fragments (fp16), dims permuted to match the gathers
        uint32_t bq[KSTEPS][2];
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
            const float *qv = sm.qt[g8] + c4 * (D / 4) + 4 * ks;
            bq[ks][0] = pack_h2(qv[0], qv[1]);
            bq[ks][1] = pack_h2(qv[2], qv[3]);
        }
        // per-lane column bounds (lane owns columns 2*c4, 2*c4+1)
        const int lo0 = sm.lo[2 * c4], hi0 = sm.hi[2 * c4];
        const int lo1 = sm.lo[2 * c4 + 1], hi1 = sm.hi[2 * c4 + 1];
        int lo_all = INT_MAX, hi_all = -1, lo_any = INT_MAX, hi_any = -1;
        bool any_real = false;
#pragma unroll
        for (int col = 0; col < kCols; ++col) {
            const int l = sm.lo[col], h = sm.hi[col];
            if (l > h) continue;     // padding / empty column
            any_real = true;
            lo_all = min(lo_all, l); hi_all = max(hi_all, h);   // union
            lo_any = lo_any == INT_MAX ? l : max(lo_any, l);     // intersection
            hi_any = hi_any == -1 ? h : min(hi_any, h);
        }
        // this item's key range, clipped to what any column can see
        const int t_begin = split * a.tiles_per_split * kTile;
        int t_end = t_begin + a.tiles_per_split * kTile;
        if (t_end > a.S_kv) t_end = a.S_kv;
        const int r_begin = max(t_begin, any_real ? (lo_all & ~(kTile - 1)) : t_end);
        const int r_end = min(t_end, any_real ? hi_all + 1 : t_begin);
        // keys every real column sees inside [t_begin, t_end)
        const int full_lo = max(t_begin, any_real ? lo_any : INT_MAX);
        const int full_hi = min(t_end - 1, hi_any);
        // per-lane bounds, restricted to this split
        const int lo0s = max(lo0, t_begin), hi0s = min(hi0, t_end - 1);
        const int lo1s = max(lo1, t_begin), hi1s = min(hi1, t_end - 1);

        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        float acc_o[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            acc_o[mt][0] = acc_o[mt][1] = acc_o[mt][2] = acc_o[mt][3] = 0.f;

        const uint8_t *kbase_g = a.kc + (int64_t)bg * a.S_kv * k_tok_bytes;
        const uint8_t *vbase_g = a.vc + (int64_t)bg * a.S_kv * v_tok_bytes;

        for (int s0 = r_begin + warp * kStep; s0 < r_end; s0 += kWarps * kStep) {
            // ---- codes of this step: keys g8 and g8+8 of each tile (K),
            //      keys 2c4, 2c4+1, 2c4+8, 2c4+9 of each tile (V)
            uint32_t kw[kStepTiles][2][KW];
            uint32_t vw[kStepTiles][4][VW];
#pragma unroll
            for (int t = 0; t < kStepTiles; ++t) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    int j = s0 + t * kTile + g8 + 8 * r;
                    j = min(j, a.S_kv - 1);
                    load_codes<NKL>(kbase_g + (int64_t)j * k_tok_bytes +
                                        (int64_t)c4 * NKL * a.kcb,
                                    a.kcb, kw[t][r]);
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    int j = s0 + t * kTile + 2 * c4 + (r & 1) + 8 * (r >> 1);
                    j = min(j, a.S_kv - 1);
                    load_codes<NVL>(vbase_g + (int64_t)j * v_tok_bytes +
                                        (int64_t)g8 * NVL * a.vcb,
                                    a.vcb, vw[t][r]);
                }
            }
            // ---- S^T = K~ Q~^T for both tiles
            float sc[kStepTiles][4];
#pragma unroll
            for (int t = 0; t < kStepTiles; ++t) {
                sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
                uint32_t af[2][KSTEPS][2];  // [row][kstep][lo/hi word]
#pragma unroll
                for (int r = 0; r < 2; ++r) {
#pragma unroll
                    for (int u = 0; u < NKL; ++u) {
                        const uint32_t code =
                            min(code_at<NKL>(kw[t][r], a.kcb, u), (uint32_t)(a.Nk - 1));
                        uint32_t w[4];
                        gather<DK>(kbase + code * (uint32_t)krow, w);
                        if constexpr (DK == 2) {
                            af[r][u >> 1][u & 1] = w[0];
                        } else if constexpr (DK == 4) {
                            af[r][u][0] = w[0];
                            af[r][u][1] = w[1];
                        } else {
                            af[r][2 * u][0] = w[0];
                            af[r][2 * u][1] = w[1];
                            af[r][2 * u + 1][0] = w[2];
                            af[r][2 * u + 1][1] = w[3];
                        }
                    }
                }
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks)
                    mma16816(sc[t], af[0][ks][0], af[1][ks][0], af[0][ks][1],
                             af[1][ks][1], bq[ks][0], bq[ks][1]);
            }
            // ---- scale, mask, online softmax (columns 2c4 and 2c4+1)
            const bool need_mask = !(s0 >= full_lo && s0 + kStep - 1 <= full_hi);
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int t = 0; t < kStepTiles; ++t) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float v = sc[t][e] * a.sl;
                    if (need_mask) {
                        const int j = s0 + t * kTile + g8 + 8 * (e >> 1);
                        const bool ok = (e & 1) ? (j >= lo1s && j <= hi1s)
                                                : (j >= lo0s && j <= hi0s);
                        v = ok ? v : -INFINITY;
                    }
                    sc[t][e] = v;
                }
                mx0 = fmaxf(mx0, fmaxf(sc[t][0], sc[t][2]));
                mx1 = fmaxf(mx1, fmaxf(sc[t][1], sc[t][3]));
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
            const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
            m0 = mn0;
            m1 = mn1;
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
                l0 *= al0;
                l1 *= al1;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    acc_o[mt][0] *= al0; acc_o[mt][2] *= al0;
                    acc_o[mt][1] *= al1; acc_o[mt][3] *= al1;
                }
            }
            uint32_t bp[kStepTiles][2];
#pragma unroll
            for (int t = 0; t < kStepTiles; ++t) {
                const float p0 = exp2f(sc[t][0] - mu0), p1 = exp2f(sc[t][1] - mu1);
                const float p2 = exp2f(sc[t][2] - mu0), p3 = exp2f(sc[t][3] - mu1);
                l0 += p0 + p2;
                l1 += p1 + p3;
                bp[t][0] = movmatrix_t(pack_h2(p0, p1));
                bp[t][1] = movmatrix_t(pack_h2(p2, p3));
            }
            // ---- O^T += V^T P^T
#pragma unroll
            for (int t = 0; t < kStepTiles; ++t) {
                // W[r][word]: value words of keys (2c4, 2c4+1, 2c4+8, 2c4+9)
                constexpr int WPL = D / 16;   // 32-bit words per lane and key
                uint32_t vwrd[4][WPL];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
#pragma unroll
                    for (int u = 0; u < NVL; ++u) {
                        const uint32_t code =
                            min(code_at<NVL>(vw[t][r], a.vcb, u), (uint32_t)(a.Nv - 1));
                        gather<DV>(vbase + code * (uint32_t)vrow, &vwrd[r][u * (DV / 2)]);
                    }
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const uint32_t a0 = __byte_perm(vwrd[0][mt], vwrd[1][mt], 0x5410);
                    const uint32_t a1 = __byte_perm(vwrd[0][mt], vwrd[1][mt], 0x7632);
                    const uint32_t a2 = __byte_perm(vwrd[2][mt], vwrd[3][mt], 0x5410);
                    const uint32_t a3 = __byte_perm(vwrd[2][mt], vwrd[3][mt], 0x7632);
                    mma16816(acc_o[mt], a0, a1, a2, a3, bp[t][0], bp[t][1]);
                }
            }
        }

        // ---- merge the warps of this CTA and write the item's partial
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        if (g8 == 0) {
            sm.m[warp][2 * c4] = m0; sm.m[warp][2 * c4 + 1] = m1;
            sm.l[warp][2 * c4] = l0; sm.l[warp][2 * c4 + 1] = l1;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int d0 = g8 * (D / 8) + 2 * mt;
            sm.o[warp][2 * c4][d0] = acc_o[mt][0];
            sm.o[warp][2 * c4 + 1][d0] = acc_o[mt][1];
            sm.o[warp][2 * c4][d0 + 1] = acc_o[mt][2];
            sm.o[warp][2 * c4 + 1][d0 + 1] = acc_o[mt][3];
        }
        __syncthreads();
        float *out = a.ws + item * (int64_t)kCols * (D + 4);
        for (int idx = tid; idx < kCols * (D + 1); idx += kThreads) {
            const int col = idx / (D + 1), d = idx % (D + 1);
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.m[w][col]);
            const float Mu = M == -INFINITY ? 0.f : M;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = exp2f(sm.m[w][col] - Mu);
                acc += f * (d < D ? sm.o[w][col][d] : sm.l[w][col]);
            }
            float *rec = out + col * (D + 4);
            if (d < D) rec[4 + d] = acc;
            else { rec[0] = M; rec[1] = acc; }
        }
    }
}

// Merge the splits of every (b, kv head, column block) and write fp16.
template <int D>
__global__ void __launch_bounds__(D)
combine_kernel(const float *__restrict__ ws, int n_split, int n_colblk, int H_kv,
               int H_q, int S_q, int G, __half *__restrict__ out) {
    const int64_t unit = blockIdx.x;      // (bg, cblk)
    const int col = blockIdx.y;
    const int cblk = (int)(unit % n_colblk);
    const int64_t bg = unit / n_colblk;
    const int cg = cblk * kCols + col;
    if (cg >= G * S_q) return;
    const int b = (int)(bg / H_kv), g = (int)(bg % H_kv);
    const int i = cg / G, gam = cg % G;
    const int d = threadIdx.x;
    const float *base = ws + (unit * n_split) * (int64_t)kCols * (D + 4) + col * (D + 4);
    const int64_t stride = (int64_t)kCols * (D + 4);
    float M = -INFINITY;
    for (int s = 0; s < n_split; ++s) M = fmaxf(M, base[s * stride]);
    float o = 0.f, l = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < n_split; ++s) {
            const float f = exp2f(base[s * stride] - M);
            l += f * base[s * stride + 1];
            o += f * base[s * stride + 4 + d];
        }
        o = l > 0.f ? o / l : 0.f;
    }
    const int hq = g * G + gam;
    out[(((int64_t)b * H_q + hq) * S_q + i) * D + d] = __float2half_rn(o);
}

int pow2_floor(int v) {
    int p = 1;
    while (p * 2 <= v) p *= 2;
    return p;
}

struct Tables {
    int k_copies, v_copies;
    size_t bytes;
};

constexpr size_t kSmemBudget = 200 * 1024;

template <int D>
size_t smem_struct() { return sizeof(Smem<D>); }

size_t smem_struct_d(int D) {
    switch (D) {
        case 32: return smem_struct<32>();
        case 64: return smem_struct<64>();
        case 128: return smem_struct<128>();
        default: return smem_struct<256>();
    }
}

// Largest replica counts (powers of two, <= 128 bytes per row) that fit.
Tables choose_tables(const vq_attend_args &a) {
    const int ek = 2 * a.k_sub_dim, ev = 2 * a.v_sub_dim;
    int kc = 128 / ek, vc = 128 / ev;
    const size_t base = smem_struct_d(a.D);
    auto total = [&](int k, int v) {
        return base + (size_t)a.k_n_centroids * k * ek +
               (size_t)a.v_n_centroids * v * ev;
    };
    while (total(kc, vc) > kSmemBudget && (kc > 1 || vc > 1)) {
        if ((size_t)a.k_n_centroids * kc * ek >= (size_t)a.v_n_centroids * vc * ev && kc > 1)
            kc /= 2;
        else if (vc > 1)
            vc /= 2;
        else
            kc /= 2;
    }
    return {kc, vc, total(kc, vc)};
}

template <int D, int DK, int DV>
cudaError_t launch_t(const DecArgs &da, const Tables &tb, int grid,
                     cudaStream_t stream) {
    auto kern = decode_kernel<D, DK, DV>;
    cudaError_t err = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tb.bytes);
    if (err != cudaSuccess) return err;
    kern<<<grid, kThreads, tb.bytes, stream>>>(da);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecArgs &da, int dk, int dv, const Tables &tb,
                     int grid, cudaStream_t s) {
#define VQ_CASE(K, V)                                                  \
    if (dk == K && dv == V) {                                          \
        if constexpr (K <= D / 4 && V <= D / 8)                        \
            return launch_t<D, K, V>(da, tb, grid, s);                 \
        else                                                           \
            return cudaErrorInvalidValue;                              \
    }
    VQ_CASE(2, 2) VQ_CASE(4, 4) VQ_CASE(8, 8) VQ_CASE(8, 4) VQ_CASE(4, 8)
    VQ_CASE(4, 2) VQ_CASE(2, 4)
#undef VQ_CASE
    return cudaErrorInvalidValue;
}

bool pair_ok(int D, int dk, int dv) {
    const bool listed = (dk == 2 && dv == 2) || (dk == 4 && dv == 4) ||
                        (dk == 8 && dv == 8) || (dk == 8 && dv == 4) ||
                        (dk == 4 && dv == 8) || (dk == 4 && dv == 2) ||
                        (dk == 2 && dv == 4);
    return listed && dk <= D / 4 && dv <= D / 8;
}

int blocks_per_sm_estimate(size_t smem) {
    int b = (int)(227 * 1024 / (smem + 1024));
    if (b > 8) b = 8;
    return b < 1 ? 1 : b;
}

}  // namespace

int decode_supported(const vq_attend_args &a) {
    if (a.D != 32 && a.D != 64 && a.D != 128 && a.D != 256) return VQ_ERR_UNSUPPORTED;
    if (!pair_ok(a.D, a.k_sub_dim, a.v_sub_dim)) return VQ_ERR_UNSUPPORTED;
    const Tables tb = choose_tables(a);
    if (tb.bytes > kSmemBudget) return VQ_ERR_UNSUPPORTED;
    return VQ_OK;
}

size_t decode_smem_bytes(const vq_attend_args &a) { return choose_tables(a).bytes; }

AttendPlan plan_decode(const vq_attend_args &a, int num_sms) {
    AttendPlan p{};
    p.cols = kCols;
    const int ncols = (a.H_q / a.H_kv) * a.S_q;
    p.n_colblk = (ncols + kCols - 1) / kCols;
    const int64_t units = (int64_t)a.B * a.H_kv * p.n_colblk;
    const int64_t tiles = (a.S_kv + kTile - 1) / kTile;
    const int64_t slots = (int64_t)num_sms * blocks_per_sm_estimate(choose_tables(a).bytes);
    // pick the split count minimising (waves * tiles per split) + a per-item
    // overhead, i.e. balance the persistent CTAs without too many partials
    int best_n = 1;
    double best_cost = 1e300;
    const int max_split = (int)((tiles + 7) / 8);   // >= 128 keys per split
    for (int n = 1; n <= 256 && n <= (max_split < 1 ? 1 : max_split); ++n) {
        const int64_t items = units * n;
        const int64_t waves = (items + slots - 1) / slots;
        const int64_t tps = (tiles + n - 1) / n;
        const double cost = (double)waves * (double)(tps + 6);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best_n = n;
        }
    }
    p.n_split = best_n;
    p.tok_per_split = (int)(((tiles + best_n - 1) / best_n) * kTile);
    p.ws_bytes = (size_t)units * best_n * kCols * (a.D + 4) * sizeof(float);
    return p;
}

AttendPlan plan_decode_capped(const vq_attend_args &a, int num_sms,
                              size_t max_ws_bytes) {
    AttendPlan p = plan_decode(a, num_sms);
    if (p.ws_bytes <= max_ws_bytes) return p;
    // fewer key splits until the partial results fit the given capacity
    const int64_t units = (int64_t)a.B * a.H_kv * p.n_colblk;
    const size_t per_split = (size_t)units * kCols * (a.D + 4) * sizeof(float);
    const int64_t tiles = (a.S_kv + kTile - 1) / kTile;
    const int64_t fit = per_split ? (int64_t)(max_ws_bytes / per_split) : 0;
    if (fit < 1) {
        p.n_split = 0;
        p.ws_bytes = per_split;   // what one split alone would need
        return p;
    }
    const int n = (int)(fit < p.n_split ? fit : p.n_split);
    p.n_split = n;
    p.tok_per_split = (int)(((tiles + n - 1) / n) * kTile);
    p.ws_bytes = per_split * (size_t)n;
    return p;
}

cudaError_t launch_decode(const vq_attend_args &a, const AttendPlan &plan,
                          cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t err;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) !=
        cudaSuccess)
        return err;
    const Tables tb = choose_tables(a);
    DecArgs da{};
    da.B = a.B; da.H_q = a.H_q; da.H_kv = a.H_kv; da.S_q = a.S_q; da.S_kv = a.S_kv;
    da.G = a.H_q / a.H_kv;
    da.q = reinterpret_cast<const __half *>(a.q_f16);
    da.kc = reinterpret_cast<const uint8_t *>(a.k_codes);
    da.kcb = a.k_code_bytes;
    da.kcbk = a.k_codebook;
    da.Nk = a.k_n_centroids;
    da.vc = reinterpret_cast<const uint8_t *>(a.v_codes);
    da.vcb = a.v_code_bytes;
    da.vcbk = a.v_codebook;
    da.Nv = a.v_n_centroids;
    da.smooth = a.smooth;
    da.smooth_mode = a.smooth_mode;
    da.sl = a.scale * kLog2e;
    da.inv_sqrt_d = (float)(1.0 / sqrt((double)a.D));
    da.causal = a.causal;
    da.window = a.sliding_window;
    da.ws = reinterpret_cast<float *>(a.workspace);
    da.n_split = plan.n_split;
    da.n_colblk = plan.n_colblk;
    da.tiles_per_split = plan.tok_per_split / kTile;
    da.n_items = (int64_t)a.B * a.H_kv * plan.n_colblk * plan.n_split;
    da.k_copies = tb.k_copies;
    da.v_copies = tb.v_copies;
    int per_sm = 1;
    int64_t grid = 0;
    {
        // occupancy of the instantiated kernel decides the persistent grid
        per_sm = blocks_per_sm_estimate(tb.bytes);
        grid = (int64_t)sms * per_sm;
        if (grid > da.n_items) grid = da.n_items;
        if (grid < 1) grid = 1;
    }
    switch (a.D) {
        case 32: err = launch_d<32>(da, a.k_sub_dim, a.v_sub_dim, tb, (int)grid, stream); break;
        case 64: err = launch_d<64>(da, a.k_sub_dim, a.v_sub_dim, tb, (int)grid, stream); break;
        case 128: err = launch_d<128>(da, a.k_sub_dim, a.v_sub_dim, tb, (int)grid, stream); break;
        case 256: err = launch_d<256>(da, a.k_sub_dim, a.v_sub_dim, tb, (int)grid, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (err != cudaSuccess) return err;
    const int64_t units = (int64_t)a.B * a.H_kv * plan.n_colblk;
    dim3 cgrid((unsigned)units, kCols);
    switch (a.D) {
        case 32: combine_kernel<32><<<cgrid, 32, 0, stream>>>(da.ws, plan.n_split, plan.n_colblk, a.H_kv, a.H_q, a.S_q, da.G, reinterpret_cast<__half *>(a.out_f16)); break;
        case 64: combine_kernel<64><<<cgrid, 64, 0, stream>>>(da.ws, plan.n_split, plan.n_colblk, a.H_kv, a.H_q, a.S_q, da.G, reinterpret_cast<__half *>(a.out_f16)); break;
        case 128: combine_kernel<128><<<cgrid, 128, 0, stream>>>(da.ws, plan.n_split, plan.n_colblk, a.H_kv, a.H_q, a.S_q, da.G, reinterpret_cast<__half *>(a.out_f16)); break;
        default: combine_kernel<256><<<cgrid, 256, 0, stream>>>(da.ws, plan.n_split, plan.n_colblk, a.H_kv, a.H_q, a.S_q, da.G, reinterpret_cast<__half *>(a.out_f16)); break;
    }
    return cudaGetLastError();
}

}  // namespace vqkv
