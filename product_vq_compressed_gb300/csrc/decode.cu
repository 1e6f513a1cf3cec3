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
//   * A unit is (b, kv head g, column block); a column is one (query head of
//     the GQA group, query row) pair, and up to 8 columns share one pass over
//     the codes, so one code fetch serves every query head of the group.
//     The (unit, 16-key tile) space is cut into equal contiguous shares, one
//     per warp of a persistent grid of one CTA per SM; each warp writes one
//     partial (m, l, o[D]) per unit it touched and per column, and the
//     combine kernel merges them and writes fp16.
//   * Both codebooks live in shared memory as fp16, replicated so that every
//     copy sits in its own bank group (lane l reads copy l mod C): the random
//     per-lane gathers are conflict-free.
//   * Codes: uint8 code rows of 16-byte multiples arrive through a per-warp
//     ring of shared-memory stages filled by cp.async.bulk (mbarrier per
//     stage, bounded waits); 10-bit packed keys of 8 dimensions have their
//     own mode; other widths are read through the read-only cache.
//   * Scores and the value sum run on warp-level tensor-core MMA
//     (m16n8k16, fp16 x fp16 -> fp32) in "swap-AB" form: S^T[16 keys x 8
//     cols] = K~[16 x D] . Q~^T and O^T[D x 8] += V_hat^T[D x 16] . P^T.
//     The fragment registers are filled straight from the gathers; head
//     dimensions are permuted (consistently on both operands) so that one
//     gather of a whole sub-vector lands in one lane's fragment.  P moves
//     from accumulator to operand layout with movmatrix.trans.
//   * Online softmax in base 2 (scale * log2 e folded into q~), per column,
//     with a reference maximum that moves only past 2^8; masks only at the
//     edges of a segment; keys no column can see are clipped away.
//   * The decode step (STEP instantiation, one cooperative launch): the new
//     tokens' encode beside the attention, per-row flags for the new code
//     rows, a grid sync and the merge of the key splits in the kernel.
#include <atomic>
#include <chrono>
#include <climits>
#include <cooperative_groups.h>
#include <math.h>

#include "vq_internal.cuh"

namespace vqkv {
namespace {

// Warps of the one CTA per SM: 12 (up to 168 registers each) for D <= 128,
// 8 for D = 256, whose accumulators need more registers per thread.
__host__ __device__ constexpr int warps_for(int D) { return D >= 256 ? 8 : 12; }
constexpr int kCols = 8;         // query columns per unit (MMA N)
constexpr int kTile = 16;        // keys per MMA tile
constexpr int kPrefetchTiles = 8;  // L2 prefetch distance
constexpr int kPfKeys = 2 * kTile * 2;  // keys per prefetch: two steps of two tiles
constexpr double kLog2e = 1.4426950408889634;
constexpr float kSlack = 8.f;    // base-2 headroom of a column's reference maximum

// ------------------------------------------------------------ primitives

// The shared-memory gathers, products and transposes below are plain asm
// (not volatile): they only read registers and the codebook tables, which
// do not change after the block's set-up barrier, so the compiler may
// schedule them freely (e.g. a tile's value gathers ahead of its softmax).
// Global loads of codes stay volatile: they must not move above the
// dependent-launch wait.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n"
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
// Codes of `cb` bytes each (1, 2), or bit-packed rows when cb = -bits: then
// the run keeps the address of its code row (packed codes are read where
// they are used; row-relative code index = run0 + i).
template <int NC>
__device__ __forceinline__ void load_codes(const uint8_t *p, int cb, uint32_t *w) {
    if (cb < 0) {
        const uint64_t a = reinterpret_cast<uint64_t>(p);
        w[0] = (uint32_t)a;
        w[1] = (uint32_t)(a >> 32);
    } else if (cb == 1) {
        load_bytes<NC>(p, w);
    } else {
        load_bytes<NC * 2>(p, w);
    }
}

template <int NC>
__device__ __forceinline__ uint32_t code_at(const uint32_t *w, int cb, int run0, int i) {
    if (cb < 0) {
        const uint32_t *row = reinterpret_cast<const uint32_t *>(
            (uint64_t)w[0] | ((uint64_t)w[1] << 32));
        const int bits = -cb, bit = (run0 + i) * bits, wi = bit >> 5, sh = bit & 31;
        uint64_t x = __ldg(row + wi);
        if (sh + bits > 32) x |= (uint64_t)__ldg(row + wi + 1) << 32;
        return (uint32_t)(x >> sh) & ((1u << bits) - 1u);
    }
    // i is a compile-time constant after unrolling
    return cb == 1 ? ((w[i >> 2] >> ((i & 3) * 8)) & 0xFFu)
                   : ((w[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu);
}

// ---- kernel modes: generic (runtime code widths, tables of any size), fast
// (uint8 codes, at most 256 centroids, one interleaved table at 64 KiB) and
// packed (keys as bit-packed rows of kPackedBits-bit codes, values uint8;
// both tables zero-padded to all 2^bits / 256 rows, one 128-byte row of
// replicas per centroid)
constexpr int kModeGeneric = 0, kModeFast = 1, kModePacked = 2;
constexpr int kPackedBits = 10;
constexpr uint32_t kPkRow = 128;   // bytes per centroid row of the packed-mode tables

// largest bit offset inside its first word of the four lanes' runs
__host__ __device__ constexpr int max_run_shift(int run) {
    int m = 0;
    for (int c = 0; c < 4; ++c) m = ((c * run) & 31) > m ? ((c * run) & 31) : m;
    return m;
}

// Run of NC packed codes of lane c4 (codes [c4 NC, c4 NC + NC) of the row):
// bits [c4 NC b, (c4 + 1) NC b) of the little-endian row of 32-bit words,
// read as the two words holding them and shifted down to bit 0 of w[0].
template <int NC>
__device__ __forceinline__ void load_packed_run(const uint8_t *row, int c4, uint32_t *w) {
    constexpr int RUN = NC * kPackedBits;
    constexpr int ROW_WORDS = (4 * RUN + 31) / 32;
    static_assert(RUN + max_run_shift(RUN) <= 64, "a lane's run must lie in two consecutive words");
    static_assert(((3 * RUN) >> 5) + 1 < ROW_WORDS, "the second word must lie in the row");
    const int b0 = c4 * RUN;
    const uint32_t *p = reinterpret_cast<const uint32_t *>(row) + (b0 >> 5);
    uint32_t x0, x1;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];\n" : "=r"(x0) : "l"(p));
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];\n" : "=r"(x1) : "l"(p + 1));
    const int sh = b0 & 31;
    w[0] = __funnelshift_r(x0, x1, sh);
    w[1] = x1 >> sh;
}

// Code i of a run loaded by load_packed_run (i is a constant once the
// caller's loop is unrolled, so one shift or funnel shift and a mask).
__device__ __forceinline__ uint32_t packed_code(const uint32_t *w, int i) {
    const int b = i * kPackedBits;
    uint32_t x;
    if (b + kPackedBits <= 32) x = w[0] >> b;
    else if (b >= 32) x = w[1] >> (b - 32);
    else x = __funnelshift_r(w[0], w[1], b);
    return x & ((1u << kPackedBits) - 1u);
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
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

// Fast-path gathers: uint8 codes and one interleaved table of 256 rows x 256
// bytes placed at shared-memory address 65536 -- row c holds the key
// centroid c replicas in bytes [0, 128) and the value centroid c replicas in
// [128, 256).  The shared address of the row for code byte i of word w plus
// the lane's replica offset (< 256) is then a single byte permute:
// bytes (off, code, 1, 0) = 65536 + code * 256 + off.
// i is a constant once the caller's loop is unrolled.
constexpr uint32_t kFastTabAddr = 65536;
__device__ __forceinline__ uint32_t row_off(uint32_t w, int i, uint32_t lane_off) {
    return __byte_perm(w, lane_off | (1u << 16), 0x7604u | ((uint32_t)i << 4));
}

template <int SUB>
__device__ __forceinline__ void gather_sh(uint32_t addr, uint32_t *w) {
    if constexpr (SUB == 2) {
        asm("ld.shared.u32 %0, [%1];\n" : "=r"(w[0]) : "r"(addr));
    } else if constexpr (SUB == 4) {
        asm("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(w[0]), "=r"(w[1]) : "r"(addr));
    } else {
        asm("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
            : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
    }
}

constexpr uint32_t kFastRow = 256;                 // bytes per interleaved row

// 16 bytes of fp16 copies of the centroid at c (SUB fp32 values): words
// (c0 c1), (c2 c3), ... repeated to fill the chunk.
template <int SUB>
__device__ __forceinline__ uint4 replica_chunk(const float *c) {
    if constexpr (SUB == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(c);
        const uint32_t w = pack_h2(v.x, v.y);
        return make_uint4(w, w, w, w);
    } else if constexpr (SUB == 4) {
        const float4 v = *reinterpret_cast<const float4 *>(c);
        const uint32_t w0 = pack_h2(v.x, v.y), w1 = pack_h2(v.z, v.w);
        return make_uint4(w0, w1, w0, w1);
    } else {
        const float4 v = *reinterpret_cast<const float4 *>(c);
        const float4 u = *reinterpret_cast<const float4 *>(c + 4);
        return make_uint4(pack_h2(v.x, v.y), pack_h2(v.z, v.w), pack_h2(u.x, u.y), pack_h2(u.z, u.w));
    }
}

__host__ __device__ __forceinline__ size_t align16(size_t v) { return (v + 15) & ~(size_t)15; }

// ------------------------------------------------------------- the kernel

struct DecArgs {
    int B, H_q, H_kv, S_q, S_kv, G;
    const __half *q;
    const uint8_t *kc;
    int kcb;           // code bytes (1, 2) or -bits of packed rows
    int krowb, vrowb;  // bytes per key / value code row
    const float *kcbk;
    int Nk;
    const uint8_t *vc;
    int vcb;
    const float *vcbk;
    int Nv;
    const float *smooth;
    int smooth_mode;
    float qscale;      // 1/sqrt(D) * scale * log2(e): applied to q~ (base-2 scores)
    int causal, window;
    int64_t stride;        // code rows per (b, kv head)
    const int32_t *kv_lens;  // keys held by each batch, or null (all S_kv)
    float *ws;         // partial records [nw][slots][kCols][D + 4]
    int n_colblk;
    int tlo, T;        // every unit scans key tiles [tlo, tlo + T)
    int64_t total;     // units * T, the flattened work
    int64_t share;     // tiles per warp (the last shares may be shorter or empty)
    int nw;            // warps sharing the work
    int slots;         // partial records per warp
    int k_copies, v_copies;
    // one decode step in one cooperative launch (vq_decode_step): encode the
    // new tokens into cache rows new_row0 .. beside the attention over the
    // rows before them, attend over the new rows once their codes are
    // written, grid sync, merge the key splits
    int step;
    const __half *k_new, *v_new;   // [B, H_kv, S_q, D]
    int new_row0;
    // per (new token, K / V): step_epoch once its code row is written (in
    // the workspace; set back to 0 after the final grid sync)
    unsigned long long *step_flags;
    unsigned long long step_epoch;   // odd, never 0
    int log2D;
    __half *out;
};

// Record of warp w for unit `unit`, column col: the warps whose shares
// overlap the unit's tiles [unit T, unit T + T) each hold one, in the slot
// of that unit among the units their share touches.
__device__ __forceinline__ float *unit_record(const DecArgs &a, int64_t unit, int64_t w, int col,
                                              int D) {
    const int64_t u0 = unit * a.T;
    const int64_t s = w * a.share;
    const int64_t slot = a.share <= a.T ? (s >= u0 ? 0 : 1) : unit - s / a.T;
    return a.ws + ((w * a.slots + slot) * kCols + col) * (int64_t)(D + 4);
}
__device__ __forceinline__ void unit_warps(const DecArgs &a, int64_t unit, int64_t *w_lo,
                                           int *n_rec) {
    const int64_t u0 = unit * a.T;
    *w_lo = u0 / a.share;
    int64_t w_hi = (u0 + a.T - 1) / a.share;
    if (w_hi > a.nw - 1) w_hi = a.nw - 1;
    *n_rec = (int)(w_hi - *w_lo + 1);
}

// Warp gw's contiguous share of the flattened (unit, tile) space is
// [gw * share, min((gw + 1) * share, total)).
__host__ __device__ __forceinline__ int64_t share_start(int64_t gw, int64_t share,
                                                         int64_t total) {
    const int64_t s = gw * share;
    return s < total ? s : total;
}

template <int D>
struct WarpScratch {
    __half qt[kCols][D];      // transformed queries (fp16 MMA operands)
    int lo[kCols], hi[kCols]; // visible key range per column
};

constexpr int kStepTiles = 2;                 // tiles per softmax step
constexpr int kStepKeys = kTile * kStepTiles;  // 32 keys

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// Codes of one step held in registers: for tile t, key rows g8 and g8 + 8
// (K side) and keys 2c4, 2c4+1, 2c4+8, 2c4+9 (V side), each the lane's
// contiguous run of sub-vector codes.
template <int D, int DK, int DV>
struct StepCodes {
    static constexpr int NKL = D / (4 * DK);
    static constexpr int NVL = D / (8 * DV);
    // room for 2-byte codes, or for a packed code row's address
    static constexpr int KW = (NKL * 2 + 3) / 4 > 2 ? (NKL * 2 + 3) / 4 : 2;
    static constexpr int VW = (NVL * 2 + 3) / 4 > 2 ? (NVL * 2 + 3) / 4 : 2;
    uint32_t k[kStepTiles][2][KW];
    uint32_t v[kStepTiles][4][VW];
};

// Row offsets (in keys) of the lane's K and V code rows inside a tile.
__device__ __forceinline__ int krow_of(int g8, int r) { return g8 + 8 * r; }
__device__ __forceinline__ int vrow_of(int c4, int r) { return 2 * c4 + (r & 1) + 8 * (r >> 1); }

template <int D, int DK, int DV, int MODE>
__device__ __forceinline__ void load_step(StepCodes<D, DK, DV> &sc, const uint8_t *kl,
                                          const uint8_t *vl, int j0, const DecArgs &a,
                                          int64_t ktb_rt, int64_t vtb_rt, int g8, int c4) {
    using SC = StepCodes<D, DK, DV>;
    constexpr bool FAST = MODE == kModeFast, PACKED = MODE == kModePacked;
    // uint8 codes (fast path; values of the packed path) and packed key rows:
    // strides are compile-time constants
    const int64_t ktb = FAST ? (int64_t)(D / DK)
                        : PACKED ? (int64_t)(4 * ((D / DK * kPackedBits + 31) / 32)) : ktb_rt;
    const int64_t vtb = FAST || PACKED ? (int64_t)(D / DV) : vtb_rt;
    auto ld_k = [&](const uint8_t *p, uint32_t *w) {
        if constexpr (FAST) load_bytes<SC::NKL>(p, w);
        else if constexpr (PACKED) load_packed_run<SC::NKL>(p, c4, w);
        else load_codes<SC::NKL>(p, a.kcb, w);
    };
    auto ld_v = [&](const uint8_t *p, uint32_t *w) {
        if constexpr (FAST || PACKED) load_bytes<SC::NVL>(p, w);
        else load_codes<SC::NVL>(p, a.vcb, w);
    };
    if (j0 + kStepKeys <= a.S_kv) {
        // one base address per step; the rows are constant offsets from it
        const uint8_t *kb = kl + (int64_t)j0 * ktb;
        const uint8_t *vb = vl + (int64_t)j0 * vtb;
#pragma unroll
        for (int t = 0; t < kStepTiles; ++t) {
#pragma unroll
            for (int r = 0; r < 2; ++r) ld_k(kb + (t * kTile + 8 * r) * ktb, sc.k[t][r]);
#pragma unroll
            for (int r = 0; r < 4; ++r)
                ld_v(vb + (t * kTile + (r & 1) + 8 * (r >> 1)) * vtb, sc.v[t][r]);
        }
    } else {  // tail of the cache: clamp rows past the last key (masked later)
#pragma unroll
        for (int t = 0; t < kStepTiles; ++t) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int j = min(j0 + t * kTile + krow_of(g8, r), a.S_kv - 1) - krow_of(g8, 0);
                ld_k(kl + (int64_t)j * ktb, sc.k[t][r]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int j = min(j0 + t * kTile + vrow_of(c4, r), a.S_kv - 1) - vrow_of(c4, 0);
                ld_v(vl + (int64_t)j * vtb, sc.v[t][r]);
            }
        }
    }
}

__device__ __forceinline__ void prefetch_l2(const uint8_t *p, uint32_t bytes) {
    if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0 && (bytes & 15u) == 0 && bytes)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes)
                     : "memory");
}

// ---- per-warp ring of code stages (uint8 code rows of 16-byte multiples)
// Lane 0 of every warp streams the K and V code rows of its next steps into
// a ring of stages in shared memory with bulk copies (cp.async.bulk, one per
// operand and step, completing on the stage's mbarrier), kRingAhead steps
// ahead of the warp; the lanes read a step's codes from its stage just
// before the step.  Tile row r of a step holds key perm_row(r), which makes
// both the key-code reads (lane rows g, g + 8) and the value-code reads
// (lane rows 2c, 2c + 1, 2c + 8, 2c + 9) of 32-byte rows bank-conflict-free.
template <int D, int DK, int DV>
struct RingCfg {
    static constexpr int KROW = D / DK, VROW = D / DV;   // code bytes per key
    static constexpr bool on = KROW % 16 == 0 && VROW % 16 == 0;
    static constexpr int STAGE = kStepKeys * (KROW + VROW);
};
constexpr uint32_t kRingAddr = 131072;        // shared address of the rings (after the table)
constexpr uint32_t kSmemLimit = 232448;       // 227 KiB of dynamic shared memory per block
constexpr uint32_t kRingPolls = 1u << 22;     // bound of every stage wait

__host__ __device__ constexpr int ring_stages(int stage_bytes, int warps) {
    return (int)((kSmemLimit - kRingAddr) / (uint32_t)(stage_bytes * warps)) > 4
               ? 4
               : (int)((kSmemLimit - kRingAddr) / (uint32_t)(stage_bytes * warps));
}

__device__ __forceinline__ int perm_row(int r) { return r ^ ((r >> 2) & 1); }

__device__ __forceinline__ void ring_bar_init(uint32_t bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void ring_expect(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n"
                 ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void ring_copy(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// bounded wait for phase `parity` of a stage's mbarrier: false if it expired
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kRingPolls; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n"
            " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}
// NB bytes of shared memory at addr (after the stage's wait: volatile)
template <int NB>
__device__ __forceinline__ void lds_bytes(uint32_t addr, uint32_t *w) {
    if constexpr (NB == 16) {
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr) : "memory");
    } else if constexpr (NB == 8) {
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(w[0]), "=r"(w[1]) : "r"(addr) : "memory");
    } else if constexpr (NB == 4) {
        asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(w[0]) : "r"(addr) : "memory");
    } else {
        unsigned short v;
        asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(addr) : "memory");
        w[0] = v;
    }
}

// A step's codes from its stage: K rows perm_row(g8) (+ 8) of each tile,
// codes [c4 NKL, c4 NKL + NKL); V rows perm_row(vrow_of(c4, r)), codes
// [g8 NVL, g8 NVL + NVL).
template <int D, int DK, int DV>
__device__ __forceinline__ void load_step_ring(StepCodes<D, DK, DV> &sc, uint32_t st, int g8,
                                               int c4) {
    using SC = StepCodes<D, DK, DV>;
    using R = RingCfg<D, DK, DV>;
    const int pk = perm_row(g8);
#pragma unroll
    for (int t = 0; t < kStepTiles; ++t) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
            lds_bytes<SC::NKL>(st + (uint32_t)((t * kTile + pk + 8 * r) * R::KROW + c4 * SC::NKL),
                               sc.k[t][r]);
#pragma unroll
        for (int r = 0; r < 4; ++r)
            lds_bytes<SC::NVL>(st + (uint32_t)(kStepKeys * R::KROW +
                                               (t * kTile + perm_row(vrow_of(c4, r))) * R::VROW +
                                               g8 * SC::NVL),
                               sc.v[t][r]);
    }
}

// The tiles of a warp's share that belong to one unit, and the keys its
// steps cover: [j_first, j_last), clipped to the keys some query row of
// batch b can see, [max(0, L - S_q - W + 1), L - 1] (no lower bound without
// a window), so ragged caches read no codes past a batch's length.
struct SegInfo {
    int64_t unit, seg_end, bg;
    int b, g, cblk, kv_len, j_first, j_last;
};
__device__ __forceinline__ SegInfo segment_at(const DecArgs &a, int64_t t, int64_t t_end) {
    SegInfo sg;
    sg.unit = t / a.T;
    sg.seg_end = min(t_end, (sg.unit + 1) * (int64_t)a.T);
    sg.cblk = (int)(sg.unit % a.n_colblk);
    sg.bg = sg.unit / a.n_colblk;
    sg.g = (int)(sg.bg % a.H_kv);
    sg.b = (int)(sg.bg / a.H_kv);
    // keys held by batch b (clamped to the cache)
    sg.kv_len = a.kv_lens ? min(max(a.kv_lens[sg.b], 0), a.S_kv) : a.S_kv;
    const int vis_lo = a.window > 0 ? max(0, sg.kv_len - a.S_q - a.window + 1) : 0;
    const int vis_end = (sg.kv_len + kTile - 1) / kTile * kTile;
    sg.j_first = max((int)((a.tlo + (t - sg.unit * (int64_t)a.T)) * kTile), vis_lo / kTile * kTile);
    sg.j_last = min((int)((a.tlo + (sg.seg_end - sg.unit * (int64_t)a.T)) * kTile),
                    vis_end);  // exclusive
    return sg;
}

// Per-warp state of one unit (batch, kv head, column block).
template <int D>
struct UnitState {
    uint32_t bq[D / 16][2];
    float acc_o[D / 16][4];
    float m0, m1, l0, l1;
    float mu0, mu1;             // exponent reference of the lane's two columns
    int lo0, hi0, lo1, hi1;     // bounds of the lane's two columns
    int lo_any, hi_any;         // keys every real column sees
    int lo_all, hi_all;         // keys some column sees
};

// Gather of code u (a compile-time index after unrolling) of a code run.
// KEY: the run holds key codes (bit-packed on the packed path).
template <int DKV, int NC, int MODE, bool KEY>
__device__ __forceinline__ void gather_code(const uint32_t *words, int u, const DecArgs &a,
                                            int cb, int N, uint32_t base, int row,
                                            const unsigned char *tab, uint32_t lane_off,
                                            uint32_t *w, int run0 = 0) {
    if constexpr (MODE == kModeFast) {
        gather_sh<DKV>(row_off(words[u >> 2], u & 3, lane_off), w);
    } else if constexpr (MODE == kModePacked) {
        // tables padded to every representable code: no clamp
        const uint32_t code = KEY ? packed_code(words, u) : (words[u >> 2] >> ((u & 3) * 8)) & 0xFFu;
        gather_sh<DKV>(base + code * kPkRow, w);
    } else {
        const uint32_t code = min(code_at<NC>(words, cb, run0, u), (uint32_t)(N - 1));
        gather<DKV>(base + code * (uint32_t)row, w);
    }
}

// One 32-key step.  MASK: the step needs the per-column key bounds (the
// first and last steps of a segment); the steps between take the unmasked
// instantiation, in which every real column sees every key.
template <int D, int DK, int DV, int MODE, bool MASK, bool PERM>
__device__ __forceinline__ void process_step(const StepCodes<D, DK, DV> &sc, int j0,
                                             UnitState<D> &u, const DecArgs &a,
                                             uint32_t kbase, uint32_t vbase, int krow,
                                             int vrow, int g8, int c4,
                                             const unsigned char *tabs, uint32_t klane,
                                             uint32_t vlane) {
    using SC = StepCodes<D, DK, DV>;
    constexpr int KSTEPS = D / 16, MT = D / 16;
    if (MASK && (j0 > u.hi_all || j0 + kStepKeys - 1 < u.lo_all)) return;  // nobody sees it

    // ---- S^T = K~ Q~^T for both tiles; even / odd k-steps accumulate
    //      separately so the four MMA chains are independent
    float s[kStepTiles][2][4];
#pragma unroll
    for (int t = 0; t < kStepTiles; ++t)
#pragma unroll
        for (int h = 0; h < 2; ++h) s[t][h][0] = s[t][h][1] = s[t][h][2] = s[t][h][3] = 0.f;
    uint32_t w8[kStepTiles][2][4];   // DK == 8: one gather serves two k-steps
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
        uint32_t f[kStepTiles][2][2];
#pragma unroll
        for (int t = 0; t < kStepTiles; ++t) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if constexpr (DK == 4) {
                    uint32_t w[2];
                    gather_code<4, SC::NKL, MODE, true>(sc.k[t][r], ks, a, a.kcb, a.Nk, kbase, krow,
                                                  tabs, klane, w, c4 * SC::NKL);
                    f[t][r][0] = w[0];
                    f[t][r][1] = w[1];
                } else if constexpr (DK == 2) {
                    gather_code<2, SC::NKL, MODE, true>(sc.k[t][r], 2 * ks, a, a.kcb, a.Nk, kbase,
                                                  krow, tabs, klane, &f[t][r][0], c4 * SC::NKL);
                    gather_code<2, SC::NKL, MODE, true>(sc.k[t][r], 2 * ks + 1, a, a.kcb, a.Nk, kbase,
                                                  krow, tabs, klane, &f[t][r][1], c4 * SC::NKL);
                } else {
                    if ((ks & 1) == 0)
                        gather_code<8, SC::NKL, MODE, true>(sc.k[t][r], ks >> 1, a, a.kcb, a.Nk,
                                                      kbase, krow, tabs, klane, w8[t][r],
                                                      c4 * SC::NKL);
                    f[t][r][0] = w8[t][r][2 * (ks & 1)];
                    f[t][r][1] = w8[t][r][2 * (ks & 1) + 1];
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kStepTiles; ++t)
            mma16816(s[t][ks & 1], f[t][0][0], f[t][1][0], f[t][0][1], f[t][1][1], u.bq[ks][0],
                     u.bq[ks][1]);
    }
    // ---- mask, online softmax for columns 2c4 and 2c4+1 (the scores are
    //      already scaled by scale * log2 e, folded into q~)
    float sc4[kStepTiles][4];
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int t = 0; t < kStepTiles; ++t) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float v = s[t][0][e] + s[t][1][e];
            if constexpr (MASK) {
                // S row g8 (+ 8) of tile t holds key perm_row(g8) (+ 8) of
                // a ring stage, key g8 (+ 8) otherwise
                const int j = j0 + t * kTile + (PERM ? perm_row(g8) : g8) + 8 * (e >> 1);
                const bool ok = (e & 1) ? (j >= u.lo1 && j <= u.hi1) : (j >= u.lo0 && j <= u.hi0);
                v = ok ? v : -INFINITY;
            }
            sc4[t][e] = v;
        }
        mx0 = fmaxf(mx0, fmaxf(sc4[t][0], sc4[t][2]));
        mx1 = fmaxf(mx1, fmaxf(sc4[t][1], sc4[t][3]));
    }
    // The reference maximum m of a column moves only when some score exceeds
    // it by more than kSlack (base 2): then the column's lanes agree on the
    // new maximum and rescale.  Otherwise p = 2^(s - m) <= 2^kSlack, which
    // fp16 holds at full relative precision; o / l does not depend on m.
    if (__any_sync(0xffffffffu, mx0 > u.m0 + kSlack || mx1 > u.m1 + kSlack)) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(u.m0, mx0), mn1 = fmaxf(u.m1, mx1);
        const float al0 = mn0 == -INFINITY ? 1.f : ex2(u.m0 - mn0);
        const float al1 = mn1 == -INFINITY ? 1.f : ex2(u.m1 - mn1);
        u.l0 *= al0;
        u.l1 *= al1;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            u.acc_o[mt][0] *= al0; u.acc_o[mt][2] *= al0;
            u.acc_o[mt][1] *= al1; u.acc_o[mt][3] *= al1;
        }
        u.m0 = mn0;
        u.m1 = mn1;
        // the exponent reference: m, or 0 while a column has seen no key
        u.mu0 = mn0 == -INFINITY ? 0.f : mn0;
        u.mu1 = mn1 == -INFINITY ? 0.f : mn1;
    }
    uint32_t bp[kStepTiles][2];
#pragma unroll
    for (int t = 0; t < kStepTiles; ++t) {
        const float p0 = ex2(sc4[t][0] - u.mu0), p1 = ex2(sc4[t][1] - u.mu1);
        const float p2 = ex2(sc4[t][2] - u.mu0), p3 = ex2(sc4[t][3] - u.mu1);
        u.l0 += p0 + p2;
        u.l1 += p1 + p3;
        bp[t][0] = movmatrix_t(pack_h2(p0, p1));
        bp[t][1] = movmatrix_t(pack_h2(p2, p3));
    }
    // ---- O^T += V_hat^T P^T, tile by tile
    constexpr int WPL = D / 16;   // 32-bit value words per lane and key
#pragma unroll
    for (int t = 0; t < kStepTiles; ++t) {
        uint32_t vw[4][WPL];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int uu = 0; uu < SC::NVL; ++uu)
                gather_code<DV, SC::NVL, MODE, false>(sc.v[t][r], uu, a, a.vcb, a.Nv, vbase, vrow,
                                               tabs, vlane, &vw[r][uu * (DV / 2)],
                                               g8 * SC::NVL);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const uint32_t a0 = __byte_perm(vw[0][mt], vw[1][mt], 0x5410);
            const uint32_t a1 = __byte_perm(vw[0][mt], vw[1][mt], 0x7632);
            const uint32_t a2 = __byte_perm(vw[2][mt], vw[3][mt], 0x5410);
            const uint32_t a3 = __byte_perm(vw[2][mt], vw[3][mt], 0x7632);
            mma16816(u.acc_o[mt], a0, a1, a2, a3, bp[t][0], bp[t][1]);
        }
    }
}

// A decode step's new code rows: written by the encoding warps, announced by
// a release store of the launch's epoch per (token, K / V); a warp that
// copies a new row first waits (bounded) for both flags of every new token
// of its (batch, KV head).  The launch is cooperative, so the encoding CTAs
// are resident while others wait.
constexpr uint32_t kFlagWaitLimit = 1u << 22;   // x ~64 ns: ~0.3 s
__device__ __forceinline__ void flag_release(unsigned long long *f, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;\n" ::"l"(f), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long flag_acquire(const unsigned long long *f) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(f) : "memory");
    return v;
}
// One lane: false when a flag was not set within the limit.
__device__ __forceinline__ bool wait_new_rows(const unsigned long long *flags,
                                              unsigned long long epoch, int64_t bg, int S_q) {
    for (int i = 0; i < 2 * S_q; ++i) {
        const unsigned long long *f = flags + 2 * bg * S_q + i;
        uint32_t it = 0;
        while (flag_acquire(f) != epoch) {
            if (++it > kFlagWaitLimit) return false;
            __nanosleep(64);
        }
    }
    return true;
}

// Encode of one new token by a group of NW warps, D = 32 E with sub-vectors
// of E dimensions (lane m owns sub-vector m), into its 32-byte uint8 code row
// (cb: the fp32 codebook, staged in shared memory by the caller): the same
// definition and decision rule as the encode kernels -- smooth and
// Walsh-Hadamard rotation (keys), nearest centroid by the direct-form fp32
// distance to every centroid, lowest index on ties, kept when the rounding
// certificate holds and decided again in float-float otherwise.  Warp `part`
// of the group scans centroids [part N / NW, (part + 1) N / NW) and leaves
// its best, second-best and index per lane in its exchange area (3 x 32
// words at xch + part * xstride); after the group's named barrier `bar_id`
// the group's first warp
// combines them in part order (so an equal distance keeps the lower index),
// takes the decision and writes the row.
template <int E, int NW>
__device__ void encode_token_group(const __half *x, const float *sm, int rotate, const float *cb,
                                   int N, uint8_t *dst, int log2D, int lane, int part,
                                   float *xch, int xstride, int bar_id) {
    const float inv_sqrt_d = 1.f / sqrtf((float)(32 * E));
    float f[E];
    load_halves<E>(x + lane * E, f);
    float asum = 0.f;
    if (rotate) {
        if (sm) {
            float sv[E];
            load_floats<E>(sm + lane * E, sv);
#pragma unroll
            for (int j = 0; j < E; ++j) f[j] *= sv[j];
        }
#pragma unroll
        for (int j = 0; j < E; ++j) {
            asum += fabsf(f[j]);
            f[j] *= inv_sqrt_d;
        }
        reg_fwht<E>(f, lane);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) asum += __shfl_xor_sync(0xffffffffu, asum, off);
    const float delta = rotate ? asum * rotation_delta_coef(log2D, inv_sqrt_d) : 0.f;
    float b = INFINITY, b2 = INFINITY;
    int bi = 0;
    const int c_lo = part * N / NW, c_hi = (part + 1) * N / NW;
#pragma unroll 8
    for (int c = c_lo; c < c_hi; ++c) {
        float cv[E];
        load_floats<E>(cb + (size_t)c * E, cv);
        float d = 0.f;
#pragma unroll
        for (int t = 0; t < E; ++t) {
            const float e = f[t] - cv[t];
            d = fmaf(e, e, d);
        }
        b2 = fminf(b2, fmaxf(b, d));
        if (d < b) { b = d; bi = c; }
    }
    if constexpr (NW > 1) {
        float *mine = xch + part * xstride;
        mine[lane] = b;
        mine[32 + lane] = b2;
        mine[64 + lane] = __int_as_float(bi);
        asm volatile("bar.sync %0, %1;\n" ::"r"(bar_id), "r"(NW * 32) : "memory");
        if (part != 0) {
            // the others' values are read before any warp of the group
            // moves on to another token
            asm volatile("bar.sync %0, %1;\n" ::"r"(bar_id), "r"(NW * 32) : "memory");
            return;
        }
#pragma unroll
        for (int w = 1; w < NW; ++w) {
            const float *theirs = xch + w * xstride;
            const float bw = theirs[lane], b2w = theirs[32 + lane];
            const int biw = __float_as_int(theirs[64 + lane]);
            const float nb2 = fminf(fminf(b2, b2w), fmaxf(b, bw));
            if (bw < b) { b = bw; bi = biw; }
            b2 = nb2;
        }
        asm volatile("bar.sync %0, %1;\n" ::"r"(bar_id), "r"(NW * 32) : "memory");
    }
    int code = bi;
    unsigned m = __ballot_sync(0xffffffffu, !code_certified<E>(b, b2, delta));
    while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const int cx = nearest_exact_e<E, E>(
            x, sm, rotate, [cb](int c, int t) { return cb[(size_t)c * E + t]; }, N, src,
            __shfl_sync(0xffffffffu, delta, src), lane);
        if (lane == src) code = cx;
    }
    dst[lane] = (uint8_t)code;
}

// Merge of the key splits inside a decode step (after the grid sync): CTA
// c takes the (unit, column, 32 output dimensions) items c, c + grid, ...;
// its warps split the item's records, each lane one output dimension: a
// warp folds its records (a batch loaded at once) into a running (m, l, o),
// and the warps' (m, l, o) are combined in shared memory (`sm` >=
// (32 kWarps + 2 kWarps) floats), out = o / l in fp16.
template <int D, int kWarps>
__device__ void merge_items(const DecArgs &a, float *sm, int warp, int lane) {
    float *part = sm;                      // [kWarps][32]: each warp's o
    float *red = sm + kWarps * 32;         // [kWarps][2]: each warp's (m, l)
    constexpr int kBatch = 16;             // records a warp loads at once
    const int64_t units = a.total / a.T;
    const int ncb = min(kCols, a.G * a.S_q);
    constexpr int nch = D / 32;
    const int64_t items = units * ncb * nch;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int ch = (int)(it % nch);
        const int64_t unit = it / nch / ncb;
        const int col = (int)(it / nch % ncb);
        const int cblk = (int)(unit % a.n_colblk);
        if (cblk * kCols + col >= a.G * a.S_q) continue;   // block-uniform
        int64_t w_lo;
        int n_rec;
        unit_warps(a, unit, &w_lo, &n_rec);
        // each warp: its records k = warp, warp + kWarps, ..., kBatch of them
        // loaded at once, folded into a running (m, l, o) rescaled once per
        // batch
        float mw = -INFINITY, lw = 0.f, ow = 0.f;
        for (int k0 = warp; k0 < n_rec; k0 += kWarps * kBatch) {
            float2 ml[kBatch];
            float ov[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int k = k0 + j * kWarps;
                if (k < n_rec) {
                    const float *r = unit_record(a, unit, w_lo + k, col, D);
                    ml[j] = __ldcg(reinterpret_cast<const float2 *>(r));
                    ov[j] = __ldcg(r + 4 + ch * 32 + lane);
                } else {
                    ml[j] = make_float2(-INFINITY, 0.f);
                    ov[j] = 0.f;
                }
            }
            float bm = mw;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) bm = fmaxf(bm, ml[j].x);
            if (bm != -INFINITY) {
                const float sc = mw == -INFINITY ? 0.f : exp2f(mw - bm);
                lw *= sc;
                ow *= sc;
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const float f = ml[j].x == -INFINITY ? 0.f : exp2f(ml[j].x - bm);
                    lw = fmaf(f, ml[j].y, lw);
                    ow = fmaf(f, ov[j], ow);
                }
                mw = bm;
            }
        }
        part[warp * 32 + lane] = ow;
        if (lane == 0) {
            red[2 * warp] = mw;
            red[2 * warp + 1] = lw;
        }
        __syncthreads();
        if (warp == 0) {
            float M = -INFINITY;
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red[2 * w]);
            float lt = 0.f, acc = 0.f;
            if (M != -INFINITY) {
                for (int w = 0; w < kWarps; ++w) {
                    const float m = red[2 * w];
                    const float f = m == -INFINITY ? 0.f : exp2f(m - M);
                    lt = fmaf(f, red[2 * w + 1], lt);
                    acc = fmaf(f, part[w * 32 + lane], acc);
                }
            }
            const int bgi = (int)(unit / a.n_colblk);
            const int b = bgi / a.H_kv, g = bgi % a.H_kv;
            const int cg = cblk * kCols + col;
            const int i = cg / a.G, hq = g * a.G + cg % a.G;
            a.out[(((int64_t)b * a.H_q + hq) * a.S_q + i) * D + ch * 32 + lane] =
                __float2half_rn(lt > 0.f ? acc / lt : 0.f);
        }
        __syncthreads();   // part[] and red[] are reused by the next item
    }
}

// STEP: the single-launch decode step (vq_decode_step): the new tokens'
// encode beside the attention (a copy of new rows waits for their flags),
// then a grid sync and the merge of the key splits (a cooperative launch);
// only the 128 / 4 / 4 fast instantiation has it.
template <int D, int DK, int DV, int MODE, bool STEP = false>
__global__ void __launch_bounds__(warps_for(D) * 32, 1)
decode_kernel(DecArgs a) {
    constexpr bool FAST = MODE == kModeFast, PACKED = MODE == kModePacked;
    static_assert(!STEP || (FAST && D == 128 && DK == 4 && DV == 4), "decode step: 128 / 4 / 4 fast");
    constexpr int kWarp0 = STEP ? kStepEncodeWarps : 0;   // first warp with a share
    constexpr int kWarps = warps_for(D), kThreads = kWarps * 32;
    constexpr int KSTEPS = D / 16, MT = D / 16;
    constexpr int EK = 2 * DK, EV = 2 * DV;
    using SC = StepCodes<D, DK, DV>;

    // shared memory: fp16 tables | per-warp scratch | fp32 staging
    //   fast path: one interleaved 256 x 256-byte table (keys | values);
    //   packed path: key table (2^kPackedBits rows) then value table (256
    //   rows), 128-byte rows, no staging;
    //   otherwise: key table (N_k rows) then value table (N_v rows)
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int krow = a.k_copies * EK, vrow = a.v_copies * EV;   // replica bytes per row
    constexpr size_t kPkKeyTab = (size_t)(1u << kPackedBits) * kPkRow;
    const size_t tab_bytes = FAST ? (size_t)0
                             : PACKED ? kPkKeyTab + 256 * (size_t)kPkRow
                                      : align16((size_t)a.Nk * krow) + align16((size_t)a.Nv * vrow);
    // fast path: scratch and staging first, the table at shared address
    // 65536 (the launch reserves 128 KiB, which always reaches past it)
    unsigned char *ktab = FAST ? smem_raw + (kFastTabAddr - (uint32_t)__cvta_generic_to_shared(smem_raw))
                               : smem_raw;
    unsigned char *vtab = FAST     ? ktab + 128
                          : PACKED ? smem_raw + kPkKeyTab
                                   : smem_raw + align16((size_t)a.Nk * krow);
    WarpScratch<D> *scratch = reinterpret_cast<WarpScratch<D> *>(smem_raw + tab_bytes);
    float *stage = reinterpret_cast<float *>(scratch + kWarps);
    // ring path (uint8 codes in rows of 16-byte multiples): the stage
    // mbarriers after the staging area, the stages from shared address 128 KiB
    using RC = RingCfg<D, DK, DV>;
    constexpr bool RING = FAST && RC::on;
    constexpr int kStages = RING ? ring_stages(RC::STAGE, kWarps) : 1;
    const uint32_t mbar0 =
        ((uint32_t)__cvta_generic_to_shared(stage + a.Nk * DK + a.Nv * DV) + 7u) & ~7u;
    if (FAST && mbar0 + (RING ? kWarps * kStages * 8 : 0) > kFastTabAddr)
        return;   // not reachable: dynamic shared memory starts near address 0
    const int kstride = FAST ? (int)kFastRow : krow;   // row strides of the tables
    const int vstride = FAST ? (int)kFastRow : vrow;
    const int nk_rows = FAST ? 256 : a.Nk, nv_rows = FAST ? 256 : a.Nv;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, c4 = lane & 3;
    // the combine may be scheduled now; it waits for this grid to finish
    pdl_launch_dependents();

    // ---- fp16 tables replicated per bank group (rows past N are zero)
    if constexpr (FAST) {
        int t0 = 0;   // first thread of the table build
        if constexpr (STEP) {
            {
                // ---- decode step: the fp32 codebooks staged, then the new
                //      tokens encoded into their cache rows by warps 0-3 (one
                //      token at a time, the codebook split over the 4 warps;
                //      tokens c, c + grid, ... on CTA c) while the other warps
                //      build the table
                const int nk_f = a.Nk * DK, nv_f = a.Nv * DV;
                for (int i = tid; i < nk_f; i += kThreads) stage[i] = a.kcbk[i];
                for (int i = tid; i < nv_f; i += kThreads) stage[nk_f + i] = a.vcbk[i];
                __syncthreads();
                pdl_wait();
                constexpr int kEncWarps = kStepEncodeWarps;
                static_assert(kThreads - kEncWarps * 32 >= 256, "one table row per builder thread");
                t0 = kEncWarps * 32;
                if (warp < kEncWarps) {
                    const int n_new = a.B * a.H_kv * a.S_q;
                    // exchange areas: the encoding warps' query scratch
                    // (unused until the attention)
                    float *xch = reinterpret_cast<float *>(scratch[0].qt);
                    constexpr int kXStride = (int)(sizeof(WarpScratch<D>) / sizeof(float));
                    static_assert(sizeof(WarpScratch<D>) % sizeof(float) == 0 &&
                                      sizeof(scratch[0].qt) >= 96 * sizeof(float),
                                  "exchange area of 96 words per warp");
                    for (int task = (int)blockIdx.x; task < 2 * n_new; task += (int)gridDim.x) {
                        const int tok = task >> 1, is_v = task & 1;
                        const int bh = tok / a.S_q, tt = tok - bh * a.S_q;
                        const int h = bh % a.H_kv;
                        const __half *x = (is_v ? a.v_new : a.k_new) + (int64_t)tok * D;
                        uint8_t *dst = const_cast<uint8_t *>(is_v ? a.vc : a.kc) +
                                       ((int64_t)bh * a.stride + a.new_row0 + tt) * 32;
                        const float *smr = is_v || a.smooth_mode == 0 ? nullptr
                                           : a.smooth_mode == 2 ? a.smooth + (size_t)h * D
                                                                : a.smooth;
                        encode_token_group<4, kEncWarps>(
                            x, smr, !is_v, is_v ? stage + a.Nk * DK : stage, is_v ? a.Nv : a.Nk,
                            dst, a.log2D, lane, warp, xch, kXStride, 1);
                        if (warp == 0) {   // the group's first warp wrote the row
                            __threadfence();
                            __syncwarp();
                            if (lane == 0) flag_release(a.step_flags + task, a.step_epoch);
                        }
                    }
                }
            }
        }
        // 256 rows x 16 chunks of 16 bytes (8 key, 8 value); every chunk of a
        // row half holds 16 / EK (16 / EV) copies of its centroid.  A thread
        // owns whole rows: both centroid loads are in flight together, then
        // the 16 stores.
        // (a decode step reads the fp32 codebooks it has staged)
        const float *kcb_src = STEP ? stage : a.kcbk;
        const float *vcb_src = STEP ? stage + a.Nk * DK : a.vcbk;
        for (int c = tid - t0; c >= 0 && c < 256; c += kThreads - t0) {
            const uint4 wk = c < a.Nk ? replica_chunk<DK>(kcb_src + c * DK) : make_uint4(0u, 0u, 0u, 0u);
            const uint4 wv = c < a.Nv ? replica_chunk<DV>(vcb_src + c * DV) : make_uint4(0u, 0u, 0u, 0u);
            uint4 *row = reinterpret_cast<uint4 *>(ktab + c * kFastRow);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                row[q] = wk;
                row[8 + q] = wv;
            }
        }
    } else if constexpr (PACKED) {
        // every row of both tables: the thread's rows' centroids are loaded
        // first, then each row's 8 chunks of 16 bytes are stored starting at
        // chunk (lane mod 8), so the lanes of a store phase hit distinct banks
        constexpr int kRows = (1 << kPackedBits) + 256;
        constexpr int kPer = (kRows + kThreads - 1) / kThreads;
        uint4 rw[kPer];
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
            const int c = tid + r * kThreads;
            const int cv = c - (1 << kPackedBits);
            rw[r] = c < a.Nk                      ? replica_chunk<DK>(a.kcbk + c * DK)
                    : cv >= 0 && cv < a.Nv ? replica_chunk<DV>(a.vcbk + cv * DV)
                                                  : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
            const int c = tid + r * kThreads;
            if (c < kRows) {
                uint4 *row = reinterpret_cast<uint4 *>(smem_raw + (size_t)c * kPkRow);
#pragma unroll
                for (int q = 0; q < 8; ++q) row[(q + lane) & 7] = rw[r];
            }
        }
    } else {
        // fp32 copy (coalesced), then the tables word by word
        const int nk_f = a.Nk * DK, nv_f = a.Nv * DV;
        for (int i = tid; i < nk_f; i += kThreads) stage[i] = a.kcbk[i];
        for (int i = tid; i < nv_f; i += kThreads) stage[nk_f + i] = a.vcbk[i];
        __syncthreads();
        for (int i = tid; i < nk_rows * (krow / 4); i += kThreads) {
            const int c = i / (krow / 4), wi = i % (krow / 4);
            const int t = ((wi * 4) % EK) / 2;
            *reinterpret_cast<uint32_t *>(ktab + (size_t)c * kstride + wi * 4) =
                c < a.Nk ? pack_h2(stage[c * DK + t], stage[c * DK + t + 1]) : 0u;
        }
        for (int i = tid; i < nv_rows * (vrow / 4); i += kThreads) {
            const int c = i / (vrow / 4), wi = i % (vrow / 4);
            const int t = ((wi * 4) % EV) / 2;
            *reinterpret_cast<uint32_t *>(vtab + (size_t)c * vstride + wi * 4) =
                c < a.Nv ? pack_h2(stage[nk_f + c * DV + t], stage[nk_f + c * DV + t + 1]) : 0u;
        }
    }
    if constexpr (STEP) {
        // a decode step: the table builders (the warps with shares) meet; the
        // encoding warps go on to the grid sync
        if (warp >= kStepEncodeWarps)
            asm volatile("bar.sync 2, %0;\n" ::"r"((kWarps - kStepEncodeWarps) * 32) : "memory");
    } else {
        __syncthreads();
    }
    // codes (and everything else below) may come from the preceding kernel:
    // wait for it to finish (a no-op unless launched as a dependent)
    pdl_wait();
    const uint32_t klane = (uint32_t)((lane % a.k_copies) * EK);
    const uint32_t vlane = (FAST ? 128u : 0u) + (uint32_t)((lane % a.v_copies) * EV);
    const uint32_t kbase = (uint32_t)__cvta_generic_to_shared(ktab) + klane;
    const uint32_t vbase = (uint32_t)__cvta_generic_to_shared(smem_raw) + (FAST ? 0u : (uint32_t)(vtab - smem_raw)) + vlane;
    const int64_t ktb = a.krowb;   // code bytes per key
    const int64_t vtb = a.vrowb;
    const int n_cols_total = a.G * a.S_q;
    WarpScratch<D> &ws = scratch[warp];

    // warps past the plan's last one have no share (they still reach the
    // grid sync of a decode step)
    const int64_t gw = warp >= kWarp0
                           ? (int64_t)blockIdx.x * (kWarps - kWarp0) + (warp - kWarp0)
                           : (int64_t)a.nw;   // an encoding warp of a decode step: no share
    int64_t t = gw < a.nw ? share_start(gw, a.share, a.total) : 0;
    const int64_t t_end = gw < a.nw ? share_start(gw + 1, a.share, a.total) : 0;
    int slot = 0;

    // ---- ring path: the producer cursor walks the warp's steps ahead of it
    const uint32_t wbar = mbar0 + (uint32_t)(warp * kStages * 8);
    const uint32_t wring = kRingAddr + (uint32_t)(warp * kStages * RC::STAGE);
    SegInfo ps{};
    int64_t pt = t;
    int pj = 0, issued = 0;
    bool pvalid = false, ring_ok = true;
    uint32_t pending = 0u, pend_par = 0u;   // stages with a copy in flight, and its phase
    auto pseek = [&]() {   // to the next step of a non-empty segment
        while (pj >= ps.j_last) {
            pt = ps.seg_end;
            if (pt >= t_end) { pvalid = false; return; }
            ps = segment_at(a, pt, t_end);
            pj = ps.j_first;
        }
    };
    // copy the next step's K and V code rows into stage issued % kStages
    // (in a decode step, rows from new_row0 on once they are written)
    int64_t new_ok_bg = -1;   // (b, kv head) whose new rows this warp has seen written
    auto issue = [&]() {
        if (!pvalid) return;
        if constexpr (STEP) {
            if (pj + kStepKeys > a.new_row0 && ps.bg != new_ok_bg) {
                bool ok = true;
                if (lane == 0) ok = wait_new_rows(a.step_flags, a.step_epoch, ps.bg, a.S_q);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {   // the records of this warp become NaN
                    ring_ok = false;
                    pvalid = false;
                    return;
                }
                new_ok_bg = ps.bg;
                // the rows were written through the generic proxy; the copies
                // read them through the async proxy
                asm volatile("fence.proxy.async.global;\n" ::: "memory");
            }
        }
        const int sidx = issued % kStages;
        const uint32_t bar = wbar + (uint32_t)(sidx * 8);
        const uint32_t st = wring + (uint32_t)(sidx * RC::STAGE);
        const int n = min(kStepKeys, a.S_kv - pj);   // rows inside the cache
        if (lane == 0) {
            // the stage was last read by this warp's lanes (generic proxy)
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            ring_expect(bar, (uint32_t)(n * (RC::KROW + RC::VROW)));
            ring_copy(st, a.kc + (ps.bg * a.stride + pj) * RC::KROW, (uint32_t)(n * RC::KROW), bar);
            ring_copy(st + kStepKeys * RC::KROW, a.vc + (ps.bg * a.stride + pj) * RC::VROW,
                      (uint32_t)(n * RC::VROW), bar);
        }
        pending |= 1u << sidx;
        pend_par = (pend_par & ~(1u << sidx)) | ((uint32_t)((issued / kStages) & 1) << sidx);
        ++issued;
        pj += kStepKeys;
        pseek();
    };
    if constexpr (RING) {
        if (lane == 0) {
            for (int k = 0; k < kStages; ++k) ring_bar_init(wbar + (uint32_t)(k * 8));
            asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        }
        __syncwarp();
        if (t < t_end) {
            ps = segment_at(a, t, t_end);
            pj = ps.j_first;
            pvalid = true;
            pseek();
        }
        // in a decode step, a copy that reads the new rows [new_row0, ..)
        // waits until they are written (the rest of the fill after the sync)
        for (int k = 0; k < kStages; ++k) {
            if (STEP && pvalid && pj + kStepKeys > a.new_row0) break;
            issue();
        }
    }
    // ---- transformed queries of a segment's unit's columns into the warp's
    //      scratch: q~ = Hn (q (.) s_g^-1) (base-2 softmax scale folded in),
    //      and each column's visible key range
    auto build_qt = [&](const SegInfo &q) {
        __syncwarp();
        for (int col = 0; col < kCols; ++col) {
            const int cg = q.cblk * kCols + col;
            if (cg < n_cols_total) {
                const int i = cg / a.G, gam = cg % a.G;
                const int hq = q.g * a.G + gam;
                const __half *qp = a.q + (((int64_t)q.b * a.H_q + hq) * a.S_q + i) * D;
                const float *sp = a.smooth_mode == 2 ? a.smooth + (size_t)q.g * D : a.smooth;
                // lane holds dims [E lane, E lane + E); FWHT by butterflies in
                // registers and xor-shuffles
                constexpr int E = D / 32;
                float f[E];
                load_halves<E>(qp + lane * E, f);
                if (a.smooth_mode != 0) {
                    float sv[E];
                    load_floats<E>(sp + lane * E, sv);
#pragma unroll
                    for (int e = 0; e < E; ++e) f[e] = f[e] / sv[e];
                }
#pragma unroll
                for (int e = 0; e < E; ++e) f[e] *= a.qscale;
                reg_fwht<E>(f, lane);
                store_halves<E>(ws.qt[col] + lane * E, f);
                if (lane == 0) {
                    const int L = q.kv_len;
                    const int q_abs = L - a.S_q + i;
                    int hi = a.causal ? q_abs : L - 1;
                    if (hi > L - 1) hi = L - 1;
                    int lo = a.window > 0 ? q_abs - a.window + 1 : 0;
                    if (lo < 0) lo = 0;
                    ws.lo[col] = lo;
                    ws.hi[col] = hi;
                }
            } else {
                for (int e = lane; e < D; e += 32) ws.qt[col][e] = __float2half_rn(0.f);
                if (lane == 0) { ws.lo[col] = 1; ws.hi[col] = 0; }   // empty
            }
            __syncwarp();
        }
    };
    bool qt_ready = false;   // the first segment's q~ already built
    // ---- decode step: the first segment's queries are transformed, then the
    //      rest of the ring is filled; a copy of new rows waits there for
    //      their flags (set by the encoding warps, which run beside this)
    if constexpr (STEP) {
        if (t < t_end) {
            build_qt(segment_at(a, t, t_end));
            qt_ready = true;
        }
        if constexpr (RING) {
            while (pvalid && issued < kStages) issue();   // nothing consumed yet
        }
    }

    int consumed = 0;

    while (t < t_end) {
        const SegInfo sg = segment_at(a, t, t_end);
        const int64_t seg_end = sg.seg_end, bg = sg.bg;
        const int cblk = sg.cblk;
        const int j_first = sg.j_first, j_last = sg.j_last;
        // the segment's first code tiles go to L2 while the queries are prepared
        const uint8_t *kg = a.kc + bg * a.stride * ktb;
        const uint8_t *vg = a.vc + bg * a.stride * vtb;
        // lane base pointers: row g8 of a tile (K), row 2c4 of a tile (V)
        // (packed rows: the row start; the run's first code index is passed on)
        const uint8_t *kl = kg + (int64_t)g8 * ktb + (a.kcb > 0 ? (int64_t)c4 * SC::NKL * a.kcb : 0);
        const uint8_t *vl = vg + (int64_t)(2 * c4) * vtb + (a.vcb > 0 ? (int64_t)g8 * SC::NVL * a.vcb : 0);
        // L2 prefetch of the keys [j, j + n) (clipped to the segment and the cache)
        auto prefetch = [&](int j, int n) {
            const int e = min(min(j + n, j_last), a.S_kv);
            if (lane == 0 && j < e) {
                prefetch_l2(kg + (int64_t)j * ktb, (uint32_t)((e - j) * ktb));
                prefetch_l2(vg + (int64_t)j * vtb, (uint32_t)((e - j) * vtb));
            }
        };
        if constexpr (!RING) prefetch(j_first, kPrefetchTiles * kTile);

        // ---- transformed queries of the unit's columns (for a decode step's
        //      first segment: built before the ring is filled)
        if (qt_ready) qt_ready = false;
        else build_qt(sg);
        UnitState<D> us;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
            const __half *qv = ws.qt[g8] + c4 * (D / 4) + 4 * ks;
            us.bq[ks][0] = *reinterpret_cast<const uint32_t *>(qv);
            us.bq[ks][1] = *reinterpret_cast<const uint32_t *>(qv + 2);
        }
        us.lo0 = ws.lo[2 * c4]; us.hi0 = ws.hi[2 * c4];
        us.lo1 = ws.lo[2 * c4 + 1]; us.hi1 = ws.hi[2 * c4 + 1];
        us.lo_all = INT_MAX; us.hi_all = -1; us.lo_any = 0; us.hi_any = INT_MAX;
        bool any_real = false;
#pragma unroll
        for (int col = 0; col < kCols; ++col) {
            const int l = ws.lo[col], h = ws.hi[col];
            if (l > h) continue;
            any_real = true;
            us.lo_all = min(us.lo_all, l); us.hi_all = max(us.hi_all, h);
            us.lo_any = max(us.lo_any, l); us.hi_any = min(us.hi_any, h);
        }
        if (!any_real) { us.lo_any = 1; us.hi_any = 0; }
        us.m0 = us.m1 = -INFINITY;
        us.mu0 = us.mu1 = 0.f;
        us.l0 = us.l1 = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            us.acc_o[mt][0] = us.acc_o[mt][1] = us.acc_o[mt][2] = us.acc_o[mt][3] = 0.f;


        // ---- stream the segment, codes double-buffered in registers
        // (a step may run past j_last by one tile; those keys belong to the
        // next share and are masked by the per-segment bounds below)
        us.lo_any = max(us.lo_any, j_first);
        us.hi_any = min(us.hi_any, j_last - 1);
        us.lo0 = max(us.lo0, j_first); us.hi0 = min(us.hi0, j_last - 1);
        us.lo1 = max(us.lo1, j_first); us.hi1 = min(us.hi1, j_last - 1);
        us.lo_all = max(us.lo_all, j_first); us.hi_all = min(us.hi_all, j_last - 1);
        // a step in [lo_any, hi_any] needs no per-column bounds
        auto step = [&](const SC &c, int jj) {
            if (jj >= us.lo_any && jj + kStepKeys - 1 <= us.hi_any)
                process_step<D, DK, DV, MODE, false, RING>(c, jj, us, a, kbase, vbase, krow, vrow,
                                                           g8, c4, smem_raw, klane, vlane);
            else
                process_step<D, DK, DV, MODE, true, RING>(c, jj, us, a, kbase, vbase, krow, vrow,
                                                          g8, c4, smem_raw, klane, vlane);
        };
        if constexpr (RING) {
            // steps from the ring: wait for the stage, read its codes, hand
            // it back to the producer (which refills it kStages steps ahead)
            for (int j = j_first; j < j_last; j += kStepKeys) {
                const int sidx = consumed % kStages;
                const uint32_t bar = wbar + (uint32_t)(sidx * 8);
                if (ring_ok) {
                    const bool ok = ring_wait(bar, (uint32_t)((consumed / kStages) & 1));
                    ring_ok = __all_sync(0xffffffffu, ok);
                    if (ring_ok) pending &= ~(1u << sidx);
                }
                SC sc;
                load_step_ring<D, DK, DV>(sc, wring + (uint32_t)(sidx * RC::STAGE), g8, c4);
                __syncwarp();
                ++consumed;
                if (ring_ok) issue();
                step(sc, j);
            }
        } else {
        SC ca, cb;
        int j = j_first;
        if (j < j_last) load_step<D, DK, DV, MODE>(ca, kl, vl, j, a, ktb, vtb, g8, c4);
        while (j < j_last) {
            if (j + kStepKeys < j_last)
                load_step<D, DK, DV, MODE>(cb, kl, vl, j + kStepKeys, a, ktb, vtb, g8, c4);
            // once per two steps (j - j_first is a multiple of 64 here): the
            // next 64 keys, kPrefetchTiles tiles ahead
            prefetch(j + kPrefetchTiles * kTile, kPfKeys);
            step(ca, j);
            j += kStepKeys;
            if (j >= j_last) break;
            if (j + kStepKeys < j_last)
                load_step<D, DK, DV, MODE>(ca, kl, vl, j + kStepKeys, a, ktb, vtb, g8, c4);
            step(cb, j);
            j += kStepKeys;
        }
        }

        // ---- this warp's partial record for the unit
        // (a stage wait that expired leaves the record, hence the output, NaN)
        if (RING && !ring_ok) us.l0 = us.l1 = NAN;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            us.l0 += __shfl_xor_sync(0xffffffffu, us.l0, off);
            us.l1 += __shfl_xor_sync(0xffffffffu, us.l1, off);
        }
        // (columns past the last real one have no record: the combine skips them)
        float *rec = a.ws + ((gw * a.slots + slot) * kCols) * (int64_t)(D + 4);
        float *rec0 = rec + (2 * c4) * (D + 4), *rec1 = rec0 + (D + 4);
        const bool real0 = cblk * kCols + 2 * c4 < n_cols_total;
        const bool real1 = cblk * kCols + 2 * c4 + 1 < n_cols_total;
        if (g8 == 0) {
            if (real0) *reinterpret_cast<float2 *>(rec0) = make_float2(us.m0, us.l0);
            if (real1) *reinterpret_cast<float2 *>(rec1) = make_float2(us.m1, us.l1);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int d0 = g8 * (D / 8) + 2 * mt;
            if (real0)
                *reinterpret_cast<float2 *>(rec0 + 4 + d0) = make_float2(us.acc_o[mt][0], us.acc_o[mt][2]);
            if (real1)
                *reinterpret_cast<float2 *>(rec1 + 4 + d0) = make_float2(us.acc_o[mt][1], us.acc_o[mt][3]);
        }
        ++slot;
        t = seg_end;
    }
    // a stage wait expired: wait (bounded) for this warp's copies still in flight
    if constexpr (RING) {
        if (!ring_ok) {
            for (int k = 0; k < kStages; ++k)
                if (pending & (1u << k)) ring_wait(wbar + (uint32_t)(k * 8), (pend_par >> k) & 1u);
        }
    }
    // ---- decode step: every record written, then the merge of the splits
    //      (the codebook table region is free now)
    if constexpr (STEP) {
        {
            cooperative_groups::this_grid().sync();   // orders the records before it
            // every wait for new rows is over: their flags back to 0 for
            // the next launch on this workspace (a replayed graph included)
            if (blockIdx.x == 0)
                for (int i = tid; i < 2 * a.B * a.H_kv * a.S_q; i += kThreads) a.step_flags[i] = 0ull;
            merge_items<D, kWarps>(a, reinterpret_cast<float *>(ktab), warp, lane);
        }
    }
}

// Merge the partial records of every (unit, column) and write fp16.  The
// records of a unit come from the warps whose shares overlap it.  One block
// of D threads per (unit, column); warp w takes output dimensions
// [32 w, 32 w + 32), one per lane.  Every lane walks the unit's records: the
// maximum M of their m, then o = sum_k 2^(m_k - M) o_k[d] and
// l = sum_k 2^(m_k - M) l_k, out = o / l.  No shared memory, no barriers
// (used when a unit has at most kNarrowRecords records).
constexpr int kMaxRecords = 2048;   // >= warps of any plan (one CTA per SM)
constexpr int kNarrowRecords = 16;  // up to this many records per unit: one lane per dimension

template <int D>
__global__ void __launch_bounds__(D)
combine_kernel(DecArgs a, __half *__restrict__ out) {
    pdl_wait();   // the records come from the decode grid
    const int64_t unit = blockIdx.x;
    const int col = blockIdx.y;
    const int cblk = (int)(unit % a.n_colblk);
    const int64_t bg = unit / a.n_colblk;
    const int cg = cblk * kCols + col;
    if (cg >= a.G * a.S_q) return;
    const int b = (int)(bg / a.H_kv), g = (int)(bg % a.H_kv);
    const int i = cg / a.G, gam = cg % a.G;
    const int d = threadIdx.x;
    const int64_t u0 = unit * a.T;
    const int64_t w_lo = u0 / a.share;
    int64_t w_hi = (u0 + a.T - 1) / a.share;
    if (w_hi > a.nw - 1) w_hi = a.nw - 1;
    int n_rec = (int)(w_hi - w_lo + 1);
    if (n_rec > kMaxRecords) n_rec = kMaxRecords;   // not reachable: see kMaxRecords
    // record of warp w for this unit: slot = unit - (first unit of w)
    auto rec_of = [&](int k) -> const float * {
        const int64_t w = w_lo + k;
        const int64_t s = w * a.share;
        const int64_t slot = a.share <= a.T ? (s >= u0 ? 0 : 1) : unit - s / a.T;
        return a.ws + ((w * a.slots + slot) * kCols + col) * (int64_t)(D + 4);
    };
    float M = -INFINITY;
#pragma unroll 8
    for (int k = 0; k < n_rec; ++k) M = fmaxf(M, rec_of(k)[0]);
    float o = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll 8
        for (int k = 0; k < n_rec; ++k) {
            const float *r = rec_of(k);
            const float f = exp2f(r[0] - M);
            l = fmaf(f, r[1], l);
            o = fmaf(f, r[4 + d], o);
        }
        o = l > 0.f ? o / l : 0.f;
    }
    const int hq = g * a.G + gam;
    out[(((int64_t)b * a.H_q + hq) * a.S_q + i) * D + d] = __float2half_rn(o);
}

// Merge for units with many records (long shares of few units): block
// (unit, column, chunk of kCombDims output dimensions), 256 threads: the
// block reduces the records' maxima and sums in parallel and keeps each
// record's rescale factor in shared memory; then 8 groups of kCombDims
// threads (one output dimension each) accumulate disjoint subsets of the
// records with many loads in flight, and the groups' sums are added.
constexpr int kCombThreads = 256;
constexpr int kCombDims = 32;

template <int D>
__global__ void __launch_bounds__(kCombThreads)
combine_wide_kernel(DecArgs a, __half *__restrict__ out) {
    constexpr int kGroups = kCombThreads / kCombDims;
    __shared__ float fac[kMaxRecords];
    __shared__ float red[kCombThreads / 32];
    __shared__ float part[kGroups][kCombDims];
    pdl_wait();   // the records come from the decode grid
    const int64_t unit = blockIdx.x;
    const int col = blockIdx.y;
    const int cblk = (int)(unit % a.n_colblk);
    const int64_t bg = unit / a.n_colblk;
    const int cg = cblk * kCols + col;
    if (cg >= a.G * a.S_q) return;
    const int b = (int)(bg / a.H_kv), g = (int)(bg % a.H_kv);
    const int i = cg / a.G, gam = cg % a.G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = (int)blockIdx.z * kCombDims + tid % kCombDims, grp = tid / kCombDims;
    const int64_t u0 = unit * a.T;
    const int64_t w_lo = u0 / a.share;
    int64_t w_hi = (u0 + a.T - 1) / a.share;
    if (w_hi > a.nw - 1) w_hi = a.nw - 1;
    int n_rec = (int)(w_hi - w_lo + 1);
    if (n_rec > kMaxRecords) n_rec = kMaxRecords;   // not reachable: see kMaxRecords
    // record of warp w for this unit: slot = unit - (first unit of w)
    auto rec_of = [&](int k) -> const float * {
        const int64_t w = w_lo + k;
        const int64_t s = w * a.share;
        const int64_t slot = a.share <= a.T ? (s >= u0 ? 0 : 1) : unit - s / a.T;
        return a.ws + ((w * a.slots + slot) * kCols + col) * (int64_t)(D + 4);
    };
    auto block_reduce = [&](float v, bool is_max) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, v, off);
            v = is_max ? fmaxf(v, o) : v + o;
        }
        __syncthreads();
        if (lane == 0) red[warp] = v;
        __syncthreads();
        v = red[0];
#pragma unroll
        for (int w = 1; w < kCombThreads / 32; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
        return v;
    };
    float M = -INFINITY;
    for (int k = tid; k < n_rec; k += kCombThreads) {
        const float m = rec_of(k)[0];
        fac[k] = m;
        M = fmaxf(M, m);
    }
    M = block_reduce(M, true);
    float o = 0.f;
    if (M != -INFINITY) {
        float l = 0.f;
        for (int k = tid; k < n_rec; k += kCombThreads) {
            const float f = exp2f(fac[k] - M);
            fac[k] = f;
            l += f * rec_of(k)[1];
        }
        l = block_reduce(l, false);   // its barriers also publish fac[]
#pragma unroll 8
        for (int k = grp; k < n_rec; k += kGroups) o += fac[k] * rec_of(k)[4 + d];
        part[grp][tid % kCombDims] = o;
        __syncthreads();
        o = 0.f;
#pragma unroll
        for (int q = 0; q < kGroups; ++q) o += part[q][tid % kCombDims];
        o = l > 0.f ? o / l : 0.f;
    }
    if (grp == 0) {
        const int hq = g * a.G + gam;
        out[(((int64_t)b * a.H_q + hq) * a.S_q + i) * D + d] = __float2half_rn(o);
    }
}

struct Tables {
    int k_copies, v_copies;
    int mode;       // kModeGeneric, kModeFast or kModePacked
    size_t bytes;
};

constexpr size_t kSmemBudget = 210 * 1024;

size_t scratch_bytes(int D) {
    switch (D) {
        case 32: return warps_for(32) * sizeof(WarpScratch<32>);
        case 64: return warps_for(64) * sizeof(WarpScratch<64>);
        case 128: return warps_for(128) * sizeof(WarpScratch<128>);
        default: return warps_for(256) * sizeof(WarpScratch<256>);
    }
}

// Shared-memory plan: the fast path (uint8 codes, N <= 256, full replicas)
// when it fits, else the largest replica counts (powers of two, <= 128
// bytes per row) that fit the budget.
Tables choose_tables(const vq_attend_args &a) {
    const int ek = 2 * a.k_sub_dim, ev = 2 * a.v_sub_dim;
    const size_t tail = scratch_bytes(a.D) +
                        sizeof(float) * ((size_t)a.k_n_centroids * a.k_sub_dim +
                                         (size_t)a.v_n_centroids * a.v_sub_dim);
    // fast path: the table sits at shared address 64 KiB, scratch, staging
    // and the ring mbarriers below it (dynamic shared memory starts within
    // the first KiB); code rows of 16-byte multiples also take the per-warp
    // rings of code stages from 128 KiB on
    const int krowb = a.D / a.k_sub_dim, vrowb = a.D / a.v_sub_dim;
    const bool ring = krowb % 16 == 0 && vrowb % 16 == 0;
    const int stage = kStepKeys * (krowb + vrowb);
    const int warps = warps_for(a.D);
    const size_t mbars = ring ? (size_t)warps * ring_stages(stage, warps) * 8 + 8 : 0;
    if (a.k_code_bytes == 1 && a.v_code_bytes == 1 && a.k_n_centroids <= 256 &&
        a.v_n_centroids <= 256 && tail + mbars + 2048 <= kFastTabAddr)
        return {128 / ek, 128 / ev, kModeFast,
                ring ? (size_t)kRingAddr + (size_t)warps * ring_stages(stage, warps) * stage
                     : 2 * (size_t)kFastTabAddr};
    // packed path: kPackedBits-bit packed keys of 8 dimensions, uint8 values
    // of 4, D = 128; tables of 128-byte rows (8 / 16 replicas), no staging
    if (a.D == 128 && a.k_sub_dim == 8 && a.v_sub_dim == 4 && a.k_code_bytes == 0 &&
        packed_code_bits(a.k_n_centroids) == kPackedBits && a.v_code_bytes == 1 &&
        a.v_n_centroids <= 256)
        return {(int)kPkRow / ek, (int)kPkRow / ev, kModePacked,
                ((size_t)1 << kPackedBits) * kPkRow + 256 * (size_t)kPkRow + scratch_bytes(a.D)};
    int kc = 128 / ek, vc = 128 / ev;
    auto total = [&](int k, int v) {
        return align16((size_t)a.k_n_centroids * k * ek) +
               align16((size_t)a.v_n_centroids * v * ev) + tail;
    };
    while (total(kc, vc) > kSmemBudget && (kc > 1 || vc > 1)) {
        if ((size_t)a.k_n_centroids * kc * ek >= (size_t)a.v_n_centroids * vc * ev && kc > 1)
            kc /= 2;
        else if (vc > 1)
            vc /= 2;
        else
            kc /= 2;
    }
    return {kc, vc, kModeGeneric, total(kc, vc)};
}

template <int D, int DK, int DV>
cudaError_t launch_t(const DecArgs &da, const Tables &tb, int grid, cudaStream_t stream) {
    void (*kern)(DecArgs) = tb.mode == kModeFast ? decode_kernel<D, DK, DV, kModeFast>
                                                 : decode_kernel<D, DK, DV, kModeGeneric>;
    if (tb.mode == kModePacked) {
        if constexpr (D == 128 && DK == 8 && DV == 4)
            kern = decode_kernel<D, DK, DV, kModePacked>;
        else
            return cudaErrorInvalidValue;
    }
    if (da.step) {
        if constexpr (D == 128 && DK == 4 && DV == 4) {
            if (tb.mode != kModeFast) return cudaErrorInvalidValue;
            kern = decode_kernel<D, DK, DV, kModeFast, true>;
        } else {
            return cudaErrorInvalidValue;
        }
    }
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)tb.bytes);
    if (err != cudaSuccess) return err;
    if (da.step) {
        // a decode step: cooperative launch (its blocks meet at a grid sync
        // and wait on one another's flags; the launch fails rather than
        // starting if they cannot all be resident at once)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(warps_for(D) * 32);
        cfg.dynamicSmemBytes = tb.bytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, da);
    }
    return launch_dependent(kern, dim3(grid), dim3(warps_for(D) * 32), tb.bytes, stream, da);
}

template <int D>
cudaError_t launch_d(const DecArgs &da, int dk, int dv, const Tables &tb, int grid,
                     cudaStream_t s) {
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

// Common key-tile range of every unit: the union of what any query row sees.
// Per-batch lengths (read on the device) can put a batch's queries anywhere
// in the cache, so then the range is the whole cache.
void tile_range(const vq_attend_args &a, int *tlo, int *T) {
    if (a.kv_lens) {
        *tlo = 0;
        *T = a.S_kv > 0 ? (a.S_kv + kTile - 1) / kTile : 1;
        return;
    }
    const int q_first = a.S_kv - a.S_q, q_last = a.S_kv - 1;
    int hi = a.causal ? q_last : a.S_kv - 1;
    int lo = a.sliding_window > 0 ? q_first - a.sliding_window + 1 : 0;
    if (lo < 0) lo = 0;
    if (hi > a.S_kv - 1) hi = a.S_kv - 1;
    if (hi < lo) { *tlo = 0; *T = 1; return; }
    *tlo = lo / kTile;
    *T = hi / kTile - *tlo + 1;
}

constexpr int kMinTilesPerWarp = 4;

}  // namespace

vq_attend_args normalize_code_widths(const vq_attend_args &a) {
    vq_attend_args n = a;
    auto fix = [](int &cb, int N, int n_sub) {
        if (cb != 0 || N < 1 || n_sub < 1) return;
        const int bits = packed_code_bits(N);
        if (bits == 8 && (n_sub * 8) % 32 == 0) cb = 1;
        if (bits == 16 && (n_sub * 16) % 32 == 0) cb = 2;
    };
    if (a.k_sub_dim > 0) fix(n.k_code_bytes, a.k_n_centroids, a.D / a.k_sub_dim);
    if (a.v_sub_dim > 0) fix(n.v_code_bytes, a.v_n_centroids, a.D / a.v_sub_dim);
    return n;
}

int decode_supported(const vq_attend_args &a) {
    if (a.D != 32 && a.D != 64 && a.D != 128 && a.D != 256) return VQ_ERR_UNSUPPORTED;
    if (!pair_ok(a.D, a.k_sub_dim, a.v_sub_dim)) return VQ_ERR_UNSUPPORTED;
    const Tables tb = choose_tables(a);
    if (tb.bytes > (tb.mode == kModeFast ? (size_t)kSmemLimit : kSmemBudget))
        return VQ_ERR_UNSUPPORTED;
    return VQ_OK;
}

size_t decode_smem_bytes(const vq_attend_args &a) { return choose_tables(a).bytes; }

// The single-launch decode step: uint8 codes of 4-dimensional sub-vectors at
// D = 128 (the shared-memory table and code-ring path), one grid of at most
// one block per SM (the persistent plan), no per-batch lengths.
int decode_step_supported(const vq_attend_args &a) {
    if (a.D != 128 || a.k_sub_dim != 4 || a.v_sub_dim != 4) return VQ_ERR_UNSUPPORTED;
    if (a.k_code_bytes != 1 || a.v_code_bytes != 1) return VQ_ERR_UNSUPPORTED;
    if (a.kv_lens) return VQ_ERR_UNSUPPORTED;
    if (choose_tables(a).mode != kModeFast) return VQ_ERR_UNSUPPORTED;
    return VQ_OK;
}

// A decode step's flags (one 8-byte word per new token and K / V) follow the
// partial records in the workspace.
size_t step_flags_offset(const AttendPlan &plan) { return (plan.ws_bytes + 15) & ~(size_t)15; }
size_t step_flags_bytes(const vq_attend_args &a) {
    return 2 * (size_t)a.B * a.H_kv * a.S_q * sizeof(unsigned long long);
}

// Work split: the (unit, key tile) space, units = (b, kv head, column
// block), is cut into equal contiguous shares, one per warp of a persistent
// grid of one CTA per SM (fewer when the problem is small).
AttendPlan plan_decode(const vq_attend_args &a, int num_sms, int reserved_warps) {
    AttendPlan p{};
    p.cols = kCols;
    const int ncols = (a.H_q / a.H_kv) * a.S_q;
    p.n_colblk = (ncols + kCols - 1) / kCols;
    int tlo = 0, T = 1;
    tile_range(a, &tlo, &T);
    p.tile_lo = tlo;
    p.tiles = T;
    const int64_t units = (int64_t)a.B * a.H_kv * p.n_colblk;
    p.total = units * T;
    const int kWarps = warps_for(a.D) - reserved_warps;   // warps with a share per CTA
    int64_t nw = (int64_t)num_sms * kWarps;
    const int64_t by_size = (p.total + kMinTilesPerWarp - 1) / kMinTilesPerWarp;
    if (nw > by_size) nw = by_size;
    if (nw > kMaxRecords) nw = kMaxRecords;   // the combine holds one factor per warp
    if (nw < 1) nw = 1;
    const int64_t share = (p.total + nw - 1) / nw;
    nw = (p.total + share - 1) / share;   // drop warps left without work
    p.n_warps = nw;
    p.share = share;
    p.grid = (int)((nw + kWarps - 1) / kWarps);
    p.slots = (int)((share + T - 1) / T + 1);
    p.n_split = 1;
    p.tok_per_split = T * kTile;
    p.ws_bytes = (size_t)nw * p.slots * kCols * (a.D + 4) * sizeof(float);
    return p;
}

AttendPlan plan_decode_capped(const vq_attend_args &a, int num_sms, size_t max_ws_bytes) {
    AttendPlan p = plan_decode(a, num_sms);
    if (p.ws_bytes <= max_ws_bytes) return p;
    // fewer warps (longer shares) until the partial records fit
    const size_t rec = (size_t)kCols * (a.D + 4) * sizeof(float);
    int64_t nw = p.n_warps;
    while (nw > 1) {
        nw = nw / 2;
        const int64_t share = (p.total + nw - 1) / nw;
        nw = (p.total + share - 1) / share;
        const int slots = (int)((share + p.tiles - 1) / p.tiles + 1);
        if ((size_t)nw * slots * rec <= max_ws_bytes) {
            p.n_warps = nw;
            p.share = share;
            p.grid = (int)((nw + warps_for(a.D) - 1) / warps_for(a.D));
            p.slots = slots;
            p.ws_bytes = (size_t)nw * slots * rec;
            return p;
        }
    }
    const int64_t units = p.total / p.tiles;
    p.n_split = 0;
    p.ws_bytes = (size_t)(units + 1) * rec;   // what a single warp would need
    return p;
}

cudaError_t launch_decode(const vq_attend_args &a, const AttendPlan &plan,
                          cudaStream_t stream, const void *k_new, const void *v_new) {
    const Tables tb = choose_tables(a);
    DecArgs da{};
    da.B = a.B; da.H_q = a.H_q; da.H_kv = a.H_kv; da.S_q = a.S_q; da.S_kv = a.S_kv;
    da.G = a.H_q / a.H_kv;
    da.q = reinterpret_cast<const __half *>(a.q_f16);
    da.kc = reinterpret_cast<const uint8_t *>(a.k_codes);
    da.kcb = a.k_code_bytes > 0 ? a.k_code_bytes : -packed_code_bits(a.k_n_centroids);
    da.krowb = a.k_code_bytes > 0 ? (a.D / a.k_sub_dim) * a.k_code_bytes
                                  : 4 * packed_row_words(a.D / a.k_sub_dim, -da.kcb);
    da.kcbk = a.k_codebook;
    da.Nk = a.k_n_centroids;
    da.vc = reinterpret_cast<const uint8_t *>(a.v_codes);
    da.vcb = a.v_code_bytes > 0 ? a.v_code_bytes : -packed_code_bits(a.v_n_centroids);
    da.vrowb = a.v_code_bytes > 0 ? (a.D / a.v_sub_dim) * a.v_code_bytes
                                  : 4 * packed_row_words(a.D / a.v_sub_dim, -da.vcb);
    da.vcbk = a.v_codebook;
    da.Nv = a.v_n_centroids;
    da.smooth = a.smooth;
    da.smooth_mode = a.smooth_mode;
    da.qscale = (float)(1.0 / sqrt((double)a.D) * (double)a.scale * kLog2e);
    da.causal = a.causal;
    da.window = a.sliding_window;
    da.stride = a.kv_stride > 0 ? a.kv_stride : a.S_kv;
    da.kv_lens = a.kv_lens;
    da.ws = reinterpret_cast<float *>(a.workspace);
    da.n_colblk = plan.n_colblk;
    da.tlo = plan.tile_lo;
    da.T = plan.tiles;
    da.total = plan.total;
    da.share = plan.share;
    da.nw = (int)plan.n_warps;
    da.slots = plan.slots;
    da.k_copies = tb.k_copies;
    da.v_copies = tb.v_copies;
    da.step = k_new != nullptr;
    da.k_new = reinterpret_cast<const __half *>(k_new);
    da.v_new = reinterpret_cast<const __half *>(v_new);
    da.new_row0 = a.S_kv - a.S_q;
    if (da.step) {
        // the new rows' flags after the records; a fresh odd epoch per launch
        // (flags left by an earlier launch are 0, and memory never written
        // by one matches an epoch only by a 2^-64 chance)
        static std::atomic<unsigned long long> epoch{
            (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() * 2ull + 1ull};
        da.step_flags = reinterpret_cast<unsigned long long *>(
            reinterpret_cast<unsigned char *>(a.workspace) + step_flags_offset(plan));
        da.step_epoch = epoch.fetch_add(2ull);
    }
    int l2d = 0;
    while ((1 << l2d) < a.D) ++l2d;
    da.log2D = l2d;
    da.out = reinterpret_cast<__half *>(a.out_f16);
    cudaError_t err;
    switch (a.D) {
        case 32: err = launch_d<32>(da, a.k_sub_dim, a.v_sub_dim, tb, plan.grid, stream); break;
        case 64: err = launch_d<64>(da, a.k_sub_dim, a.v_sub_dim, tb, plan.grid, stream); break;
        case 128: err = launch_d<128>(da, a.k_sub_dim, a.v_sub_dim, tb, plan.grid, stream); break;
        case 256: err = launch_d<256>(da, a.k_sub_dim, a.v_sub_dim, tb, plan.grid, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (err != cudaSuccess || da.step) return err;   // a step merges in its own launch
    const int64_t units = plan.total / plan.tiles;
    const int cols = min(kCols, da.G * da.S_q);   // real columns of a column block
    __half *out = reinterpret_cast<__half *>(a.out_f16);
    // records per unit: at most ceil(T / share) + 1
    const int64_t recs = (plan.tiles + plan.share - 1) / plan.share + 1;
    if (recs > kNarrowRecords) {
        const dim3 cgrid((unsigned)units, (unsigned)cols, (unsigned)(a.D / kCombDims));
        const dim3 cblock(kCombThreads);
        switch (a.D) {
            case 32: return launch_dependent(combine_wide_kernel<32>, cgrid, cblock, 0, stream, da, out);
            case 64: return launch_dependent(combine_wide_kernel<64>, cgrid, cblock, 0, stream, da, out);
            case 128: return launch_dependent(combine_wide_kernel<128>, cgrid, cblock, 0, stream, da, out);
            default: return launch_dependent(combine_wide_kernel<256>, cgrid, cblock, 0, stream, da, out);
        }
    }
    const dim3 cgrid((unsigned)units, (unsigned)cols);
    const dim3 cblock((unsigned)a.D);
    switch (a.D) {
        case 32: return launch_dependent(combine_kernel<32>, cgrid, cblock, 0, stream, da, out);
        case 64: return launch_dependent(combine_kernel<64>, cgrid, cblock, 0, stream, da, out);
        case 128: return launch_dependent(combine_kernel<128>, cgrid, cblock, 0, stream, da, out);
        default: return launch_dependent(combine_kernel<256>, cgrid, cblock, 0, stream, da, out);
    }
}

}  // namespace vqkv
