// prefill.cu -- attention over the coded cache for long query blocks on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Page: "Metal Kernels API", section "Fused SDPA", metal_fused_sdpa (SDPA on
// the dequantised cache without materialising it; causal alignment to the
// tail of the cache; sliding window; GQA), with the raw-query semantics of
// VecInferKVCache.fused_sdpa; the prefill-shaped loop over key tiles follows
// the companion kernel described under rabitq_prefill_attend (both products
// on matrix tiles, keys and values decoded inside the tile loop).
//
// The kernel below (prefill_pair_kernel) serves every GQA group size:
//   * Q~ = Hn (q (.) s_g^-1) * scale * log2(e) is built once per CTA (FWHT in
//     registers) and stored as the A operand in the canonical K-major,
//     128-byte-swizzled shared-memory layout (fp16).
//   * For every tile of 128 keys, K~ and V_hat are rebuilt from the uint8
//     codes and fp16 codebook replicas in shared memory as [keys x D] tiles
//     (one key row per thread, 128-byte swizzle): K~ is the K-major B operand
//     of S = Q~ K~^T, V_hat the MN-major B operand of O = P V_hat.
//   * tcgen05.mma kind::f16, M = N = 128, K = 16 per instruction, fp32
//     accumulation in tensor memory.
//   * Online softmax in base 2 per row, with a reference maximum that moves
//     only when a score exceeds it by more than 2^8.
//   * Key tiles that no row of the CTA can see are skipped; masks are applied
//     only on tiles that need them.
// Every mbarrier wait is bounded: if one expires the CTA writes NaN rows,
// waits (bounded) for its own MMAs once more, frees its tensor memory and
// exits, so a fault shows up in the output instead of hanging the GPU.
#include <cuda.h>
#include <math.h>

#include <mutex>

#include "vq_internal.cuh"

namespace vqkv {
namespace {

constexpr int kRows = 128;        // query rows per CTA (MMA M)
constexpr int kKeys = 128;        // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kD = 128;           // head dimension of this kernel
constexpr int kSub = 4;           // sub-vector size of both codebooks
constexpr uint32_t kTileBytes = kRows * kD * 2;  // one fp16 operand tile, 32 KiB
constexpr uint32_t kHalfTile = kTileBytes / 2;   // 64-element K half, 16 KiB
constexpr uint32_t kTabKBytes = 256 * 128;       // key centroids: 16 fp16 replicas per row
constexpr uint32_t kTabVBytes = 256 * 64;        // value centroids: 8 fp16 replicas per row
constexpr uint32_t kCodeTile = kKeys * 32;       // one tile's K (or V) codes, 4 KiB
constexpr uint32_t kStageBytes = 2 * kCodeTile;  // a ring stage: K codes | V codes
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr float kSlack = 8.f;     // base-2 headroom of a row's reference maximum

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;             // leading byte offset (unused when swizzled)
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset
    d |= (uint64_t)1 << 46;             // version
    d |= (uint64_t)2 << 61;             // 128-byte swizzle
    return d;
}

// Shared-memory matrix descriptor for an MN-major operand with the 128-byte
// swizzle: 64 MN elements (128 bytes) per row, one row per K index, 8-row
// groups 1024 bytes apart (stride byte offset, along K), 64-element MN
// blocks `mn_stride` bytes apart (leading byte offset).
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t saddr, uint32_t mn_stride) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((mn_stride >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptors, kind::f16: fp16 A and B, fp32 D, M = 128,
// N = 128; A K-major; B K-major (S = Q~ K~^T) or MN-major (O = P V_hat).
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kKeys >> 3) << 17) |
                            ((uint32_t)(kRows >> 4) << 24);
constexpr uint32_t kIdescBmn = kIdesc | (1u << 16);

// 32 consecutive fp32 columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
          "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Byte offset of the 16-byte chunk `chunk` (8 fp16 along K) of row `row` in a
// K-major operand tile made of two 64-element K halves of [128 rows x 128 B]
// with the 128-byte swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw_off(int row, int chunk) {
    const int half = chunk >> 3, c = chunk & 7;
    return (uint32_t)(half * kHalfTile + row * 128 + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(addr), "r"(a), "r"(b),
                 "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

struct PrefillArgs {
    int B, H_q, H_kv, S_q, S_kv, G;
    const __half *q;
    const uint8_t *kc, *vc;       // uint8 codes, 32 per key
    const float *kcb, *vcb;       // [Nk, 4], [Nv, 4] fp32
    int Nk, Nv;
    const float *smooth;
    int smooth_mode;
    float qscale;                 // scale * log2(e) / sqrt(D), folded into Q~
    int causal, window;
    int64_t stride;               // code rows per (b, kv head)
    const int32_t *kv_lens;       // keys held by each batch, or null (all S_kv)
    __half *out;
};

// ------------------------------------------------------------------ two heads per CTA
//
// prefill_pair_kernel: one CTA = (batch, two query heads of one KV group,
// tile of 128 query rows), 416 threads in four roles; an odd group's last
// pair has a single head (head B's warps idle, its products skipped).  The
// two heads share the rebuilt K~ and V_hat tiles of their KV head, and the
// two heads' products and softmaxes interleave so that the tensor cores run
// one head's product while the CUDA cores run the other head's softmax.
//   * warps 0-3 / 4-7: softmax of head A / head B; thread = query row r
//     (tensor-memory lane r), the whole 128-score row of a tile.  P (fp16) is
//     written back into the first 64 columns of the row's own score columns
//     and is read from there as the A operand of O += P V_hat.
//   * warps 8-11: rebuild of K~(j) (one buffer) and V_hat(j) (two buffers)
//     from the codes, one key row per thread; codes of tile j+1 load ahead.
//   * warp 12: tensor-memory allocation and every tcgen05.mma, in the order
//     S_A(j), S_B(j), then per tile PV_A(j), S_A(j+1), PV_B(j), S_B(j+1).
//     The whole warp runs the loop (its waits and operand descriptors stay
//     warp-uniform) and one elected lane issues each instruction.  A score
//     block is overwritten only after the product that read its P has
//     completed.
// Tensor memory (512 columns): S_A | S_B | O_A | O_B.  O stays in tensor
// memory for the whole key range; when a row's reference maximum moves, the
// softmax thread rescales its P columns already written in this tile and its
// O row (the previous P V_hat of that head has completed by then: the score
// block it waits for was issued after it).
// Every wait is bounded and also gives up once another role has failed; the
// verdict is CTA-wide (NaN rows), and the MMA warp drains its products
// before tensor memory is freed.

constexpr int kPairThreads = 416;
constexpr int kRebuildWarp = 8;   // first warp of the rebuild role
constexpr int kMmaWarp = 12;
constexpr int kPairCols = 512;    // tensor-memory columns
enum PairBar {
    kBarSA, kBarSB,       // score block of head A / B complete (commit)
    kBarOA, kBarOB,       // P V_hat of head A / B complete (commit)
    kBarPA, kBarPB,       // P of head A / B written (one arrival per warp)
    kBarK,                // K~ written (one arrival per warp)
    kBarV0, kBarV1,       // V_hat buffer 0 / 1 written (one arrival per warp)
    kBarVF0, kBarVF1,     // V_hat buffer 0 / 1 free again (commit)
    kBarDrain,            // every issued product complete (commit)
    kBarC0, kBarC1,       // code stage 0 / 1 loaded (tensor copies, transaction bytes)
    kBarE0, kBarE1,       // code stage 0 / 1 read (one arrival per rebuild warp)
    kNumPairBars
};

__device__ __forceinline__ uint32_t mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void warp_arrive(uint32_t bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Bounded wait by a whole warp: every lane polls and all leave together.
// False on timeout (which raises the CTA's failure flag) or once another
// role has raised it.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *fail) {
    for (uint32_t it = 0; it < kWaitLimit; ++it) {
        if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
        if ((it & 255u) == 255u && __any_sync(0xffffffffu, *fail != 0)) return false;
    }
    *fail = 1;
    return false;
}

// Products D (tensor memory) += A x B with A in shared memory (ss) or in
// tensor memory (ts, K-major) and B in shared memory, and the commit, each
// issued by one lane of a converged warp (elect.sync): the warp runs the
// issue loop together, so its operand descriptors stay warp-uniform and a
// product costs a few instructions.
__device__ __forceinline__ void mma_ss_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred e, p;\n .reg .b32 lid;\n"
        " elect.sync lid|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred e, p;\n .reg .b32 lid;\n"
        " elect.sync lid|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void commit_elect(uint32_t bar) {
    asm volatile(
        "{\n .reg .pred e;\n .reg .b32 lid;\n elect.sync lid|e, 0xffffffff;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n"
        ::"r"(bar) : "memory");
}

// 16 consecutive 32-bit columns of this thread's lane, load and store.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// 64 consecutive fp32 columns of this thread's lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float *v) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
          "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
          "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
          "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]),
          "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]),
          "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
          "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
          "r"(r[13]), "r"(r[14]), "r"(r[15]) : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
        ::"r"(taddr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),
          "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]),
          "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
          "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]),
          "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]),
          "f"(v[31]) : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// In-register Walsh-Hadamard butterflies h = 1 .. 32 over 64 values.
__device__ __forceinline__ void fwht64(float *x) {
#pragma unroll
    for (int h = 1; h < 64; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            if ((i & h) == 0) {
                const float u = x[i], v = x[i + h];
                x[i] = u + v;
                x[i + h] = u - v;
            }
        }
    }
}

// One tile of code rows (128 rows of 32 bytes, starting at row `row` of the
// tensor map's [rows x 32 bytes] view of a code buffer) into shared memory by
// the tensor copy engine, completing on `bar` (rows past the buffer read as
// zero).  The innermost coordinate is 0: 16-byte aligned.
__device__ __forceinline__ void tma_code_tile(uint32_t dst, const CUtensorMap *map, int row,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n"
                 ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__global__ void __launch_bounds__(kPairThreads, 1)
prefill_pair_kernel(PrefillArgs a, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned: Q~_A | Q~_B | K~ | V_hat 0 | V_hat 1 | key table |
    // value table | code ring (2 stages) | misc
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *gbase = smem_raw + (base - raw);
    const uint32_t sQ = base, sK = base + 2 * kTileBytes, sV = base + 3 * kTileBytes,
                   sTabK = base + 5 * kTileBytes, sTabV = sTabK + kTabKBytes,
                   sRing = sTabV + kTabVBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(gbase + (sRing - base) + 2 * kStageBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumPairBars);
    volatile int *fail = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *rs = reinterpret_cast<float *>(tmem_slot + 2);   // [kD] 1 / s_g
    const uint32_t bar0 = smem_u32(bars);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qt = blockIdx.x, b = blockIdx.z;
    // blockIdx.y = (KV group g, pair of its query heads): heads hq0 (A) and
    // hq0 + 1 (B); an odd group's last pair has no head B
    const int pairs = (a.G + 1) / 2;
    const int g = blockIdx.y / pairs;
    const int hq0 = g * a.G + 2 * (blockIdx.y - g * pairs);
    const bool has_b = hq0 + 1 < (g + 1) * a.G;
    const int q0 = qt * kRows;

    // ---- key tiles visible to some row of the tile (shared by both heads;
    //      batch b holds L keys)
    const int L = a.kv_lens ? min(max(a.kv_lens[b], 0), a.S_kv) : a.S_kv;
    const int last_row = min(q0 + kRows, a.S_q) - 1;
    const int qa_first = L - a.S_q + q0, qa_last = L - a.S_q + last_row;
    const int cta_lo = a.window > 0 ? max(0, qa_first - a.window + 1) : 0;
    const int cta_hi = min(a.causal ? qa_last : L - 1, L - 1);
    const int all_lo = a.window > 0 ? max(0, qa_last - a.window + 1) : 0;   // seen by every row
    const int all_hi = min(a.causal ? qa_first : L - 1, L - 1);
    const int t_first = cta_lo / kKeys;
    const int t_last = cta_hi < cta_lo ? t_first - 1 : cta_hi / kKeys;   // none: empty range
    const int n_tiles = t_last - t_first + 1;

    // code tiles come from a ring of two stages filled by the tensor copy
    // engine: tile t_first + i in stage i mod 2, its copy issued (by the
    // first rebuild thread) once every rebuild warp has read tile i - 2
    const int64_t bg = (int64_t)b * a.H_kv + g;
    const int code_row0 = (int)(bg * a.stride);   // tensor-map row of key 0 of (b, g)
    const bool producer = tid == kRebuildWarp * 32;
    auto issue_codes = [&](int tile) {   // producer only
        const int st = (tile - t_first) & 1;
        const uint32_t dst = sRing + (uint32_t)st * kStageBytes;
        mbar_expect_tx(bar(kBarC0 + st), kStageBytes);
        tma_code_tile(dst, &tm_k, code_row0 + tile * kKeys, bar(kBarC0 + st));
        tma_code_tile(dst + kCodeTile, &tm_v, code_row0 + tile * kKeys, bar(kBarC0 + st));
    };
    uint32_t kcw[8], vcw[8];   // rebuild role: the 32 K and V codes of its key row

    // ---- prologue, the roles side by side: the MMA warp allocates tensor
    //      memory and sets up the barriers; the rebuild warps start the first
    //      tile's code loads, then build the codebook replicas; the softmax
    //      warps build Q~ (their own smooth reciprocals)
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                     ::"r"(smem_u32(tmem_slot)), "r"(kPairCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
        if (lane == 0) {
            for (int i = 0; i < kBarC0; ++i) {
                const bool commit = i == kBarSA || i == kBarSB || i == kBarOA || i == kBarOB ||
                                    i == kBarVF0 || i == kBarVF1 || i == kBarDrain;
                mbar_init(bar(i), commit ? 1u : 4u);
            }
            *fail = 0;
            asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        }
    } else if (warp >= kRebuildWarp) {
        // the copies of the first two tiles' codes (in flight during the
        // table build), then the fp16 codebook replicas: key table row c =
        // centroid c x16, value table row c = centroid c x8
        const int t = tid - kRebuildWarp * 32;
        if (producer) {
            // the ring's barriers, then the first two tiles' copies
            mbar_init(bar(kBarC0), 1u);
            mbar_init(bar(kBarC1), 1u);
            mbar_init(bar(kBarE0), 4u);
            mbar_init(bar(kBarE1), 4u);
            asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
            fence_proxy_async();
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
            if (n_tiles > 0) issue_codes(t_first);
            if (n_tiles > 1) issue_codes(t_first + 1);
        }
        for (int c = t; c < 256; c += 128) {
            uint32_t k0 = 0u, k1 = 0u, v0 = 0u, v1 = 0u;
            if (c < a.Nk) {
                const float4 f = *reinterpret_cast<const float4 *>(a.kcb + c * kSub);
                k0 = pack_h2(f.x, f.y);
                k1 = pack_h2(f.z, f.w);
            }
            if (c < a.Nv) {
                const float4 f = *reinterpret_cast<const float4 *>(a.vcb + c * kSub);
                v0 = pack_h2(f.x, f.y);
                v1 = pack_h2(f.z, f.w);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) sts128(sTabK + (uint32_t)c * 128u + q * 16u, k0, k1, k0, k1);
#pragma unroll
            for (int q = 0; q < 4; ++q) sts128(sTabV + (uint32_t)c * 64u + q * 16u, v0, v1, v0, v1);
        }
    } else {
        // smooth reciprocals of the group (threads of head A), shared by
        // the eight softmax warps through a named barrier
        if (tid < kD) {
            const float *sp = a.smooth_mode == 2 ? a.smooth + (size_t)g * kD : a.smooth;
            rs[tid] = a.smooth_mode != 0 ? 1.f / sp[tid] : 1.f;
        }
        asm volatile("bar.sync 1, 256;\n" ::: "memory");
        if (warp < 4 || has_b) {
            // ---- Q~ row r of head h (fp16, swizzled A operand): each half's
            //      butterflies below 64 in registers, the first half parked in
            //      the K~ / V_hat region (free until the loop), then the stage
            //      h = 64 pairs the halves: x[i], x[i + 64] -> sum, difference.
            const int h = warp >> 2, r = tid & (kRows - 1), row = q0 + r;
            float *xs = reinterpret_cast<float *>(gbase + 2 * kTileBytes) + h * (kD / 2) * kRows;
            const __half *qp = a.q + (((int64_t)b * a.H_q + hq0 + h) * a.S_q + row) * kD;
            // both halves' loads in flight before the first butterflies
            uint4 raw[kD / 8];
#pragma unroll
            for (int e = 0; e < kD / 8; ++e)
                raw[e] = row < a.S_q ? *reinterpret_cast<const uint4 *>(qp + 8 * e)
                                     : make_uint4(0u, 0u, 0u, 0u);
            float x[kD / 2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int e = 0; e < kD / 2; e += 8) {
                    const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw[(half * 64 + e) / 8]);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 f = __half22float2(h2[k]);
                        x[e + 2 * k] = f.x * rs[half * 64 + e + 2 * k];
                        x[e + 2 * k + 1] = f.y * rs[half * 64 + e + 2 * k + 1];
                    }
                }
                fwht64(x);
                if (half == 0) {
#pragma unroll
                    for (int e = 0; e < kD / 2; ++e) xs[e * kRows + r] = x[e];
                }
            }
            const uint32_t sQh = sQ + (uint32_t)h * kTileBytes;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                float lo8[8], hi8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float u = xs[(ch * 8 + k) * kRows + r], v = x[ch * 8 + k];
                    lo8[k] = (u + v) * a.qscale;
                    hi8[k] = (u - v) * a.qscale;
                }
                sts128(sQh + sw_off(r, ch), pack_h2(lo8[0], lo8[1]), pack_h2(lo8[2], lo8[3]),
                       pack_h2(lo8[4], lo8[5]), pack_h2(lo8[6], lo8[7]));
                sts128(sQh + sw_off(r, 8 + ch), pack_h2(hi8[0], hi8[1]), pack_h2(hi8[2], hi8[3]),
                       pack_h2(hi8[4], hi8[5]), pack_h2(hi8[6], hi8[7]));
            }
            fence_proxy_async();
        }
    }
    tc_fence_before();
    __syncthreads();   // tensor memory, barriers, tables and Q~ ready; scratch free
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // softmax role: head h, row r (tensor-memory lane r)
    const int h = (warp >> 2) & 1, r = tid & (kRows - 1), row = q0 + r;
    const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lanes + (uint32_t)(h * kKeys);
    const uint32_t t_o = tmem + lanes + (uint32_t)(2 * kKeys + h * kD);
    float l = 0.f;
    if (warp < kRebuildWarp) {
        // ================= softmax of head h, row r
        const int q_abs = L - a.S_q + row;
        const int t_end = h == 0 || has_b ? t_last : t_first - 1;   // no head B: no tiles
        int hi = a.causal ? q_abs : L - 1;
        hi = min(hi, L - 1);
        int lo = a.window > 0 ? max(0, q_abs - a.window + 1) : 0;
        if (row >= a.S_q) { lo = 1; hi = 0; }
        float m = -INFINITY;
        uint32_t ph = 0;
        for (int tile = t_first; tile <= t_end; ++tile) {
            if (!warp_wait(bar(kBarSA + h), ph, fail)) break;
            ph ^= 1;
            tc_fence_after();
            const int j0 = tile * kKeys;
            const bool full = j0 >= all_lo && j0 + kKeys - 1 <= all_hi;
            float alpha_o = 1.f;   // rescale owed by this row's O
            // the row in two 64-column halves (one tcgen05.ld each); P of half
            // c goes to columns [32 c, 32 c + 32), all of them already read
#pragma unroll 1
            for (int c = 0; c < kKeys / 64; ++c) {
                float sv[64];
                tmem_ld64(t_s + c * 64, sv);
                if (!full) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const int j = j0 + c * 64 + i;
                        sv[i] = (j >= lo && j <= hi) ? sv[i] : -INFINITY;
                    }
                }
                // four independent maximum chains
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int i = 0; i < 64; i += 8) {
                    mx0 = max3f(mx0, sv[i], sv[i + 1]);
                    mx1 = max3f(mx1, sv[i + 2], sv[i + 3]);
                    mx2 = max3f(mx2, sv[i + 4], sv[i + 5]);
                    mx3 = max3f(mx3, sv[i + 6], sv[i + 7]);
                }
                const float cmax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                // the reference maximum moves only past kSlack (base 2)
                const bool moves = cmax > m + kSlack;
                if (__any_sync(0xffffffffu, moves)) {
                    const float alpha = moves ? ex2(m - cmax) : 1.f;   // 0 from -inf
                    if (moves) {
                        l *= alpha;
                        alpha_o *= alpha;
                        m = cmax;
                    }
                    // P columns already written in this tile, rescaled
                    if (c > 0) tmem_wait_st();
                    for (int cc = 0; cc < 2 * c; ++cc) {
                        uint32_t pw[16];
                        tmem_ld16(t_s + cc * 16, pw);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 f = __half22float2(*reinterpret_cast<__half2 *>(&pw[i]));
                            pw[i] = pack_h2(f.x * alpha, f.y * alpha);
                        }
                        tmem_st16(t_s + cc * 16, pw);
                    }
                }
                const float base_m = m == -INFINITY ? 0.f : m;
                float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float p0 = ex2(sv[q * 32 + i] - base_m);
                        const float p1 = ex2(sv[q * 32 + i + 1] - base_m);
                        const float p2 = ex2(sv[q * 32 + i + 2] - base_m);
                        const float p3 = ex2(sv[q * 32 + i + 3] - base_m);
                        ls0 += p0 + p1;
                        ls1 += p2 + p3;
                        pk[i / 2] = pack_h2(p0, p1);
                        pk[i / 2 + 1] = pack_h2(p2, p3);
                    }
                    tmem_st16(t_s + c * 32 + q * 16, pk);
                }
                l += ls0 + ls1;
            }
            // the row's O (all earlier tiles' P V_hat, complete) follows the
            // moved maximum; on the first tile the product overwrites O
            if (tile > t_first && __any_sync(0xffffffffu, alpha_o != 1.f)) {
#pragma unroll 1
                for (int c = 0; c < kD / 32; ++c) {
                    float ov[32];
                    tmem_ld32(t_o + c * 32, ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] *= alpha_o;
                    tmem_st32(t_o + c * 32, ov);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(bar(kBarPA + h));
        }
        __syncwarp();
    } else if (warp < kMmaWarp) {
        // ================= rebuild of K~ and V_hat, key row r of each tile
        const int r = tid - kRebuildWarp * 32;
        // gather address of code byte i of word w: a byte permute gives
        // code * 256 + o, shifted down to the table's row size -- key rows of
        // 128 bytes (the lane's replica (lane mod 16) * 8, o = 2x that),
        // value rows of 64 bytes (replica (lane mod 8) * 8, o = 4x that)
        const uint32_t ok2 = (uint32_t)((lane & 15) * 16), ov4 = (uint32_t)((lane & 7) * 32);
        auto build_row = [&](const uint32_t *cw, uint32_t dst, uint32_t tab, uint32_t o, int sh) {
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                const uint32_t w = cw[ch >> 1];
                const uint32_t i0 = (uint32_t)(ch & 1) * 2u;
                const uint2 e0 = lds64(tab + (__byte_perm(w, o, 0x6504u | (i0 << 4)) >> sh));
                const uint2 e1 = lds64(tab + (__byte_perm(w, o, 0x6504u | ((i0 + 1u) << 4)) >> sh));
                sts128(dst + sw_off(r, ch), e0.x, e0.y, e1.x, e1.y);
            }
        };
        uint32_t ph_sb = 0, ph_vf = 0;   // ph_vf: bit b = parity of V_hat buffer b
        int issued = n_tiles > 1 ? t_first + 1 : t_last;   // last tile whose copy was issued
        int consumed = t_first - 1;                           // last tile read from the ring
        for (int tile = t_first; tile <= t_last; ++tile) {
            const int i = tile - t_first, st = i & 1;
            // this tile's codes (row r of its stage), then the stage back to
            // the producer, which refills it with tile + 2
            if (!warp_wait(bar(kBarC0 + st), (uint32_t)((i >> 1) & 1), fail)) break;
            consumed = tile;
            {
                const uint32_t src = sRing + (uint32_t)st * kStageBytes + (uint32_t)r * 32u;
                const uint4 c0 = lds128(src), c1 = lds128(src + 16);
                const uint4 d0 = lds128(src + kCodeTile), d1 = lds128(src + kCodeTile + 16);
                kcw[0] = c0.x; kcw[1] = c0.y; kcw[2] = c0.z; kcw[3] = c0.w;
                kcw[4] = c1.x; kcw[5] = c1.y; kcw[6] = c1.z; kcw[7] = c1.w;
                vcw[0] = d0.x; vcw[1] = d0.y; vcw[2] = d0.z; vcw[3] = d0.w;
                vcw[4] = d1.x; vcw[5] = d1.y; vcw[6] = d1.z; vcw[7] = d1.w;
            }
            warp_arrive(bar(kBarE0 + st));
            if (warp == kRebuildWarp && tile + 2 <= t_last) {
                if (!warp_wait(bar(kBarE0 + st), (uint32_t)((i >> 1) & 1), fail)) break;
                if (producer) {
                    fence_proxy_async();   // the stage's reads before the copy's writes
                    issue_codes(tile + 2);
                }
                issued = tile + 2;
                __syncwarp();
            }
            if (i > 0) {   // the score blocks of the previous tile read K~
                if (!warp_wait(bar(has_b ? kBarSB : kBarSA), ph_sb, fail)) break;
                ph_sb ^= 1;
            }
            build_row(kcw, sK, sTabK, ok2, 1);
            fence_proxy_async();
            warp_arrive(bar(kBarK));
            const int vb = i & 1;
            if (i > 1) {   // the products of tile - 2 read this V_hat buffer
                if (!warp_wait(bar(kBarVF0 + vb), (ph_vf >> vb) & 1u, fail)) break;
                ph_vf ^= 1u << vb;
            }
            build_row(vcw, sV + (uint32_t)vb * kTileBytes, sTabV, ov4, 2);
            fence_proxy_async();
            warp_arrive(bar(kBarV0 + vb));
        }
        // after a failure: the producer's warp waits (bounded, whatever the
        // failure flag) for its copies still in flight before the CTA can end
        if (warp == kRebuildWarp) {
            for (int tile = consumed + 1; tile <= issued; ++tile) {
                const int i = tile - t_first;
                bool done = false;
                for (uint32_t it = 0; it < kWaitLimit && !done; ++it)
                    done = __all_sync(0xffffffffu, mbar_try(bar(kBarC0 + (i & 1)), (uint32_t)((i >> 1) & 1)));
            }
        }
        __syncwarp();
    } else {
        // ================= tensor-core issue: the warp runs the loop (uniform
        // waits and descriptors), one elected lane issues each instruction.
        // A descriptor's start address is its low 14 bits (address / 16), so
        // an operand offset is added to a base descriptor as offset / 16.
        if (n_tiles > 0) {
            const uint64_t dq0 = smem_desc(sQ), dq1 = smem_desc(sQ + kTileBytes);
            const uint64_t dk = smem_desc(sK);
            const uint64_t dv0 = smem_desc_mn(sV, kHalfTile), dv1 = smem_desc_mn(sV + kTileBytes, kHalfTile);
            auto issue_s = [&](int hh) {
                const uint64_t dq = hh ? dq1 : dq0;
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    const uint32_t off = (uint32_t)((ks >> 2) * kHalfTile + (ks & 3) * 32);
                    mma_ss_elect(tmem + (uint32_t)(hh * kKeys), dq + (off >> 4), dk + (off >> 4),
                                 kIdesc, ks > 0);
                }
                commit_elect(bar(kBarSA + hh));
            };
            auto issue_pv = [&](int hh, int vb, bool acc) {
                const uint64_t dv = vb ? dv1 : dv0;
#pragma unroll
                for (int ks = 0; ks < kKeys / 16; ++ks) {
                    // A = P: keys 16 ks .. 16 ks + 15 in columns 8 ks .. 8 ks + 7
                    mma_ts_elect(tmem + (uint32_t)(2 * kKeys + hh * kD),
                                 tmem + (uint32_t)(hh * kKeys + ks * 8),
                                 dv + (uint64_t)(ks * 128), kIdescBmn, (acc || ks > 0) ? 1u : 0u);
                }
                commit_elect(bar(kBarOA + hh));
            };
            uint32_t ph_k = 0, ph_v = 0, ph_p[2] = {0u, 0u}, ph_o[2] = {0u, 0u};   // ph_v: bit b per buffer
            bool ok = warp_wait(bar(kBarK), ph_k, fail);
            ph_k ^= 1;
            if (ok) {
                tc_fence_after();
                issue_s(0);
                if (has_b) issue_s(1);
            }
            for (int tile = t_first; ok && tile <= t_last; ++tile) {
                const int i = tile - t_first, vb = i & 1;
                const bool more = tile < t_last;
                if (!(ok = warp_wait(bar(kBarV0 + vb), (ph_v >> vb) & 1u, fail))) break;
                ph_v ^= 1u << vb;
                if (!(ok = warp_wait(bar(kBarPA), ph_p[0], fail))) break;
                ph_p[0] ^= 1;
                tc_fence_after();
                issue_pv(0, vb, i > 0);
                if (more) {
                    if (!(ok = warp_wait(bar(kBarK), ph_k, fail))) break;
                    ph_k ^= 1;
                    if (!(ok = warp_wait(bar(kBarOA), ph_o[0], fail))) break;
                    ph_o[0] ^= 1;
                    tc_fence_after();
                    issue_s(0);
                }
                if (has_b) {
                    if (!(ok = warp_wait(bar(kBarPB), ph_p[1], fail))) break;
                    ph_p[1] ^= 1;
                    tc_fence_after();
                    issue_pv(1, vb, i > 0);
                }
                commit_elect(bar(kBarVF0 + vb));
                if (more && has_b) {
                    if (!(ok = warp_wait(bar(kBarOB), ph_o[1], fail))) break;
                    ph_o[1] ^= 1;
                    tc_fence_after();
                    issue_s(1);
                }
            }
            // every product issued completes before the output is read and
            // tensor memory is freed
            commit_elect(bar(kBarDrain));
            bool drained = false;
            for (uint32_t it = 0; it < kWaitLimit && !drained; ++it)
                drained = __all_sync(0xffffffffu, mbar_try(bar(kBarDrain), 0u));
            if (!drained && lane == 0) *fail = 1;
        }
        __syncwarp();
    }
    if (warp < kRebuildWarp && (h == 0 || has_b)) {
        // ---- output row r of head h, as soon as the head's last P V_hat has
        //      completed (the other head's last tile may still be running).
        //      Its completion is phase n_tiles - 1 of the head's O barrier:
        //      this warp saw S(last) complete, which was issued only after
        //      phase n_tiles - 2 had completed, so the parity wait cannot
        //      match an earlier phase.  (tcgen05.ld is warp-collective: every
        //      lane loads, only rows of the query block are stored.)
        bool have_o = n_tiles > 0 && *fail == 0;
        if (have_o) have_o = warp_wait(bar(kBarOA + h), (uint32_t)((n_tiles - 1) & 1), fail);
        tc_fence_after();
        const bool failed = *fail != 0;
        have_o = have_o && !failed;
        const float inv = failed ? __int_as_float(0x7fc00000) : (l > 0.f ? 1.f / l : 0.f);
        __half *op = a.out + (((int64_t)b * a.H_q + hq0 + h) * a.S_q + row) * kD;
#pragma unroll 1
        for (int c = 0; c < kD / 32; ++c) {
            float ov[32];
            if (have_o) {
                tmem_ld32(t_o + c * 32, ov);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) ov[i] = 0.f;
            }
            if (row < a.S_q) {
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const float *p = ov + ch * 8;
                    uint4 v;
                    v.x = pack_h2(p[0] * inv, p[1] * inv);
                    v.y = pack_h2(p[2] * inv, p[3] * inv);
                    v.z = pack_h2(p[4] * inv, p[5] * inv);
                    v.w = pack_h2(p[6] * inv, p[7] * inv);
                    *reinterpret_cast<uint4 *>(op + c * 32 + ch * 8) = v;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n"
                     ::"r"(tmem), "r"(kPairCols));
    }
}

size_t prefill_pair_smem_bytes() {
    return 5 * (size_t)kTileBytes + kTabKBytes + kTabVBytes + 2 * (size_t)kStageBytes +
           kNumPairBars * 8 + 8 + kD * sizeof(float) + 1024;   // + alignment slack
}

// cuTensorMapEncodeTiled, looked up once through the runtime (the library
// links no driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Tensor map of a uint8 code buffer seen as [rows x 32 bytes]; tiles of
// 128 rows.
bool code_tensor_map(CUtensorMap *m, const void *codes, uint64_t rows) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {32, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {32};
    const cuuint32_t box[2] = {32, (cuuint32_t)kKeys};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(codes), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int prefill_supported(const vq_attend_args &a) {
    if (a.D != kD || a.k_sub_dim != kSub || a.v_sub_dim != kSub) return VQ_ERR_UNSUPPORTED;
    if (a.k_code_bytes != 1 || a.v_code_bytes != 1) return VQ_ERR_UNSUPPORTED;
    if (a.k_n_centroids > 256 || a.v_n_centroids > 256) return VQ_ERR_UNSUPPORTED;
    if (a.S_q < 64) return VQ_ERR_UNSUPPORTED;
    // code tiles are addressed by 32-bit tensor-map row coordinates
    const int64_t stride = a.kv_stride > 0 ? a.kv_stride : a.S_kv;
    if ((int64_t)a.B * a.H_kv * stride + kKeys >= ((int64_t)1 << 31)) return VQ_ERR_UNSUPPORTED;
    return VQ_OK;
}

cudaError_t launch_prefill(const vq_attend_args &a, cudaStream_t stream) {
    PrefillArgs p{};
    p.B = a.B; p.H_q = a.H_q; p.H_kv = a.H_kv; p.S_q = a.S_q; p.S_kv = a.S_kv;
    p.G = a.H_q / a.H_kv;
    p.q = reinterpret_cast<const __half *>(a.q_f16);
    p.kc = reinterpret_cast<const uint8_t *>(a.k_codes);
    p.vc = reinterpret_cast<const uint8_t *>(a.v_codes);
    p.kcb = a.k_codebook;
    p.vcb = a.v_codebook;
    p.Nk = a.k_n_centroids;
    p.Nv = a.v_n_centroids;
    p.smooth = a.smooth;
    p.smooth_mode = a.smooth_mode;
    p.qscale = (float)((double)a.scale * 1.4426950408889634 / sqrt((double)kD));
    p.causal = a.causal;
    p.window = a.sliding_window;
    p.stride = a.kv_stride > 0 ? a.kv_stride : a.S_kv;
    p.kv_lens = a.kv_lens;
    p.out = reinterpret_cast<__half *>(a.out_f16);
    const unsigned q_tiles = (unsigned)((a.S_q + kRows - 1) / kRows);
    // up to two query heads of one KV group per CTA
    const size_t smem = prefill_pair_smem_bytes();
    cudaError_t err = cudaFuncSetAttribute(prefill_pair_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    CUtensorMap tmk, tmv;
    const uint64_t rows = (uint64_t)a.B * a.H_kv * (uint64_t)p.stride;
    if (!code_tensor_map(&tmk, a.k_codes, rows) || !code_tensor_map(&tmv, a.v_codes, rows))
        return cudaErrorInvalidValue;
    dim3 grid(q_tiles, (unsigned)(a.H_kv * ((p.G + 1) / 2)), (unsigned)a.B);
    prefill_pair_kernel<<<grid, kPairThreads, smem, stream>>>(p, tmk, tmv);
    return cudaGetLastError();
}

}  // namespace vqkv
