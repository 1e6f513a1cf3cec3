/*
 * vqkv.h -- C ABI of libvqkv.so, a product-vector-quantised KV cache for
 * NVIDIA GB300 (sm_103a).
 *
 * The operations follow three documentation pages of a VecInfer-style cache:
 *   "Metal Kernels API" (veloxquant.dev/docs/api/metal-api), sections
 *     "VecInfer kernels" and "Fused SDPA";
 *   "Metal GPU Kernels" guide (veloxquant.dev/docs/guides/metal-kernels),
 *     section "Fused SDPA kernel";
 *   "veloxquant_mlx.cache.vecinfer_cache module" (VecInferKVCache).
 * Each entry point below names the passage that defines it.
 *
 * Conventions shared by every entry point
 *   - Tensors are caller-owned, contiguous, row-major, and live in device
 *     memory (or memory the device can address).  The library allocates
 *     nothing and keeps no state between calls; scratch space, where an
 *     operation needs it, is passed in by the caller.
 *   - fp16 tensors are IEEE binary16 (passed as void*); codebooks, smooth
 *     factors and fp32 outputs are IEEE binary32.
 *   - Codes are unsigned integers of `code_bytes` bytes each: 1 (uint8,
 *     n_centroids <= 256) or 2 (uint16, n_centroids <= 65536); or
 *     code_bytes = 0: bit-packed rows (page "veloxquant_mlx.cache.
 *     vecinfer_cache module": (D / sub_dim) * b / 8 bytes per token).  Then
 *     b = ceil(log2 n_centroids) (at least 1, n_centroids <= 65536) bits per
 *     code, the D / sub_dim codes of one vector form a little-endian bit
 *     stream (code m in bits [m b, m b + b)), and every vector's row is padded
 *     to whole 32-bit words: a "[..., D/sub_dim]" code tensor becomes
 *     "[..., ceil(D/sub_dim * b / 32)]" words.
 *   - Every pointer must be 16-byte aligned (vectorised 128-bit accesses).
 *   - Checks run in this order: sizes (VQ_ERR_SHAPE), limits
 *     (VQ_ERR_UNSUPPORTED), then -- unless the problem is empty, which
 *     returns VQ_OK without reading any pointer -- pointers (VQ_ERR_NULL)
 *     and alignment (VQ_ERR_ALIGN), then workspace size.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  All work is enqueued asynchronously on it; arguments are
 *     validated on the host before anything is enqueued, so an error status
 *     means nothing was launched (except VQ_ERR_CUDA, which reports a failed
 *     launch).
 *   - The attention kernels are launched as programmatic dependents: when
 *     the preceding work on the stream is a vq_encode_* call, they may start
 *     staging their codebooks while that encode finishes, and read every
 *     other input (codes, queries, smooth factors) only after it completed.
 *     So an attention call's codebooks must not be outputs of the encode call
 *     enqueued just before it (codes and reconstructions never are).
 *   - The library never aborts, exits or traps on the device.
 */
#ifndef VQKV_H_
#define VQKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VQ_API __attribute__((visibility("default")))
#else
#define VQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VQ_OK = 0,
    VQ_ERR_NULL = -1,        /* a required pointer is NULL                   */
    VQ_ERR_SHAPE = -2,       /* inconsistent sizes (e.g. D % sub_dim != 0)   */
    VQ_ERR_UNSUPPORTED = -3, /* valid request outside this build's limits    */
    VQ_ERR_ALIGN = -4,       /* a pointer is not 16-byte aligned             */
    VQ_ERR_WORKSPACE = -5,   /* workspace missing or smaller than required   */
    VQ_ERR_CUDA = -6         /* a CUDA launch or query failed                */
} vq_status;

/* Static, human-readable description of a status code (never NULL). */
VQ_API const char *vq_status_str(int status);

/*
 * Key encode.  Page: "Metal Kernels API", section "VecInfer kernels",
 * vecinfer_encode_decode_metal (smooth -> Walsh-Hadamard transform -> VQ
 * encode -> dequant -> inverse-WHT -> inverse-smooth), with the search of
 * vecinfer_quantize_metal; the module summary of
 * "veloxquant_mlx.cache.vecinfer_cache" describes the same smooth + rotation.
 *
 *   keys_f16   [B, H, S, D] fp16.
 *   codebook   [n_centroids, sub_dim] fp32, shared by all sub-vector
 *              positions and heads.
 *   smooth     smooth_mode 0: NULL (no smoothing); 1: [D]; 2: [H, D] fp32,
 *              finite and non-zero.
 *   codes      [B, H, S, D/sub_dim] of code_bytes each (output).
 *   k_hat_f16  [B, H, S, D] fp16 reconstruction (output) or NULL to skip.
 *
 * Per vector x of head h: y = Hn (s_h (.) x) with Hn the normalised
 * Sylvester-Hadamard matrix; code_m = the nearest centroid of sub-vector
 * y[m*sub_dim : (m+1)*sub_dim] by squared Euclidean distance, the lowest
 * index on ties; k_hat = s_h^-1 (.) Hn concat_m codebook[code_m], rounded to
 * fp16 (nearest even).  The search runs in fp32; a decision that a rigorous
 * bound on the fp32 rounding (of y and of the distances) cannot certify is
 * taken again in float-float arithmetic (about 44 significant bits), so a
 * code differs from the exact nearest centroid of the exact y only where
 * two squared distances agree to about 1e-10 relative.
 *
 * Errors: VQ_ERR_NULL (keys, codebook, codes, or smooth when smooth_mode
 * != 0), VQ_ERR_SHAPE (a size < 0, D % sub_dim != 0, smooth_mode not in
 * 0..2, code_bytes not 1 or 2), VQ_ERR_UNSUPPORTED (D not a power of two in
 * [32, 512], sub_dim not in {1, 2, 4, 8, 16}, n_centroids < 1 or above the
 * code width, or a codebook larger than 160 KiB), VQ_ERR_ALIGN, VQ_ERR_CUDA.
 * B, H or S equal to 0 is a no-op (pointers may then be NULL).
 */
VQ_API int vq_encode_keys(const void *keys_f16, int B, int H, int S, int D,
                   const float *codebook, int n_centroids, int sub_dim,
                   const float *smooth, int smooth_mode, void *codes,
                   int code_bytes, void *k_hat_f16, void *stream);

/*
 * Value encode.  Page: "Metal Kernels API", section "VecInfer kernels",
 * vecinfer_encode_decode_simple_metal, the value-side sibling of the key
 * encoder without the smooth and Hadamard steps.
 *
 * Same arguments, limits and errors as vq_encode_keys without smooth: per
 * vector, code_m = nearest centroid of x[m*sub_dim : (m+1)*sub_dim] (squared
 * distance, lowest index on ties, decided as for keys); v_hat (optional) =
 * concat_m codebook[code_m] rounded to fp16.
 */
VQ_API int vq_encode_values(const void *values_f16, int B, int H, int S, int D,
                     const float *codebook, int n_centroids, int sub_dim,
                     void *codes, int code_bytes, void *v_hat_f16,
                     void *stream);

/*
 * Cache append.  Page: "veloxquant_mlx.cache.vecinfer_cache module",
 * VecInferKVCache.update_and_fetch (new tokens are encoded and stored after
 * the ones already cached).  The same encodes as vq_encode_keys and
 * vq_encode_values, with the codes written into a preallocated cache:
 *
 *   codes      [B, H, capacity, D/sub_dim] (output rows offset .. offset+S-1
 *              of every (b, h); the other rows are not touched).
 *   capacity   rows per (b, h) of the code buffer.
 *   offset     first row written: token t of the call goes to row offset + t.
 *
 * Everything else (inputs [B, H, S, D], the optional fp16 reconstruction
 * [B, H, S, D], limits, errors) is as in the calls above; in addition
 * VQ_ERR_SHAPE when capacity < 0, offset < 0 or offset + S > capacity.
 * vq_encode_keys(...) equals vq_encode_keys_into(..., capacity = S,
 * offset = 0, ...).
 */
VQ_API int vq_encode_keys_into(const void *keys_f16, int B, int H, int S, int D,
                               const float *codebook, int n_centroids, int sub_dim,
                               const float *smooth, int smooth_mode, void *codes,
                               int code_bytes, int capacity, int offset, void *k_hat_f16,
                               void *stream);
VQ_API int vq_encode_values_into(const void *values_f16, int B, int H, int S, int D,
                                 const float *codebook, int n_centroids, int sub_dim,
                                 void *codes, int code_bytes, int capacity, int offset,
                                 void *v_hat_f16, void *stream);

/*
 * Codebook gather.  Page: "Metal Kernels API", section "VecInfer kernels",
 * vecinfer_dequant_metal.
 *
 *   codes   [n_vectors, n_sub] of code_bytes each.
 *   out     [n_vectors, n_sub * sub_dim]: fp32 when out_is_f32 != 0, else
 *           fp16 (nearest even).
 * out[v, m*sub_dim + t] = codebook[codes[v, m], t].  A code >= n_centroids
 * is a caller error: its output row is undefined, but every memory access
 * stays in bounds (the code is clamped).
 * Errors: VQ_ERR_NULL, VQ_ERR_SHAPE (negative sizes, n_sub or sub_dim < 1,
 * code_bytes not 1 or 2), VQ_ERR_UNSUPPORTED (n_centroids above the code
 * width), VQ_ERR_ALIGN, VQ_ERR_CUDA.  n_vectors == 0 is a no-op.
 */
VQ_API int vq_dequant(const void *codes, int code_bytes, int64_t n_vectors, int n_sub,
               const float *codebook, int n_centroids, int sub_dim, void *out,
               int out_is_f32, void *stream);

/*
 * Arguments of attention over the coded cache.  Page: "Metal Kernels API",
 * section "Fused SDPA", metal_fused_sdpa, with the query semantics of
 * VecInferKVCache.fused_sdpa ("veloxquant_mlx.cache.vecinfer_cache module"):
 * the caller passes the raw query; the library applies the dual transform
 * q~ = Hn (q (.) s_g^-1) itself, so that q~ . K~^T equals q . K_hat^T.
 *
 *   q_f16      [B, H_q, S_q, D] fp16, untransformed.
 *   k_codes    [B, H_kv, kv_stride, D/k_sub_dim] key codes (k_code_bytes
 *              each), produced by vq_encode_keys with k_codebook and smooth;
 *              rows 0 .. S_kv-1 of every (b, kv head) are the cache.
 *   v_codes    [B, H_kv, kv_stride, D/v_sub_dim] value codes.
 *   kv_stride  rows per (b, kv head) of the code buffers (a preallocated
 *              cache's capacity); 0 means S_kv.  Must be 0 or >= S_kv.
 *   kv_lens    NULL, or device int32 [B]: batch b holds kv_lens[b] <= S_kv
 *              cached keys (its rows 0 .. kv_lens[b]-1); its queries align
 *              to that length (q_abs = kv_lens[b] - S_q + i).  Values are
 *              clamped to [0, S_kv] on the device; a query with no visible
 *              key gets a zero row.  NULL: every batch holds S_kv keys.
 *   smooth     key smooth factors, as in vq_encode_keys.
 *   scale      softmax scale (typically 1/sqrt(D)).
 *   causal     != 0: queries align to the tail of the cache, row i sits at
 *              q_abs = S_kv - S_q + i and sees keys j <= q_abs.
 *   sliding_window  > 0: row i sees only keys j > q_abs - sliding_window
 *              (the window ends at, and includes, the query's position).
 *   out_f16    [B, H_q, S_q, D] fp16 (output).
 *   workspace  device scratch of at least vq_attend_workspace_bytes(args)
 *              bytes, 16-byte aligned; may be NULL when that size is 0.
 * Query head h reads KV head h / (H_q / H_kv).  Softmax accumulates in fp32.
 * The key and value codebooks are independent (sizes may differ).
 */
typedef struct {
    int B, H_q, H_kv, S_q, S_kv, D;
    const void *q_f16;
    const void *k_codes;
    int k_code_bytes;
    const float *k_codebook;
    int k_n_centroids, k_sub_dim;
    const void *v_codes;
    int v_code_bytes;
    const float *v_codebook;
    int v_n_centroids, v_sub_dim;
    const float *smooth;
    int smooth_mode;
    float scale;
    int causal;
    int sliding_window;
    void *out_f16;
    void *workspace;
    size_t workspace_bytes;
    int kv_stride;
    const int32_t *kv_lens;
} vq_attend_args;

/*
 * Scratch bytes vq_decode_attend / vq_prefill_attend / vq_decode_step need
 * for `args` on the current device: the split-KV partial results, or for a
 * single-launch decode step its partial results and the flags of its new
 * rows, whichever is larger (0 if none).  Depends only on the sizes in args
 * and on the device's SM count.  Returns 0 for a NULL args.
 */
VQ_API size_t vq_attend_workspace_bytes(const vq_attend_args *args);

/*
 * Attention over the coded cache on CUDA cores + warp-level MMA, split
 * across the key axis with a combine pass (flash-decoding).  Any S_q.
 * Page: "Metal Kernels API", section "Fused SDPA", metal_fused_sdpa.
 *
 * Errors: VQ_ERR_NULL, VQ_ERR_SHAPE (negative sizes, H_kv == 0 or
 * H_q % H_kv != 0, D % sub_dim != 0, S_q > S_kv when causal or windowed,
 * S_kv == 0 with S_q > 0, negative window, bad smooth_mode or code width,
 * kv_stride < 0 or 0 < kv_stride < S_kv),
 * VQ_ERR_UNSUPPORTED (D not a power of two in [32, 256], sub_dim not in
 * {2, 4, 8}, codebooks over the on-chip limit, n_centroids above the code
 * width), VQ_ERR_ALIGN, VQ_ERR_WORKSPACE, VQ_ERR_CUDA.
 */
VQ_API int vq_decode_attend(const vq_attend_args *args, void *stream);

/*
 * One decode step of the cache in one launch.  Page "veloxquant_mlx.cache.
 * vecinfer_cache module", VecInferKVCache.update_and_fetch (the new tokens
 * are encoded and stored after the cached ones) followed by its fused_sdpa
 * over the updated cache.
 *
 *   k_new_f16, v_new_f16  [B, H_kv, S_q, D] fp16: the keys and values of the
 *              S_q new tokens (the tokens of the queries).
 *   args       as for vq_decode_attend, with S_kv counting the new tokens:
 *              their codes are written into rows S_kv - S_q .. S_kv - 1 of
 *              every (b, kv head) of k_codes / v_codes (the other rows are
 *              not touched), encoded exactly as vq_encode_keys_into (with
 *              k_codebook, smooth) and vq_encode_values_into (v_codebook)
 *              would; then every query attends over rows 0 .. S_kv - 1 as
 *              in vq_decode_attend.  kv_lens must be NULL.
 * With D = 128, 4-dimensional sub-vectors, uint8 codes and codebooks of at
 * most 256 centroids this is one cooperative launch: the encode beside the
 * attention over the rows before the new ones (a reader of a new row waits,
 * bounded, for a per-row flag in the workspace that the encode sets), then a
 * grid sync and the merge of the key splits; other shapes run as the three
 * calls on the same stream.  The workspace is sized by
 * vq_attend_workspace_bytes for these args (the single launch keeps its
 * partial records and flags inside that size); it must not be in use by
 * another call at the same time.  The launch leaves the flags cleared, so
 * a workspace can serve consecutive steps and a captured CUDA graph.
 * Errors: those of vq_decode_attend and of the encodes; VQ_ERR_SHAPE when
 * S_q > S_kv, VQ_ERR_UNSUPPORTED when kv_lens is given, VQ_ERR_NULL /
 * VQ_ERR_ALIGN for the new tokens, VQ_ERR_CUDA when the launch fails (e.g.
 * the grid cannot be resident at once).
 */
VQ_API int vq_decode_step(const vq_attend_args *args, const void *k_new_f16,
                          const void *v_new_f16, void *stream);

/*
 * Same operation through the tcgen05 tensor-core path (code tiles brought
 * into shared memory by tensor copies, key/value tiles rebuilt from them,
 * Q~K~^T and PV on the tensor cores, accumulators in tensor memory).  Used
 * when S_q >= 64; smaller S_q, shapes outside the tensor-core kernel's
 * limits (D != 128, sub_dim != 4, codes wider than one byte), and code
 * buffers of 2^31 rows or more (B * H_kv * rows, the tensor copies' row
 * coordinate), are served by vq_decode_attend with the same arguments.
 * Each block runs two query heads of a KV group (sharing the rebuilt
 * tiles); with an odd GQA group size H_q / H_kv the last block of a group
 * runs a single head.  Page: "Metal
 * Kernels API", section "Fused SDPA", metal_fused_sdpa; the prefill-shaped
 * tile loop follows the companion described under rabitq_prefill_attend.
 * Errors as vq_decode_attend.
 */
VQ_API int vq_prefill_attend(const vq_attend_args *args, void *stream);

/*
 * Allocation-free variant of vq_decode_attend.  The documentation pages have
 * no counterpart: this is a service of this library for callers that cannot
 * allocate device memory -- for example a plug-in inside a host application
 * that owns all GPU memory, a runtime that fixes its memory plan before the
 * model runs, or a latency-critical decode loop that must not call
 * cudaMalloc (which can synchronise the device).
 *
 * Same arguments, results and errors as vq_decode_attend, except that
 * args->workspace and args->workspace_bytes are ignored: the split-KV
 * partial results go to a scratch array of VQ_NOALLOC_SCRATCH_BYTES compiled
 * into the library, which every GPU that loads the library keeps until the
 * process exits.  The library allocates nothing, here or anywhere.
 *   - A problem fits exactly when
 *       (B * H_kv * ceil(H_q / H_kv * S_q / 8) + 1) * 8 * (D + 4) * 4
 *         <= VQ_NOALLOC_SCRATCH_BYTES
 *     (its partial results with a single key split); problems whose regular
 *     split (vq_attend_workspace_bytes) needs more than the array run with
 *     fewer, longer splits.  A problem that does not fit returns
 *     VQ_ERR_WORKSPACE before anything is launched; use vq_decode_attend
 *     with a workspace for those.
 *   - All calls share the array: calls whose work overlaps on the GPU (other
 *     streams or host threads) race on it; order them on one stream or with
 *     events.  Every call overwrites what it reads, so no clearing is needed.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it with the
 *     id of the device's context; make that first call before any stream
 *     capture.  A call that finds another context current (after
 *     cudaDeviceReset, or a primary context released and re-created) looks
 *     the address up again: make that call outside a stream capture too.
 */
#define VQ_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
VQ_API int vq_decode_attend_noalloc(const vq_attend_args *args, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* VQKV_H_ */
