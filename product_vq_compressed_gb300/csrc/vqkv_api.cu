// vqkv_api.cu -- the extern "C" entry points of libvqkv.so: synchronous
// argument validation, launch planning, and launches on the caller's stream.
// Declarations and the meaning of every argument: include/vqkv.h.
#include <stdint.h>

#include "vq_internal.cuh"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

int ilog2(int v) {
    int r = 0;
    while ((1 << r) < v) ++r;
    return r;
}

// code_bytes: 1 (uint8), 2 (uint16), 0 (bit-packed rows of ceil(log2 N)-bit codes)
int code_capacity_ok(int n_centroids, int code_bytes) {
    if (code_bytes != 0 && code_bytes != 1 && code_bytes != 2) return VQ_ERR_SHAPE;
    if (n_centroids < 1) return VQ_ERR_UNSUPPORTED;
    const int64_t cap = code_bytes == 1 ? 256 : 65536;
    if ((int64_t)n_centroids > cap) return VQ_ERR_UNSUPPORTED;
    return VQ_OK;
}

int encode_common(const void *x, int B, int H, int S, int D,
                  const float *codebook, int N, int sub_dim, const float *smooth,
                  int smooth_mode, void *codes, int code_bytes, int capacity, int offset,
                  void *xhat, int rotate, void *stream) {
    if (smooth_mode < 0 || smooth_mode > 2) return VQ_ERR_SHAPE;
    if (B < 0 || H < 0 || S < 0 || D < 1 || sub_dim < 1) return VQ_ERR_SHAPE;
    if (capacity < 0 || offset < 0 || (int64_t)offset + S > capacity) return VQ_ERR_SHAPE;
    if (D % sub_dim != 0) return VQ_ERR_SHAPE;
    int rc = code_capacity_ok(N, code_bytes);
    if (rc != VQ_OK) return rc;
    if (!pow2(D) || D < 32 || D > 512) return VQ_ERR_UNSUPPORTED;
    if (!(sub_dim == 1 || sub_dim == 2 || sub_dim == 4 || sub_dim == 8 || sub_dim == 16))
        return VQ_ERR_UNSUPPORTED;
    if ((size_t)N * sub_dim * sizeof(float) > 160u * 1024u) return VQ_ERR_UNSUPPORTED;
    const int64_t n_vec = (int64_t)B * H * S;
    if (n_vec == 0) return VQ_OK;  // empty problem: no pointer is read
    if (!x || !codebook || !codes) return VQ_ERR_NULL;
    if (smooth_mode != 0 && !smooth) return VQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(codebook) || !aligned16(codes) ||
        (xhat && !aligned16(xhat)) || (smooth && !aligned16(smooth)))
        return VQ_ERR_ALIGN;
    vqkv::EncodeParams p{};
    p.x = reinterpret_cast<const __half *>(x);
    p.n_vec = n_vec;
    p.H = H;
    p.S = S;
    p.D = D;
    p.log2D = ilog2(D);
    p.codebook = codebook;
    p.N = N;
    p.sub_dim = sub_dim;
    p.smooth = smooth_mode ? smooth : nullptr;
    p.smooth_mode = smooth_mode;
    p.rotate = rotate;
    p.codes = codes;
    p.code_bytes = code_bytes;
    p.code_bits = code_bytes == 0 ? vqkv::packed_code_bits(N) : 0;
    p.row_words = code_bytes == 0 ? vqkv::packed_row_words(D / sub_dim, p.code_bits) : 0;
    p.xhat = reinterpret_cast<__half *>(xhat);
    p.div_S = vqkv::make_fastdiv((uint32_t)(S > 0 ? S : 1));
    p.div_H = vqkv::make_fastdiv((uint32_t)(H > 0 ? H : 1));
    p.cap = capacity;
    p.off = offset;
    return vqkv::launch_encode(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? VQ_OK
               : VQ_ERR_CUDA;
}

int current_sms(int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return VQ_ERR_CUDA;
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return VQ_ERR_CUDA;
    return VQ_OK;
}

int decode_impl(const vq_attend_args *a, void *stream) {
    int rc = vqkv::attend_validate(a);
    if (rc != VQ_OK) return rc;
    if ((int64_t)a->B * a->H_q * a->S_q == 0) return VQ_OK;
    int sms = 0;
    rc = current_sms(&sms);
    if (rc != VQ_OK) return rc;
    const vqkv::AttendPlan plan = vqkv::plan_decode(*a, sms);
    if (!a->workspace || a->workspace_bytes < plan.ws_bytes) return VQ_ERR_WORKSPACE;
    return vqkv::launch_decode(*a, plan, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? VQ_OK
               : VQ_ERR_CUDA;
}

}  // namespace

namespace vqkv {
// Argument checks shared by every attention entry point (decode, prefill,
// and the allocation-free decode); the workspace size is checked by the
// caller, which knows its plan.
int attend_validate(const vq_attend_args *a) {
    if (!a) return VQ_ERR_NULL;
    if (a->B < 0 || a->H_q < 0 || a->H_kv < 0 || a->S_q < 0 || a->S_kv < 0 ||
        a->D < 1 || a->sliding_window < 0)
        return VQ_ERR_SHAPE;
    if (a->H_kv == 0 || a->H_q % a->H_kv != 0) return VQ_ERR_SHAPE;
    if (a->k_sub_dim < 1 || a->v_sub_dim < 1) return VQ_ERR_SHAPE;
    if (a->D % a->k_sub_dim != 0 || a->D % a->v_sub_dim != 0) return VQ_ERR_SHAPE;
    if (a->smooth_mode < 0 || a->smooth_mode > 2) return VQ_ERR_SHAPE;
    if ((a->causal || a->sliding_window > 0) && a->S_q > a->S_kv) return VQ_ERR_SHAPE;
    if (a->kv_stride < 0 || (a->kv_stride > 0 && a->kv_stride < a->S_kv)) return VQ_ERR_SHAPE;
    if (a->S_kv == 0 && a->S_q > 0 && a->B > 0 && a->H_q > 0) return VQ_ERR_SHAPE;
    int rc = code_capacity_ok(a->k_n_centroids, a->k_code_bytes);
    if (rc != VQ_OK) return rc;
    rc = code_capacity_ok(a->v_n_centroids, a->v_code_bytes);
    if (rc != VQ_OK) return rc;
    if (!pow2(a->D)) return VQ_ERR_UNSUPPORTED;
    rc = vqkv::decode_supported(*a);
    if (rc != VQ_OK) return rc;
    if ((int64_t)a->B * a->H_q * a->S_q == 0) return VQ_OK;  // nothing to read
    if (!a->q_f16 || !a->k_codes || !a->k_codebook || !a->v_codes ||
        !a->v_codebook || !a->out_f16)
        return VQ_ERR_NULL;
    if (a->smooth_mode != 0 && !a->smooth) return VQ_ERR_NULL;
    if (!aligned16(a->q_f16) || !aligned16(a->k_codes) || !aligned16(a->k_codebook) ||
        !aligned16(a->v_codes) || !aligned16(a->v_codebook) || !aligned16(a->out_f16) ||
        (a->smooth && !aligned16(a->smooth)) ||
        (a->workspace && !aligned16(a->workspace)))
        return VQ_ERR_ALIGN;
    return VQ_OK;
}

}  // namespace vqkv

extern "C" {

const char *vq_status_str(int status) {
    switch (status) {
        case VQ_OK: return "ok";
        case VQ_ERR_NULL: return "a required pointer is NULL";
        case VQ_ERR_SHAPE: return "inconsistent or invalid sizes";
        case VQ_ERR_UNSUPPORTED: return "request outside the supported limits";
        case VQ_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case VQ_ERR_WORKSPACE: return "workspace missing or too small";
        case VQ_ERR_CUDA: return "CUDA launch or query failed";
        default: return "unknown status";
    }
}

int vq_encode_keys(const void *keys_f16, int B, int H, int S, int D,
                   const float *codebook, int n_centroids, int sub_dim,
                   const float *smooth, int smooth_mode, void *codes,
                   int code_bytes, void *k_hat_f16, void *stream) {
    return encode_common(keys_f16, B, H, S, D, codebook, n_centroids, sub_dim,
                         smooth, smooth_mode, codes, code_bytes, S, 0, k_hat_f16, 1,
                         stream);
}

int vq_encode_keys_into(const void *keys_f16, int B, int H, int S, int D,
                        const float *codebook, int n_centroids, int sub_dim,
                        const float *smooth, int smooth_mode, void *codes,
                        int code_bytes, int capacity, int offset, void *k_hat_f16,
                        void *stream) {
    return encode_common(keys_f16, B, H, S, D, codebook, n_centroids, sub_dim,
                         smooth, smooth_mode, codes, code_bytes, capacity, offset,
                         k_hat_f16, 1, stream);
}

int vq_encode_values(const void *values_f16, int B, int H, int S, int D,
                     const float *codebook, int n_centroids, int sub_dim,
                     void *codes, int code_bytes, void *v_hat_f16,
                     void *stream) {
    return encode_common(values_f16, B, H, S, D, codebook, n_centroids, sub_dim,
                         nullptr, 0, codes, code_bytes, S, 0, v_hat_f16, 0, stream);
}

int vq_encode_values_into(const void *values_f16, int B, int H, int S, int D,
                          const float *codebook, int n_centroids, int sub_dim,
                          void *codes, int code_bytes, int capacity, int offset,
                          void *v_hat_f16, void *stream) {
    return encode_common(values_f16, B, H, S, D, codebook, n_centroids, sub_dim,
                         nullptr, 0, codes, code_bytes, capacity, offset, v_hat_f16, 0,
                         stream);
}

int vq_dequant(const void *codes, int code_bytes, int64_t n_vectors, int n_sub,
               const float *codebook, int n_centroids, int sub_dim, void *out,
               int out_is_f32, void *stream) {
    if (n_vectors < 0 || n_sub < 1 || sub_dim < 1) return VQ_ERR_SHAPE;
    int rc = code_capacity_ok(n_centroids, code_bytes);
    if (rc != VQ_OK) return rc;
    if (n_vectors == 0) return VQ_OK;  // empty problem: no pointer is read
    if (!codes || !codebook || !out) return VQ_ERR_NULL;
    if (!aligned16(codes) || !aligned16(codebook) || !aligned16(out)) return VQ_ERR_ALIGN;
    vqkv::DequantParams p{};
    p.codes = codes;
    p.code_bytes = code_bytes;
    p.code_bits = code_bytes == 0 ? vqkv::packed_code_bits(n_centroids) : 0;
    p.row_words = code_bytes == 0 ? vqkv::packed_row_words(n_sub, p.code_bits) : 0;
    p.n_vec = n_vectors;
    p.n_sub = n_sub;
    p.codebook = codebook;
    p.N = n_centroids;
    p.sub_dim = sub_dim;
    p.out = out;
    p.out_is_f32 = out_is_f32 != 0;
    return vqkv::launch_dequant(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? VQ_OK
               : VQ_ERR_CUDA;
}

size_t vq_attend_workspace_bytes(const vq_attend_args *args) {
    // Sized for the split-KV path, which both entry points may take.
    if (!args) return 0;
    const vq_attend_args n = vqkv::normalize_code_widths(*args);
    const vq_attend_args *a = &n;
    if (a->H_kv <= 0 || a->H_q <= 0 || a->H_q % a->H_kv != 0 || a->D < 1 ||
        a->S_q <= 0 || a->B <= 0 || a->S_kv <= 0 || a->k_sub_dim < 1 ||
        a->v_sub_dim < 1 || vqkv::decode_supported(*a) != VQ_OK)
        return 0;
    int sms = 0;
    if (current_sms(&sms) != VQ_OK) return 0;
    // the larger of the split-KV plan's records and what a single-launch
    // decode step keeps there (its own plan's records, which has fewer warps
    // with longer shares, then the flags of its new rows)
    const size_t attend = vqkv::plan_decode(*a, sms).ws_bytes;
    const size_t step =
        vqkv::step_flags_offset(vqkv::plan_decode(*a, sms, vqkv::kStepEncodeWarps)) +
        vqkv::step_flags_bytes(*a);
    return attend > step ? attend : step;
}

int vq_decode_attend(const vq_attend_args *args, void *stream) {
    if (!args) return VQ_ERR_NULL;
    const vq_attend_args n = vqkv::normalize_code_widths(*args);
    return decode_impl(&n, stream);
}

int vq_decode_step(const vq_attend_args *in, const void *k_new_f16, const void *v_new_f16,
                   void *stream) {
    if (!in) return VQ_ERR_NULL;
    const vq_attend_args n = vqkv::normalize_code_widths(*in);
    const vq_attend_args *a = &n;
    int rc = vqkv::attend_validate(a);
    if (rc != VQ_OK) return rc;
    if (a->S_q > a->S_kv) return VQ_ERR_SHAPE;   // the new tokens are cache rows
    if (a->kv_lens) return VQ_ERR_UNSUPPORTED;   // one append offset for every batch
    if ((int64_t)a->B * a->H_q * a->S_q == 0) return VQ_OK;
    if (!k_new_f16 || !v_new_f16) return VQ_ERR_NULL;
    if (!aligned16(k_new_f16) || !aligned16(v_new_f16)) return VQ_ERR_ALIGN;
    int sms = 0;
    rc = current_sms(&sms);
    if (rc != VQ_OK) return rc;
    const bool one_launch = vqkv::decode_step_supported(*a) == VQ_OK;
    // the single launch keeps kStepEncodeWarps warps of every CTA for the
    // encode (fewer warps with shares); vq_attend_workspace_bytes covers its
    // records and flags as well as the separate calls' records
    const vqkv::AttendPlan plan =
        vqkv::plan_decode(*a, sms, one_launch ? vqkv::kStepEncodeWarps : 0);
    const size_t need = one_launch ? vqkv::step_flags_offset(plan) + vqkv::step_flags_bytes(*a)
                                   : plan.ws_bytes;
    if (!a->workspace || a->workspace_bytes < need) return VQ_ERR_WORKSPACE;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (one_launch)
        return vqkv::launch_decode(*a, plan, st, k_new_f16, v_new_f16) == cudaSuccess ? VQ_OK
                                                                                 : VQ_ERR_CUDA;
    // other shapes: the appends and the attention as separate launches
    const int cap = a->kv_stride > 0 ? a->kv_stride : a->S_kv;
    const int off = a->S_kv - a->S_q;
    rc = encode_common(k_new_f16, a->B, a->H_kv, a->S_q, a->D, a->k_codebook, a->k_n_centroids,
                       a->k_sub_dim, a->smooth, a->smooth_mode, const_cast<void *>(a->k_codes),
                       in->k_code_bytes, cap, off, nullptr, 1, stream);
    if (rc != VQ_OK) return rc;
    rc = encode_common(v_new_f16, a->B, a->H_kv, a->S_q, a->D, a->v_codebook, a->v_n_centroids,
                       a->v_sub_dim, nullptr, 0, const_cast<void *>(a->v_codes),
                       in->v_code_bytes, cap, off, nullptr, 0, stream);
    if (rc != VQ_OK) return rc;
    return vqkv::launch_decode(*a, plan, st) == cudaSuccess ? VQ_OK : VQ_ERR_CUDA;
}

int vq_prefill_attend(const vq_attend_args *in, void *stream) {
    if (!in) return VQ_ERR_NULL;
    const vq_attend_args n = vqkv::normalize_code_widths(*in);
    const vq_attend_args *args = &n;
    int rc = vqkv::attend_validate(args);
    if (rc != VQ_OK) return rc;
    if (vqkv::prefill_supported(*args) != VQ_OK) return decode_impl(args, stream);
    if ((int64_t)args->B * args->H_q * args->S_q == 0) return VQ_OK;
    return vqkv::launch_prefill(*args, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? VQ_OK
               : VQ_ERR_CUDA;
}

}  // extern "C"
