/*
 * vq_oracle.c -- plain, slow, float64 CPU oracle for the product-VQ KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library; it is written from the documentation pages alone:
 *
 *   [API]   "Metal Kernels API" (veloxquant.dev/docs/api/metal-api),
 *           section "VecInfer kernels" (vecinfer_quantize_metal,
 *           vecinfer_dequant_metal, vecinfer_encode_decode_metal and its
 *           value-side "simple" sibling) and section "Fused SDPA"
 *           (metal_fused_sdpa, supports_shape); section "RaBitQ kernels",
 *           rabitq_prefill_attend, for the causal alignment convention that
 *           the page says fused_sdpa shares.
 *   [CACHE] "veloxquant_mlx.cache.vecinfer_cache module", the module summary
 *           (smooth scaling + Walsh-Hadamard rotation of keys, product VQ,
 *           per-token storage formula) and VecInferKVCache.fused_sdpa (raw,
 *           untransformed queries in; the dual transform is internal).
 *
 * Every step is the definition written out, in the order the pages give it,
 * with no blocking, fusion or reordering:
 *   - the Hadamard matrix is built by Sylvester's doubling and applied as an
 *     explicit D x D matrix-vector product (never a butterfly);
 *   - squared distances use the direct form sum_t (y_t - c_t)^2;
 *   - argmin keeps the first (lowest) index among equal distances;
 *   - attention reconstructs K_hat = s^-1 (.) H^T dequant(codes) and runs a
 *     textbook max-subtracted softmax with exp() from libm.
 *
 * Readings of points the pages leave open (all of them are listed, with the
 * reasons, in the design notes of the repository):
 *   - smooth multiplies keys before the rotation and divides queries (and
 *     K_hat) after it; H is the normalised Sylvester matrix (natural order);
 *   - ties go to the lowest index;
 *   - the causal mask aligns queries to the tail of the cache:
 *     q_abs = S_kv - S_q + i, key j is visible iff j <= q_abs;
 *   - a sliding window W > 0 keeps the W keys ending at the query's own
 *     position: q_abs - W < j;  with causal off only that lower bound holds;
 *   - GQA maps query head h to KV head h / (H_q / H_kv).
 *
 * Float64 throughout; the caller converts fp16 inputs exactly to double and
 * rounds outputs to fp16 itself.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENOMEM (-2)

static int is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

/*
 * Normalised Sylvester-Hadamard matrix, row-major D x D:
 *   H_1 = [1],  H_2n = [[H_n, H_n], [H_n, -H_n]],  Hn = H_D / sqrt(D).
 * [API] vecinfer_encode_decode_metal takes H_mat, a [D, D] Walsh-Hadamard
 * matrix; [CACHE] calls the step a Walsh-Hadamard rotation (so it must be
 * orthonormal, hence the 1/sqrt(D)).
 */
int orc_hadamard(int D, double *Hn) {
    if (!is_pow2(D) || !Hn) return ORC_EINVAL;
    Hn[0] = 1.0;
    for (int n = 1; n < D; n *= 2) {
        /* grow the top-left n x n block to 2n x 2n, in place, row stride D */
        for (int r = 0; r < n; r++) {
            for (int c = 0; c < n; c++) {
                double v = Hn[(size_t)r * D + c];
                Hn[(size_t)r * D + (c + n)] = v;
                Hn[(size_t)(r + n) * D + c] = v;
                Hn[(size_t)(r + n) * D + (c + n)] = -v;
            }
        }
    }
    double inv = 1.0 / sqrt((double)D);
    for (size_t i = 0; i < (size_t)D * D; i++) Hn[i] *= inv;
    return ORC_OK;
}

/* smooth factor for (head h, channel t); mode 0 none, 1 [D], 2 [H, D] */
static double smooth_at(const double *smooth, int mode, int D, int h, int t) {
    if (mode == 0 || !smooth) return 1.0;
    if (mode == 1) return smooth[t];
    return smooth[(size_t)h * D + t];
}

/*
 * Forward transform of one key vector: y = Hn . (s_h (.) x).
 * [API] vecinfer_encode_decode_metal: "smooth -> Walsh-Hadamard transform".
 * With rotate == 0 (values, the "simple" variant without smooth or
 * Hadamard) y = x.
 */
static void forward_transform(const double *x, int D, const double *Hn,
                              const double *smooth, int mode, int h,
                              int rotate, double *tmp, double *y) {
    if (!rotate) {
        memcpy(y, x, sizeof(double) * (size_t)D);
        return;
    }
    for (int t = 0; t < D; t++) tmp[t] = smooth_at(smooth, mode, D, h, t) * x[t];
    for (int r = 0; r < D; r++) {
        double acc = 0.0;
        for (int t = 0; t < D; t++) acc += Hn[(size_t)r * D + t] * tmp[t];
        y[r] = acc;
    }
}

/*
 * Inverse transform: x_hat = s_h^-1 (.) Hn^T . y_hat.
 * [API] vecinfer_encode_decode_metal: "dequant -> inverse-WHT ->
 * inverse-smooth".  Hn^T is written out (it equals Hn, but the oracle does
 * not rely on that).
 */
static void inverse_transform(const double *yhat, int D, const double *Hn,
                              const double *smooth, int mode, int h,
                              int rotate, double *xhat) {
    if (!rotate) {
        memcpy(xhat, yhat, sizeof(double) * (size_t)D);
        return;
    }
    for (int t = 0; t < D; t++) {
        double acc = 0.0;
        for (int r = 0; r < D; r++) acc += Hn[(size_t)r * D + t] * yhat[r];
        xhat[t] = acc / smooth_at(smooth, mode, D, h, t);
    }
}

/*
 * Squared Euclidean distance, direct form.
 * [API] vecinfer_quantize_metal computes squared distances to every centroid.
 */
static double sqdist(const double *y, const double *c, int d) {
    double acc = 0.0;
    for (int t = 0; t < d; t++) {
        double e = y[t] - c[t];
        acc += e * e;
    }
    return acc;
}

/*
 * Nearest centroid of one sub-vector: the first index reaching the minimum
 * distance.  Also reports the best and the second-best distance (the second
 * best over all other indices; equal to the best when there is a tie).
 * [API] vecinfer_quantize_metal returns codebook indices of the nearest
 * centroid for each sub-vector of size sub_dim.
 */
static int32_t nearest(const double *y, const double *codebook, int N, int d,
                       double *best_out, double *second_out) {
    int32_t best_i = 0;
    double best = INFINITY, second = INFINITY;
    for (int c = 0; c < N; c++) {
        double dist = sqdist(y, codebook + (size_t)c * d, d);
        if (dist < best) {
            second = best;
            best = dist;
            best_i = c;
        } else if (dist < second) {
            second = dist;
        }
    }
    if (best_out) *best_out = best;
    if (second_out) *second_out = second;
    return best_i;
}

/*
 * Encode n_vec vectors of size D.
 *   x          [n_vec, D]           input (fp16 values converted to double)
 *   head       [n_vec]              KV head of each vector (for smooth [H, D])
 *   smooth     [H, D] (mode 2), [D] (mode 1) or NULL (mode 0)
 *   rotate     1: keys (smooth + Hadamard), 0: values (plain sub-vector VQ)
 *   codebook   [N, d]               shared by every sub-vector position
 * Outputs (any may be NULL except codes):
 *   codes      [n_vec, D/d]         int32 nearest-centroid indices
 *   d1, d2     [n_vec, D/d]         best / second-best squared distance
 *   y_out      [n_vec, D]           the transformed vector the search ran on
 *   xhat       [n_vec, D]           reconstruction from the oracle's codes:
 *                                   s^-1 (.) Hn^T concat_m codebook[code_m]
 * [API] vecinfer_encode_decode_metal (keys), its "simple" value-side sibling
 * (values), vecinfer_quantize_metal (the search itself).
 */
int orc_encode(const double *x, int64_t n_vec, int D, const int32_t *head,
               const double *smooth, int smooth_mode, int rotate,
               const double *codebook, int N, int d, int32_t *codes,
               double *d1, double *d2, double *y_out, double *xhat) {
    if (!x || !codes || !codebook || n_vec < 0 || D <= 0 || N <= 0 || d <= 0 ||
        D % d != 0)
        return ORC_EINVAL;
    if (rotate && !is_pow2(D)) return ORC_EINVAL;
    if (smooth_mode != 0 && !smooth) return ORC_EINVAL;
    int n_sub = D / d;
    double *Hn = NULL;
    double *tmp = malloc(sizeof(double) * (size_t)D);
    double *y = malloc(sizeof(double) * (size_t)D);
    double *yhat = malloc(sizeof(double) * (size_t)D);
    if (rotate) Hn = malloc(sizeof(double) * (size_t)D * D);
    if (!tmp || !y || !yhat || (rotate && !Hn)) {
        free(tmp); free(y); free(yhat); free(Hn);
        return ORC_ENOMEM;
    }
    if (rotate) orc_hadamard(D, Hn);
    for (int64_t v = 0; v < n_vec; v++) {
        int h = head ? head[v] : 0;
        forward_transform(x + (size_t)v * D, D, Hn, smooth, smooth_mode, h,
                          rotate, tmp, y);
        if (y_out) memcpy(y_out + (size_t)v * D, y, sizeof(double) * (size_t)D);
        for (int m = 0; m < n_sub; m++) {
            double b, s;
            int32_t c = nearest(y + (size_t)m * d, codebook, N, d, &b, &s);
            codes[(size_t)v * n_sub + m] = c;
            if (d1) d1[(size_t)v * n_sub + m] = b;
            if (d2) d2[(size_t)v * n_sub + m] = s;
            memcpy(yhat + (size_t)m * d, codebook + (size_t)c * d,
                   sizeof(double) * (size_t)d);
        }
        if (xhat)
            inverse_transform(yhat, D, Hn, smooth, smooth_mode, h, rotate,
                              xhat + (size_t)v * D);
    }
    free(tmp); free(y); free(yhat); free(Hn);
    return ORC_OK;
}

/*
 * Codebook gather: out[v, m*d + t] = codebook[codes[v, m], t].
 * [API] vecinfer_dequant_metal ("a codebook gather").
 * Returns ORC_EINVAL if any code is outside [0, N).
 */
int orc_dequant(const int32_t *codes, int64_t n_vec, int n_sub,
                const double *codebook, int N, int d, double *out) {
    if (!codes || !codebook || !out || n_vec < 0 || n_sub <= 0 || N <= 0 ||
        d <= 0)
        return ORC_EINVAL;
    for (int64_t v = 0; v < n_vec; v++) {
        for (int m = 0; m < n_sub; m++) {
            int32_t c = codes[(size_t)v * n_sub + m];
            if (c < 0 || c >= N) return ORC_EINVAL;
            for (int t = 0; t < d; t++)
                out[((size_t)v * n_sub + m) * d + t] =
                    codebook[(size_t)c * d + t];
        }
    }
    return ORC_OK;
}

/*
 * Reconstruction from given codes (keys: rotate = 1, values: rotate = 0):
 *   xhat = s_h^-1 (.) Hn^T dequant(codes).
 * [API] vecinfer_encode_decode_metal, second half of its pipeline.
 */
int orc_reconstruct(const int32_t *codes, int64_t n_vec, int D,
                    const int32_t *head, const double *smooth, int smooth_mode,
                    int rotate, const double *codebook, int N, int d,
                    double *xhat) {
    if (!codes || !codebook || !xhat || D % d != 0) return ORC_EINVAL;
    if (rotate && !is_pow2(D)) return ORC_EINVAL;
    if (smooth_mode != 0 && !smooth) return ORC_EINVAL;
    int n_sub = D / d;
    double *yhat = malloc(sizeof(double) * (size_t)D);
    double *Hn = rotate ? malloc(sizeof(double) * (size_t)D * D) : NULL;
    if (!yhat || (rotate && !Hn)) {
        free(yhat); free(Hn);
        return ORC_ENOMEM;
    }
    if (rotate) orc_hadamard(D, Hn);
    int rc = ORC_OK;
    for (int64_t v = 0; v < n_vec && rc == ORC_OK; v++) {
        rc = orc_dequant(codes + (size_t)v * n_sub, 1, n_sub, codebook, N, d,
                         yhat);
        if (rc == ORC_OK)
            inverse_transform(yhat, D, Hn, smooth, smooth_mode,
                              head ? head[v] : 0, rotate,
                              xhat + (size_t)v * D);
    }
    free(yhat); free(Hn);
    return rc;
}

/*
 * Mask of the fused attention: key j is visible to query row i iff
 *   (!causal || j <= q_abs) && (W == 0 || j > q_abs - W),
 *   q_abs = S_kv - S_q + i.
 * [API] metal_fused_sdpa: causal "queries align to the tail of S_kv";
 * sliding_window "only attend to the last sliding_window keys before each
 * query position"; rabitq_prefill_attend spells the alignment out
 * (q_abs = (S_kv - S_q) + q_pos, slot j masked whenever j > q_abs).
 */
static int visible(int64_t j, int64_t q_abs, int causal, int64_t W) {
    if (causal && j > q_abs) return 0;
    if (W > 0 && j <= q_abs - W) return 0;
    return 1;
}

/*
 * Attention over the compressed cache, for a list of query rows.
 *   q        [B, H_q, S_q, D]   raw (untransformed) queries
 *   k_codes  [B, H_kv, S_kv, D/dk], v_codes [B, H_kv, S_kv, D/dv]  int32
 *   k_cb [Nk, dk], v_cb [Nv, dv], smooth (key smooth, see orc_encode)
 *   rows     [n_rows, 3]        (b, h_q, i) triples
 *   out      [n_rows, D]        float64 attention output
 * Per row: g = h_q / (H_q / H_kv);  K_hat_j = s_g^-1 (.) Hn^T dequant(k_j);
 * V_hat_j = dequant(v_j);  s_j = scale * <q, K_hat_j> over the visible set;
 * p = softmax(s) (max-subtracted, exp from libm);  out = sum_j p_j V_hat_j.
 * An empty visible set gives a zero row.
 * [API] metal_fused_sdpa ("mathematically identical to running standard SDPA
 * on the dequantized fp16 K_hat"); [CACHE] VecInferKVCache.fused_sdpa takes
 * the untransformed q.  The oracle never forms the transformed query or a
 * lookup table, so agreement with a table-based kernel checks the dual
 * transform as well.
 * K_hat of the (b, g) pair last used is kept between rows, so rows sorted
 * by (b, h_q) reuse it.
 */
int orc_attend_rows(const double *q, int B, int H_q, int H_kv, int S_q,
                    int S_kv, int D, const int32_t *k_codes,
                    const double *k_cb, int Nk, int dk, const int32_t *v_codes,
                    const double *v_cb, int Nv, int dv, const double *smooth,
                    int smooth_mode, double scale, int causal,
                    int sliding_window, const int32_t *rows, int64_t n_rows,
                    double *out) {
    if (!q || !k_codes || !k_cb || !v_codes || !v_cb || !rows || !out)
        return ORC_EINVAL;
    if (B < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv != 0 || S_q < 0 ||
        S_kv < 0 || D <= 0 || dk <= 0 || dv <= 0 || D % dk != 0 ||
        D % dv != 0 || !is_pow2(D) || sliding_window < 0)
        return ORC_EINVAL;
    if (smooth_mode != 0 && !smooth) return ORC_EINVAL;
    int G = H_q / H_kv, nk = D / dk, nv = D / dv;
    double *Hn = malloc(sizeof(double) * (size_t)D * D);
    double *Khat = malloc(sizeof(double) * ((size_t)S_kv * D + 1));
    double *yhat = malloc(sizeof(double) * (size_t)D);
    double *vhat = malloc(sizeof(double) * (size_t)D);
    double *sc = malloc(sizeof(double) * ((size_t)S_kv + 1));
    if (!Hn || !Khat || !yhat || !vhat || !sc) {
        free(Hn); free(Khat); free(yhat); free(vhat); free(sc);
        return ORC_ENOMEM;
    }
    orc_hadamard(D, Hn);
    int have_b = -1, have_g = -1, rc = ORC_OK;
    for (int64_t r = 0; r < n_rows && rc == ORC_OK; r++) {
        int b = rows[3 * r], hq = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || hq < 0 || hq >= H_q || i < 0 || i >= S_q) {
            rc = ORC_EINVAL;
            break;
        }
        int g = hq / G;
        if (b != have_b || g != have_g) {
            for (int64_t j = 0; j < S_kv && rc == ORC_OK; j++) {
                const int32_t *kc =
                    k_codes + (((size_t)b * H_kv + g) * S_kv + j) * nk;
                rc = orc_dequant(kc, 1, nk, k_cb, Nk, dk, yhat);
                if (rc == ORC_OK)
                    inverse_transform(yhat, D, Hn, smooth, smooth_mode, g, 1,
                                      Khat + (size_t)j * D);
            }
            have_b = b;
            have_g = g;
        }
        if (rc != ORC_OK) break;
        const double *qr = q + (((size_t)b * H_q + hq) * S_q + i) * D;
        int64_t q_abs = (int64_t)S_kv - S_q + i;
        double mx = -INFINITY;
        int64_t n_vis = 0;
        for (int64_t j = 0; j < S_kv; j++) {
            if (!visible(j, q_abs, causal, sliding_window)) continue;
            double acc = 0.0;
            for (int t = 0; t < D; t++) acc += qr[t] * Khat[(size_t)j * D + t];
            sc[j] = scale * acc;
            if (sc[j] > mx) mx = sc[j];
            n_vis++;
        }
        double *o = out + (size_t)r * D;
        for (int t = 0; t < D; t++) o[t] = 0.0;
        if (n_vis == 0) continue;
        double denom = 0.0;
        for (int64_t j = 0; j < S_kv; j++) {
            if (!visible(j, q_abs, causal, sliding_window)) continue;
            sc[j] = exp(sc[j] - mx);
            denom += sc[j];
        }
        for (int64_t j = 0; j < S_kv && rc == ORC_OK; j++) {
            if (!visible(j, q_abs, causal, sliding_window)) continue;
            const int32_t *vc =
                v_codes + (((size_t)b * H_kv + g) * S_kv + j) * nv;
            rc = orc_dequant(vc, 1, nv, v_cb, Nv, dv, vhat);
            double p = sc[j] / denom;
            for (int t = 0; t < D; t++) o[t] += p * vhat[t];
        }
    }
    free(Hn); free(Khat); free(yhat); free(vhat); free(sc);
    return rc;
}

/*
 * Lookup-table score (asymmetric MIPS) for one query against one coded key:
 *   q~ = Hn . (q (.) s_g^-1),  LUT[m][c] = scale * <q~_m, C_k[c]>,
 *   score = sum_m LUT[m][code_m].
 * [API] "compute_query_lut (asymmetric-MIPS query-codebook LUT precompute)"
 * and metal_fused_sdpa's requirement q_tilde @ K_tilde.T == q @ K_hat.T.
 * The oracle's attention never uses this; it exists so that a test can check
 * the identity against the explicit reconstruction above.
 */
int orc_lut_score(const double *q, int D, const double *smooth, int smooth_mode,
                  int g, const double *k_cb, int Nk, int dk,
                  const int32_t *code, double scale, double *score) {
    if (!q || !k_cb || !code || !score || !is_pow2(D) || D % dk != 0)
        return ORC_EINVAL;
    if (smooth_mode != 0 && !smooth) return ORC_EINVAL;
    int nk = D / dk;
    double *Hn = malloc(sizeof(double) * (size_t)D * D);
    double *qs = malloc(sizeof(double) * (size_t)D);
    double *qt = malloc(sizeof(double) * (size_t)D);
    if (!Hn || !qs || !qt) {
        free(Hn); free(qs); free(qt);
        return ORC_ENOMEM;
    }
    orc_hadamard(D, Hn);
    for (int t = 0; t < D; t++) qs[t] = q[t] / smooth_at(smooth, smooth_mode, D, g, t);
    for (int r = 0; r < D; r++) {
        double acc = 0.0;
        for (int t = 0; t < D; t++) acc += Hn[(size_t)r * D + t] * qs[t];
        qt[r] = acc;
    }
    double total = 0.0;
    int rc = ORC_OK;
    for (int m = 0; m < nk; m++) {
        int32_t c = code[m];
        if (c < 0 || c >= Nk) { rc = ORC_EINVAL; break; }
        double lut = 0.0;
        for (int t = 0; t < dk; t++) lut += qt[m * dk + t] * k_cb[(size_t)c * dk + t];
        total += scale * lut;
    }
    *score = total;
    free(Hn); free(qs); free(qt);
    return rc;
}
