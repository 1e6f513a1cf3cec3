"""Pins of the float64 oracle against facts fixed outside the oracle itself.

Each test checks the oracle against something it does not compute: a library
routine (scipy's Sylvester Hadamard), a closed form, a hand-worked example
under tests/golden/, an exact round trip, brute force on tiny inputs, or an
invariant.  Together they are chosen so that a plausible slip in the oracle
-- a wrong normalisation, smooth applied the wrong way round, a dropped
mask bound, an off-by-one alignment, a wrong GQA map, an unnormalised
softmax, a tie broken to the wrong side -- fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _hn(D):
    """Normalised Sylvester Hadamard from scipy (a library routine)."""
    return scipy.linalg.hadamard(D).astype(np.float64) / math.sqrt(D)


# ----------------------------------------------------------------- Hadamard

@pytest.mark.parametrize("D", [1, 2, 4, 8, 16, 32, 64, 128, 256, 512])
def test_hadamard_equals_scipy_sylvester(oracle, D):
    assert np.array_equal(oracle.hadamard(D) * math.sqrt(D),
                          scipy.linalg.hadamard(D).astype(np.float64))


@pytest.mark.parametrize("D", [4, 32, 128])
def test_hadamard_popcount_closed_form(oracle, D):
    H = oracle.hadamard(D) * math.sqrt(D)
    i, j = np.meshgrid(np.arange(D), np.arange(D), indexing="ij")
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    assert np.array_equal(np.rint(H), (-1.0) ** pc)


@pytest.mark.parametrize("D", [8, 64, 512])
def test_hadamard_integer_orthogonality(oracle, D):
    Hpm = np.rint(oracle.hadamard(D) * math.sqrt(D)).astype(np.int64)
    assert set(np.unique(Hpm)) == {-1, 1}
    assert np.array_equal(Hpm @ Hpm.T, D * np.eye(D, dtype=np.int64))
    Hn = oracle.hadamard(D)
    assert np.allclose(Hn @ Hn, np.eye(D), atol=1e-14, rtol=0)


# ------------------------------------------------------------ golden examples

def test_golden_encode_handworked(oracle):
    g = json.load(open(os.path.join(GOLDEN, "encode_d4_handworked.json")))
    x = np.array(g["x"])[None, :]
    r = oracle.encode(x, np.array(g["codebook"]), heads=np.zeros(1, np.int32),
                      smooth=np.array(g["smooth_D"]), rotate=True,
                      want_y=True, want_xhat=True)
    assert r["codes"][0].tolist() == g["codes"]
    assert np.allclose(r["y"][0], g["y"], atol=1e-15)
    assert np.allclose(r["d1"][0], g["d1"], atol=1e-15)
    assert np.allclose(r["d2"][0], g["d2"], atol=1e-15)
    assert np.allclose(r["xhat"][0], g["xhat"], atol=1e-15)


def test_golden_attend_handworked(oracle):
    g = json.load(open(os.path.join(GOLDEN, "attend_d4_handworked.json")))
    D = g["D"]
    kc = np.array(g["k_codes"], np.int32)[None, None]
    vc = np.array(g["v_codes"], np.int32)[None, None]
    for case in g["cases"]:
        S_q = case["S_q"]
        q = np.tile(np.array(g["q_row"]), (1, 1, S_q, 1))
        out = oracle.attend(q, kc, np.array(g["k_codebook"]), vc,
                            np.array(g["v_codebook"]), None, g["scale"],
                            causal=case["causal"],
                            sliding_window=case["window"])
        assert out.shape == (1, 1, S_q, D)
        assert np.allclose(out[0, 0], np.array(case["out"]), atol=1e-14), case


# -------------------------------------------------------------- nearest code

def _brute_nearest(y, cb):
    """Lowest index of the minimum exact squared distance, plus top-2."""
    dists = [sum((a - b) ** 2 for a, b in zip(y, c)) for c in cb]
    best = min(dists)
    idx = dists.index(best)
    rest = dists[:idx] + dists[idx + 1:]
    return idx, best, (min(rest) if rest else math.inf)


@pytest.mark.parametrize("d", [1, 2, 4])
def test_argmin_brute_force_integer_points(oracle, d):
    rng = np.random.default_rng(100 + d)
    N = 12
    cb = rng.integers(-3, 4, size=(N, d)).astype(np.float64)
    cb[5] = cb[2]          # duplicated centroid: index 2 must win
    cb[9] = cb[0]
    n_sub = 8 // d if d <= 8 else 1
    x = rng.integers(-4, 5, size=(300, n_sub * d)).astype(np.float64)
    # points exactly halfway between two centroids (equidistant)
    x[0, :d] = (cb[1] + cb[3]) / 2.0
    x[1, :d] = cb[2]
    r = oracle.encode(x, cb, rotate=False)
    for v in range(x.shape[0]):
        for m in range(n_sub):
            y = x[v, m * d:(m + 1) * d].tolist()
            idx, best, second = _brute_nearest(y, cb.tolist())
            assert r["codes"][v, m] == idx
            assert r["d1"][v, m] == best
            assert r["d2"][v, m] == second


def test_argmin_ties_lowest_index_all_equal(oracle):
    cb = np.zeros((7, 2))
    r = oracle.encode(np.array([[1.0, 2.0]]), cb, rotate=False)
    assert r["codes"][0, 0] == 0 and r["d1"][0, 0] == r["d2"][0, 0] == 5.0


# ------------------------------------------------------------ exact round trip

@pytest.mark.parametrize("smooth_mode", [0, 1, 2])
@pytest.mark.parametrize("D,d,N", [(32, 4, 16), (64, 4, 256), (128, 8, 1024),
                                   (256, 2, 64)])
def test_encode_exact_round_trip(oracle, smooth_mode, D, d, N):
    """Codebook holds the transformed sub-vectors -> encode returns them.

    x = s^-1 (.) Hn . concat_m C[code_m] with Hn from scipy; encoding x must
    give back exactly those codes (distance 0) and reconstruct x.
    """
    rng = np.random.default_rng(D * 10 + d + smooth_mode)
    H = 3
    cb = rng.standard_normal((N, d))
    codes = rng.integers(0, N, size=(2, H, 5, D // d))
    y = cb[codes].reshape(2, H, 5, D)
    if smooth_mode == 0:
        smooth, s_b = None, np.ones((1, H, 1, D))
    elif smooth_mode == 1:
        smooth = rng.uniform(0.5, 2.0, D)
        s_b = np.broadcast_to(smooth, (1, H, 1, D))
    else:
        smooth = rng.uniform(0.5, 2.0, (H, D))
        s_b = smooth[None, :, None, :]
    x = (y @ _hn(D).T) / s_b
    r = oracle.encode(x, cb, smooth=smooth, rotate=True, want_xhat=True,
                      want_y=True)
    assert np.array_equal(r["codes"], codes)
    assert np.max(r["d1"]) < 1e-24
    assert np.allclose(r["y"], y, atol=1e-12, rtol=0)
    assert np.allclose(r["xhat"], x, atol=1e-12, rtol=0)


def test_encode_round_trip_survives_fp16_input(oracle):
    """Cast to fp16, the inputs still encode to the same codes when every
    centroid is farther from the others than the fp16 perturbation."""
    rng = np.random.default_rng(7)
    D, d, N, H = 64, 4, 32, 2
    cb = rng.standard_normal((N, d)) * 4.0
    gaps = [np.linalg.norm(cb[a] - cb[b]) for a in range(N) for b in range(a)]
    codes = rng.integers(0, N, size=(1, H, 40, D // d))
    smooth = rng.uniform(0.5, 2.0, (H, D))
    x = (cb[codes].reshape(1, H, 40, D) @ _hn(D).T) / smooth[None, :, None, :]
    x16 = x.astype(np.float16).astype(np.float64)
    # perturbation in the rotated domain: ||Hn (s (.) dx)|| = ||s (.) dx||
    pert = np.max(np.linalg.norm((x16 - x) * smooth[None, :, None, :], axis=-1))
    assert 2 * pert < min(gaps)
    r = oracle.encode(x16, cb, smooth=smooth, rotate=True, want_xhat=True)
    assert np.array_equal(r["codes"], codes)
    assert np.allclose(oracle.to_f16(r["xhat"]).astype(np.float64), x16,
                       atol=2e-3, rtol=1e-2)


# -------------------------------------------------------------- dequant

def test_dequant_is_numpy_gather(oracle):
    rng = np.random.default_rng(3)
    cb = rng.standard_normal((256, 4))
    codes = rng.integers(0, 256, size=(3, 5, 32))
    out = oracle.dequant(codes, cb)
    assert np.array_equal(out, cb[codes].reshape(3, 5, 128))


def test_dequant_rejects_out_of_range(oracle):
    with pytest.raises(ValueError):
        oracle.dequant(np.array([[0, 4]]), np.zeros((4, 2)))


# ---------------------------------------------------------- LUT identity

@pytest.mark.parametrize("smooth_mode", [0, 1, 2])
def test_lut_score_equals_explicit_dot(oracle, smooth_mode):
    """sum_m LUT[m][code_m] == scale * <q, K_hat> (dual transform)."""
    rng = np.random.default_rng(11 + smooth_mode)
    D, d, N, H = 128, 4, 256, 4
    cb = rng.standard_normal((N, d))
    smooth = (None if smooth_mode == 0 else
              rng.uniform(0.5, 2.0, D) if smooth_mode == 1 else
              rng.uniform(0.5, 2.0, (H, D)))
    for trial in range(6):
        g = trial % H
        q = rng.standard_normal(D)
        code = rng.integers(0, N, D // d)
        khat = oracle.reconstruct(code[None], cb, heads=np.array([g]),
                                  smooth=smooth, rotate=True)[0]
        scale = 1 / math.sqrt(D)
        expect = scale * float(q @ khat)
        got = oracle.lut_score(q, smooth, g, cb, code, scale)
        assert abs(got - expect) <= 1e-12 * max(1.0, abs(expect))


# ------------------------------------------------------------- attention

def _visible(S_q, S_kv, causal, W):
    i = np.arange(S_q)[:, None]
    j = np.arange(S_kv)[None, :]
    q_abs = S_kv - S_q + i
    vis = np.ones((S_q, S_kv), bool)
    if causal:
        vis &= j <= q_abs
    if W > 0:
        vis &= j > q_abs - W
    return vis


@pytest.mark.parametrize("causal,W,S_q", [(True, 0, 1), (True, 0, 7),
                                          (True, 5, 9), (False, 0, 4),
                                          (False, 6, 4), (True, 3, 33)])
def test_one_centroid_codebook_gives_uniform_weights(oracle, causal, W, S_q):
    """With a single key centroid every score is equal, so the output is the
    plain mean of the visible V_hat rows."""
    rng = np.random.default_rng(21)
    B, H_kv, G, S_kv, D, dv = 2, 2, 3, 40, 32, 4
    kcb = rng.standard_normal((1, 8))
    vcb = rng.standard_normal((16, dv))
    kc = np.zeros((B, H_kv, S_kv, D // 8), np.int32)
    vc = rng.integers(0, 16, size=(B, H_kv, S_kv, D // dv))
    q = rng.standard_normal((B, H_kv * G, S_q, D))
    smooth = rng.uniform(0.5, 2, (H_kv, D))
    out = oracle.attend(q, kc, kcb, vc, vcb, smooth, 0.3, causal, W)
    vis = _visible(S_q, S_kv, causal, W)
    vhat = vcb[vc].reshape(B, H_kv, S_kv, D)
    for b in range(B):
        for h in range(H_kv * G):
            for i in range(S_q):
                expect = vhat[b, h // G][vis[i]].mean(axis=0)
                assert np.allclose(out[b, h, i], expect, atol=1e-13)


@pytest.mark.parametrize("causal,W,S_q,G", [(True, 0, 1, 1), (True, 0, 6, 2),
                                            (True, 4, 6, 4), (False, 0, 3, 2),
                                            (False, 5, 3, 1), (True, 100, 5, 2)])
def test_attention_matches_textbook_softmax(oracle, causal, W, S_q, G):
    """Keys whose transformed sub-vectors are codebook entries make K_hat
    known exactly (x below); the oracle must then equal softmax(scale q x^T)
    V_hat computed with scipy, for every (b, h_q, row)."""
    rng = np.random.default_rng(31 + S_q + G)
    B, H_kv, S_kv, D, dk, dv, Nk, Nv = 2, 2, 24, 32, 4, 2, 64, 32
    kcb = rng.standard_normal((Nk, dk))
    vcb = rng.standard_normal((Nv, dv))
    kc = rng.integers(0, Nk, size=(B, H_kv, S_kv, D // dk))
    vc = rng.integers(0, Nv, size=(B, H_kv, S_kv, D // dv))
    smooth = rng.uniform(0.5, 2, (H_kv, D))
    x = (kcb[kc].reshape(B, H_kv, S_kv, D) @ _hn(D).T) / smooth[None, :, None, :]
    vhat = vcb[vc].reshape(B, H_kv, S_kv, D)
    q = rng.standard_normal((B, H_kv * G, S_q, D))
    scale = 0.7
    out = oracle.attend(q, kc, kcb, vc, vcb, smooth, scale, causal, W)
    vis = _visible(S_q, S_kv, causal, W)
    for b in range(B):
        for h in range(H_kv * G):
            for i in range(S_q):
                s = scale * (x[b, h // G] @ q[b, h, i])
                p = scipy.special.softmax(np.where(vis[i], s, -np.inf))
                assert np.allclose(out[b, h, i], p @ vhat[b, h // G],
                                   atol=1e-12, rtol=1e-12)


def test_window_at_least_cache_equals_no_window(oracle):
    rng = np.random.default_rng(5)
    kcb, vcb = rng.standard_normal((16, 4)), rng.standard_normal((16, 4))
    kc = rng.integers(0, 16, (1, 1, 30, 8))
    vc = rng.integers(0, 16, (1, 1, 30, 8))
    q = rng.standard_normal((1, 1, 4, 32))
    a = oracle.attend(q, kc, kcb, vc, vcb, None, 0.5, True, 0)
    for W in (30, 31, 1000):
        assert np.array_equal(a, oracle.attend(q, kc, kcb, vc, vcb, None, 0.5,
                                               True, W))


def test_attend_rows_subset_matches_full(oracle):
    rng = np.random.default_rng(8)
    kcb, vcb = rng.standard_normal((16, 4)), rng.standard_normal((16, 4))
    kc = rng.integers(0, 16, (2, 2, 20, 8))
    vc = rng.integers(0, 16, (2, 2, 20, 8))
    q = rng.standard_normal((2, 4, 3, 32))
    full = oracle.attend(q, kc, kcb, vc, vcb, None, 0.5, True, 7)
    rows = np.array([[1, 3, 2], [0, 0, 0], [1, 2, 1]])
    part = oracle.attend_rows(q, kc, kcb, vc, vcb, None, 0.5, True, 7, rows)
    for r, (b, h, i) in enumerate(rows):
        assert np.array_equal(part[r], full[b, h, i])


# ---------------------------------------------------------- storage formula

@pytest.mark.parametrize("D,dk,N", [(128, 4, 256), (64, 4, 256), (128, 8, 1024),
                                    (128, 2, 16)])
def test_storage_per_token(D, dk, N):
    """Bytes per token and head: (D/d_k) * b_k / 8 with b_k = log2(N)
    (vecinfer_cache module summary).  Byte-aligned widths (8, 16 bits)
    store exactly that; narrower codes sit in the next byte-aligned word
    (4-bit codes in uint8 take 2x, 10-bit codes in uint16 take 1.6x)."""
    from product_vq_compressed_gb300.workloads import small_spec
    b_k = int(math.log2(N))
    formula = (D / dk) * b_k / 8
    spec = small_spec(0, D=D, k_d=dk, k_N=N)
    stored = (D // dk) * np.dtype(spec.k_code_dtype).itemsize
    if b_k in (8, 16):
        assert stored == formula
    else:
        container = 1 if N <= 256 else 2
        assert stored == (D // dk) * container and stored > formula
    if (D, dk, N) == (128, 4, 256):
        assert formula == 32.0
    if (D, dk, N) == (128, 8, 1024):
        assert formula == 20.0
