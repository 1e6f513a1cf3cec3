"""GPU parity of key / value encode and dequant against the float64 oracle.

Codes must equal the oracle's except where the oracle's two best distances
are a near tie (relative gap < 1e-6, oracle/parity.py); every other
mismatch fails, including the scaled-up and outlier cases.
Reconstructions are held to
|err| <= 2e-3 + 1e-2 |ref|.  Sizes span several 512-sub-vector tiles and a
ragged tail; the full-size workloads are checked on sampled vectors.
"""
import numpy as np
import pytest
import torch

from _gpu_helpers import DEV, check_encode, dev
from product_vq_compressed_gb300 import binding as vq
from product_vq_compressed_gb300.workloads import WORKLOADS, make_inputs, small_spec

pytestmark = pytest.mark.gpu

CASES = [
    # D, sub_dim, N, smooth_mode, B, H, S
    (64, 4, 256, 2, 1, 2, 256),      # tiny-like
    (128, 4, 256, 2, 1, 3, 77),      # ragged: 77 tokens, 16 per tile
    (128, 8, 1024, 2, 2, 2, 129),    # uint16 codes
    (32, 2, 16, 1, 1, 4, 300),
    (256, 8, 64, 0, 1, 2, 61),
    (512, 16, 128, 2, 1, 1, 9),      # one token per tile
    (128, 1, 32, 2, 1, 1, 12),
    (64, 16, 512, 1, 1, 2, 50),
    (64, 4, 4096, 2, 1, 1, 40),      # codebook too large for the tensor-core screen
]


@pytest.mark.parametrize("D,d,N,mode,B,H,S", CASES)
@pytest.mark.parametrize("with_hat", [False, True])
def test_encode_keys_parity(D, d, N, mode, B, H, S, with_hat):
    spec = small_spec(D * 7 + d + N % 97, B=B, H_q=H, H_kv=H, D=D, S_kv=S,
                      k_N=N, k_d=d, smooth_mode=mode,
                      key_outliers=(1, D // 2), outlier_scale=8.0)
    inp = make_inputs(spec)
    kc, kh = vq.encode_keys(dev(inp["keys"]), dev(inp["k_codebook"]), d,
                            dev(inp["smooth"]), want_k_hat=with_hat)
    torch.cuda.synchronize()
    assert kc.dtype == (torch.uint8 if N <= 256 else torch.uint16)
    res = check_encode(inp["keys"], inp["k_codebook"], d, inp["smooth"], True,
                       kc.cpu().numpy(), None if kh is None else kh.cpu().numpy())
    assert res["mismatch"] == res["near_tie"], res


@pytest.mark.parametrize("D,d,N,mode,B,H,S", CASES[:5])
def test_encode_values_parity(D, d, N, mode, B, H, S):
    spec = small_spec(D + d + N, B=B, H_q=H, H_kv=H, D=D, S_kv=S, v_N=N, v_d=d)
    inp = make_inputs(spec)
    vc, vh = vq.encode_values(dev(inp["values"]), dev(inp["v_codebook"]), d,
                              want_v_hat=True)
    torch.cuda.synchronize()
    res = check_encode(inp["values"], inp["v_codebook"], d, None, False,
                       vc.cpu().numpy(), vh.cpu().numpy())
    assert res["near_tie"] == res["mismatch"]


def test_encode_uint16_codes_for_small_codebook():
    spec = small_spec(5, D=64, S_kv=40, k_N=16, k_d=4)
    inp = make_inputs(spec)
    codes = torch.empty((1, 2, 40, 16), dtype=torch.uint16, device=DEV)
    vq.encode_keys(dev(inp["keys"]), dev(inp["k_codebook"]), 4,
                   dev(inp["smooth"]), codes=codes)
    torch.cuda.synchronize()
    check_encode(inp["keys"], inp["k_codebook"], 4, inp["smooth"], True,
                 codes.cpu().numpy().astype(np.int64), None)


def test_encode_single_vector_and_empty():
    spec = small_spec(6, D=128, S_kv=1, H_q=1, H_kv=1)
    inp = make_inputs(spec)
    kc, kh = vq.encode_keys(dev(inp["keys"]), dev(inp["k_codebook"]), 4,
                            dev(inp["smooth"]), want_k_hat=True)
    torch.cuda.synchronize()
    check_encode(inp["keys"], inp["k_codebook"], 4, inp["smooth"], True,
                 kc.cpu().numpy(), kh.cpu().numpy())
    empty = torch.empty((1, 2, 0, 128), dtype=torch.float16, device=DEV)
    c, _ = vq.encode_keys(empty, dev(inp["k_codebook"]), 4, None)
    assert c.shape == (1, 2, 0, 32)


def test_encode_round_trip_is_exact_on_gpu():
    """Keys built from codebook entries encode back to the same codes."""
    import scipy.linalg
    rng = np.random.default_rng(9)
    D, d, N, H, S = 128, 4, 256, 2, 64
    cb = (rng.standard_normal((N, d)) * 3).astype(np.float32)
    codes = rng.integers(0, N, size=(1, H, S, D // d))
    smooth = rng.uniform(0.5, 2, (H, D)).astype(np.float32)
    Hn = scipy.linalg.hadamard(D) / np.sqrt(D)
    x = (cb[codes].reshape(1, H, S, D).astype(np.float64) @ Hn.T) / smooth[None, :, None, :]
    x16 = x.astype(np.float16)
    kc, _ = vq.encode_keys(dev(x16), dev(cb), d, dev(smooth))
    torch.cuda.synchronize()
    # fp16 rounding of x moves points by ~1e-3; the codebook spacing is far
    # larger, so every code must come back
    assert np.array_equal(kc.cpu().numpy().astype(np.int64), codes)


@pytest.mark.parametrize("code_bytes,N,d", [(1, 256, 4), (2, 1024, 8), (1, 16, 2)])
@pytest.mark.parametrize("f32", [True, False])
def test_dequant_bit_exact(code_bytes, N, d, f32):
    import oracle
    rng = np.random.default_rng(N + d)
    cb = rng.standard_normal((N, d)).astype(np.float32)
    dt = np.uint8 if code_bytes == 1 else np.uint16
    codes = rng.integers(0, N, size=(3, 5, 37, 128 // d)).astype(dt)
    out = vq.dequant(dev(codes), dev(cb), out_f32=f32)
    torch.cuda.synchronize()
    ref = oracle.dequant(codes.astype(np.int64), cb)
    if f32:
        assert np.array_equal(out.cpu().numpy(), ref.astype(np.float32))
    else:
        assert np.array_equal(out.cpu().numpy().view(np.uint16),
                              oracle.to_f16(ref).view(np.uint16))


@pytest.mark.parametrize("name", ["tiny", "decode-1seq", "bulk-encode"])
def test_encode_full_size_sampled(name):
    """Full-size workloads, codes and k_hat on a sample of vectors (plus the
    first and last), in the launch configuration the benchmark uses."""
    spec = WORKLOADS[name]
    inp = make_inputs(spec)
    with_hat = name != "decode-1seq"
    kc, kh = vq.encode_keys(dev(inp["keys"]), dev(inp["k_codebook"]), spec.k_d,
                            dev(inp["smooth"]), want_k_hat=with_hat)
    vc, _ = vq.encode_values(dev(inp["values"]), dev(inp["v_codebook"]), spec.v_d)
    torch.cuda.synchronize()
    n = spec.B * spec.H_kv * spec.enc_len
    rng = np.random.default_rng(123)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 1500)]))
    rk = check_encode(inp["keys"], inp["k_codebook"], spec.k_d, inp["smooth"],
                      True, kc.cpu().numpy(),
                      None if kh is None else kh.cpu().numpy(), rows=rows)
    rv = check_encode(inp["values"], inp["v_codebook"], spec.v_d, None, False,
                      vc.cpu().numpy(), None, rows=rows)
    print(name, "keys", rk, "values", rv)
    assert rk["mismatch"] == rk["near_tie"] and rv["mismatch"] == rv["near_tie"]


def _encode_case(seed, D, d, N, x_scale, cb_scale, H=2, S=70, cb=None):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((1, H, S, D)) * x_scale).astype(np.float16)
    if cb is None:
        cb = (rng.standard_normal((N, d)) * cb_scale).astype(np.float32)
    smooth = rng.uniform(0.5, 2.0, (H, D)).astype(np.float32)
    kc, kh = vq.encode_keys(dev(x), dev(cb), d, dev(smooth), want_k_hat=True)
    torch.cuda.synchronize()
    res = check_encode(x, cb, d, smooth, True, kc.cpu().numpy(), kh.cpu().numpy())
    return kc.cpu().numpy().astype(np.int64), res


@pytest.mark.parametrize("D,d,N,x_scale,cb_scale", [
    (128, 4, 100, 1.0, 1.0),       # N not a multiple of 32: padded columns
    (64, 2, 1, 1.0, 1.0),          # a single centroid
    (128, 8, 33, 1.0, 1.0),
    (256, 2, 256, 1.0, 1.0),
    (128, 4, 256, 3000.0, 3000.0), # beyond the range of the fp16 operand split
    (128, 4, 256, 3000.0, 1.0),    # large sub-vectors, ordinary codebook
    (64, 4, 256, 1e-4, 1e-4),      # fp16-subnormal split parts
])
def test_encode_screening_edge_cases(D, d, N, x_scale, cb_scale):
    codes, res = _encode_case(D + N + d, D, d, N, x_scale, cb_scale)
    assert res["mismatch"] == res["near_tie"], res
    if N == 1:
        assert (codes == 0).all()


@pytest.mark.parametrize("layout", ["adjacent", "far"])
def test_encode_duplicate_centroids_take_lowest_index(layout):
    """Exact duplicates tie in every arithmetic; the lower index must win."""
    rng = np.random.default_rng(31)
    base = rng.standard_normal((128, 4)).astype(np.float32)
    cb = np.repeat(base, 2, axis=0) if layout == "adjacent" else np.concatenate([base, base])
    codes, res = _encode_case(32, 128, 4, 256, 1.0, 1.0, cb=cb)
    if layout == "adjacent":
        assert (codes % 2 == 0).all()
    else:
        assert (codes < 128).all()


@pytest.mark.parametrize("d,N,rotate", [
    (4, 256, True),     # tensor-core screen, keys
    (4, 256, False),    # tensor-core screen, values
    (8, 1024, True),    # tensor-core screen, uint16 codes
    (16, 64, True),     # CUDA-core search
    (4, 4096, True),    # CUDA-core search, large codebook
])
def test_encode_close_pairs_are_decided_exactly(d, N, rotate):
    """Codebooks with two centroids at almost the same distance from a
    sub-vector: the relative gap of the squared distances (about 4e-6 for
    keys, 2e-6 for values) is above the near-tie threshold (1e-6), so the
    code must equal the oracle's, but below what the fp32 rotation and
    distances can order; the kernels must decide these sub-vectors in
    higher precision."""
    import scipy.linalg
    rng = np.random.default_rng(1000 + d * 7 + N + rotate)
    D, H, S = 128, 2, 16
    x16 = rng.standard_normal((1, H, S, D)).astype(np.float16)
    smooth = rng.uniform(0.5, 2.0, (H, D)).astype(np.float32) if rotate else None
    x = x16.astype(np.float64)
    if rotate:
        Hn = scipy.linalg.hadamard(D) / np.sqrt(D)
        y = (x * smooth[None, :, None, :]) @ Hn
    else:
        y = x
    subs = y.reshape(-1, d)
    n_pairs = min(N // 4, len(subs))
    pick = rng.choice(len(subs), n_pairs, replace=False)
    # the rest of the codebook: far away from every sub-vector
    fill = rng.standard_normal((N, d))
    cb = 40.0 * fill / np.linalg.norm(fill, axis=1, keepdims=True)
    eps = 2e-6 if rotate else 1e-6
    slots = rng.permutation(N)[:2 * n_pairs].reshape(n_pairs, 2)
    for k, sv in enumerate(pick):
        u = rng.standard_normal((2, d))
        u /= np.linalg.norm(u, axis=1, keepdims=True)
        near, far = slots[k] if rng.random() < 0.5 else slots[k][::-1]
        cb[near] = subs[sv] + u[0]
        cb[far] = subs[sv] + (1.0 + eps) * u[1]
    cb = cb.astype(np.float32)
    if rotate:
        codes, _ = vq.encode_keys(dev(x16), dev(cb), d, dev(smooth))
    else:
        codes, _ = vq.encode_values(dev(x16), dev(cb), d)
    torch.cuda.synchronize()
    res = check_encode(x16, cb, d, smooth, rotate, codes.cpu().numpy(), None)
    assert res["mismatch"] == res["near_tie"], res
