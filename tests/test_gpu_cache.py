"""GPU parity of the cache-append encode (codes written into a preallocated
cache at a row offset), of attention over a cache whose buffers hold more
rows than S_kv (kv_stride), and of per-batch cache lengths (kv_lens).

Pages: "veloxquant_mlx.cache.vecinfer_cache module" (update_and_fetch:
new tokens are encoded and stored after the cached ones; attention runs
over the stored codes).  Expected values come from the float64 oracle on
the compact cache of each batch.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu_helpers import DEV, check_encode, dev
from oracle import parity
from product_vq_compressed_gb300 import binding as vq

pytestmark = pytest.mark.gpu

SENTINEL = 0xAB


def _rng_inputs(seed, B, H, S, D, N, d, H_q=None, S_q=1):
    rng = np.random.default_rng(seed)
    keys = rng.standard_normal((B, H, S, D)).astype(np.float16)
    values = rng.standard_normal((B, H, S, D)).astype(np.float16)
    smooth = rng.uniform(0.5, 2.0, (H, D)).astype(np.float32)
    kcb = rng.standard_normal((N, d)).astype(np.float32)
    vcb = rng.standard_normal((N, d)).astype(np.float32)
    q = rng.standard_normal((B, H_q or H, S_q, D)).astype(np.float16)
    return rng, keys, values, smooth, kcb, vcb, q


@pytest.mark.parametrize("N,d,offset,cap", [(256, 4, 37, 200), (1024, 8, 0, 61),
                                             (256, 2, 150, 200)])
def test_encode_into_writes_only_its_rows(N, d, offset, cap):
    B, H, S, D = 2, 3, 50 if cap > 61 else 61, 128
    _, keys, values, smooth, kcb, vcb, _ = _rng_inputs(N + offset, B, H, S, D, N, d)
    def sentinel_buf():   # filled through a signed view (fill of uint16 is not universal)
        if N <= 256:
            return torch.full((B, H, cap, D // d), SENTINEL, dtype=torch.uint8, device=DEV)
        return torch.full((B, H, cap, D // d), SENTINEL, dtype=torch.int16,
                          device=DEV).view(vq.code_dtype(N))
    kbuf, vbuf = sentinel_buf(), sentinel_buf()
    _, kh = vq.encode_keys_into(dev(keys), dev(kcb), d, dev(smooth), kbuf, offset,
                                want_k_hat=True)
    vq.encode_values_into(dev(values), dev(vcb), d, vbuf, offset)
    ref_k, ref_kh = vq.encode_keys(dev(keys), dev(kcb), d, dev(smooth), want_k_hat=True)
    ref_v, _ = vq.encode_values(dev(values), dev(vcb), d)
    torch.cuda.synchronize()
    kb = kbuf.cpu().numpy().astype(np.int64)
    vb = vbuf.cpu().numpy().astype(np.int64)
    # the written rows are the plain encode's codes, the rest is untouched
    assert np.array_equal(kb[:, :, offset:offset + S], ref_k.cpu().numpy().astype(np.int64))
    assert np.array_equal(vb[:, :, offset:offset + S], ref_v.cpu().numpy().astype(np.int64))
    assert np.array_equal(kh.cpu().numpy().view(np.uint16), ref_kh.cpu().numpy().view(np.uint16))
    outside = np.concatenate([kb[:, :, :offset], kb[:, :, offset + S:],
                              vb[:, :, :offset], vb[:, :, offset + S:]], axis=2)
    assert np.all(outside == SENTINEL)
    # and they are the oracle's codes
    res = check_encode(keys, kcb, d, smooth, True, kb[:, :, offset:offset + S],
                       kh.cpu().numpy())
    assert res["mismatch"] == res["near_tie"], res


def test_encode_into_rejects_overflow():
    keys = torch.zeros((1, 1, 10, 64), dtype=torch.float16, device=DEV)
    cb = torch.zeros((16, 4), dtype=torch.float32, device=DEV)
    buf = torch.zeros((1, 1, 12, 16), dtype=torch.uint8, device=DEV)
    with pytest.raises(vq.VQError):
        vq.encode_keys_into(keys, cb, 4, None, buf, 3)   # 3 + 10 > 12
    with pytest.raises(vq.VQError):
        vq.encode_keys_into(keys, cb, 4, None, buf, -1)


def _cache(rng, B, H, rows, n, N):
    return (rng.integers(0, N, size=(B, H, rows, n)).astype(np.uint8),
            rng.integers(0, N, size=(B, H, rows, n)).astype(np.uint8))


def _oracle_per_batch(q, kc, vc, kcb, vcb, smooth, scale, causal, window, lens):
    B, H_q, S_q, D = q.shape
    out = np.zeros((B, H_q, S_q, D))
    for b in range(B):
        L = lens[b]
        out[b] = oracle.attend(q[b:b + 1], kc[b:b + 1, :, :L], kcb, vc[b:b + 1, :, :L],
                               vcb, smooth, scale, causal, window)[0]
    return out


@pytest.mark.parametrize("entry,S_q,window", [("decode", 1, 0), ("decode", 5, 40),
                                              ("prefill", 128, 0), ("prefill", 96, 200)])
def test_attend_strided_cache_and_kv_lens(entry, S_q, window):
    """Codes in buffers of `rows` > S_kv rows (garbage past S_kv) and
    per-batch lengths, against the oracle on each batch's compact cache."""
    B, H_kv, H_q, D, d, N = 3, 2, 8, 128, 4, 256
    S_kv, rows = 333, 380
    rng, _, _, smooth, kcb, vcb, q = _rng_inputs(S_q * 7 + window, B, H_kv, 1, D, N, d,
                                                 H_q=H_q, S_q=S_q)
    kc, vc = _cache(rng, B, H_kv, rows, D // d, N)
    lens = [S_kv, 290, max(S_q, 70)]
    scale = 1.0 / np.sqrt(D)
    fn = vq.decode_attend if entry == "decode" else vq.prefill_attend
    kl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = fn(dev(q), dev(kc), dev(kcb), dev(vc), dev(vcb), dev(smooth), scale,
             causal=True, sliding_window=window, s_kv=S_kv, kv_lens=kl)
    out_full = fn(dev(q), dev(kc), dev(kcb), dev(vc), dev(vcb), dev(smooth), scale,
                  causal=True, sliding_window=window, s_kv=S_kv)
    torch.cuda.synchronize()
    ref = _oracle_per_batch(q, kc, vc, kcb, vcb, smooth, scale, True, window, lens)
    ok, err, _ = parity.allclose_report(out.cpu().numpy().astype(np.float64), oracle.to_f16(ref).astype(np.float64))
    assert ok, f"kv_lens max |err| {err}"
    ref_full = _oracle_per_batch(q, kc, vc, kcb, vcb, smooth, scale, True, window, [S_kv] * B)
    ok, err, _ = parity.allclose_report(out_full.cpu().numpy().astype(np.float64),
                                        oracle.to_f16(ref_full).astype(np.float64))
    assert ok, f"strided max |err| {err}"


@pytest.mark.parametrize("entry,S_q", [("decode", 4), ("prefill", 128)])
def test_kv_lens_shorter_than_queries_gives_zero_rows(entry, S_q):
    """A batch holding fewer keys than it has causal query rows: the rows
    before the first key see nothing and come out zero (the oracle's empty
    visible set); lengths past S_kv are clamped."""
    B, H_kv, H_q, D, d, N = 2, 1, 2, 128, 4, 256
    S_kv = 300
    rng, _, _, smooth, kcb, vcb, q = _rng_inputs(11 + S_q, B, H_kv, 1, D, N, d,
                                                 H_q=H_q, S_q=S_q)
    kc, vc = _cache(rng, B, H_kv, S_kv, D // d, N)
    L0 = S_q // 2
    kl = torch.tensor([L0, 10 * S_kv], dtype=torch.int32, device=DEV)
    fn = vq.decode_attend if entry == "decode" else vq.prefill_attend
    out = fn(dev(q), dev(kc), dev(kcb), dev(vc), dev(vcb), dev(smooth), 1 / np.sqrt(D),
             causal=True, kv_lens=kl).cpu().numpy().astype(np.float64)
    torch.cuda.synchronize()
    ref = _oracle_per_batch(q, kc, vc, kcb, vcb, smooth, 1 / np.sqrt(D), True, 0,
                            [L0, S_kv])
    assert np.all(out[0, :, :S_q - L0] == 0.0)
    ok, err, _ = parity.allclose_report(out, oracle.to_f16(ref).astype(np.float64))
    assert ok, f"max |err| {err}"
