"""Bit-packed codes (code_bytes 0 at the boundary; int32 token rows in the
binding): b = ceil(log2 N) bits per code, code m of a token row in bits
[m b, m b + b) of its 32-bit words, rows padded to whole words.  Page
"veloxquant_mlx.cache.vecinfer_cache module": per-token storage
(D / d) * b / 8 bytes, e.g. 20 bytes for 16 ten-bit codes.

The packing below is this test's own (numpy); encode must write exactly the
packed form of the codes the byte-code encode writes, dequant must read it
back, and attention over packed caches must match the oracle over the same
codes.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu_helpers import DEV, check_encode, dev
from oracle import parity
from product_vq_compressed_gb300 import binding as vq

pytestmark = pytest.mark.gpu


def bits_for(N):
    b = 1
    while (1 << b) < N:
        b += 1
    return b


def pack(codes, bits):
    n_sub = codes.shape[-1]
    words = (n_sub * bits + 31) // 32
    flat = codes.reshape(-1, n_sub).astype(np.uint64)
    out = np.zeros((flat.shape[0], words + 1), np.uint64)
    for m in range(n_sub):
        w, sh = divmod(m * bits, 32)
        v = flat[:, m] << np.uint64(sh)
        out[:, w] |= v & np.uint64(0xFFFFFFFF)
        out[:, w + 1] |= v >> np.uint64(32)
    return out[:, :words].astype(np.uint32).view(np.int32).reshape(codes.shape[:-1] + (words,))


def unpack(rows, n_sub, bits):
    words = rows.shape[-1]
    flat = rows.reshape(-1, words).view(np.uint32).astype(np.uint64)
    flat = np.concatenate([flat, np.zeros((flat.shape[0], 1), np.uint64)], axis=1)
    out = np.zeros((flat.shape[0], n_sub), np.int64)
    for m in range(n_sub):
        w, sh = divmod(m * bits, 32)
        v = (flat[:, w] | (flat[:, w + 1] << np.uint64(32))) >> np.uint64(sh)
        out[:, m] = (v & np.uint64((1 << bits) - 1)).astype(np.int64)
    return out.reshape(rows.shape[:-1] + (n_sub,))


def test_pack_helpers_round_trip():
    rng = np.random.default_rng(0)
    for bits, n_sub in [(10, 16), (4, 32), (3, 21), (16, 5), (1, 64)]:
        c = rng.integers(0, 1 << bits, size=(3, 7, n_sub))
        assert np.array_equal(unpack(pack(c, bits), n_sub, bits), c)


@pytest.mark.parametrize("N,d,D", [(1024, 8, 128), (16, 4, 128), (1000, 4, 64), (5, 2, 32),
                                   (256, 4, 128)])
def test_encode_packed_equals_byte_codes(N, d, D):
    rng = np.random.default_rng(N + d)
    B, H, S = 2, 3, 77
    keys = rng.standard_normal((B, H, S, D)).astype(np.float16)
    values = rng.standard_normal((B, H, S, D)).astype(np.float16)
    smooth = rng.uniform(0.5, 2.0, (H, D)).astype(np.float32)
    cb = rng.standard_normal((N, d)).astype(np.float32)
    kp, _ = vq.encode_keys(dev(keys), dev(cb), d, dev(smooth), packed=True)
    kb, _ = vq.encode_keys(dev(keys), dev(cb), d, dev(smooth))
    vp, _ = vq.encode_values(dev(values), dev(cb), d, packed=True)
    vb, _ = vq.encode_values(dev(values), dev(cb), d)
    torch.cuda.synchronize()
    bits, n_sub = bits_for(N), D // d
    assert kp.dtype == torch.int32 and kp.shape[-1] == (n_sub * bits + 31) // 32
    kbn = kb.cpu().numpy().astype(np.int64)
    assert np.array_equal(kp.cpu().numpy(), pack(kbn, bits))
    assert np.array_equal(vp.cpu().numpy(), pack(vb.cpu().numpy().astype(np.int64), bits))
    res = check_encode(keys, cb, d, smooth, True, unpack(kp.cpu().numpy(), n_sub, bits), None)
    assert res["mismatch"] == res["near_tie"], res
    # dequant of packed rows equals dequant of the byte codes
    out_p = vq.dequant(kp, dev(cb), n_sub=n_sub)
    out_b = vq.dequant(kb, dev(cb))
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_b)


def test_encode_into_packed_rows():
    rng = np.random.default_rng(3)
    N, d, D, H, S, cap, off = 1024, 8, 128, 2, 40, 100, 33
    keys = rng.standard_normal((1, H, S, D)).astype(np.float16)
    smooth = rng.uniform(0.5, 2.0, (H, D)).astype(np.float32)
    cb = rng.standard_normal((N, d)).astype(np.float32)
    words = vq.packed_row_words(D // d, N)
    buf = torch.full((1, H, cap, words), -7, dtype=torch.int32, device=DEV)
    vq.encode_keys_into(dev(keys), dev(cb), d, dev(smooth), buf, off)
    ref, _ = vq.encode_keys(dev(keys), dev(cb), d, dev(smooth), packed=True)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.array_equal(b[:, :, off:off + S], ref.cpu().numpy())
    assert np.all(b[:, :, :off] == -7) and np.all(b[:, :, off + S:] == -7)


@pytest.mark.parametrize("Nk,dk,Nv,dv,S_q,entry", [(1024, 8, 16, 4, 1, "decode"),
                                                   (1000, 4, 256, 4, 3, "decode"),
                                                   (1024, 8, 256, 4, 1, "decode"),
                                                   (600, 8, 200, 4, 2, "decode"),
                                                   (256, 4, 256, 4, 128, "prefill"),
                                                   (1024, 8, 100, 4, 80, "prefill"),
                                                   (1024, 8, 256, 4, 80, "prefill")])
def test_attend_over_packed_cache(Nk, dk, Nv, dv, S_q, entry):
    rng = np.random.default_rng(Nk + Nv + S_q)
    B, H_kv, H_q, D, S_kv = 2, 2, 4, 128, 300
    kcb = rng.standard_normal((Nk, dk)).astype(np.float32)
    vcb = rng.standard_normal((Nv, dv)).astype(np.float32)
    smooth = rng.uniform(0.5, 2.0, (H_kv, D)).astype(np.float32)
    q = rng.standard_normal((B, H_q, S_q, D)).astype(np.float16)
    kc = rng.integers(0, Nk, size=(B, H_kv, S_kv, D // dk))
    vc = rng.integers(0, Nv, size=(B, H_kv, S_kv, D // dv))
    kp = dev(pack(kc, bits_for(Nk)))
    vp = dev(pack(vc, bits_for(Nv)))
    fn = vq.decode_attend if entry == "decode" else vq.prefill_attend
    out = fn(dev(q), kp, dev(kcb), vp, dev(vcb), dev(smooth), 1 / np.sqrt(D), causal=True,
             sliding_window=0)
    torch.cuda.synchronize()
    ref = oracle.attend(q, kc, kcb, vc, vcb, smooth, 1 / np.sqrt(D), True, 0)
    ok, err, _ = parity.allclose_report(out.cpu().numpy().astype(np.float64),
                                        oracle.to_f16(ref).astype(np.float64))
    assert ok, f"max |err| {err}"


def _oracle_per_batch(q, kc, vc, kcb, vcb, smooth, scale, window, lens):
    out = np.zeros(q.shape, np.float64)
    for b, L in enumerate(lens):
        out[b] = oracle.attend(q[b:b + 1], kc[b:b + 1, :, :L], kcb, vc[b:b + 1, :, :L], vcb,
                               smooth, scale, True, window)[0]
    return out


@pytest.mark.parametrize("S_q,window,Nk", [(1, 0, 1024), (1, 300, 1024), (4, 100, 777)])
def test_packed_key_path_gqa_window_lengths(S_q, window, Nk):
    """The packed-key decode path (10-bit key codes of 8 dimensions, uint8
    value codes of 4, D = 128): GQA, sliding window, per-batch lengths, a
    buffer of more rows than S_kv, codes at both ends of the code range,
    a ragged last tile, against the oracle on each batch's compact cache."""
    rng = np.random.default_rng(Nk + window + S_q)
    B, H_kv, H_q, D, dk, dv, Nv = 3, 2, 8, 128, 8, 4, 256
    S_kv, rows = 1000, 1037
    kcb = rng.standard_normal((Nk, dk)).astype(np.float32)
    vcb = rng.standard_normal((Nv, dv)).astype(np.float32)
    smooth = rng.uniform(0.5, 2.0, (H_kv, D)).astype(np.float32)
    q = rng.standard_normal((B, H_q, S_q, D)).astype(np.float16)
    kc = rng.integers(0, Nk, size=(B, H_kv, rows, D // dk))
    vc = rng.integers(0, Nv, size=(B, H_kv, rows, D // dv))
    kc[:, :, ::7] = Nk - 1          # the last code in every lane position
    kc[:, :, 3::11] = 0
    kp = dev(pack(kc, bits_for(Nk)))
    vp = dev(vc.astype(np.uint8))
    lens = [S_kv, 517, 33]
    kl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    scale = 1 / np.sqrt(D)
    out = vq.decode_attend(dev(q), kp, dev(kcb), vp, dev(vcb), dev(smooth), scale, causal=True,
                           sliding_window=window, s_kv=S_kv, kv_lens=kl)
    full = vq.decode_attend(dev(q), kp, dev(kcb), vp, dev(vcb), dev(smooth), scale,
                            causal=True, sliding_window=window, s_kv=S_kv)
    torch.cuda.synchronize()
    ref = _oracle_per_batch(q, kc, vc, kcb, vcb, smooth, scale, window, lens)
    ok, err, _ = parity.allclose_report(out.cpu().numpy().astype(np.float64),
                                        oracle.to_f16(ref).astype(np.float64))
    assert ok, f"kv_lens max |err| {err}"
    ref = _oracle_per_batch(q, kc, vc, kcb, vcb, smooth, scale, window, [S_kv] * B)
    ok, err, _ = parity.allclose_report(full.cpu().numpy().astype(np.float64),
                                        oracle.to_f16(ref).astype(np.float64))
    assert ok, f"max |err| {err}"


def test_gqa_decode_packed_full_size_whole_groups():
    """The 10-bit packed-key decode workload at full size (B=32, H_q=32,
    H_kv=8, S_kv=32768) in the launch the benchmark times: every query head
    of the first and the last batch, against the oracle over the same codes.
    The cache is packed here, batch by batch, by this file's own packer."""
    from _gpu_helpers import oracle_attend_rows_parallel
    from product_vq_compressed_gb300.workloads import WORKLOADS, make_inputs
    spec = WORKLOADS["gqa-decode-packed"]
    inp = make_inputs(spec)
    kc = inp["k_codes"]
    bits = bits_for(spec.k_N)
    kp = np.concatenate([pack(kc[b:b + 1], bits) for b in range(spec.B)])
    out = vq.decode_attend(dev(inp["q"]), dev(kp), dev(inp["k_codebook"]),
                           dev(inp["v_codes"]), dev(inp["v_codebook"]), dev(inp["smooth"]),
                           spec.sm_scale, causal=spec.causal, sliding_window=spec.window)
    torch.cuda.synchronize()
    rows = np.array([(b, h, 0) for b in (0, spec.B - 1) for h in range(spec.H_q)])
    ref = oracle_attend_rows_parallel(inp, spec, rows, kc, inp["v_codes"])
    got = out.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    ok, err, excess = parity.allclose_report(got, ref)
    assert ok, f"max |err| {err}, worst excess {excess}"
