"""One decode step of the cache in one launch (vq_decode_step): the new
tokens' keys and values are encoded into the cache rows after the cached
ones, then every query attends over the updated cache.

Page: "veloxquant_mlx.cache.vecinfer_cache module", VecInferKVCache.
update_and_fetch followed by fused_sdpa.  Checks, against the float64
oracle: the new rows' codes (equal except at near ties), the rows that must
not change, and the attention output over the updated cache (computed by
the oracle from its own codes); against the separate calls (encode_into +
decode_attend): the same cache and an output within the tolerance; and a
CUDA-graph capture of the single launch that replays bit for bit.
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


def _case(seed, B, H_q, H_kv, S_kv, S_q, cap, D=128, d=4, N=256):
    rng = np.random.default_rng(seed)
    x = dict(
        smooth=rng.uniform(0.5, 2.0, (H_kv, D)).astype(np.float32),
        kcb=rng.standard_normal((N, d)).astype(np.float32),
        vcb=rng.standard_normal((N, d)).astype(np.float32),
        kc=rng.integers(0, N, (B, H_kv, cap, D // d)).astype(np.uint8),
        vc=rng.integers(0, N, (B, H_kv, cap, D // d)).astype(np.uint8),
        k_new=rng.standard_normal((B, H_kv, S_q, D)).astype(np.float16),
        v_new=rng.standard_normal((B, H_kv, S_q, D)).astype(np.float16),
        q=rng.standard_normal((B, H_q, S_q, D)).astype(np.float16),
        S_kv=S_kv, S_q=S_q, d=d, D=D)
    x["k_new"][..., 5] *= 8   # an outlier channel
    # rows the step must not touch
    x["kc"][:, :, S_kv:] = SENTINEL
    x["vc"][:, :, S_kv:] = SENTINEL
    return x


CASES = [
    # B, H_q, H_kv, S_kv, S_q, cap
    (1, 8, 8, 8192, 1, 8256),      # the decode-append shape
    (4, 32, 8, 2000, 1, 2048),     # GQA group 4
    (2, 8, 2, 700, 3, 710),        # three new tokens per sequence
]


@pytest.mark.parametrize("B,H_q,H_kv,S_kv,S_q,cap", CASES)
def test_decode_step_matches_oracle_and_separate_calls(B, H_q, H_kv, S_kv, S_q, cap):
    x = _case(B * 1000 + S_kv, B, H_q, H_kv, S_kv, S_q, cap)
    d, D = x["d"], x["D"]
    kcb, vcb, smooth = dev(x["kcb"]), dev(x["vcb"]), dev(x["smooth"])
    kbuf, vbuf = dev(x["kc"]), dev(x["vc"])
    out = vq.decode_step(dev(x["q"]), dev(x["k_new"]), dev(x["v_new"]), kbuf, kcb, vbuf, vcb,
                         smooth, 1 / np.sqrt(D), s_kv=S_kv)
    # the separate calls on copies of the original cache
    kb2, vb2 = dev(x["kc"]), dev(x["vc"])
    vq.encode_keys_into(dev(x["k_new"]), kcb, d, smooth, kb2, S_kv - S_q)
    vq.encode_values_into(dev(x["v_new"]), vcb, d, vb2, S_kv - S_q)
    ref2 = vq.decode_attend(dev(x["q"]), kb2, kcb, vb2, vcb, smooth, 1 / np.sqrt(D), s_kv=S_kv)
    torch.cuda.synchronize()
    kb, vb = kbuf.cpu().numpy(), vbuf.cpu().numpy()
    assert np.array_equal(kb, kb2.cpu().numpy()) and np.array_equal(vb, vb2.cpu().numpy())
    # untouched rows
    assert np.array_equal(kb[:, :, :S_kv - S_q], x["kc"][:, :, :S_kv - S_q])
    assert np.array_equal(vb[:, :, :S_kv - S_q], x["vc"][:, :, :S_kv - S_q])
    assert np.all(kb[:, :, S_kv:] == SENTINEL) and np.all(vb[:, :, S_kv:] == SENTINEL)
    # the new rows: the oracle's codes except at near ties
    new = slice(S_kv - S_q, S_kv)
    rk = check_encode(x["k_new"], x["kcb"], d, x["smooth"], True, kb[:, :, new], None)
    rv = check_encode(x["v_new"], x["vcb"], d, None, False, vb[:, :, new], None)
    assert rk["mismatch"] == rk["near_tie"] and rv["mismatch"] == rv["near_tie"]
    got = out.float().cpu().numpy()
    ok, err, _ = parity.allclose_report(got, ref2.float().cpu().numpy())
    assert ok, f"step vs separate calls: max |err| {err}"
    # attention over the updated cache, the new rows encoded by the oracle
    ko = oracle.encode(x["k_new"], x["kcb"], smooth=x["smooth"])["codes"]
    vo = oracle.encode(x["v_new"], x["vcb"], rotate=False)["codes"]
    kc_ref = x["kc"][:, :, :S_kv].astype(np.int64)
    vc_ref = x["vc"][:, :, :S_kv].astype(np.int64)
    kc_ref[:, :, new] = ko
    vc_ref[:, :, new] = vo
    ref = oracle.attend(x["q"], kc_ref, x["kcb"], vc_ref, x["vcb"], x["smooth"], 1 / np.sqrt(D),
                        causal=True)
    if rk["mismatch"] == 0 and rv["mismatch"] == 0:
        ok, err, _ = parity.allclose_report(got, oracle.to_f16(ref).astype(np.float64))
        assert ok, f"step vs oracle: max |err| {err}"


@pytest.mark.parametrize("S_q,window", [(1, 500), (2, 1), (3, 130)])
def test_decode_step_with_a_sliding_window(S_q, window):
    """A sliding window (the new rows are always inside it; a window of 1
    leaves each query only its own row): the step against the separate calls
    and against the oracle over the updated cache."""
    B, H_q, H_kv, S_kv, cap = 2, 8, 2, 3000, 3010
    x = _case(S_q * 100 + window, B, H_q, H_kv, S_kv, S_q, cap)
    d, D = x["d"], x["D"]
    kcb, vcb, smooth = dev(x["kcb"]), dev(x["vcb"]), dev(x["smooth"])
    kbuf, vbuf = dev(x["kc"]), dev(x["vc"])
    out = vq.decode_step(dev(x["q"]), dev(x["k_new"]), dev(x["v_new"]), kbuf, kcb, vbuf, vcb,
                         smooth, 1 / np.sqrt(D), sliding_window=window, s_kv=S_kv)
    kb2, vb2 = dev(x["kc"]), dev(x["vc"])
    vq.encode_keys_into(dev(x["k_new"]), kcb, d, smooth, kb2, S_kv - S_q)
    vq.encode_values_into(dev(x["v_new"]), vcb, d, vb2, S_kv - S_q)
    ref2 = vq.decode_attend(dev(x["q"]), kb2, kcb, vb2, vcb, smooth, 1 / np.sqrt(D),
                            sliding_window=window, s_kv=S_kv)
    torch.cuda.synchronize()
    assert torch.equal(kbuf, kb2) and torch.equal(vbuf, vb2)
    got = out.float().cpu().numpy()
    ok, err, _ = parity.allclose_report(got, ref2.float().cpu().numpy())
    assert ok, f"step vs separate calls: max |err| {err}"
    kb, vb = kbuf.cpu().numpy(), vbuf.cpu().numpy()
    ref = oracle.attend(x["q"], kb[:, :, :S_kv].astype(np.int64), x["kcb"],
                        vb[:, :, :S_kv].astype(np.int64), x["vcb"], x["smooth"], 1 / np.sqrt(D),
                        causal=True, sliding_window=window)
    ok, err, _ = parity.allclose_report(got, oracle.to_f16(ref).astype(np.float64))
    assert ok, f"step vs oracle: max |err| {err}"


@pytest.mark.parametrize("smooth_mode", [0, 1])
def test_decode_step_smooth_layouts(smooth_mode):
    """No smooth, and one smooth vector [D] shared by the heads: the new
    keys' codes against the oracle's (near ties only), the caches against
    the separate calls, the output against the oracle."""
    B, H_q, H_kv, S_kv, S_q, cap = 1, 8, 4, 900, 1, 960
    x = _case(50 + smooth_mode, B, H_q, H_kv, S_kv, S_q, cap)
    d, D = x["d"], x["D"]
    sm = None if smooth_mode == 0 else x["smooth"][0].copy()
    kcb, vcb = dev(x["kcb"]), dev(x["vcb"])
    smd = None if sm is None else dev(sm)
    kbuf, vbuf = dev(x["kc"]), dev(x["vc"])
    out = vq.decode_step(dev(x["q"]), dev(x["k_new"]), dev(x["v_new"]), kbuf, kcb, vbuf, vcb,
                         smd, 1 / np.sqrt(D), s_kv=S_kv)
    kb2, vb2 = dev(x["kc"]), dev(x["vc"])
    vq.encode_keys_into(dev(x["k_new"]), kcb, d, smd, kb2, S_kv - S_q)
    vq.encode_values_into(dev(x["v_new"]), vcb, d, vb2, S_kv - S_q)
    torch.cuda.synchronize()
    assert torch.equal(kbuf, kb2) and torch.equal(vbuf, vb2)
    kb, vb = kbuf.cpu().numpy(), vbuf.cpu().numpy()
    new = slice(S_kv - S_q, S_kv)
    rk = check_encode(x["k_new"], x["kcb"], d, sm, True, kb[:, :, new], None)
    assert rk["mismatch"] == rk["near_tie"]
    ref = oracle.attend(x["q"], kb[:, :, :S_kv].astype(np.int64), x["kcb"],
                        vb[:, :, :S_kv].astype(np.int64), x["vcb"], sm, 1 / np.sqrt(D),
                        causal=True)
    ok, err, _ = parity.allclose_report(out.float().cpu().numpy(),
                                        oracle.to_f16(ref).astype(np.float64))
    assert ok, f"step vs oracle: max |err| {err}"


def test_decode_step_on_a_workspace_of_stale_bytes():
    """The single launch's new rows are announced through flags in the
    workspace; a workspace that holds arbitrary bytes (here random ones,
    as left by other calls) and a second step on the same workspace give
    the same result as the separate calls."""
    x = _case(31, 2, 8, 2, 1500, 1, 1600)
    d, D, S_kv = x["d"], x["D"], x["S_kv"]
    kcb, vcb, smooth = dev(x["kcb"]), dev(x["vcb"]), dev(x["smooth"])
    kbuf, vbuf = dev(x["kc"]), dev(x["vc"])
    q = dev(x["q"])
    out = torch.empty_like(q)
    args = vq.make_attend_args(q, kbuf, kcb, vbuf, vcb, smooth, 1 / np.sqrt(D), True, 0, out,
                               s_kv=S_kv)
    n = max(vq.attend_workspace_bytes(args), 16)
    ws = torch.from_numpy(np.random.default_rng(3).integers(0, 256, n, dtype=np.uint8)).to(DEV)
    kb2, vb2 = dev(x["kc"]), dev(x["vc"])
    for step in range(2):
        k_new = x["k_new"] if step == 0 else x["k_new"][..., ::-1].copy()
        v_new = x["v_new"] if step == 0 else x["v_new"][..., ::-1].copy()
        vq.decode_step(q, dev(k_new), dev(v_new), kbuf, kcb, vbuf, vcb, smooth, 1 / np.sqrt(D),
                       out=out, workspace=ws, s_kv=S_kv)
        vq.encode_keys_into(dev(k_new), kcb, d, smooth, kb2, S_kv - 1)
        vq.encode_values_into(dev(v_new), vcb, d, vb2, S_kv - 1)
        ref = vq.decode_attend(q, kb2, kcb, vb2, vcb, smooth, 1 / np.sqrt(D), s_kv=S_kv)
        torch.cuda.synchronize()
        assert torch.equal(kbuf, kb2) and torch.equal(vbuf, vb2), step
        ok, err, _ = parity.allclose_report(out.float().cpu().numpy(), ref.float().cpu().numpy())
        assert ok, f"step {step}: max |err| {err}"


def test_decode_step_other_shapes_run_as_separate_calls():
    """D = 64 has no single-launch path: the same result through the three
    calls on the stream."""
    x = _case(77, 1, 4, 2, 300, 1, 320, D=64)
    d, D = x["d"], x["D"]
    kcb, vcb, smooth = dev(x["kcb"]), dev(x["vcb"]), dev(x["smooth"])
    kbuf, vbuf = dev(x["kc"]), dev(x["vc"])
    out = vq.decode_step(dev(x["q"]), dev(x["k_new"]), dev(x["v_new"]), kbuf, kcb, vbuf, vcb,
                         smooth, 1 / np.sqrt(D), s_kv=300)
    torch.cuda.synchronize()
    kb = kbuf.cpu().numpy()
    rk = check_encode(x["k_new"], x["kcb"], d, x["smooth"], True, kb[:, :, 299:300], None)
    assert rk["mismatch"] == rk["near_tie"]
    kc_ref = kb[:, :, :300].astype(np.int64)
    vc_ref = vbuf.cpu().numpy()[:, :, :300].astype(np.int64)
    ref = oracle.attend(x["q"], kc_ref, x["kcb"], vc_ref, x["vcb"], x["smooth"], 1 / np.sqrt(D),
                        causal=True)
    ok, err, _ = parity.allclose_report(out.float().cpu().numpy(), oracle.to_f16(ref).astype(np.float64))
    assert ok, err


def test_decode_step_replays_as_a_graph():
    """The single launch captured into a CUDA graph: each replay with
    refreshed inputs equals the eager call bit for bit."""
    x = _case(5, 1, 8, 8, 512, 1, 576)
    D = x["D"]
    kcb, vcb, smooth = dev(x["kcb"]), dev(x["vcb"]), dev(x["smooth"])
    rng = np.random.default_rng(6)
    sets = [(rng.standard_normal((1, 8, 1, D)).astype(np.float16),
             rng.standard_normal((1, 8, 1, D)).astype(np.float16),
             rng.standard_normal((1, 8, 1, D)).astype(np.float16)) for _ in range(3)]
    kbuf, vbuf = dev(x["kc"]), dev(x["vc"])
    k_in, v_in, q_in = (dev(a) for a in sets[0])
    out = torch.empty_like(q_in)
    args = vq.make_attend_args(q_in, kbuf, kcb, vbuf, vcb, smooth, 1 / np.sqrt(D), True, 0, out,
                               s_kv=512)
    ws = torch.empty(max(vq.attend_workspace_bytes(args), 16), dtype=torch.uint8, device=DEV)

    def step(stream=None):
        vq.decode_step(q_in, k_in, v_in, kbuf, kcb, vbuf, vcb, smooth, 1 / np.sqrt(D), out=out,
                       workspace=ws, stream=stream, s_kv=512)

    eager = []
    for k, v, q in sets:
        k_in.copy_(dev(k)); v_in.copy_(dev(v)); q_in.copy_(dev(q))
        step()
        torch.cuda.synchronize()
        eager.append((out.clone(), kbuf.clone(), vbuf.clone()))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(stream=s)   # warm-up on the capture stream
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(stream=s)
    for (k, v, q), (o_ref, kb_ref, vb_ref) in zip(sets, eager):
        k_in.copy_(dev(k)); v_in.copy_(dev(v)); q_in.copy_(dev(q))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, o_ref)
        assert torch.equal(kbuf, kb_ref) and torch.equal(vbuf, vb_ref)
