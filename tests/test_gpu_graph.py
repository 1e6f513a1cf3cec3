"""A single-token decode step with cache append (vq_encode_keys_into,
vq_encode_values_into, vq_decode_attend) captured once into a CUDA graph
and replayed: every replay must reproduce the eager calls bit for bit, with
the step's inputs refreshed in place between replays.  The attention kernels
are programmatic dependents of the encodes; the capture keeps those edges.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu_helpers import DEV, dev
from oracle import parity
from product_vq_compressed_gb300 import binding as vq

pytestmark = pytest.mark.gpu


def _inputs(seed, H=4, D=128, d=4, N=256, S_kv=300, cap=320):
    rng = np.random.default_rng(seed)
    return dict(
        smooth=rng.uniform(0.5, 2.0, (H, D)).astype(np.float32),
        kcb=rng.standard_normal((N, d)).astype(np.float32),
        vcb=rng.standard_normal((N, d)).astype(np.float32),
        kc=rng.integers(0, N, (1, H, cap, D // d)).astype(np.uint8),
        vc=rng.integers(0, N, (1, H, cap, D // d)).astype(np.uint8),
        new=[(rng.standard_normal((1, H, 1, D)).astype(np.float16),
              rng.standard_normal((1, H, 1, D)).astype(np.float16),
              rng.standard_normal((1, H, 1, D)).astype(np.float16)) for _ in range(3)],
        S_kv=S_kv, d=d)


def test_decode_append_step_replays_as_a_graph():
    x = _inputs(41)
    S_kv, d = x["S_kv"], x["d"]
    kcb, vcb, smooth = dev(x["kcb"]), dev(x["vcb"]), dev(x["smooth"])
    kbuf, vbuf = dev(x["kc"]), dev(x["vc"])
    k_in, v_in, q_in = (dev(a) for a in x["new"][0])
    out = torch.empty_like(q_in)
    args = vq.make_attend_args(q_in, kbuf, kcb, vbuf, vcb, smooth, 1 / np.sqrt(128),
                               True, 0, out, s_kv=S_kv)
    ws = torch.empty(max(vq.attend_workspace_bytes(args), 16), dtype=torch.uint8, device=DEV)

    def step(stream=None):
        vq.encode_keys_into(k_in, kcb, d, smooth, kbuf, S_kv - 1, stream=stream)
        vq.encode_values_into(v_in, vcb, d, vbuf, S_kv - 1, stream=stream)
        vq.decode_attend(q_in, kbuf, kcb, vbuf, vcb, smooth, 1 / np.sqrt(128), out=out,
                         workspace=ws, stream=stream, s_kv=S_kv)

    # eager reference for every input set
    eager = []
    for k, v, q in x["new"]:
        k_in.copy_(dev(k)); v_in.copy_(dev(v)); q_in.copy_(dev(q))
        step()
        torch.cuda.synchronize()
        eager.append((out.clone(), kbuf.clone(), vbuf.clone()))

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(stream=s)                       # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(stream=s)
    for idx, (k, v, q) in enumerate(x["new"]):
        k_in.copy_(dev(k)); v_in.copy_(dev(v)); q_in.copy_(dev(q))
        g.replay()
        torch.cuda.synchronize()
        o_ref, kb_ref, vb_ref = eager[idx]
        assert torch.equal(out.view(torch.int16), o_ref.view(torch.int16)), idx
        assert torch.equal(kbuf, kb_ref) and torch.equal(vbuf, vb_ref), idx

    # and the replayed step is the oracle's attention over the appended cache,
    # the appended row encoded by the oracle (the GPU's codes for it must be
    # the oracle's up to the accepted near ties)
    k, v, q = x["new"][-1]
    H, D = k.shape[1], k.shape[3]
    ok_k = oracle.encode(k.reshape(H, D), x["kcb"], heads=np.arange(H), smooth=x["smooth"])
    ok_v = oracle.encode(v.reshape(H, D), x["vcb"], rotate=False)
    kc = x["kc"][:, :, :S_kv].copy()
    vc = x["vc"][:, :, :S_kv].copy()
    kc[0, :, S_kv - 1] = ok_k["codes"]
    vc[0, :, S_kv - 1] = ok_v["codes"]
    gpu_k = kbuf.cpu().numpy()[0, :, S_kv - 1].astype(np.int64)
    gpu_v = vbuf.cpu().numpy()[0, :, S_kv - 1].astype(np.int64)
    if not (np.array_equal(gpu_k, ok_k["codes"]) and np.array_equal(gpu_v, ok_v["codes"])):
        pytest.skip("appended token at a near tie: codes differ within the accepted bound")
    ref = oracle.attend(q, kc, x["kcb"], vc, x["vcb"], x["smooth"], 1 / np.sqrt(128), True, 0)
    ok, err, _ = parity.allclose_report(out.cpu().numpy().astype(np.float64),
                                        oracle.to_f16(ref).astype(np.float64))
    assert ok, f"max |err| {err}"
