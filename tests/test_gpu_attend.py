"""GPU parity of attention over the coded cache against the float64 oracle.

Both sides get the same codes (drawn uniformly, or encoded by the oracle),
so the comparison isolates the attention kernel.  Outputs are fp16 and held
to |err| <= 2e-3 + 1e-2 |ref|.  Small cases span several 16-key tiles, key
splits and column blocks, with ragged tails; full-size workloads are checked
on sampled rows and on whole query tiles / whole GQA groups in the launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

from _gpu_helpers import DEV, dev, oracle_attend_rows, oracle_attend_rows_parallel, run_attend
import oracle
from oracle import parity
from product_vq_compressed_gb300 import binding as vq
from product_vq_compressed_gb300.workloads import WORKLOADS, make_inputs, small_spec

pytestmark = pytest.mark.gpu


def _all_rows(spec):
    b, h, i = np.meshgrid(np.arange(spec.B), np.arange(spec.H_q),
                          np.arange(spec.S_q), indexing="ij")
    return np.stack([b.ravel(), h.ravel(), i.ravel()], axis=1)


def _check(spec, inp, out, rows=None):
    rows = _all_rows(spec) if rows is None else np.asarray(rows)
    ref = oracle_attend_rows(inp, spec, rows, inp["k_codes"], inp["v_codes"])
    got = out.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    ok, err, excess = parity.allclose_report(got, ref)
    assert ok, f"max |err| {err}, worst excess {excess}"
    return err


SMALL = [
    # D, dk, dv, Nk, Nv, B, H_q, H_kv, S_kv, S_q, causal, window
    (128, 4, 4, 256, 256, 1, 8, 8, 777, 1, True, 0),
    (128, 4, 4, 256, 256, 2, 32, 8, 1000, 1, True, 0),      # GQA 4
    (64, 4, 4, 256, 256, 1, 2, 2, 256, 1, True, 0),         # tiny-like
    (128, 8, 4, 1024, 256, 1, 8, 1, 530, 3, True, 0),       # GQA 8, S_q 3
    (32, 2, 2, 16, 16, 2, 4, 4, 333, 5, True, 7),
    (256, 8, 8, 64, 128, 1, 4, 2, 129, 2, False, 0),
    (128, 4, 8, 256, 512, 1, 6, 3, 200, 4, False, 9),
    (64, 2, 4, 128, 256, 1, 3, 1, 64, 64, True, 0),         # square causal
    (128, 4, 4, 256, 256, 1, 4, 1, 300, 130, True, 100),    # many columns
    (128, 4, 4, 256, 256, 1, 2, 2, 1, 1, True, 0),          # single key
    (128, 4, 2, 256, 64, 1, 2, 1, 50, 10, True, 1),         # window 1
    (128, 4, 4, 256, 256, 1, 2, 2, 90, 7, True, 1000),      # window > S_kv
]


@pytest.mark.parametrize("D,dk,dv,Nk,Nv,B,H_q,H_kv,S_kv,S_q,causal,W", SMALL)
@pytest.mark.parametrize("entry", ["decode", "prefill"])
def test_attend_small(D, dk, dv, Nk, Nv, B, H_q, H_kv, S_kv, S_q, causal, W, entry):
    spec = small_spec(D + S_kv + S_q, B=B, H_q=H_q, H_kv=H_kv, D=D, S_kv=S_kv,
                      S_q=S_q, k_N=Nk, k_d=dk, v_N=Nv, v_d=dv, causal=causal,
                      window=W, draw_keys=False, draw_values=False,
                      draw_codes=True)
    inp = make_inputs(spec)
    out = run_attend(entry, inp, spec, inp["k_codes"], inp["v_codes"])
    torch.cuda.synchronize()
    _check(spec, inp, out)


def test_attend_max_codes_and_smooth_modes():
    """Codes at N-1 and every smooth layout."""
    for mode in (0, 1, 2):
        spec = small_spec(40 + mode, H_q=4, H_kv=2, D=128, S_kv=120, S_q=2,
                          smooth_mode=mode, draw_keys=False, draw_values=False,
                          draw_codes=True)
        inp = make_inputs(spec)
        inp["k_codes"][..., ::3] = spec.k_N - 1
        inp["v_codes"][..., ::5] = spec.v_N - 1
        out = run_attend("decode", inp, spec, inp["k_codes"], inp["v_codes"])
        torch.cuda.synchronize()
        _check(spec, inp, out)


def test_attend_over_oracle_encoded_cache():
    """Encode with the oracle, attend on the GPU: the end-to-end meaning of
    q . K_hat^T through the dual transform."""
    spec = WORKLOADS["tiny"]
    inp = make_inputs(spec)
    ko = oracle.encode(inp["keys"], inp["k_codebook"], smooth=inp["smooth"])
    vo = oracle.encode(inp["values"], inp["v_codebook"], rotate=False)
    inp["k_codes"] = ko["codes"].astype(np.uint8)
    inp["v_codes"] = vo["codes"].astype(np.uint8)
    out = run_attend("decode", inp, spec, inp["k_codes"], inp["v_codes"])
    torch.cuda.synchronize()
    _check(spec, inp, out)


def test_one_centroid_gives_mean_of_values_full_size():
    """Property at full batched-decode size: a one-entry key codebook makes
    every score equal, so each output is the mean of the visible V_hat rows."""
    spec = WORKLOADS["gqa-decode"]
    inp = make_inputs(spec)
    kcb = inp["k_codebook"][:1].copy()
    kc = np.zeros_like(inp["k_codes"])
    out = vq.decode_attend(dev(inp["q"]), dev(kc), dev(kcb), dev(inp["v_codes"]),
                           dev(inp["v_codebook"]), dev(inp["smooth"]),
                           spec.sm_scale, causal=True)
    vhat = vq.dequant(dev(inp["v_codes"]), dev(inp["v_codebook"]), out_f32=True)
    mean = vhat.double().mean(dim=2)                       # [B, H_kv, D]
    ref = mean.repeat_interleave(spec.G, dim=1)[:, :, None, :]
    torch.cuda.synchronize()
    err = (out.double() - ref).abs()
    assert bool((err <= 2e-3 + 1e-2 * ref.abs()).all()), float(err.max())


@pytest.mark.parametrize("name,entry,n_bg,rows_per",
                         [("decode-1seq", "decode", 8, 1),
                          ("gqa-decode", "decode", 3, 4),
                          ("chunked-prefill", "prefill", 2, 6),
                          ("chunked-prefill", "decode", 1, 4)])
def test_attend_full_size_sampled(name, entry, n_bg, rows_per):
    spec = WORKLOADS[name]
    inp = make_inputs(spec)
    if name == "decode-1seq":
        ko = oracle.encode(inp["keys"], inp["k_codebook"], smooth=inp["smooth"])
        vo = oracle.encode(inp["values"], inp["v_codebook"], rotate=False)
        inp["k_codes"] = ko["codes"].astype(np.uint8)
        inp["v_codes"] = vo["codes"].astype(np.uint8)
    out = run_attend(entry, inp, spec, inp["k_codes"], inp["v_codes"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    rows = []
    bgs = rng.choice(spec.B * spec.H_kv, size=min(n_bg, spec.B * spec.H_kv),
                     replace=False)
    for bg in bgs:
        b, g = divmod(int(bg), spec.H_kv)
        for _ in range(rows_per):
            h = g * spec.G + int(rng.integers(0, spec.G))
            i = int(rng.integers(0, spec.S_q))
            rows.append((b, h, i))
    rows.append((0, 0, spec.S_q - 1))
    err = _check(spec, inp, out, rows)
    print(name, entry, "rows", len(rows), "max |err|", err)


def test_chunked_prefill_full_size_whole_tiles():
    """Chunked prefill at full size through the tensor-core kernel (the
    launch the benchmark times): every row of whole 128-row query tiles for
    both heads of a CTA's head pair -- the first tile, the second, the last,
    and a middle tile of the last KV group.  The sliding window's lower bound
    cuts the first key tile of every query tile."""
    spec = WORKLOADS["chunked-prefill"]
    inp = make_inputs(spec)
    out = run_attend("prefill", inp, spec, inp["k_codes"], inp["v_codes"])
    torch.cuda.synchronize()
    last = spec.S_q // 128 - 1
    plan = [(0, (0, 1)), (1, (0, 1)), (last, (2, 3)), (7, (spec.H_q - 2, spec.H_q - 1))]
    rows = np.array([(0, h, i) for t, hs in plan for h in hs
                     for i in range(128 * t, 128 * t + 128)])
    ref = oracle_attend_rows_parallel(inp, spec, rows, inp["k_codes"], inp["v_codes"])
    got = out.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    ok, err, excess = parity.allclose_report(got, ref)
    assert ok, f"max |err| {err}, worst excess {excess}"


@pytest.mark.parametrize("name", ["gqa-decode", "gqa-decode-ragged"])
def test_gqa_decode_full_size_whole_batches(name):
    """Batched GQA decode at full size: all 32 query heads (every KV head's
    group) of the first and the last batch."""
    spec = WORKLOADS[name]
    inp = make_inputs(spec)
    kv_lens = inp.get("kv_lens")
    out = vq.decode_attend(dev(inp["q"]), dev(inp["k_codes"]), dev(inp["k_codebook"]),
                           dev(inp["v_codes"]), dev(inp["v_codebook"]), dev(inp["smooth"]),
                           spec.sm_scale, causal=spec.causal, sliding_window=spec.window,
                           kv_lens=dev(kv_lens))
    torch.cuda.synchronize()
    rows = np.array([(b, h, 0) for b in (0, spec.B - 1) for h in range(spec.H_q)])
    ref = oracle_attend_rows_parallel(inp, spec, rows, inp["k_codes"], inp["v_codes"])
    got = out.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    ok, err, excess = parity.allclose_report(got, ref)
    assert ok, f"max |err| {err}, worst excess {excess}"


def test_workspace_too_small_is_rejected():
    spec = small_spec(77, H_q=2, H_kv=2, D=128, S_kv=100, draw_keys=False,
                      draw_values=False, draw_codes=True)
    inp = make_inputs(spec)
    q = dev(inp["q"])
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(vq.VQError) as e:
        vq.decode_attend(q, dev(inp["k_codes"]), dev(inp["k_codebook"]),
                         dev(inp["v_codes"]), dev(inp["v_codebook"]),
                         dev(inp["smooth"]), workspace=ws)
    assert e.value.status == vq.VQ_ERR_WORKSPACE
