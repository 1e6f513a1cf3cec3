"""vq_decode_attend_noalloc: decode attention without a caller workspace.

Some callers cannot allocate device memory at all -- a plug-in living inside
a host application that owns every byte of GPU memory, a runtime whose
memory plan is fixed before the model runs, or a latency-critical decode
loop that must never call cudaMalloc because it can synchronise the device.
For them the library offers a variant of vq_decode_attend that keeps its
split-KV partial results in a fixed scratch array built into the library.

These tests call that entry point through the C ABI and compare it with the
regular entry point (given a workspace) on the same inputs, within the
tolerance of the other attention tests, |a - b| <= 2e-3 + 1e-2 |b|, for two
calls in a row (the array keeps the previous call's contents, which must not
matter), and with the float64 oracle on sampled rows.  One case is too large
for the array with the regular split and runs with fewer, longer key splits.
The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from _gpu_helpers import oracle_attend_rows_parallel
from oracle import parity
from product_vq_compressed_gb300 import binding as vq
from product_vq_compressed_gb300.workloads import WORKLOADS, make_inputs, small_spec

pytestmark = pytest.mark.gpu


def _to_dev(inp):
    return {k: torch.from_numpy(np.ascontiguousarray(v)).cuda()
            for k, v in inp.items() if isinstance(v, np.ndarray)}


def _noalloc_call(d, spec, out):
    """vq_decode_attend_noalloc through the C ABI; no workspace passed."""
    a = vq.make_attend_args(d["q"], d["k_codes"], d["k_codebook"], d["v_codes"],
                            d["v_codebook"], d.get("smooth"), spec.sm_scale,
                            spec.causal, spec.window, out, workspace=None)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return vq.lib().vq_decode_attend_noalloc(ctypes.byref(a), stream)


def _within(a, b):
    a, b = a.double(), b.double()
    return bool(((a - b).abs() <= 2e-3 + 1e-2 * b.abs()).all())


def _uncapped_workspace_bytes(d, spec):
    a = vq.make_attend_args(d["q"], d["k_codes"], d["k_codebook"], d["v_codes"],
                            d["v_codebook"], d.get("smooth"), spec.sm_scale,
                            spec.causal, spec.window, d["q"], workspace=None)
    return vq.attend_workspace_bytes(a)


NOALLOC_SCRATCH_BYTES = 32 << 20   # VQ_NOALLOC_SCRATCH_BYTES in include/vqkv.h


@pytest.mark.parametrize("spec,capped", [
    (small_spec(501, B=4, H_q=32, H_kv=8, D=128, S_kv=4096, draw_keys=False,
                draw_values=False, draw_codes=True), False),
    (small_spec(502, B=2, H_q=4, H_kv=2, D=64, S_kv=700, S_q=3, window=100,
                draw_keys=False, draw_values=False, draw_codes=True), False),
    (WORKLOADS["gqa-decode"], False),
    # about 38 MiB of partial results with the regular split: the array
    # takes it only with half the warps (longer shares, more slots per warp)
    (small_spec(504, B=768, H_q=8, H_kv=8, D=128, S_kv=1024, draw_keys=False,
                draw_values=False, draw_codes=True), True),
], ids=["gqa-4096", "windowed-sq3", "gqa-decode-full", "capped-split"])
def test_noalloc_matches_regular_entry_point_twice(spec, capped):
    inp = make_inputs(spec)
    d = _to_dev(inp)
    assert (_uncapped_workspace_bytes(d, spec) > NOALLOC_SCRATCH_BYTES) == capped
    rng = np.random.default_rng(11)
    for call in range(2):
        if call == 1:  # new queries: stale scratch from call 0 must not leak
            d["q"] = torch.randn_like(d["q"].float()).half()
            inp["q"] = d["q"].cpu().numpy()
        ref = vq.decode_attend(d["q"], d["k_codes"], d["k_codebook"], d["v_codes"],
                               d["v_codebook"], d.get("smooth"), spec.sm_scale,
                               spec.causal, spec.window)
        out = torch.full_like(d["q"], float("nan"))
        st = _noalloc_call(d, spec, out)
        torch.cuda.synchronize()
        assert st == vq.VQ_OK, vq.lib().vq_status_str(st)
        assert _within(out, ref), float((out.double() - ref.double()).abs().max())
        # and the float64 oracle on rows of two (batch, kv head) pairs
        rows = []
        for bg in rng.choice(spec.B * spec.H_kv, size=2, replace=False):
            b, g = divmod(int(bg), spec.H_kv)
            rows += [(b, g * spec.G + h, i) for h in range(spec.G) for i in range(spec.S_q)]
        rows = np.array(rows)
        oref = oracle_attend_rows_parallel(inp, spec, rows, inp["k_codes"], inp["v_codes"])
        got = out.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
        ok, err, _ = parity.allclose_report(got, oref)
        assert ok, f"oracle max |err| {err}"


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Partial results that do not fit the built-in array even with one key
    split are refused with VQ_ERR_WORKSPACE before anything is launched."""
    spec = small_spec(503, B=1024, H_q=8, H_kv=8, D=128, S_kv=16,
                      draw_keys=False, draw_values=False, draw_codes=True)
    d = _to_dev(make_inputs(spec))
    out = torch.zeros_like(d["q"])
    st = _noalloc_call(d, spec, out)
    torch.cuda.synchronize()
    assert st == vq.VQ_ERR_WORKSPACE
    assert bool((out == 0).all())
