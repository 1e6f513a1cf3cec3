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
matter).  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("spec", [
    small_spec(501, B=4, H_q=32, H_kv=8, D=128, S_kv=4096, draw_keys=False,
               draw_values=False, draw_codes=True),
    small_spec(502, B=2, H_q=4, H_kv=2, D=64, S_kv=700, S_q=3, window=100,
               draw_keys=False, draw_values=False, draw_codes=True),
    WORKLOADS["gqa-decode"],
], ids=["gqa-4096", "windowed-sq3", "gqa-decode-full"])
def test_noalloc_matches_regular_entry_point_twice(spec):
    inp = make_inputs(spec)
    d = _to_dev(inp)
    for call in range(2):
        if call == 1:  # new queries: stale scratch from call 0 must not leak
            d["q"] = torch.randn_like(d["q"].float()).half()
        ref = vq.decode_attend(d["q"], d["k_codes"], d["k_codebook"], d["v_codes"],
                               d["v_codebook"], d.get("smooth"), spec.sm_scale,
                               spec.causal, spec.window)
        out = torch.full_like(d["q"], float("nan"))
        st = _noalloc_call(d, spec, out)
        torch.cuda.synchronize()
        assert st == vq.VQ_OK, vq.lib().vq_status_str(st)
        assert _within(out, ref), float((out.double() - ref.double()).abs().max())


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
