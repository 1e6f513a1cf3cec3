"""GPU parity of the tensor-core prefill kernels against the float64 oracle.

Query blocks of 64 rows or more with D = 128, 4-dimensional sub-vectors and
uint8 codes take the tensor-core path: two query heads of a KV group per CTA,
and a single head in the last CTA of an odd group.  The cases span
several key tiles with ragged tails, windows and causal bounds that cut
tiles, the three smooth modes, and a cache whose scores grow along the keys
so that every row's reference maximum moves between and within key tiles
(the rescaling of P and of the running output).
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu_helpers import dev, oracle_attend_rows, run_attend
from oracle import parity
from product_vq_compressed_gb300 import binding as vq
from product_vq_compressed_gb300.workloads import make_inputs, small_spec

pytestmark = pytest.mark.gpu

CASES = [
    # B, H_q, H_kv, S_kv, S_q, causal, window, smooth_mode
    (1, 2, 1, 700, 200, True, 0, 2),       # group 2, ragged query block
    (2, 8, 2, 1000, 128, True, 300, 2),    # group 4, window cutting tiles
    (1, 8, 1, 517, 64, False, 0, 1),       # group 8, not causal
    (1, 4, 2, 128, 128, True, 0, 0),       # one key tile exactly
    (1, 2, 1, 4101, 96, True, 1000, 2),    # long cache, window
    (1, 4, 4, 333, 130, True, 0, 0),       # group 1: single-head CTAs
    (1, 6, 2, 450, 256, True, 129, 2),     # group 3: a pair and a single head
    (1, 4, 1, 2000, 384, True, 200, 2),    # three query tiles: the last CTA pair half empty
    (2, 4, 2, 1500, 640, False, 300, 2),   # five query tiles, window, not causal
]


@pytest.mark.parametrize("B,H_q,H_kv,S_kv,S_q,causal,window,smooth_mode", CASES)
def test_prefill_matches_oracle(B, H_q, H_kv, S_kv, S_q, causal, window, smooth_mode):
    spec = small_spec(S_kv * 3 + S_q + H_q, B=B, H_q=H_q, H_kv=H_kv, D=128, S_kv=S_kv,
                      S_q=S_q, causal=causal, window=window, smooth_mode=smooth_mode,
                      draw_keys=False, draw_values=False, draw_codes=True)
    inp = make_inputs(spec)
    out = run_attend("prefill", inp, spec, inp["k_codes"], inp["v_codes"])
    torch.cuda.synchronize()
    b, h, i = np.meshgrid(np.arange(B), np.arange(H_q), np.arange(S_q), indexing="ij")
    rows = np.stack([b.ravel(), h.ravel(), i.ravel()], axis=1)
    ref = oracle_attend_rows(inp, spec, rows, inp["k_codes"], inp["v_codes"])
    got = out.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    ok, err, excess = parity.allclose_report(got, ref)
    assert ok, f"max |err| {err}, worst excess {excess}"


@pytest.mark.parametrize("H_q,H_kv,causal", [(4, 2, True), (4, 2, False), (3, 1, True)])
def test_prefill_growing_scores_move_the_maximum(H_q, H_kv, causal):
    """q = 64 e_0 makes the rotated query constant over the dimensions, and
    key j's centroids (c / 64 in every dimension, exact in fp16, so that
    rounding only scales all scores alike) grow with j: the score rises by
    about 1.44 (base 2) per level and 12 every 32 keys, past the reference
    maximum's headroom of 8, so every row moves its maximum in every chunk
    of the scores it sees."""
    D, N, S_kv, S_q = 128, 256, 1000, 192
    rng = np.random.default_rng(77 + H_q)
    level = np.minimum(np.arange(S_kv) * N // S_kv, N - 1)
    kcb = np.repeat((np.arange(N) / 64.0)[:, None], 4, axis=1).astype(np.float32)
    vcb = rng.standard_normal((N, 4)).astype(np.float32)
    kc = np.broadcast_to(level[None, None, :, None], (1, H_kv, S_kv, D // 4)).astype(np.uint8)
    vc = rng.integers(0, N, (1, H_kv, S_kv, D // 4)).astype(np.uint8)
    q = np.zeros((1, H_q, S_q, D), np.float16)
    q[..., 0] = 64.0
    scale = 1.0 / np.sqrt(D)
    out = vq.prefill_attend(dev(q), dev(kc), dev(kcb), dev(vc), dev(vcb), None, scale,
                            causal=causal, sliding_window=0)
    torch.cuda.synchronize()
    ref = oracle.attend(q, kc, kcb, vc, vcb, None, scale, causal, 0)
    ok, err, _ = parity.allclose_report(out.cpu().numpy().astype(np.float64),
                                        oracle.to_f16(ref).astype(np.float64))
    assert ok, f"max |err| {err}"


@pytest.mark.parametrize("H_q,H_kv", [(4, 2), (3, 3)])
def test_prefill_empty_cache_batch_is_zero(H_q, H_kv):
    """A batch holding no keys (kv_lens 0): its CTAs have no key tile and
    write exact zeros; the other batch is the oracle's attention over its
    own length (even and odd group sizes)."""
    D, N, S_kv, S_q = 128, 256, 400, 130
    spec = small_spec(31 + H_q, B=2, H_q=H_q, H_kv=H_kv, D=D, S_kv=S_kv, S_q=S_q,
                      causal=True, draw_keys=False, draw_values=False, draw_codes=True)
    inp = make_inputs(spec)
    lens = torch.tensor([0, 333], dtype=torch.int32, device="cuda:0")
    out = vq.prefill_attend(dev(inp["q"]), dev(inp["k_codes"]), dev(inp["k_codebook"]),
                            dev(inp["v_codes"]), dev(inp["v_codebook"]), dev(inp["smooth"]),
                            spec.sm_scale, causal=True, kv_lens=lens)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(got[0] == 0.0)
    ref = oracle.attend(inp["q"][1:], inp["k_codes"][1:, :, :333], inp["k_codebook"],
                        inp["v_codes"][1:, :, :333], inp["v_codebook"], inp["smooth"],
                        spec.sm_scale, True, 0)
    ok, err, _ = parity.allclose_report(got[1:], oracle.to_f16(ref).astype(np.float64))
    assert ok, f"max |err| {err}"
