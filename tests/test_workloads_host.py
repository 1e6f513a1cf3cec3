"""The seeded synthetic inputs: the named workloads' sizes, and the recipe
(deterministic per seed, outlier channels, per-batch lengths, code ranges)
on small specs of the same fields.  No GPU."""
import dataclasses

import numpy as np
import pytest

from product_vq_compressed_gb300.workloads import WORKLOADS, make_inputs, small_spec

SIZES = {
    # name: (B, H_q, H_kv, D, S_kv, S_q, k_N, k_d, v_N, v_d, window)
    "tiny": (1, 2, 2, 64, 256, 1, 256, 4, 256, 4, 0),
    "decode-1seq": (1, 8, 8, 128, 8192, 1, 256, 4, 256, 4, 0),
    "bulk-encode": (4, 32, 32, 128, 8192, 1, 1024, 8, 256, 4, 0),
    "bulk-encode-packed": (4, 32, 32, 128, 8192, 1, 1024, 8, 256, 4, 0),
    "gqa-decode": (32, 32, 8, 128, 32768, 1, 256, 4, 256, 4, 0),
    "gqa-decode-ragged": (32, 32, 8, 128, 32768, 1, 256, 4, 256, 4, 0),
    "gqa-decode-packed": (32, 32, 8, 128, 32768, 1, 1024, 8, 256, 4, 0),
    "chunked-prefill": (1, 32, 8, 128, 18432, 2048, 256, 4, 256, 4, 4096),
    "decode-append": (1, 8, 8, 128, 8192, 1, 256, 4, 256, 4, 0),
}


@pytest.mark.parametrize("name", sorted(SIZES))
def test_named_workload_sizes(name):
    s = WORKLOADS[name]
    got = (s.B, s.H_q, s.H_kv, s.D, s.S_kv, s.S_q, s.k_N, s.k_d, s.v_N, s.v_d, s.window)
    assert got == SIZES[name]
    assert s.H_q % s.H_kv == 0 and s.D % s.k_d == 0 and s.D % s.v_d == 0


def test_packed_and_append_fields():
    assert WORKLOADS["bulk-encode-packed"].packed_keys
    assert WORKLOADS["gqa-decode-packed"].packed_keys and WORKLOADS["gqa-decode-packed"].draw_codes
    assert WORKLOADS["gqa-decode-ragged"].ragged
    a = WORKLOADS["decode-append"]
    assert a.S_enc == 1 and a.capacity == a.S_kv + 64


def test_inputs_are_deterministic_per_seed():
    s = small_spec(5, B=2, H_q=4, H_kv=2, D=64, S_kv=40, S_q=3, draw_codes=True,
                   outlier_frac=0.05, outlier_scale=6.0, ragged=True)
    a, b = make_inputs(s), make_inputs(s)
    for k, v in a.items():
        if isinstance(v, np.ndarray):
            assert np.array_equal(v, b[k]), k
    c = make_inputs(dataclasses.replace(s, seed=6))
    assert not np.array_equal(a["q"], c["q"])


def test_outlier_channels_are_scaled():
    """outlier_frac of the channels (rounded) are drawn with outlier_scale
    times the standard deviation of the others, in keys and in values."""
    s = small_spec(9, B=2, H_q=2, H_kv=2, D=128, S_kv=2048, outlier_frac=0.02,
                   outlier_scale=10.0)
    inp = make_inputs(s)
    for name, ch_key in (("keys", "key_outlier_channels"), ("values", "value_outlier_channels")):
        ch = inp[ch_key]
        assert len(ch) == round(0.02 * 128) and len(set(ch)) == len(ch)
        x = inp[name].astype(np.float64)
        std = x.reshape(-1, 128).std(axis=0)
        others = np.setdiff1d(np.arange(128), ch)
        ratio = std[ch].mean() / std[others].mean()
        assert 9.0 < ratio < 11.0, (name, ratio)


def test_ragged_lengths_and_code_ranges():
    s = small_spec(3, B=64, H_q=4, H_kv=2, D=64, S_kv=100, k_N=1000, k_d=8, v_N=200, v_d=4,
                   draw_keys=False, draw_values=False, draw_codes=True, ragged=True)
    inp = make_inputs(s)
    lens = inp["kv_lens"]
    assert lens.dtype == np.int32 and lens.shape == (64,)
    assert lens.min() >= 50 and lens.max() <= 100
    kc, vc = inp["k_codes"], inp["v_codes"]
    assert kc.dtype == np.uint16 and vc.dtype == np.uint8
    assert kc.shape == (64, 2, 100, 8) and vc.shape == (64, 2, 100, 16)
    assert kc.max() < 1000 and vc.max() < 200
    assert inp["k_codebook"].shape == (1000, 8) and inp["v_codebook"].shape == (200, 4)


@pytest.mark.parametrize("mode,shape", [(0, None), (1, (64,)), (2, (2, 64))])
def test_smooth_layouts(mode, shape):
    s = small_spec(4, H_q=2, H_kv=2, D=64, S_kv=8, smooth_mode=mode)
    sm = make_inputs(s)["smooth"]
    if shape is None:
        assert sm is None
    else:
        assert sm.shape == shape and sm.min() >= 0.5 and sm.max() <= 2.0
