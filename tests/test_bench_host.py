"""Host logic of bench.py that needs no GPU: the bit packing it applies to
drawn codes of packed-key workloads, and the algorithmic bytes it divides by.

Packed layout (page "veloxquant_mlx.cache.vecinfer_cache module", storage
of b-bit codes): code m of a token row occupies bits [m b, m b + b) of the
row's little-endian 32-bit words.  The check below builds each row bit by
bit in plain Python, independently of the vectorised packer.
"""
import numpy as np
import torch

import bench
from product_vq_compressed_gb300.workloads import WORKLOADS


def _row_bit_by_bit(codes, bits):
    words = (len(codes) * bits + 31) // 32
    out = [0] * words
    for m, c in enumerate(codes):
        for k in range(bits):
            if (int(c) >> k) & 1:
                pos = m * bits + k
                out[pos // 32] |= 1 << (pos % 32)
    return [w - (1 << 32) if w >= (1 << 31) else w for w in out]


def test_pack_rows_matches_bit_by_bit_packing():
    rng = np.random.default_rng(0)
    for n, N in [(16, 1024), (32, 1000), (5, 8), (7, 65536), (16, 2)]:
        bits = bench._bits(N)
        codes = rng.integers(0, N, size=(3, 2, n))
        codes[0, 0, :] = N - 1
        got = bench.pack_rows(torch.from_numpy(codes), bits, torch).numpy()
        assert got.dtype == np.int32
        for idx in np.ndindex(codes.shape[:-1]):
            assert got[idx].tolist() == _row_bit_by_bit(codes[idx], bits), (n, N, idx)


def test_unpack_rows_inverts_pack_rows():
    rng = np.random.default_rng(1)
    for n, N in [(16, 1024), (32, 1000), (7, 65536), (5, 3)]:
        bits = bench._bits(N)
        codes = rng.integers(0, N, size=(4, 3, n))
        rows = bench.pack_rows(torch.from_numpy(codes), bits, torch).numpy()
        assert np.array_equal(bench.unpack_rows(rows, n, bits), codes)


def test_bits_per_code():
    assert [bench._bits(n) for n in (2, 3, 4, 256, 257, 1000, 1024, 1025)] == \
        [1, 2, 2, 8, 9, 10, 10, 11]


def test_packed_decode_algorithmic_bytes():
    """20-byte packed key rows + 32-byte value rows per token-head, plus q and out."""
    s = WORKLOADS["gqa-decode-packed"]
    _, bound, byts, unit = bench.algorithmic("gqa-decode-packed", s)
    assert bound == "hbm" and unit == "GB/s"
    assert byts == s.B * s.H_kv * s.S_kv * (20 + 32) + 2 * s.B * s.H_q * s.S_q * s.D * 2


def test_prefill_flops_count_every_visible_key():
    """chunked-prefill: 4 D FLOPs (QK^T and PV, a multiply-add each) per query
    head, query row and visible key.  The visible keys of each row come
    from the mask's definition (causal: j <= q_abs; window W: j > q_abs - W;
    q_abs = S_kv - S_q + i), counted row by row."""
    s = WORKLOADS["chunked-prefill"]
    _, bound, flops, unit = bench.algorithmic("chunked-prefill", s)
    assert bound == "tensor" and unit == "TFLOP/s"
    q_abs = s.S_kv - s.S_q + np.arange(s.S_q)
    lo = np.maximum(0, q_abs - s.window + 1) if s.window else np.zeros_like(q_abs)
    hi = q_abs if s.causal else np.full_like(q_abs, s.S_kv - 1)
    visible = int(np.sum(hi - lo + 1))
    assert flops == 4 * s.D * s.H_q * s.B * visible


def test_decode_bytes_are_the_codes_read_once():
    """gqa-decode: one uint8 code per sub-vector of every cached key and
    value, per KV head, plus the fp16 queries read and outputs written;
    ragged caches count their own lengths."""
    s = WORKLOADS["gqa-decode"]
    _, bound, byts, _ = bench.algorithmic("gqa-decode", s)
    assert bound == "hbm"
    assert byts == s.B * s.H_kv * s.S_kv * (s.D // s.k_d + s.D // s.v_d) + \
        2 * s.B * s.H_q * s.S_q * s.D * 2
    r = WORKLOADS["gqa-decode-ragged"]
    lens = np.array([r.S_kv // 2, r.S_kv, 5] + [r.S_kv - 1] * (r.B - 3))
    _, _, rb, _ = bench.algorithmic("gqa-decode-ragged", r, lens)
    assert rb == r.H_kv * int(lens.sum()) * 64 + 2 * r.B * r.H_q * r.S_q * r.D * 2


def test_encode_flops_one_multiply_add_per_dimension_and_candidate():
    s = WORKLOADS["decode-1seq"]
    kernel, bound, flops, _ = bench.algorithmic("decode-1seq", s)
    assert kernel == "encode" and bound == "alu"
    n_sub = s.B * s.H_kv * s.S_kv * (s.D // s.k_d)
    assert flops == 2 * s.k_d * s.k_N * n_sub



def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the contract's keys, on the workload's own metric."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                        "decode-append", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300,
                       cwd=__import__("os").path.dirname(bench.__file__))
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    metric, unit = bench.METRICS["decode-append"][0], bench.METRICS["decode-append"][1]
    assert d["impl"] == "reference" and d["metric"] == metric and d["unit"] == unit
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 1, 0)
    assert d["vs_baseline"] is None and d["data"] == "synthetic" and d["dtype"] == "f64"
    assert d["config"]["workload"] == "decode-append"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
