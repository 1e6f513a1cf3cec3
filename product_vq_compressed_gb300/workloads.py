"""Seeded synthetic inputs shaped like the documented workloads.

This module only draws random numbers (numpy ``default_rng``, PCG64); it holds
none of the method's arithmetic, so the oracle tests and the CUDA path can
both take their inputs from it.

Named workloads (sizes from the documented configurations):

==================  =========================================================
``tiny``            B=1, H_q=H_kv=2, D=64, S_kv=256, S_q=1; key channels
                    {3,17,40,61} scaled x8; 256x4 codebooks; scale 1/8; seed 0
``decode-1seq``     B=1, H_q=H_kv=8, D=128, S_kv=8192, S_q=1; 256x4 codebooks;
                    8192 new keys to encode, values pre-encoded; seed 1
``bulk-encode``     keys and values [4,32,8192,128], 3 of 128 channels x10
                    (drawn separately for keys and values); key codebook
                    1024x8 (uint16 codes), value codebook 256x4; seed 2
``gqa-decode``      B=32, H_q=32, H_kv=8, D=128, S_kv=32768, S_q=1; uniform
                    uint8 codes; 256x4 codebooks; seed 3
``chunked-prefill`` B=1, H_q=32, H_kv=8, D=128, S_q=2048 queries after 16384
                    cached tokens (cache holds 18432 coded tokens), sliding
                    window 4096, causal; uniform uint8 codes; seed 4
``decode-append``   one decode step of B=1, H_q=H_kv=8, D=128: the new token's
                    key and value are encoded into row 8191 of a cache of
                    capacity 8256 rows, then one query per head attends over
                    the 8192 cached tokens; uniform uint8 codes for the
                    cache; seed 5
``gqa-decode-ragged`` gqa-decode with per-sequence cache lengths drawn
                    uniformly in [S_kv / 2, S_kv]; seed 6
``bulk-encode-packed`` bulk-encode with the key codes stored as 10-bit packed
                    rows (20 bytes per token-head); the same inputs (seed 2)
``gqa-decode-packed`` gqa-decode over a cache of 10-bit packed key codes
                    (1024x8 key codebook, 20 bytes per token-head) and uint8
                    value codes (256x4, 32 bytes); uniform codes; seed 7
==================  =========================================================

Draw order (only what a workload uses): keys, values, outlier channels,
smooth, key codebook, value codebook, q, key codes, value codes, per-batch
cache lengths.
Values: fp16 from N(0,1) (drawn in float32, cast to fp16 after any outlier
scaling); smooth: float32 uniform[0.5, 2] per (KV head, channel); codebooks:
float32 N(0,1); codes: uniform integers in [0, N).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np


@dataclasses.dataclass
class Spec:
    """Shape and distribution of one synthetic workload."""

    name: str
    B: int
    H_q: int
    H_kv: int
    D: int
    S_kv: int                     # keys in the cache attended over
    S_q: int = 1
    k_N: int = 256                # key codebook size
    k_d: int = 4                  # key sub-vector size
    v_N: int = 256
    v_d: int = 4
    scale: Optional[float] = None  # default 1/sqrt(D)
    causal: bool = True
    window: int = 0
    seed: int = 0
    smooth_mode: int = 2          # 0 none, 1 [D], 2 [H_kv, D]
    # which tensors the workload draws
    draw_keys: bool = True
    draw_values: bool = True
    draw_codes: bool = False      # uniform random K/V codes instead of keys
    S_enc: Optional[int] = None   # keys/values per (b, head) to encode
    key_outliers: Sequence[int] = ()   # fixed outlier channels (keys)
    outlier_scale: float = 1.0
    outlier_frac: float = 0.0     # fraction of channels drawn as outliers
    capacity: Optional[int] = None  # rows per (b, kv head) of the code buffers
    packed_keys: bool = False     # key codes stored as bit-packed rows
    ragged: bool = False          # per-batch cache lengths in [S_kv / 2, S_kv]

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def sm_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    @property
    def n_k(self) -> int:
        return self.D // self.k_d

    @property
    def n_v(self) -> int:
        return self.D // self.v_d

    @property
    def k_code_dtype(self):
        return np.uint8 if self.k_N <= 256 else np.uint16

    @property
    def v_code_dtype(self):
        return np.uint8 if self.v_N <= 256 else np.uint16

    @property
    def enc_len(self) -> int:
        return self.S_kv if self.S_enc is None else self.S_enc


WORKLOADS = {
    "tiny": Spec("tiny", B=1, H_q=2, H_kv=2, D=64, S_kv=256, scale=1.0 / 8,
                 seed=0, key_outliers=(3, 17, 40, 61), outlier_scale=8.0),
    "decode-1seq": Spec("decode-1seq", B=1, H_q=8, H_kv=8, D=128, S_kv=8192,
                        seed=1),
    "bulk-encode": Spec("bulk-encode", B=4, H_q=32, H_kv=32, D=128, S_kv=8192,
                        k_N=1024, k_d=8, v_N=256, v_d=4, seed=2,
                        outlier_frac=0.02, outlier_scale=10.0),
    "bulk-encode-packed": Spec("bulk-encode-packed", B=4, H_q=32, H_kv=32, D=128, S_kv=8192,
                               k_N=1024, k_d=8, v_N=256, v_d=4, seed=2,
                               outlier_frac=0.02, outlier_scale=10.0, packed_keys=True),
    "gqa-decode": Spec("gqa-decode", B=32, H_q=32, H_kv=8, D=128, S_kv=32768,
                       seed=3, draw_keys=False, draw_values=False,
                       draw_codes=True),
    "chunked-prefill": Spec("chunked-prefill", B=1, H_q=32, H_kv=8, D=128,
                            S_kv=16384 + 2048, S_q=2048, window=4096, seed=4,
                            draw_keys=False, draw_values=False,
                            draw_codes=True),
    "decode-append": Spec("decode-append", B=1, H_q=8, H_kv=8, D=128, S_kv=8192,
                          S_enc=1, capacity=8192 + 64, seed=5, draw_codes=True),
    "gqa-decode-packed": Spec("gqa-decode-packed", B=32, H_q=32, H_kv=8, D=128,
                              S_kv=32768, k_N=1024, k_d=8, v_N=256, v_d=4, seed=7,
                              draw_keys=False, draw_values=False, draw_codes=True,
                              packed_keys=True),
    "gqa-decode-ragged": Spec("gqa-decode-ragged", B=32, H_q=32, H_kv=8, D=128,
                              S_kv=32768, seed=6, draw_keys=False,
                              draw_values=False, draw_codes=True, ragged=True),
}


def _normal_f16(rng, shape, outlier_channels=(), outlier_scale=1.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if len(outlier_channels):
        x[..., list(outlier_channels)] *= np.float32(outlier_scale)
    return x.astype(np.float16)


def make_inputs(spec: Spec) -> dict:
    """Draw every input of ``spec`` in the documented order.

    Returns numpy arrays: ``keys``/``values`` fp16 [B, H_kv, S_enc, D] (when
    drawn), ``smooth`` float32 [H_kv, D] (or [D], or None), ``k_codebook``
    float32 [k_N, k_d], ``v_codebook`` float32 [v_N, v_d], ``q`` fp16
    [B, H_q, S_q, D], and ``k_codes``/``v_codes`` [B, H_kv, S_kv, n] in
    uint8/uint16 (when drawn).
    """
    rng = np.random.default_rng(spec.seed)
    out = {}
    enc_shape = (spec.B, spec.H_kv, spec.enc_len, spec.D)
    keys = values = None
    if spec.draw_keys:
        keys = rng.standard_normal(size=enc_shape, dtype=np.float32)
    if spec.draw_values:
        values = rng.standard_normal(size=enc_shape, dtype=np.float32)
    k_out = list(spec.key_outliers)
    v_out = []
    if spec.outlier_frac > 0:
        n_out = int(round(spec.outlier_frac * spec.D))
        k_out = sorted(rng.choice(spec.D, size=n_out, replace=False).tolist())
        v_out = sorted(rng.choice(spec.D, size=n_out, replace=False).tolist())
    if keys is not None:
        if k_out:
            keys[..., k_out] *= np.float32(spec.outlier_scale)
        out["keys"] = keys.astype(np.float16)
        del keys
    if values is not None:
        if v_out:
            values[..., v_out] *= np.float32(spec.outlier_scale)
        out["values"] = values.astype(np.float16)
        del values
    out["key_outlier_channels"] = k_out
    out["value_outlier_channels"] = v_out
    if spec.smooth_mode == 2:
        out["smooth"] = rng.uniform(0.5, 2.0, size=(spec.H_kv, spec.D)).astype(np.float32)
    elif spec.smooth_mode == 1:
        out["smooth"] = rng.uniform(0.5, 2.0, size=(spec.D,)).astype(np.float32)
    else:
        out["smooth"] = None
    out["k_codebook"] = rng.standard_normal(size=(spec.k_N, spec.k_d), dtype=np.float32)
    out["v_codebook"] = rng.standard_normal(size=(spec.v_N, spec.v_d), dtype=np.float32)
    out["q"] = rng.standard_normal(
        size=(spec.B, spec.H_q, spec.S_q, spec.D), dtype=np.float32).astype(np.float16)
    if spec.draw_codes:
        out["k_codes"] = rng.integers(0, spec.k_N, size=(spec.B, spec.H_kv, spec.S_kv, spec.n_k),
                                      dtype=spec.k_code_dtype)
        out["v_codes"] = rng.integers(0, spec.v_N, size=(spec.B, spec.H_kv, spec.S_kv, spec.n_v),
                                      dtype=spec.v_code_dtype)
    if spec.ragged:
        out["kv_lens"] = rng.integers(spec.S_kv // 2, spec.S_kv + 1, size=spec.B).astype(np.int32)
    return out


def small_spec(seed: int, **kw) -> Spec:
    """A small parity-test workload; keyword arguments override the fields."""
    base = dict(name=f"small-{seed}", B=1, H_q=2, H_kv=2, D=64, S_kv=200,
                seed=seed)
    base.update(kw)
    return Spec(**base)
