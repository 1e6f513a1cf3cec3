"""Parity rules between the CUDA path and the float64 oracle.

TEST INFRASTRUCTURE ONLY (imported by the tests, the smoke check and the
benchmark's CPU leg).

Codes.  A code is an integer decided by floating point, so a kernel that
computes in fp32 may pick a different centroid than the float64 oracle only
when two candidates are too close for fp32 to order them.  A GPU code g that
differs from the oracle's code o is accepted when either
  * near tie (the stated rule): the oracle's best and second-best squared
    distances differ by less than 1e-6 relative, (d2 - d1) < 1e-6 * d2; or
  * fp32 bound: d_g - d_o <= E_g + E_o, where E_c bounds |d~_c - d_c|, the
    error of the kernel's fp32 distance to centroid c (derivation below).
Both counts are reported; anything else fails.

fp32 error bound (u = 2^-24, gamma_k = k u / (1 - k u)), for the kernel's
arithmetic on a key vector x of head h with smooth s and D = 2^L:
  u_t = fl(fl(x_t s_t) * fl(1/sqrt D))          relative error <= 3u
  y~  = FWHT(u) in L stages of fp32 add/sub      |y~_r - y_r(u)| <= gamma_L sum|u_i|
  => |y~_r - y_r| <= delta = (gamma_L (1 + 3u) + 3u) * sum_i |x_i s_i| / sqrt D
  d~_c = fp32 sum_t (y~_t - c_t)^2 (subtract, fused multiply-add chain)
  => |d~_c - d_c| <= E_c = A_c + gamma_{d+2} (d_c + A_c),
     A_c = 2 delta sum_t |y_t - c_t| + d delta^2.
Values are not rotated: x is exact in fp32, delta = 0.
"""
from __future__ import annotations

import math

import numpy as np

U = 2.0 ** -24
NEAR_TIE_REL = 1e-6


def _gamma(k):
    return k * U / (1 - k * U)


def transform_error_bound(x, smooth, D, rotate=True):
    """delta per vector (x [n, D] float64, smooth [n, D] float64 or None)."""
    if not rotate:
        return np.zeros(x.shape[0])
    L = int(round(math.log2(D)))
    xs = np.abs(x) * (np.abs(smooth) if smooth is not None else 1.0)
    return (_gamma(L) * (1 + 3 * U) + 3 * U) * xs.sum(axis=1) / math.sqrt(D)


def check_codes(gpu_codes, oracle_out, x=None, smooth_rows=None, rotate=True,
                codebook=None):
    """Compare GPU codes with the oracle's.

    gpu_codes: int array [n, n_sub]; oracle_out: dict from oracle.encode with
    ``want_y=True`` (flattened to [n, ...]); x: the fp16 inputs as float64
    [n, D]; smooth_rows: smooth factors per input row [n, D] (keys) or None.
    Returns a dict of counts; raises AssertionError on an unjustified
    mismatch.
    """
    o_codes = np.asarray(oracle_out["codes"]).reshape(gpu_codes.shape)
    g = np.asarray(gpu_codes).astype(np.int64)
    mism = np.argwhere(g != o_codes)
    n = g.shape[0]
    res = {"subvectors": int(g.size), "mismatch": int(len(mism)),
           "near_tie": 0, "fp32_bound": 0}
    if len(mism) == 0:
        return res
    cb = np.asarray(codebook, dtype=np.float64)
    d = cb.shape[1]
    y = np.asarray(oracle_out["y"]).reshape(n, -1)
    D = y.shape[1]
    d1 = np.asarray(oracle_out["d1"]).reshape(g.shape)
    d2 = np.asarray(oracle_out["d2"]).reshape(g.shape)
    delta = transform_error_bound(np.asarray(x, dtype=np.float64).reshape(n, D),
                                  None if smooth_rows is None else
                                  np.asarray(smooth_rows, dtype=np.float64).reshape(n, D),
                                  D, rotate)
    gam = _gamma(d + 2)
    bad = []
    for v, m in mism:
        ys = y[v, m * d:(m + 1) * d]
        cg, co = cb[g[v, m]], cb[o_codes[v, m]]
        dg = float(((ys - cg) ** 2).sum())
        do = float(((ys - co) ** 2).sum())
        if (d2[v, m] - d1[v, m]) < NEAR_TIE_REL * d2[v, m]:
            res["near_tie"] += 1
            continue
        A_g = 2 * delta[v] * np.abs(ys - cg).sum() + d * delta[v] ** 2
        A_o = 2 * delta[v] * np.abs(ys - co).sum() + d * delta[v] ** 2
        E = A_g + gam * (dg + A_g) + A_o + gam * (do + A_o)
        if dg - do <= E * (1 + 1e-9) + 1e-12 * max(do, 1e-300):
            res["fp32_bound"] += 1
        else:
            bad.append((int(v), int(m), int(g[v, m]), int(o_codes[v, m]), dg, do, E))
    assert not bad, f"{len(bad)} unjustified code mismatches, first: {bad[:3]}"
    return res


def allclose_report(got, ref, atol=2e-3, rtol=1e-2):
    """|got - ref| <= atol + rtol |ref| elementwise; returns (ok, max_err,
    worst excess)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    lim = atol + rtol * np.abs(ref)
    ok = bool(np.all(err <= lim))
    return ok, float(err.max(initial=0.0)), float((err - lim).max(initial=-np.inf))
