"""Parity rules between the CUDA path and the float64 oracle.

TEST INFRASTRUCTURE ONLY (imported by the tests, the smoke check and the
benchmark's CPU leg).

Codes.  A code is an integer decided by floating point.  The stated rule:
a GPU code may differ from the oracle's only where the oracle's best and
second-best squared distances are a near tie, (d2 - d1) < 1e-6 * d2
(relative).  Those mismatches are counted and reported; any other
mismatch fails.  (The kernels decide in fp32 and re-decide in fp64 every
sub-vector whose fp32 decision a rigorous error bound cannot certify, so
that nothing wider than a near tie is needed.)
"""
from __future__ import annotations

import numpy as np

NEAR_TIE_REL = 1e-6


def check_codes(gpu_codes, oracle_out, **_unused):
    """Compare GPU codes with the oracle's.

    gpu_codes: int array [n, n_sub]; oracle_out: dict from oracle.encode
    (flattened to [n, ...]) with the best and second-best distances d1, d2.
    Returns {"subvectors", "mismatch", "near_tie"}; raises AssertionError on
    a mismatch that is not a near tie.
    """
    o_codes = np.asarray(oracle_out["codes"]).reshape(gpu_codes.shape)
    g = np.asarray(gpu_codes).astype(np.int64)
    mism = np.argwhere(g != o_codes)
    res = {"subvectors": int(g.size), "mismatch": int(len(mism)), "near_tie": 0}
    if len(mism) == 0:
        return res
    d1 = np.asarray(oracle_out["d1"]).reshape(g.shape)
    d2 = np.asarray(oracle_out["d2"]).reshape(g.shape)
    bad = []
    for v, m in mism:
        if (d2[v, m] - d1[v, m]) < NEAR_TIE_REL * d2[v, m]:
            res["near_tie"] += 1
        else:
            bad.append((int(v), int(m), int(g[v, m]), int(o_codes[v, m]),
                        float(d1[v, m]), float(d2[v, m])))
    assert not bad, f"{len(bad)} code mismatches that are not near ties, first: {bad[:3]}"
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
