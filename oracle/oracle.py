"""ctypes marshalling for the float64 C oracle (``vq_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
CPU-baseline leg of the benchmark, never by the product path.

Nothing here does any of the method's arithmetic.  It converts inputs to
float64 / int32 (fp16 -> float64 is exact), calls the C functions and, where
a page fixes an fp16 output, rounds float64 results to fp16 with numpy's
round-to-nearest-even cast.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libvq_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile ``vq_oracle.c`` with gcc (IEEE float64, no FMA contraction)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.orc_hadamard.argtypes = [i32, _dp]
            lib.orc_encode.argtypes = [_dp, i64, i32, _ip, _dp, i32, i32, _dp,
                                       i32, i32, _ip, _dp, _dp, _dp, _dp]
            lib.orc_dequant.argtypes = [_ip, i64, i32, _dp, i32, i32, _dp]
            lib.orc_reconstruct.argtypes = [_ip, i64, i32, _ip, _dp, i32, i32,
                                            _dp, i32, i32, _dp]
            lib.orc_attend_rows.argtypes = [
                _dp, i32, i32, i32, i32, i32, i32, _ip, _dp, i32, i32, _ip,
                _dp, i32, i32, _dp, i32, f64, i32, i32, _ip, i64, _dp]
            lib.orc_lut_score.argtypes = [_dp, i32, _dp, i32, i32, _dp, i32,
                                          i32, _ip, f64, _dp]
            for fn in ("orc_hadamard", "orc_encode", "orc_dequant",
                       "orc_reconstruct", "orc_attend_rows", "orc_lut_score"):
                getattr(lib, fn).restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a, kind):
    if a is None:
        return None
    return a.ctypes.data_as(kind)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"oracle {name} failed with status {rc}")


def to_f16(a) -> np.ndarray:
    """Round float64 to fp16, round-to-nearest-even (numpy's cast)."""
    return np.asarray(a, dtype=np.float64).astype(np.float16)


def hadamard(D: int) -> np.ndarray:
    """Normalised Sylvester-Hadamard matrix [D, D] (float64)."""
    out = np.zeros((D, D), dtype=np.float64)
    _check(_load().orc_hadamard(D, _p(out, _dp)), "hadamard")
    return out


def _smooth_args(smooth):
    if smooth is None:
        return None, 0
    s = _f64(smooth)
    return s, (1 if s.ndim == 1 else 2)


def encode(x, codebook, heads=None, smooth=None, rotate=True,
           want_y=False, want_xhat=False):
    """Encode vectors x [..., D] against codebook [N, d].

    ``heads`` gives the KV head of every vector (same leading shape as x);
    when x is [B, H, S, D] and heads is None it is derived from axis 1.
    Returns a dict with int32 ``codes`` [..., D/d], float64 ``d1``/``d2``
    (best / second-best squared distance), and optionally ``y`` (the
    transformed vector) and ``xhat`` (float64 reconstruction from the
    oracle's own codes).
    """
    x = _f64(x)
    cb = _f64(codebook)
    N, d = cb.shape
    D = x.shape[-1]
    lead = x.shape[:-1]
    n_vec = int(np.prod(lead)) if lead else 1
    if heads is None:
        if x.ndim == 4:
            heads = np.broadcast_to(
                np.arange(x.shape[1], dtype=np.int32)[None, :, None], lead)
        else:
            heads = np.zeros(lead, dtype=np.int32)
    hv = _i32(np.broadcast_to(heads, lead)).reshape(-1)
    s, mode = _smooth_args(smooth)
    n_sub = D // d
    codes = np.zeros((n_vec, n_sub), dtype=np.int32)
    d1 = np.zeros((n_vec, n_sub))
    d2 = np.zeros((n_vec, n_sub))
    y = np.zeros((n_vec, D)) if want_y else None
    xh = np.zeros((n_vec, D)) if want_xhat else None
    rc = _load().orc_encode(_p(x, _dp), n_vec, D, _p(hv, _ip), _p(s, _dp),
                            mode, int(bool(rotate)), _p(cb, _dp), N, d,
                            _p(codes, _ip), _p(d1, _dp), _p(d2, _dp),
                            _p(y, _dp), _p(xh, _dp))
    _check(rc, "encode")
    out = {"codes": codes.reshape(lead + (n_sub,)),
           "d1": d1.reshape(lead + (n_sub,)),
           "d2": d2.reshape(lead + (n_sub,))}
    if want_y:
        out["y"] = y.reshape(lead + (D,))
    if want_xhat:
        out["xhat"] = xh.reshape(lead + (D,))
    return out


def dequant(codes, codebook) -> np.ndarray:
    """Codebook gather [..., n_sub] -> [..., n_sub*d] (float64)."""
    c = _i32(codes)
    cb = _f64(codebook)
    N, d = cb.shape
    lead = c.shape[:-1]
    n_sub = c.shape[-1]
    n_vec = int(np.prod(lead)) if lead else 1
    out = np.zeros((n_vec, n_sub * d))
    _check(_load().orc_dequant(_p(c, _ip), n_vec, n_sub, _p(cb, _dp), N, d,
                               _p(out, _dp)), "dequant")
    return out.reshape(lead + (n_sub * d,))


def reconstruct(codes, codebook, heads=None, smooth=None, rotate=True):
    """s^-1 (.) Hn^T dequant(codes) for keys (rotate) or dequant for values."""
    c = _i32(codes)
    cb = _f64(codebook)
    N, d = cb.shape
    lead = c.shape[:-1]
    D = c.shape[-1] * d
    n_vec = int(np.prod(lead)) if lead else 1
    if heads is None:
        if c.ndim == 4:
            heads = np.broadcast_to(
                np.arange(c.shape[1], dtype=np.int32)[None, :, None], lead)
        else:
            heads = np.zeros(lead, dtype=np.int32)
    hv = _i32(np.broadcast_to(heads, lead)).reshape(-1)
    s, mode = _smooth_args(smooth)
    out = np.zeros((n_vec, D))
    _check(_load().orc_reconstruct(_p(c, _ip), n_vec, D, _p(hv, _ip),
                                   _p(s, _dp), mode, int(bool(rotate)),
                                   _p(cb, _dp), N, d, _p(out, _dp)),
           "reconstruct")
    return out.reshape(lead + (D,))


def attend_rows(q, k_codes, k_codebook, v_codes, v_codebook, smooth, scale,
                causal, sliding_window, rows, H_kv=None):
    """Attention output (float64 [n_rows, D]) for (b, h_q, i) rows.

    q [B, H_q, S_q, D] (raw); k_codes [B, H_kv, S_kv, D/dk]; v_codes
    [B, H_kv, S_kv, D/dv].  Rows are processed in the given order; sort them
    by (b, h_q) so the oracle reuses each K_hat reconstruction.
    """
    qf = _f64(q)
    B, H_q, S_q, D = qf.shape
    kc = _i32(k_codes)
    vc = _i32(v_codes)
    H_kv = kc.shape[1] if H_kv is None else H_kv
    S_kv = kc.shape[2]
    kcb = _f64(k_codebook)
    vcb = _f64(v_codebook)
    s, mode = _smooth_args(smooth)
    r = _i32(rows).reshape(-1, 3)
    out = np.zeros((r.shape[0], D))
    rc = _load().orc_attend_rows(
        _p(qf, _dp), B, H_q, H_kv, S_q, S_kv, D, _p(kc, _ip), _p(kcb, _dp),
        kcb.shape[0], kcb.shape[1], _p(vc, _ip), _p(vcb, _dp), vcb.shape[0],
        vcb.shape[1], _p(s, _dp), mode, float(scale), int(bool(causal)),
        int(sliding_window), _p(r, _ip), r.shape[0], _p(out, _dp))
    _check(rc, "attend_rows")
    return out


def attend(q, k_codes, k_codebook, v_codes, v_codebook, smooth, scale,
           causal=True, sliding_window=0):
    """Attention output for every row, float64 [B, H_q, S_q, D]."""
    B, H_q, S_q, D = np.shape(q)
    bb, hh, ii = np.meshgrid(np.arange(B), np.arange(H_q), np.arange(S_q),
                             indexing="ij")
    rows = np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1)
    out = attend_rows(q, k_codes, k_codebook, v_codes, v_codebook, smooth,
                      scale, causal, sliding_window, rows)
    return out.reshape(B, H_q, S_q, D)


def lut_score(q_row, smooth, g, k_codebook, code_row, scale) -> float:
    """Lookup-table score sum_m LUT[m][code_m] for one raw query row."""
    qf = _f64(q_row)
    D = qf.shape[-1]
    kcb = _f64(k_codebook)
    s, mode = _smooth_args(smooth)
    c = _i32(code_row)
    out = ctypes.c_double(0.0)
    _check(_load().orc_lut_score(_p(qf, _dp), D, _p(s, _dp), mode, int(g),
                                 _p(kcb, _dp), kcb.shape[0], kcb.shape[1],
                                 _p(c, _ip), float(scale), ctypes.byref(out)),
           "lut_score")
    return out.value
