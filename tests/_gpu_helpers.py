"""Shared helpers of the GPU parity tests (inputs to device, oracle calls)."""
import numpy as np
import torch

import oracle
from oracle import parity
from product_vq_compressed_gb300 import binding as vq

DEV = "cuda:0"


def dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def check_encode(x16, codebook, sub_dim, smooth, rotate, gpu_codes, gpu_hat,
                 rows=None):
    """Oracle-check codes (and the fp16 reconstruction) of x16 [B, H, S, D].

    rows: optional flat vector indices to check (a sample); all otherwise.
    Returns the parity counts.
    """
    B, H, S, D = x16.shape
    n = B * H * S
    xf = x16.reshape(n, D)
    heads = np.broadcast_to(np.arange(H)[None, :, None], (B, H, S)).reshape(n)
    if rows is None:
        rows = np.arange(n)
    rows = np.asarray(rows)
    o = oracle.encode(xf[rows], codebook, heads=heads[rows],
                      smooth=smooth if rotate else None, rotate=rotate,
                      want_y=True, want_xhat=gpu_hat is not None)
    g = gpu_codes.reshape(n, -1)[rows].astype(np.int64)
    res = parity.check_codes(g, o)
    if gpu_hat is not None:
        # compare the reconstruction where every code of the vector agrees;
        # vectors with a justified code difference are counted above
        same = (g == o["codes"]).all(axis=1)
        ref = oracle.to_f16(o["xhat"][same]).astype(np.float64)
        got = gpu_hat.reshape(n, D)[rows][same].astype(np.float64)
        ok, err, _ = parity.allclose_report(got, ref)
        assert ok, f"reconstruction max |err| {err}"
        res["hat_checked"] = int(same.sum())
        res["hat_max_err"] = err
    return res


def oracle_attend_rows(inp, spec, rows, k_codes, v_codes, causal=None,
                       window=None):
    """Float64 attention for (b, h_q, i) rows, sorted by (b, h_q)."""
    rows = np.asarray(rows)
    order = np.lexsort((rows[:, 2], rows[:, 1], rows[:, 0]))
    out = np.zeros((len(rows), spec.D))
    out[order] = oracle.attend_rows(
        inp["q"], k_codes, inp["k_codebook"], v_codes, inp["v_codebook"],
        inp["smooth"], spec.sm_scale, spec.causal if causal is None else causal,
        spec.window if window is None else window, rows[order])
    return out


def run_attend(entry, inp, spec, k_codes, v_codes, causal=None, window=None):
    fn = vq.decode_attend if entry == "decode" else vq.prefill_attend
    return fn(dev(inp["q"]), dev(k_codes), dev(inp["k_codebook"]), dev(v_codes),
              dev(inp["v_codebook"]), dev(inp["smooth"]), spec.sm_scale,
              causal=spec.causal if causal is None else causal,
              sliding_window=spec.window if window is None else window)


def oracle_attend_rows_parallel(inp, spec, rows, k_codes, v_codes, workers=None):
    """oracle_attend_rows for many rows of a full-size workload: the rows of
    each (batch, KV head) go to the oracle with that head's slice of the
    inputs only, one thread per (batch, KV head) (the C oracle releases the
    GIL).  Per-batch cache lengths are applied by slicing the codes."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    rows = np.asarray(rows)
    G = spec.G
    groups = {}
    for k, (b, h, i) in enumerate(rows):
        groups.setdefault((int(b), int(h) // G), []).append(k)
    out = np.zeros((len(rows), spec.D))
    sm = inp["smooth"]

    def one(key):
        b, g = key
        ks = groups[key]
        kc, vc = k_codes[b:b + 1, g:g + 1], v_codes[b:b + 1, g:g + 1]
        if "kv_lens" in inp:
            L = int(inp["kv_lens"][b])
            kc, vc = kc[:, :, :L], vc[:, :, :L]
        local = np.array([[0, rows[k, 1] - g * G, rows[k, 2]] for k in ks])
        order = np.lexsort((local[:, 2], local[:, 1]))
        res = oracle.attend_rows(
            inp["q"][b:b + 1, g * G:(g + 1) * G], kc, inp["k_codebook"], vc,
            inp["v_codebook"], None if sm is None else (sm if sm.ndim == 1 else sm[g:g + 1]),
            spec.sm_scale, spec.causal, spec.window, local[order])
        out[np.asarray(ks)[order]] = res

    n = workers or min(len(groups), max(1, len(os.sched_getaffinity(0))))
    with ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(one, list(groups)))
    return out
