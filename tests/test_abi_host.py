"""Host-side checks of the C ABI (no GPU needed).

The library must build for sm_103a, export every function that
include/vqkv.h declares, and reject bad arguments synchronously -- before
any CUDA call -- with the documented status codes.  Pointers here are fake
addresses that the library never dereferences on these error paths.
"""
import ctypes
import os
import re

import pytest

from product_vq_compressed_gb300 import binding as vq
from product_vq_compressed_gb300 import build as vqbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include",
                      "vqkv.h")
FAKE = 0x10000          # 16-byte aligned fake device address
FAKE_MIS = 0x10008      # misaligned


@pytest.fixture(scope="module")
def L():
    vqbuild.build_library()
    return vq.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"VQ_API\s+[\w\s\*]+?\b(vq_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert names == set(vq.EXPORTED)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    for st in range(0, -7, -1):
        s = L.vq_status_str(st)
        assert s and s.decode() != "unknown status"
    assert L.vq_status_str(-99).decode() == "unknown status"


def _enc(L, **kw):
    a = dict(keys=FAKE, B=1, H=2, S=8, D=128, cb=FAKE, N=256, sub=4,
             smooth=FAKE, mode=2, codes=FAKE, code_bytes=1, khat=None)
    a.update(kw)
    return L.vq_encode_keys(a["keys"], a["B"], a["H"], a["S"], a["D"], a["cb"],
                            a["N"], a["sub"], a["smooth"], a["mode"], a["codes"],
                            a["code_bytes"], a["khat"], None)


def test_encode_argument_errors(L):
    assert _enc(L, keys=None) == vq.VQ_ERR_NULL
    assert _enc(L, codes=None) == vq.VQ_ERR_NULL
    assert _enc(L, smooth=None) == vq.VQ_ERR_NULL
    assert _enc(L, mode=3) == vq.VQ_ERR_SHAPE
    assert _enc(L, S=-1) == vq.VQ_ERR_SHAPE
    assert _enc(L, D=128, sub=3) == vq.VQ_ERR_SHAPE
    assert _enc(L, code_bytes=4) == vq.VQ_ERR_SHAPE
    assert _enc(L, N=257, code_bytes=1) == vq.VQ_ERR_UNSUPPORTED
    assert _enc(L, N=65537, code_bytes=2) == vq.VQ_ERR_UNSUPPORTED
    assert _enc(L, N=0) == vq.VQ_ERR_UNSUPPORTED
    assert _enc(L, D=96, sub=4) == vq.VQ_ERR_UNSUPPORTED
    assert _enc(L, D=1024, sub=4) == vq.VQ_ERR_UNSUPPORTED
    assert _enc(L, D=16, sub=4) == vq.VQ_ERR_UNSUPPORTED
    assert _enc(L, D=128, sub=32) == vq.VQ_ERR_UNSUPPORTED
    assert _enc(L, N=65536, code_bytes=2, sub=4) == vq.VQ_ERR_UNSUPPORTED  # 1 MiB codebook
    assert _enc(L, keys=FAKE_MIS) == vq.VQ_ERR_ALIGN
    assert _enc(L, codes=FAKE_MIS) == vq.VQ_ERR_ALIGN
    assert _enc(L, khat=FAKE_MIS) == vq.VQ_ERR_ALIGN
    # empty problems are a no-op that touches nothing
    assert _enc(L, B=0) == vq.VQ_OK
    assert _enc(L, S=0) == vq.VQ_OK
    assert _enc(L, S=0, keys=None, codes=None, cb=None) == vq.VQ_OK
    assert _enc(L, S=0, D=96) == vq.VQ_ERR_UNSUPPORTED
    assert L.vq_encode_values(FAKE, 1, 1, 0, 64, FAKE, 16, 4, FAKE, 1, None,
                              None) == vq.VQ_OK
    assert L.vq_encode_values(FAKE, 1, 1, 4, 64, FAKE, 16, 4, None, 1, None,
                              None) == vq.VQ_ERR_NULL


def test_encode_into_argument_errors(L):
    def f(S=8, cap=16, off=0, values=False):
        if values:
            return L.vq_encode_values_into(FAKE, 1, 2, S, 128, FAKE, 256, 4, FAKE, 1,
                                           cap, off, None, None)
        return L.vq_encode_keys_into(FAKE, 1, 2, S, 128, FAKE, 256, 4, FAKE, 2, FAKE,
                                     1, cap, off, None, None)
    assert f(cap=16, off=9) == vq.VQ_ERR_SHAPE        # 9 + 8 rows > 16
    assert f(off=-1) == vq.VQ_ERR_SHAPE
    assert f(cap=-1) == vq.VQ_ERR_SHAPE
    assert f(cap=7) == vq.VQ_ERR_SHAPE
    assert f(values=True, cap=10, off=3) == vq.VQ_ERR_SHAPE
    assert f(S=0, cap=4, off=4) == vq.VQ_OK             # empty: nothing written


def test_dequant_argument_errors(L):
    assert L.vq_dequant(None, 1, 4, 32, FAKE, 256, 4, FAKE, 1, None) == vq.VQ_ERR_NULL
    assert L.vq_dequant(None, 1, 0, 32, None, 256, 4, None, 1, None) == vq.VQ_OK
    assert L.vq_dequant(FAKE, 3, 4, 32, FAKE, 256, 4, FAKE, 1, None) == vq.VQ_ERR_SHAPE
    assert L.vq_dequant(FAKE, 1, -1, 32, FAKE, 256, 4, FAKE, 1, None) == vq.VQ_ERR_SHAPE
    assert L.vq_dequant(FAKE, 1, 4, 0, FAKE, 256, 4, FAKE, 1, None) == vq.VQ_ERR_SHAPE
    assert L.vq_dequant(FAKE, 1, 4, 32, FAKE, 300, 4, FAKE, 1, None) == vq.VQ_ERR_UNSUPPORTED
    assert L.vq_dequant(FAKE_MIS, 1, 4, 32, FAKE, 256, 4, FAKE, 1, None) == vq.VQ_ERR_ALIGN
    assert L.vq_dequant(FAKE, 1, 0, 32, FAKE, 256, 4, FAKE, 1, None) == vq.VQ_OK


def _args(**kw):
    a = vq.AttendArgs()
    base = dict(B=2, H_q=8, H_kv=2, S_q=1, S_kv=100, D=128, q_f16=FAKE,
                k_codes=FAKE, k_code_bytes=1, k_codebook=FAKE,
                k_n_centroids=256, k_sub_dim=4, v_codes=FAKE, v_code_bytes=1,
                v_codebook=FAKE, v_n_centroids=256, v_sub_dim=4, smooth=FAKE,
                smooth_mode=2, scale=0.1, causal=1, sliding_window=0,
                out_f16=FAKE, workspace=FAKE, workspace_bytes=1 << 30)
    base.update(kw)
    for k, v in base.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("fn", ["vq_decode_attend", "vq_prefill_attend"])
def test_attend_argument_errors(L, fn):
    call = lambda **kw: getattr(L, fn)(ctypes.byref(_args(**kw)), None)  # noqa: E731
    assert getattr(L, fn)(None, None) == vq.VQ_ERR_NULL
    assert call(q_f16=0) == vq.VQ_ERR_NULL
    assert call(out_f16=0) == vq.VQ_ERR_NULL
    assert call(smooth=0) == vq.VQ_ERR_NULL
    assert call(H_q=6, H_kv=4) == vq.VQ_ERR_SHAPE
    assert call(H_kv=0) == vq.VQ_ERR_SHAPE
    assert call(k_sub_dim=3) == vq.VQ_ERR_SHAPE
    assert call(S_q=101) == vq.VQ_ERR_SHAPE                 # causal, S_q > S_kv
    assert call(S_q=101, causal=0, sliding_window=5) == vq.VQ_ERR_SHAPE
    assert call(S_kv=0) == vq.VQ_ERR_SHAPE
    assert call(sliding_window=-1) == vq.VQ_ERR_SHAPE
    assert call(smooth_mode=5) == vq.VQ_ERR_SHAPE
    assert call(k_code_bytes=3) == vq.VQ_ERR_SHAPE
    assert call(k_n_centroids=300) == vq.VQ_ERR_UNSUPPORTED
    assert call(D=96) == vq.VQ_ERR_UNSUPPORTED
    assert call(D=512) == vq.VQ_ERR_UNSUPPORTED
    assert call(k_sub_dim=16, v_sub_dim=16) == vq.VQ_ERR_UNSUPPORTED
    assert call(k_n_centroids=65536, k_code_bytes=2) == vq.VQ_ERR_UNSUPPORTED
    assert call(kv_stride=50) == vq.VQ_ERR_SHAPE     # rows per head < S_kv
    assert call(kv_stride=-1) == vq.VQ_ERR_SHAPE
    assert call(q_f16=FAKE_MIS) == vq.VQ_ERR_ALIGN
    assert call(workspace=FAKE_MIS) == vq.VQ_ERR_ALIGN
    assert L.vq_attend_workspace_bytes(None) == 0
    assert call(B=0, q_f16=0, out_f16=0) == vq.VQ_OK


def test_library_has_sm103a_code(L):
    """The build targets sm_103a (the only -gencode in the build flags)."""
    assert vqbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.getsize(vqbuild.LIB_PATH) > 100_000


def test_decode_step_argument_errors(L):
    """vq_decode_step: the attention checks, then its own, before any launch."""
    step = lambda kn=FAKE, vn=FAKE, **kw: L.vq_decode_step(  # noqa: E731
        ctypes.byref(_args(**kw)), kn, vn, None)
    assert L.vq_decode_step(None, FAKE, FAKE, None) == vq.VQ_ERR_NULL
    assert step(H_q=6, H_kv=4) == vq.VQ_ERR_SHAPE
    assert step(S_q=101) == vq.VQ_ERR_SHAPE
    assert step(S_q=101, causal=0) == vq.VQ_ERR_SHAPE      # new tokens are cache rows
    assert step(D=96) == vq.VQ_ERR_UNSUPPORTED
    assert step(kv_lens=FAKE) == vq.VQ_ERR_UNSUPPORTED
    assert step(kn=None) == vq.VQ_ERR_NULL
    assert step(vn=None) == vq.VQ_ERR_NULL
    assert step(kn=FAKE_MIS) == vq.VQ_ERR_ALIGN
    assert step(q_f16=FAKE_MIS) == vq.VQ_ERR_ALIGN
    assert step(B=0, q_f16=0, out_f16=0, kn=None, vn=None) == vq.VQ_OK
