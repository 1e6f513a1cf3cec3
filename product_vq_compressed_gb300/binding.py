"""Thin Python binding of libvqkv.so (ctypes).

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch supplies device memory and the current stream.  The
function names mirror the C entry points declared in include/vqkv.h.

If the shared library has not been built, importing works but every call
raises ``VQError`` naming the missing file; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

from . import build as _build

VQ_OK = 0
VQ_ERR_NULL = -1
VQ_ERR_SHAPE = -2
VQ_ERR_UNSUPPORTED = -3
VQ_ERR_ALIGN = -4
VQ_ERR_WORKSPACE = -5
VQ_ERR_CUDA = -6

EXPORTED = ("vq_status_str", "vq_encode_keys", "vq_encode_values",
            "vq_encode_keys_into", "vq_encode_values_into",
            "vq_dequant", "vq_attend_workspace_bytes", "vq_decode_attend",
            "vq_prefill_attend", "vq_decode_attend_noalloc", "vq_decode_step")


class VQError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


class AttendArgs(ctypes.Structure):
    """Mirror of vq_attend_args."""

    _fields_ = [
        ("B", ctypes.c_int), ("H_q", ctypes.c_int), ("H_kv", ctypes.c_int),
        ("S_q", ctypes.c_int), ("S_kv", ctypes.c_int), ("D", ctypes.c_int),
        ("q_f16", ctypes.c_void_p),
        ("k_codes", ctypes.c_void_p), ("k_code_bytes", ctypes.c_int),
        ("k_codebook", ctypes.c_void_p),
        ("k_n_centroids", ctypes.c_int), ("k_sub_dim", ctypes.c_int),
        ("v_codes", ctypes.c_void_p), ("v_code_bytes", ctypes.c_int),
        ("v_codebook", ctypes.c_void_p),
        ("v_n_centroids", ctypes.c_int), ("v_sub_dim", ctypes.c_int),
        ("smooth", ctypes.c_void_p), ("smooth_mode", ctypes.c_int),
        ("scale", ctypes.c_float), ("causal", ctypes.c_int),
        ("sliding_window", ctypes.c_int),
        ("out_f16", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("kv_stride", ctypes.c_int), ("kv_lens", ctypes.c_void_p),
    ]


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """The loaded ctypes library (raises if it was never built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise VQError(VQ_ERR_CUDA,
                          f"libvqkv.so not built ({path}); run "
                          "product_vq_compressed_gb300.build.build_library()")
        L = ctypes.CDLL(path)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.vq_status_str.argtypes = [i32]
        L.vq_status_str.restype = ctypes.c_char_p
        L.vq_encode_keys.argtypes = [vp, i32, i32, i32, i32, vp, i32, i32, vp,
                                     i32, vp, i32, vp, vp]
        L.vq_encode_values.argtypes = [vp, i32, i32, i32, i32, vp, i32, i32,
                                       vp, i32, vp, vp]
        L.vq_encode_keys_into.argtypes = [vp, i32, i32, i32, i32, vp, i32, i32, vp,
                                          i32, vp, i32, i32, i32, vp, vp]
        L.vq_encode_values_into.argtypes = [vp, i32, i32, i32, i32, vp, i32, i32,
                                            vp, i32, i32, i32, vp, vp]
        L.vq_dequant.argtypes = [vp, i32, i64, i32, vp, i32, i32, vp, i32, vp]
        L.vq_attend_workspace_bytes.argtypes = [ctypes.POINTER(AttendArgs)]
        L.vq_attend_workspace_bytes.restype = ctypes.c_size_t
        L.vq_decode_attend.argtypes = [ctypes.POINTER(AttendArgs), vp]
        L.vq_prefill_attend.argtypes = [ctypes.POINTER(AttendArgs), vp]
        L.vq_decode_attend_noalloc.argtypes = [ctypes.POINTER(AttendArgs), vp]
        L.vq_decode_step.argtypes = [ctypes.POINTER(AttendArgs), vp, vp, vp]
        for fn in ("vq_encode_keys", "vq_encode_values", "vq_encode_keys_into",
                   "vq_encode_values_into", "vq_dequant",
                   "vq_decode_attend", "vq_prefill_attend",
                   "vq_decode_attend_noalloc", "vq_decode_step"):
            getattr(L, fn).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != VQ_OK:
        raise VQError(status, f"{what}: {lib().vq_status_str(status).decode()}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def code_dtype(n_centroids: int) -> torch.dtype:
    return torch.uint8 if n_centroids <= 256 else torch.uint16


def packed_code_bits(n_centroids: int) -> int:
    """Bits per code of bit-packed codes: 2^bits >= n_centroids, bits >= 1."""
    b = 1
    while (1 << b) < n_centroids:
        b += 1
    return b


def packed_row_words(n_sub: int, n_centroids: int) -> int:
    """32-bit words per token row of n_sub bit-packed codes."""
    return (n_sub * packed_code_bits(n_centroids) + 31) // 32


def _code_bytes(t: torch.Tensor) -> int:
    """1 (uint8 codes), 2 (uint16 codes) or 0: int32 tensors hold bit-packed
    token rows (code m of a row in bits [m b, m b + b) of its 32-bit words)."""
    return 0 if t.dtype == torch.int32 else t.element_size()


def _smooth_mode(smooth: Optional[torch.Tensor]) -> int:
    if smooth is None:
        return 0
    return 1 if smooth.dim() == 1 else 2


def _new_codes(B, H, S, n_sub, N, packed, device):
    if packed:
        return torch.empty((B, H, S, packed_row_words(n_sub, N)), dtype=torch.int32,
                           device=device)
    return torch.empty((B, H, S, n_sub), dtype=code_dtype(N), device=device)


def encode_keys(keys: torch.Tensor, codebook: torch.Tensor, sub_dim: int,
                smooth: Optional[torch.Tensor] = None,
                codes: Optional[torch.Tensor] = None,
                k_hat: Optional[torch.Tensor] = None, want_k_hat: bool = False,
                stream=None, packed: bool = False) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """vq_encode_keys on keys [B, H, S, D] fp16; returns (codes, k_hat).
    packed: codes as bit-packed int32 token rows."""
    B, H, S, D = keys.shape
    N = codebook.shape[0]
    if codes is None:
        codes = _new_codes(B, H, S, D // sub_dim, N, packed, keys.device)
    if k_hat is None and want_k_hat:
        k_hat = torch.empty_like(keys)
    st = lib().vq_encode_keys(_ptr(keys), B, H, S, D, _ptr(codebook), N,
                              sub_dim, _ptr(smooth), _smooth_mode(smooth),
                              _ptr(codes), _code_bytes(codes), _ptr(k_hat),
                              _stream(stream))
    _check(st, "vq_encode_keys")
    return codes, k_hat


def encode_values(values: torch.Tensor, codebook: torch.Tensor, sub_dim: int,
                  codes: Optional[torch.Tensor] = None,
                  v_hat: Optional[torch.Tensor] = None,
                  want_v_hat: bool = False, stream=None, packed: bool = False):
    """vq_encode_values on values [B, H, S, D] fp16; returns (codes, v_hat)."""
    B, H, S, D = values.shape
    N = codebook.shape[0]
    if codes is None:
        codes = _new_codes(B, H, S, D // sub_dim, N, packed, values.device)
    if v_hat is None and want_v_hat:
        v_hat = torch.empty_like(values)
    st = lib().vq_encode_values(_ptr(values), B, H, S, D, _ptr(codebook), N,
                                sub_dim, _ptr(codes), _code_bytes(codes),
                                _ptr(v_hat), _stream(stream))
    _check(st, "vq_encode_values")
    return codes, v_hat


def encode_keys_into(keys: torch.Tensor, codebook: torch.Tensor, sub_dim: int,
                     smooth: Optional[torch.Tensor], codes: torch.Tensor, offset: int,
                     k_hat: Optional[torch.Tensor] = None, want_k_hat: bool = False,
                     stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """vq_encode_keys_into: keys [B, H, S, D] into rows offset .. offset+S-1
    of the preallocated codes [B, H, capacity, D / sub_dim]."""
    B, H, S, D = keys.shape
    if k_hat is None and want_k_hat:
        k_hat = torch.empty_like(keys)
    st = lib().vq_encode_keys_into(_ptr(keys), B, H, S, D, _ptr(codebook),
                                   codebook.shape[0], sub_dim, _ptr(smooth),
                                   _smooth_mode(smooth), _ptr(codes), _code_bytes(codes),
                                   codes.shape[2], int(offset), _ptr(k_hat), _stream(stream))
    _check(st, "vq_encode_keys_into")
    return codes, k_hat


def encode_values_into(values: torch.Tensor, codebook: torch.Tensor, sub_dim: int,
                       codes: torch.Tensor, offset: int,
                       v_hat: Optional[torch.Tensor] = None, want_v_hat: bool = False,
                       stream=None):
    """vq_encode_values_into: values [B, H, S, D] into rows offset .. of codes."""
    B, H, S, D = values.shape
    if v_hat is None and want_v_hat:
        v_hat = torch.empty_like(values)
    st = lib().vq_encode_values_into(_ptr(values), B, H, S, D, _ptr(codebook),
                                     codebook.shape[0], sub_dim, _ptr(codes),
                                     _code_bytes(codes), codes.shape[2], int(offset),
                                     _ptr(v_hat), _stream(stream))
    _check(st, "vq_encode_values_into")
    return codes, v_hat


def dequant(codes: torch.Tensor, codebook: torch.Tensor,
            out: Optional[torch.Tensor] = None, out_f32: bool = True,
            stream=None, n_sub: Optional[int] = None) -> torch.Tensor:
    """vq_dequant: codes [..., n_sub] -> [..., n_sub * sub_dim]; packed int32
    rows [..., words] need n_sub."""
    N, d = codebook.shape
    if n_sub is None:
        n_sub = codes.shape[-1]
    # vectors: all leading dimensions (one row of codes, or of packed words, each)
    n_vec = codes.numel() // codes.shape[-1] if codes.shape[-1] else 0
    if out is None:
        out = torch.empty(codes.shape[:-1] + (n_sub * d,),
                          dtype=torch.float32 if out_f32 else torch.float16,
                          device=codes.device)
    st = lib().vq_dequant(_ptr(codes), _code_bytes(codes), n_vec, n_sub,
                          _ptr(codebook), N, d, _ptr(out),
                          int(out.dtype == torch.float32), _stream(stream))
    _check(st, "vq_dequant")
    return out


def make_attend_args(q, k_codes, k_codebook, v_codes, v_codebook, smooth,
                     scale, causal=True, sliding_window=0, out=None,
                     workspace=None, s_kv=None, kv_lens=None) -> AttendArgs:
    """k_codes / v_codes [B, H_kv, rows, n_sub]: the first s_kv rows (all when
    None) are the cache; kv_lens: optional device int32 [B] per-batch lengths."""
    B, H_q, S_q, D = q.shape
    _, H_kv, rows, _ = k_codes.shape
    if v_codes.shape[2] != rows:
        raise ValueError("k_codes and v_codes must have the same row count")
    S_kv = rows if s_kv is None else int(s_kv)
    if kv_lens is not None and (kv_lens.dtype != torch.int32 or not kv_lens.is_contiguous()
                                or kv_lens.numel() != B):
        raise ValueError("kv_lens must be a contiguous int32 tensor of B elements")
    a = AttendArgs()
    a.B, a.H_q, a.H_kv, a.S_q, a.S_kv, a.D = B, H_q, H_kv, S_q, S_kv, D
    a.q_f16 = q.data_ptr()
    a.k_codes = k_codes.data_ptr()
    a.k_code_bytes = _code_bytes(k_codes)
    a.k_codebook = k_codebook.data_ptr()
    a.k_n_centroids, a.k_sub_dim = k_codebook.shape
    a.v_codes = v_codes.data_ptr()
    a.v_code_bytes = _code_bytes(v_codes)
    a.v_codebook = v_codebook.data_ptr()
    a.v_n_centroids, a.v_sub_dim = v_codebook.shape
    a.smooth = 0 if smooth is None else smooth.data_ptr()
    a.smooth_mode = _smooth_mode(smooth)
    a.scale = float(scale)
    a.causal = int(bool(causal))
    a.sliding_window = int(sliding_window)
    a.out_f16 = 0 if out is None else out.data_ptr()
    a.workspace = 0 if workspace is None else workspace.data_ptr()
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    a.kv_stride = rows
    a.kv_lens = 0 if kv_lens is None else kv_lens.data_ptr()
    return a


def attend_workspace_bytes(args: AttendArgs) -> int:
    return int(lib().vq_attend_workspace_bytes(ctypes.byref(args)))


def _attend(fn_name, q, k_codes, k_codebook, v_codes, v_codebook, smooth,
            scale=None, causal=True, sliding_window=0, out=None,
            workspace=None, stream=None, s_kv=None, kv_lens=None):
    D = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    a = make_attend_args(q, k_codes, k_codebook, v_codes, v_codebook, smooth,
                         scale, causal, sliding_window, out, workspace, s_kv, kv_lens)
    if workspace is None:
        need = attend_workspace_bytes(a)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            a.workspace = workspace.data_ptr()
            a.workspace_bytes = need
    st = getattr(lib(), fn_name)(ctypes.byref(a), _stream(stream))
    _check(st, fn_name)
    return out


def decode_attend(q, k_codes, k_codebook, v_codes, v_codebook, smooth,
                  scale=None, causal=True, sliding_window=0, out=None,
                  workspace=None, stream=None, s_kv=None, kv_lens=None) -> torch.Tensor:
    """vq_decode_attend; raw q [B, H_q, S_q, D] fp16 -> out (same shape).
    s_kv: cached rows of the code buffers (all when None); kv_lens: optional
    device int32 [B] per-batch lengths."""
    return _attend("vq_decode_attend", q, k_codes, k_codebook, v_codes,
                   v_codebook, smooth, scale, causal, sliding_window, out,
                   workspace, stream, s_kv, kv_lens)


def decode_step(q, k_new, v_new, k_codes, k_codebook, v_codes, v_codebook, smooth,
                scale=None, causal=True, sliding_window=0, out=None, workspace=None,
                stream=None, s_kv=None) -> torch.Tensor:
    """vq_decode_step: encode k_new / v_new [B, H_kv, S_q, D] into rows
    s_kv - S_q .. s_kv - 1 of the code buffers, then attend (one launch)."""
    D = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    for t in (k_new, v_new):
        if t.dtype != torch.float16 or not t.is_contiguous():
            raise VQError(VQ_ERR_SHAPE, "k_new / v_new must be contiguous fp16")
    a = make_attend_args(q, k_codes, k_codebook, v_codes, v_codebook, smooth, scale, causal,
                         sliding_window, out, workspace, s_kv, None)
    if workspace is None:
        need = attend_workspace_bytes(a)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            a.workspace = workspace.data_ptr()
            a.workspace_bytes = need
    st = lib().vq_decode_step(ctypes.byref(a), k_new.data_ptr(), v_new.data_ptr(),
                              _stream(stream))
    _check(st, "vq_decode_step")
    return out


def prefill_attend(q, k_codes, k_codebook, v_codes, v_codebook, smooth,
                   scale=None, causal=True, sliding_window=0, out=None,
                   workspace=None, stream=None, s_kv=None, kv_lens=None) -> torch.Tensor:
    """vq_prefill_attend (tensor-core path for S_q >= 64); s_kv and kv_lens
    as in decode_attend."""
    return _attend("vq_prefill_attend", q, k_codes, k_codebook, v_codes,
                   v_codebook, smooth, scale, causal, sliding_window, out,
                   workspace, stream, s_kv, kv_lens)
