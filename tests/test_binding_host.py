"""Host logic of the ctypes binding that needs no GPU: how the attention
arguments are marshalled into the C struct (vq_attend_args of vqkv.h)."""
import pytest
import torch

from product_vq_compressed_gb300 import binding as vq


def test_attend_args_marshalling():
    """The binding's argument marshalling on CPU tensors: sizes from the
    shapes, code widths from the dtypes (uint8 1, uint16 2, int32 rows of
    packed codes 0), the smooth layout from its rank, the cache rows as
    kv_stride with s_kv counting the attended ones, flags and pointers."""
    q = torch.zeros((2, 8, 3, 128), dtype=torch.float16)
    kc = torch.zeros((2, 4, 50, 5), dtype=torch.int32)        # packed 10-bit keys
    vc = torch.zeros((2, 4, 50, 32), dtype=torch.uint8)
    kcb = torch.zeros((1000, 8))
    vcb = torch.zeros((256, 4))
    out = torch.zeros_like(q)
    ws = torch.zeros(64, dtype=torch.uint8)
    lens = torch.tensor([40, 45], dtype=torch.int32)
    for smooth, mode in ((None, 0), (torch.ones(128), 1), (torch.ones(4, 128), 2)):
        a = vq.make_attend_args(q, kc, kcb, vc, vcb, smooth, 0.25, causal=False,
                                sliding_window=7, out=out, workspace=ws, s_kv=45, kv_lens=lens)
        assert (a.B, a.H_q, a.H_kv, a.S_q, a.S_kv, a.D) == (2, 8, 4, 3, 45, 128)
        assert (a.k_code_bytes, a.v_code_bytes) == (0, 1)
        assert (a.k_n_centroids, a.k_sub_dim, a.v_n_centroids, a.v_sub_dim) == (1000, 8, 256, 4)
        assert a.smooth_mode == mode and (a.smooth or 0) == (0 if smooth is None else smooth.data_ptr())
        assert a.kv_stride == 50 and a.causal == 0 and a.sliding_window == 7
        assert abs(a.scale - 0.25) < 1e-7
        assert a.workspace == ws.data_ptr() and a.workspace_bytes == 64
        assert a.kv_lens == lens.data_ptr() and a.out_f16 == out.data_ptr()
    a = vq.make_attend_args(q, torch.zeros((2, 4, 50, 16), dtype=torch.uint16), kcb, vc, vcb,
                            None, 1.0)
    assert a.k_code_bytes == 2 and a.S_kv == 50 and a.kv_lens is None and a.workspace is None
    with pytest.raises(ValueError):
        vq.make_attend_args(q, kc, kcb, vc[:, :, :49], vcb, None, 1.0)
    with pytest.raises(ValueError):
        vq.make_attend_args(q, kc, kcb, vc, vcb, None, 1.0, kv_lens=lens.to(torch.int64))
