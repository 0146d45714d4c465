"""rk_segpaged_decode_noalloc: decode for callers that cannot allocate device memory (a
plugin whose host hands it no allocator, or a latency-critical caller that must not call
cudaMalloc).  Its scratch is a fixed array inside the library; its results must match
rk_segpaged_decode run with a caller workspace, on two calls in a row (the array keeps
the previous call's contents, which must not leak into the next call).

Collected last on purpose, so a run that stops at the first failure has run every other
test first.  It passes on its own in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import rk_oracle as O
from workloads import synth
from workloads.device import attn_to_device

pytestmark = pytest.mark.gpu

ATOL, RTOL_L2 = 3e-2, 5e-3   # the attention tolerance of the parity tests


@pytest.fixture(scope="module")
def rk():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from head_aware_paged_rope_b300 import build as b
    b.build()
    import head_aware_paged_rope_b300 as m
    f = m.LIB.rk_segpaged_decode_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(m.AttnArgs), ctypes.c_void_p]
    return m


def _close(a, b):
    a, b = a.float().cpu().numpy(), b.float().cpu().numpy()
    assert np.abs(a - b).max() <= ATOL
    assert np.linalg.norm(a - b) <= RTOL_L2 * max(np.linalg.norm(b), 1e-30)


def test_noalloc_decode_matches_workspace_decode_twice(rk):
    stream = torch.cuda.current_stream().cuda_stream
    batches = [synth.decode_microbench(B=6, ctx=3001, Hq=32, Hkv=8, window=256, sink=4, seed=7).attn,
               synth.decode_microbench(B=3, ctx=1500, Hq=32, Hkv=8, window=100, sink=0, seed=8).attn]
    for batch in batches:   # two calls in a row, different sizes, the second reusing the array
        ref = attn_to_device(batch, "cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        rk.segpaged_decode(ref.args(rk, decode=True, status=st))
        got = attn_to_device(batch, "cuda")
        got.out.fill_(float("nan"))
        got.lse.fill_(float("nan"))
        code = rk.LIB.rk_segpaged_decode_noalloc(ctypes.byref(got.args(rk, decode=True, status=st)), stream)
        torch.cuda.synchronize()
        assert code == 0 and int(st.item()) == 0
        _close(got.out, ref.out)
        assert torch.allclose(got.lse, ref.lse, atol=1e-3, rtol=0)
        # and against the oracle, on a few rows
        res = O.segpaged_attention(batch, rows=[(0, 0), (batch.B - 1, batch.Hkv - 1)])
        G = batch.Hq // batch.Hkv
        for (t, h), (o, _) in res.items():
            assert np.abs(got.out[t, h * G:(h + 1) * G].float().cpu().numpy() - o).max() <= ATOL


def test_noalloc_decode_rejects_sizes_beyond_its_scratch(rk):
    # 4096 sequences x 8 KV heads need far more than the fixed scratch: rejected before any launch
    a = rk.AttnArgs(q=1, cu_seqlens_q=None, seq_len=1, k_pool=1, v_pool=1, n_pool_pages=10, page_table=1,
                    page_logical=None, n_pages=1, head_class=1, window=1, sink=None, B=4096, Hq=64, Hkv=8,
                    d=128, P=16, max_pages=4, total_q=4096, max_q=1, scale=0.0, out=1, lse=None, status=None)
    assert rk.segpaged_decode_workspace_size(a) > (16 << 20)
    assert rk.LIB.rk_segpaged_decode_noalloc(ctypes.byref(a), None) == 2   # RK_ERR_UNSUPPORTED
