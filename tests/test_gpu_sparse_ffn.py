"""GPU parity of the token-level sparse FFN (rk_sparse_ffn, through the C ABI) against the
fp64 oracle: the kept tokens bit for bit (index work), FFN outputs of kept tokens within
max-abs 3e-2 and relative L2 5e-3 (bf16 output; the gated activation is rounded to bf16
before W_down), and exact zeros for the skipped tokens ("小红书 RedKnot", section 3, third
component)."""
import numpy as np
import pytest
import torch

from oracle import rk_oracle as O
from workloads import synth
from workloads.device import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rk():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from head_aware_paged_rope_b300 import build as b
    b.build()
    import head_aware_paged_rope_b300 as m
    return m


def _run(rk, w):
    dev = "cuda"
    x = to_device(w.x, dev)
    out = torch.full(x.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    kept = torch.full((max(w.keep, 1),), -1, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    args = rk.sparse_ffn_args(x, torch.from_numpy(w.importance).to(dev), to_device(w.w_gate, dev),
                              to_device(w.w_up, dev), to_device(w.w_down, dev), out, kept, keep=w.keep, status=st)
    rk.sparse_ffn(args)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out.float().cpu().numpy(), kept.cpu().numpy()[:w.keep]


def _check(w, out, kept, rows=None):
    want, ref = O.sparse_ffn(w.x, w.importance, w.keep, w.w_gate, w.w_up, w.w_down, rows=rows)
    assert np.array_equal(kept, want)
    skipped = np.ones(len(w.importance), dtype=bool)
    skipped[want] = False
    assert np.all(out[skipped] == 0)
    if ref:
        got = np.stack([out[t] for t in ref])
        exp = np.stack(list(ref.values()))
        assert np.abs(got - exp).max() <= 3e-2
        assert np.linalg.norm(got - exp) <= 5e-3 * np.linalg.norm(exp)


@pytest.mark.parametrize("T,d_model,d_ff,frac", [(300, 256, 512, 0.46), (2000, 1024, 2048, 0.5), (129, 512, 384, 1.0)])
def test_sparse_ffn_small(rk, T, d_model, d_ff, frac):
    # ragged M tiles (kept counts not multiples of 128), several N tiles and K steps
    w = synth.sparse_ffn_workload(seed=T, T=T, d_model=d_model, d_ff=d_ff, keep_frac=frac)
    out, kept = _run(rk, w)
    _check(w, out, kept)


def test_sparse_ffn_ties_and_nothing_kept(rk):
    w = synth.sparse_ffn_workload(seed=3, T=1000, d_model=256, d_ff=256, keep_frac=0.31, ties=True)
    assert len(np.unique(w.importance)) < 200                       # many equal scores
    out, kept = _run(rk, w)
    _check(w, out, kept)
    w.keep = 0
    out, _ = _run(rk, w)
    assert np.all(out == 0)


@pytest.mark.slow
def test_sparse_ffn_qwen3_32b_shape_sampled(rk):
    # the full Qwen3-32B feed-forward block over 4096 tokens, half kept; sampled rows
    w = synth.sparse_ffn_workload()
    out, kept = _run(rk, w)
    rng = np.random.default_rng(5)
    rows = rng.choice(len(w.importance), 24, replace=False).tolist()
    _check(w, out, kept, rows=rows)
