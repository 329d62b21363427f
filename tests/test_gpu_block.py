"""GPU: the block front end (Q = X Wq^T and V = X Wv^T per head, then the forward, in one
tensor-core kernel) through the C ABI against the oracle's, element by element, on small
shapes with ragged tiles and on the two ViT block workloads at full size (every slice); plus
bit-stability, the guard band after H and the rejected calls."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import gen
from tests.conftest import gpu_available
from tests.gpu_util import assert_parity, to_device, to_host64

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch
    import linear_complexity_anchor_gb300 as pkg
    pkg.load()
    return pkg, torch, oracle_mod


def _bw(B, heads, n, m, dm, recipe="normal"):
    base = gen.WORKLOADS["deit_base"].with_(name="block", B=B, heads=heads, n=n, m=m, d=64, recipe=recipe)
    return gen.BlockWorkload("block", base, dm, "test shape")


def _device(x, torch):
    return {k: to_device(v, "bf16", torch) for k, v in x.items()}


def _oracle(orc, bw, x, slices=None):
    """Oracle H of the listed slices (all by default), one slice per host thread."""
    w = bw.w
    X = gen.to_float64(x["X"], "bf16")
    Wq, Wv, U = (gen.to_float64(x[k], "bf16") for k in ("Wq", "Wv", "U"))
    slices = range(w.slices) if slices is None else slices

    def one(s):
        b, h = divmod(s, w.heads)
        return s, orc.block_slice(X[b], Wq[h], Wv[h], U[h], w.scale)

    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        return dict(ex.map(one, list(slices)))


def _check(H, bw, refs, what):
    w = bw.w
    Hc = H.cpu()
    for s, ref in sorted(refs.items()):
        b, h = divmod(s, w.heads)
        assert_parity(to_host64(Hc[b, h]), ref, "bf16", f"{what} slice ({b},{h})")


# (B, heads, n, m, dm): one 64-column chunk; the DeiT-Base width; exactly one tile; a second
# tile of one token; a single token and a single anchor; two full tiles; long chunk loops;
# few anchors
_SHAPES = [(1, 1, 196, 16, 64), (2, 3, 197, 49, 768), (2, 2, 128, 64, 128), (1, 2, 129, 32, 192),
           (3, 1, 1, 1, 64), (2, 6, 256, 30, 384), (1, 2, 77, 64, 1024), (2, 2, 200, 5, 512)]


@pytest.mark.parametrize("shape", _SHAPES)
def test_block_matches_oracle(env, shape):
    pkg, torch, orc = env
    bw = _bw(*shape)
    x = gen.make_block_inputs(bw, seed=sum(shape))
    t = _device(x, torch)
    H = pkg.block_forward(t["X"], t["Wq"], t["Wv"], t["U"], scale=bw.w.scale)
    torch.cuda.synchronize()
    assert pkg.device_error() == 0
    _check(H, bw, _oracle(orc, bw, x), f"block {shape}")


@pytest.mark.parametrize("name", sorted(gen.BLOCK_WORKLOADS))
def test_block_workload_every_slice(env, name):
    """The bench's launch (full size), every slice against the oracle."""
    pkg, torch, orc = env
    bw = gen.BLOCK_WORKLOADS[name]
    x = gen.make_block_inputs(bw, seed=0)
    t = _device(x, torch)
    H = pkg.block_forward(t["X"], t["Wq"], t["Wv"], t["U"], scale=bw.w.scale)
    torch.cuda.synchronize()
    assert pkg.device_error() == 0
    for s0 in range(0, bw.w.slices, 256):
        _check(H, bw, _oracle(orc, bw, x, range(s0, min(bw.w.slices, s0 + 256))), name)


def test_block_bit_stable_and_guard_band(env):
    pkg, torch, _ = env
    bw = _bw(3, 4, 150, 40, 256)
    w = bw.w
    x = gen.make_block_inputs(bw, seed=5)
    t = _device(x, torch)
    numel = w.slices * w.n * w.d
    buf = torch.full((numel + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    H = buf[:numel].view(w.B, w.heads, w.n, w.d)
    pkg.block_forward(t["X"], t["Wq"], t["Wv"], t["U"], H=H, scale=w.scale)
    H2 = pkg.block_forward(t["X"], t["Wq"], t["Wv"], t["U"], scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(H.view(torch.int16), H2.view(torch.int16))
    assert bool((buf[numel:] == 7.0).all()), "the kernel wrote past the end of H"
    assert pkg.device_error() == 0


def test_block_constant_values_and_rejections(env):
    """All value weights on one embedding column and that column constant per batch entry:
    V is constant over the tokens, so every H row equals it; then rejected calls leave
    nothing behind and a valid call still matches."""
    pkg, torch, orc = env
    bw = _bw(2, 2, 180, 20, 128)
    w = bw.w
    x = gen.make_block_inputs(bw, seed=9)
    X = gen.bf16_to_f32(x["X"]).copy()
    X[:, :, 3] = np.array([1.5, -0.75])[:, None]
    x["X"] = gen.round_bf16(X)
    Wv = np.zeros(x["Wv"].shape, dtype=np.float32)
    Wv[:, :, 3] = 0.5
    x["Wv"] = gen.round_bf16(Wv)
    t = _device(x, torch)
    H = pkg.block_forward(t["X"], t["Wq"], t["Wv"], t["U"], scale=w.scale)
    torch.cuda.synchronize()
    want = np.broadcast_to(np.array([0.75, -0.375])[:, None, None, None], (w.B, w.heads, w.n, w.d))
    assert_parity(to_host64(H), want, "bf16", "constant values")
    bad = pkg.anchor_attn_block_forward_ptr(t["X"].data_ptr(), t["Wq"].data_ptr(), t["Wv"].data_ptr(),
                                            t["U"].data_ptr(), t["X"].data_ptr(), w.B, w.heads, w.n, w.m, 64, 128,
                                            w.scale, 0)
    assert bad == 3  # H on top of X
    assert pkg.anchor_attn_block_forward_ptr(0, 0, 0, 0, 0, w.B, w.heads, 300, w.m, 64, 128, w.scale, 0) == 2
    torch.cuda.synchronize()
    assert pkg.device_error() == 0
    H2 = pkg.block_forward(t["X"], t["Wq"], t["Wv"], t["U"], scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(H.view(torch.int16), H2.view(torch.int16))
