"""GPU: the masked (causal) variant through the C ABI against the oracle's, element by element,
plus the properties that hold at any size: the last row equals the unmasked forward's, the
first row is its own value, and changing later tokens leaves earlier rows unchanged."""
import numpy as np
import pytest

import gen
from tests.conftest import gpu_available
from tests.gpu_util import assert_parity, to_device, to_host64, widen

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch
    import linear_complexity_anchor_gb300 as pkg
    pkg.load()
    return pkg, torch, oracle_mod


def _w(dtype, B, heads, n, m, d):
    return gen.WORKLOADS["vit14_f32"].with_(name="causal", B=B, heads=heads, n=n, m=m, d=d, dtype=dtype)


_SHAPES = [(1, 1, 196, 16, 64), (2, 3, 197, 49, 64), (1, 2, 1100, 64, 64), (1, 2, 700, 128, 128), (2, 2, 65, 30, 32),
           (3, 1, 1, 8, 16), (1, 1, 2, 5, 16), (1, 2, 1537, 100, 64)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", _SHAPES)
def test_causal_matches_oracle(env, dtype, shape):
    pkg, torch, orc = env
    w = _w(dtype, *shape)
    x = gen.make_inputs(w, seed=sum(shape))
    t = {k: to_device(x[k], dtype, torch) for k in "QUV"}
    H = pkg.causal_forward(t["Q"], t["U"], t["V"], scale=w.scale)
    Hf = pkg.forward(t["Q"], t["U"], t["V"], scale=w.scale)
    torch.cuda.synchronize()
    xx = widen(x, dtype)
    assert_parity(to_host64(H), orc.causal(xx["Q"], xx["U"], xx["V"], w.scale), dtype, f"causal {dtype} {shape}")
    assert pkg.device_error() == 0
    # the last token sees every token; the first only itself
    assert_parity(to_host64(H[:, :, -1]), to_host64(Hf[:, :, -1]), dtype, "last row against the forward")
    assert_parity(to_host64(H[:, :, 0]), gen.to_float64(x["V"], dtype)[:, :, 0], dtype, "first row")


def test_causal_ignores_later_tokens(env):
    pkg, torch, _ = env
    w = _w("bf16", 2, 2, 1300, 64, 64)
    x = gen.make_inputs(w, seed=21)
    t = {k: to_device(x[k], "bf16", torch) for k in "QUV"}
    H1 = pkg.causal_forward(t["Q"], t["U"], t["V"], scale=w.scale)
    Q2, V2 = t["Q"].clone(), t["V"].clone()
    Q2[:, :, 900:] += 1.0
    V2[:, :, 900:] -= 1.0
    H2 = pkg.causal_forward(Q2, t["U"], V2, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(H1[:, :, :900].view(torch.int16), H2[:, :, :900].view(torch.int16))
    assert not torch.equal(H1[:, :, 900:], H2[:, :, 900:])
