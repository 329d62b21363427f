"""GPU: the approximation-error diagnostic through the C ABI.  Full softmax attention against
the oracle's, the per-slice relative Frobenius error against the oracle's metric, and the
diagnostic itself (anchor attention against full attention on deit_base-style inputs, whose
anchors are rows of the keys plus noise) against the same computed by the oracle."""
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


def _inputs(dtype, B, heads, n, m, d, seed):
    w = gen.WORKLOADS["deit_base"].with_(name="diag", B=B, heads=heads, n=n, m=m, d=d, dtype=dtype)
    x = gen.make_inputs(w, seed=seed)
    x["K"] = gen.make_keys(w, seed=seed)
    return w, x


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 3, 197, 49, 64), (1, 2, 1100, 64, 128), (3, 1, 1, 8, 16), (2, 2, 63, 8, 32),
                                   (1, 1, 65, 8, 64), (1, 2, 200, 8, 64)])
def test_full_attention_matches_oracle(env, dtype, shape):
    pkg, torch, orc = env
    w, x = _inputs(dtype, *shape, seed=sum(shape))
    t = {k: to_device(x[k], dtype, torch) for k in "QKV"}
    H = pkg.full_forward(t["Q"], t["K"], t["V"], scale=w.scale)
    torch.cuda.synchronize()
    ref = orc.full_attention(*(gen.to_float64(x[k], dtype) for k in "QKV"), w.scale)
    assert_parity(to_host64(H), ref, dtype, f"full attention {dtype} {shape}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_relative_error_metric(env, dtype):
    pkg, torch, orc = env
    w, x = _inputs(dtype, 3, 2, 300, 49, 64, seed=4)
    t = {k: to_device(x[k], dtype, torch) for k in "QUV"}
    Ha = pkg.forward(t["Q"], t["U"], t["V"], scale=w.scale)
    Hb = pkg.forward(t["Q"], t["U"], t["Q"], scale=w.scale)  # any second tensor of the shape
    err = pkg.relative_error(Ha, Hb)
    torch.cuda.synchronize()
    ref = orc.relative_frobenius(to_host64(Ha), to_host64(Hb))
    assert np.allclose(err.double().cpu().numpy(), ref, rtol=1e-5, atol=1e-7)
    zero = pkg.relative_error(Ha, Ha)
    assert float(zero.abs().max()) == 0.0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_diagnostic_matches_oracle(env, dtype):
    """||H_full - H_anchor||_F / ||H_full||_F per slice, the GPU's against the oracle's."""
    pkg, torch, orc = env
    w, x = _inputs(dtype, 4, 12, 197, 49, 64, seed=0)
    t = {k: to_device(x[k], dtype, torch) for k in "QUVK"}
    Hf = pkg.full_forward(t["Q"], t["K"], t["V"], scale=w.scale)
    Ha = pkg.forward(t["Q"], t["U"], t["V"], scale=w.scale)
    err = pkg.relative_error(Hf, Ha).double().cpu().numpy()
    xx = {k: gen.to_float64(x[k], dtype) for k in "QUVK"}
    ref = orc.relative_frobenius(orc.full_attention(xx["Q"], xx["K"], xx["V"], w.scale),
                                 orc.forward(xx["Q"], xx["U"], xx["V"], w.scale))
    tol = 1e-5 + 1e-5 * ref if dtype == "f32" else 5e-3 + 2e-2 * ref
    assert np.all(np.abs(err - ref) <= tol), f"max difference {np.abs(err - ref).max():.3e} (errors {ref.min():.3f}..{ref.max():.3f})"
