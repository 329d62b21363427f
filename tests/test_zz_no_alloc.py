"""The allocation-free entry point, anchor_attn_forward_static_scratch.

It serves callers that may not allocate device memory during a call (an engine plugin's
enqueue step, a loop with a fixed memory budget): its workspace is a fixed array compiled
into the library.  Checked here through the C ABI against the oracle and against
anchor_attn_forward on the same inputs, on two calls in a row (the second on other data, so
stale contents of the shared array would show), and for the size limit.  Collected last on
purpose.
"""
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


def _inputs(torch, w, seed):
    x = gen.make_inputs(w, seed=seed)
    return x, {k: to_device(x[k], "bf16", torch) for k in "QUV"}


@pytest.mark.parametrize("shape", [(2, 3, 1100, 40, 64), (1, 4, 2000, 20, 64), (2, 2, 700, 128, 128),
                                   (3, 2, 197, 30, 64)])
def test_static_scratch_matches_oracle(env, shape):
    pkg, torch, orc = env
    B, heads, n, m, d = shape
    w = gen.WORKLOADS["vit14_f32"].with_(name="noalloc", B=B, heads=heads, n=n, m=m, d=d, dtype="bf16")
    for call, seed in enumerate((31, 32)):
        x, t = _inputs(torch, w, seed)
        H_ref = torch.empty_like(t["Q"])
        H_new = torch.full_like(t["Q"], float("nan"))
        args = (t["Q"].data_ptr(), t["U"].data_ptr(), t["V"].data_ptr())
        st_ref = pkg.anchor_attn_forward_ptr(*args, H_ref.data_ptr(), B, heads, n, m, d, w.scale, 0)
        st_new = pkg.anchor_attn_forward_static_scratch_ptr(*args, H_new.data_ptr(), B, heads, n, m, d, w.scale, 0)
        torch.cuda.synchronize()
        assert st_ref == 0 and st_new == 0, (st_ref, st_new)
        xx = widen(x, "bf16")
        ref = orc.forward(xx["Q"], xx["U"], xx["V"], w.scale)
        assert_parity(to_host64(H_new), ref, "bf16", f"static scratch call {call + 1} against the oracle")
        assert_parity(to_host64(H_new), to_host64(H_ref), "bf16", f"static scratch call {call + 1} against the forward")


def test_static_scratch_rejects_oversize(env):
    pkg, torch, _ = env
    cap = pkg.static_scratch_bytes()
    assert cap == 16 << 20
    # 64 slices x 32 chunks x (128*128 + 128) floats >> 16 MiB
    B, heads, n, m, d = 4, 16, 16384, 128, 128
    need = 4 * B * heads * (((n + 511) // 512) * (m * d + m) + m * d)
    assert need > cap
    Q = torch.zeros((B, heads, n, d), dtype=torch.bfloat16, device="cuda")
    U = torch.zeros((heads, m, d), dtype=torch.bfloat16, device="cuda")
    H = torch.full_like(Q, 7.0)
    st = pkg.anchor_attn_forward_static_scratch_ptr(Q.data_ptr(), U.data_ptr(), Q.data_ptr(), H.data_ptr(),
                                                    B, heads, n, m, d, 0.1, 0)
    torch.cuda.synchronize()
    assert st == 6 and pkg.status_string(st).startswith("problem exceeds")
    assert bool((H == 7.0).all())
