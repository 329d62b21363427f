"""GPU: the tensor-core variant's schedules and its bounded waits, through the C ABI.

Pass 2 either reads back the A tiles pass 1 stored or recomputes A from Q; the recomputing
plan also takes pass-2 work most-recently-reduced slice first.  The workloads pick it only
when every slice's A copy would not fit half of L2, so the test entry forces it on small
shapes here: the result must match the oracle, and be bit-identical to the stored-A plan's
(same chunks; both pass the same bf16 A to the same MMAs).

The bounded waits are exercised the allowed way: the test entry keeps one slice's W' from
ever being published, with a 1 ms limit on waits for other CTAs.  The waits for it give up,
set bit 1 of the device error word and the CTAs leave; the next normal call on the same
context must be correct.
"""
import numpy as np
import pytest

import gen
from tests.conftest import gpu_available
from tests.gpu_util import assert_slices, oracle_slices, to_device

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch
    import linear_complexity_anchor_gb300 as pkg
    pkg.load()
    assert pkg.device_error() == 0
    return pkg, torch, oracle_mod


def _w(B, heads, n, m, d):
    return gen.WORKLOADS["det_800x1344"].with_(name="sched", B=B, heads=heads, n=n, m=m, d=d)


def _test_call(pkg, torch, t, w, H, hold=-1, wait_ns=2_000_000_000, force_recompute=True):
    st = pkg.anchor_attn_test_forward_ptr(t["Q"].data_ptr(), t["U"].data_ptr(), t["V"].data_ptr(), H.data_ptr(),
                                          w.B, w.heads, w.n, w.m, w.d, w.scale, hold, wait_ns, force_recompute, 0)
    torch.cuda.synchronize()
    return st


def _oracle_slices(orc, x, w, H, picks, what):
    assert_slices(H.cpu(), w, oracle_slices(orc, w, x, picks), what)


# (B, heads, n, m, d): ragged last tiles, masked anchors, both D, chunk counts from 2 to 33;
# the last four give most CTAs several pass-1 and pass-2 items, which interleave pass-1 and
# pass-2 tiles of different slices in one CTA (the single-A-buffer layouts share nothing
# between them: H is staged in the epilogue's own buffer)
_RECOMPUTE = [(1, 4, 4096, 64, 64), (2, 3, 4200, 64, 64), (1, 2, 1100, 49, 64), (2, 2, 3000, 100, 64),
           (1, 3, 2500, 128, 128), (2, 2, 5000, 33, 128), (1, 1, 16384, 128, 128), (3, 1, 700, 64, 64),
           (4, 4, 8192, 64, 128), (4, 4, 8192, 128, 128), (8, 4, 4096, 64, 64), (16, 8, 2048, 100, 64)]


@pytest.mark.parametrize("shape", _RECOMPUTE)
def test_recompute_plan_matches_oracle_and_stored_plan(env, shape):
    pkg, torch, orc = env
    w = _w(*shape)
    plan = pkg.query_plan("bf16", *shape)
    assert plan["variant"] in ("umma", "stream", "split_tc")
    x = gen.make_inputs(w, seed=sum(shape))
    t = {k: to_device(x[k], "bf16", torch) for k in "QUV"}
    H = torch.full_like(t["Q"], float("nan"))
    assert _test_call(pkg, torch, t, w, H) == 0
    assert pkg.device_error() == 0
    _oracle_slices(orc, x, w, H, range(w.slices), "recompute")
    H2 = pkg.forward(t["Q"], t["U"], t["V"], scale=w.scale)
    torch.cuda.synchronize()
    if plan["variant"] == "umma":
        assert torch.equal(H.view(torch.int16), H2.view(torch.int16)), \
            f"recompute and {'stored' if plan['stored_a'] else 'default'} plans differ"
    else:  # another kernel and summation order: against the oracle instead
        _oracle_slices(orc, x, w, H2, range(w.slices), plan["variant"])


def test_workload_plans(env):
    pkg, _, _ = env
    w = gen.WORKLOADS["long_16k"]
    assert not pkg.query_plan("bf16", w.B, w.heads, w.n, w.m, w.d)["stored_a"]
    w = gen.WORKLOADS["det_800x1344"]
    assert pkg.query_plan("bf16", w.B, w.heads, w.n, w.m, w.d)["stored_a"]


@pytest.mark.parametrize("force_recompute", [True, False])
def test_wait_for_a_held_reduction_gives_up(env, force_recompute):
    """One slice's W' is never published and waits for other CTAs are limited to 1 ms: the
    waits give up (bit 1), the kernel ends, and the context stays usable."""
    pkg, torch, orc = env
    w = _w(1, 4, 4096, 64, 64)
    x = gen.make_inputs(w, seed=77)
    t = {k: to_device(x[k], "bf16", torch) for k in "QUV"}
    H = torch.zeros_like(t["Q"])
    assert _test_call(pkg, torch, t, w, H, hold=2, wait_ns=1_000_000, force_recompute=force_recompute) == 0
    code = pkg.device_error()
    assert code & 2, f"device error word {code:#x}: the held reduction's wait did not give up"
    assert pkg.device_error() == 0, "reading the error word clears it"
    # the same context runs the next call correctly
    H2 = pkg.forward(t["Q"], t["U"], t["V"], scale=w.scale)
    torch.cuda.synchronize()
    assert pkg.device_error() == 0
    _oracle_slices(orc, x, w, H2, range(w.slices), "after a held call")


def test_test_entry_rejects_other_variants(env):
    pkg, torch, _ = env
    w = _w(1, 1, 300, 20, 64)      # m < 32: CUDA-core variant
    Q = torch.zeros((1, 1, 300, 64), dtype=torch.bfloat16, device="cuda")
    U = torch.zeros((1, 20, 64), dtype=torch.bfloat16, device="cuda")
    H = torch.zeros_like(Q)
    st = pkg.anchor_attn_test_forward_ptr(Q.data_ptr(), U.data_ptr(), Q.data_ptr(), H.data_ptr(), 1, 1, 300, 20, 64,
                                          w.scale, -1, 1000, True, 0)
    assert st == 2
    st = pkg.anchor_attn_test_forward_ptr(Q.data_ptr(), U.data_ptr(), Q.data_ptr(), H.data_ptr(), 1, 1, 300, 20, 64,
                                          w.scale, -1, 0, True, 0)
    assert st == 1
