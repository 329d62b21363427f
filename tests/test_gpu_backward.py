"""GPU: the backward (dQ, dU, dV) through the C ABI against the oracle's backward, element by
element, on the same seeded inputs (the oracle's backward is pinned by finite differences of
the forward oracle in test_oracle_backward_pins.py).  bf16 with d = 64 or 128 and m <= 128 runs
on the tensor cores (one CTA per slice at d = 64 with m <= 64, runs of tiles over every SM
otherwise); the rest, and fp32, on CUDA cores."""
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
    assert pkg.device_error() == 0
    return pkg, torch, oracle_mod


def _case(env, dtype, B, heads, n, m, d, seed, dH=None, scale=None):
    pkg, torch, orc = env
    w = gen.WORKLOADS["vit14_f32"].with_(name="bwd", B=B, heads=heads, n=n, m=m, d=d, dtype=dtype)
    x = gen.make_inputs(w, seed=seed)
    if dH is None:
        dH = gen.make_inputs(w.with_(name="bwd_dh"), seed=seed + 1000)["V"]
    t = {k: to_device(x[k], dtype, torch) for k in "QUV"}
    tdH = to_device(dH, dtype, torch)
    sc = w.scale if scale is None else scale
    dQ, dU, dV = pkg.backward(t["Q"], t["U"], t["V"], tdH, scale=sc)
    torch.cuda.synchronize()
    ref = orc.backward(*(gen.to_float64(a, dtype) for a in (x["Q"], x["U"], x["V"], dH)), sc)
    return (dQ, dU, dV), ref, (t, tdH, sc)


_SHAPES = [(1, 1, 196, 16, 64), (2, 3, 197, 30, 64), (1, 2, 700, 64, 64), (2, 2, 1100, 20, 64),
           (1, 2, 513, 128, 128), (2, 1, 129, 49, 128), (3, 2, 7, 1, 16), (1, 1, 2, 33, 32), (1, 2, 300, 256, 64)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", _SHAPES)
def test_backward_matches_oracle(env, dtype, shape):
    got, ref, _ = _case(env, dtype, *shape, seed=sum(shape))
    bar = "f32_bwd" if dtype == "f32" else dtype
    for name, g, r in zip(("dQ", "dU", "dV"), got, ref):
        assert_parity(to_host64(g), r, bar, f"{name} {dtype} {shape}")
    assert env[0].device_error() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_constant_upstream_rows(env, dtype):
    """dH with constant rows: dQ = dU = 0 and dV = dH (S_t keeps column sums)."""
    w = gen.WORKLOADS["vit14_f32"].with_(name="bwd", B=2, heads=2, n=600, m=40, d=64, dtype=dtype)
    x = gen.make_inputs(w, seed=3)
    dH = np.ascontiguousarray(np.broadcast_to(x["V"][:, :, :1, :], x["V"].shape))
    (dQ, dU, dV), ref, _ = _case(env, dtype, 2, 2, 600, 40, 64, seed=3, dH=dH)
    bar = "f32_bwd" if dtype == "f32" else dtype
    for name, g, r in zip(("dQ", "dU", "dV"), (dQ, dU, dV), ref):
        if name == "dV":
            assert_parity(to_host64(g), r, bar, f"{name} constant rows")
        else:  # exactly zero in exact arithmetic: rounding only, against the gradients' scale
            scale = float(np.abs(gen.to_float64(dH, dtype)).max())
            assert float(to_host64(g).__abs__().max()) <= (1e-5 if dtype == "f32" else 1e-2) * scale, name
    assert_parity(to_host64(dV), gen.to_float64(dH, dtype), bar, "dV = dH")


# tensor-core path: one token; exactly one tile; a second tile of one token; a long slice;
# one anchor; many batch entries summed into dU
_TC_SHAPES = [(3, 2, 1, 7, 64), (2, 2, 128, 64, 64), (1, 3, 129, 49, 64), (1, 1, 2000, 64, 64), (2, 2, 300, 1, 64),
              (16, 2, 197, 33, 64)]


@pytest.mark.parametrize("shape", _TC_SHAPES)
def test_backward_tensor_core_shapes(env, shape):
    got, ref, _ = _case(env, "bf16", *shape, seed=sum(shape) + 1)
    for name, g, r in zip(("dQ", "dU", "dV"), got, ref):
        assert_parity(to_host64(g), r, "bf16", f"{name} {shape}")
    assert env[0].device_error() == 0


# d = 128 tensor-core path: one token; exactly one tile; a ragged second tile; a long slice
# cut into many items; one anchor; many batch entries summed into dU; fewer anchors than 64
_WIDE_SHAPES = [(3, 2, 1, 7, 128), (2, 2, 128, 128, 128), (1, 3, 129, 49, 128), (1, 1, 2000, 128, 128),
                (2, 2, 300, 1, 128), (16, 2, 197, 100, 128), (1, 2, 5000, 40, 128)]


# the same kernels at d = 64 with more than 64 anchors (one token; a ragged second tile; a long
# slice cut into many runs; the most anchors)
_WIDE64_SHAPES = [(3, 1, 1, 70, 64), (2, 2, 300, 100, 64), (2, 2, 1100, 65, 64), (1, 3, 2000, 128, 64),
                  (1, 2, 129, 128, 64)]


@pytest.mark.parametrize("shape", _WIDE64_SHAPES)
def test_backward_wide_d64_shapes(env, shape):
    got, ref, _ = _case(env, "bf16", *shape, seed=sum(shape) + 3)
    for name, g, r in zip(("dQ", "dU", "dV"), got, ref):
        assert_parity(to_host64(g), r, "bf16", f"{name} {shape}")
    assert env[0].device_error() == 0


@pytest.mark.parametrize("shape", _WIDE_SHAPES)
def test_backward_wide_tensor_core_shapes(env, shape):
    got, ref, _ = _case(env, "bf16", *shape, seed=sum(shape) + 2)
    for name, g, r in zip(("dQ", "dU", "dV"), got, ref):
        assert_parity(to_host64(g), r, "bf16", f"{name} {shape}")
    assert env[0].device_error() == 0


def test_backward_long_16k_sampled_heads(env):
    """Full size (4 x 16 slices of 16384 tokens, 128 anchors, d = 128): dQ and dV of every
    batch entry of four heads (16 of the 64 slices) element by element, and those heads' dU
    against the sum of their four slices' shares."""
    pkg, torch, orc = env
    w = gen.WORKLOADS["long_16k"]
    x = gen.make_inputs(w, seed=0)
    dH = gen.make_inputs(w.with_(name="bwd_dh"), seed=1000)["V"]
    t = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
    dQ, dU, dV = pkg.backward(t["Q"], t["U"], t["V"], to_device(dH, w.dtype, torch), scale=w.scale)
    torch.cuda.synchronize()
    assert pkg.device_error() == 0
    heads = [0, 5, 10, w.heads - 1]
    dQh = {(b, h): to_host64(dQ[b, h]) for b in range(w.B) for h in heads}
    dVh = {(b, h): to_host64(dV[b, h]) for b in range(w.B) for h in heads}
    dUh = to_host64(dU)
    U = gen.to_float64(x["U"], w.dtype)

    def one(bh):
        b, h = bh
        f = lambda a: gen.to_float64(a[b, h], w.dtype)
        return bh, orc.slice_backward(f(x["Q"]), U[h], f(x["V"]), f(dH), w.scale)

    dU_ref = {h: np.zeros(U.shape[1:]) for h in heads}
    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        for (b, h), (rq, ru, rv) in ex.map(one, [(b, h) for b in range(w.B) for h in heads]):
            assert_parity(dQh[b, h], rq, w.dtype, f"long_16k dQ slice ({b},{h})")
            assert_parity(dVh[b, h], rv, w.dtype, f"long_16k dV slice ({b},{h})")
            dU_ref[h] += ru
    for h in heads:
        assert_parity(dUh[h], dU_ref[h], w.dtype, f"long_16k dU head {h}")


@pytest.mark.parametrize("name", ["deit_small", "deit_base", "det_800x1344"])
def test_backward_workload_every_slice(env, name):
    """Full size: every slice's dQ and dV against the oracle element by element, and dU
    against the sum of every slice's share (the oracle runs one slice per host core)."""
    pkg, torch, orc = env
    w = gen.WORKLOADS[name]
    x = gen.make_inputs(w, seed=0)
    dH = gen.make_inputs(w.with_(name="bwd_dh"), seed=1000)["V"]
    t = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
    dQ, dU, dV = pkg.backward(t["Q"], t["U"], t["V"], to_device(dH, w.dtype, torch), scale=w.scale)
    torch.cuda.synchronize()
    assert pkg.device_error() == 0
    dQh, dVh, dUh = to_host64(dQ), to_host64(dV), to_host64(dU)
    U = gen.to_float64(x["U"], w.dtype)

    def one(s):
        b, h = divmod(s, w.heads)
        f = lambda a: gen.to_float64(a[b, h], w.dtype)
        return s, orc.slice_backward(f(x["Q"]), U[h], f(x["V"]), f(dH), w.scale)

    dU_ref = np.zeros(U.shape)
    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        for s, (rq, ru, rv) in ex.map(one, range(w.slices)):
            b, h = divmod(s, w.heads)
            assert_parity(dQh[b, h], rq, w.dtype, f"{name} dQ slice ({b},{h})")
            assert_parity(dVh[b, h], rv, w.dtype, f"{name} dV slice ({b},{h})")
            dU_ref[h] += ru
    assert_parity(dUh, dU_ref, w.dtype, f"{name} dU")


def test_backward_bit_stable(env):
    pkg, torch, _ = env
    # tensor-core paths (one CTA per slice at d = 64, m <= 64; runs of tiles at d = 64 with more
    # anchors and at d = 128) and the CUDA-core path (more than 128 anchors)
    for shape in [(2, 3, 1500, 64, 64), (2, 3, 1500, 100, 64), (2, 3, 1500, 100, 128), (2, 3, 1500, 200, 64)]:
        got1, _, (t, tdH, sc) = _case(env, "bf16", *shape, seed=9)
        got2 = pkg.backward(t["Q"], t["U"], t["V"], tdH, scale=sc)
        torch.cuda.synchronize()
        for a, b in zip(got1, got2):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_backward_empty_and_rejected(env):
    pkg, torch, _ = env
    U = torch.ones((2, 4, 64), dtype=torch.bfloat16, device="cuda")
    dU = torch.full_like(U, 5.0)
    Q = torch.zeros((0, 2, 10, 64), dtype=torch.bfloat16, device="cuda")
    st = pkg.anchor_attn_backward_ptr(0, U.data_ptr(), 0, 0, 0, dU.data_ptr(), 0, 0, 2, 10, 4, 64, 0.125, 0)
    torch.cuda.synchronize()
    assert st == 0 and bool((dU == 0).all()), "no batch entries: dU is zero"
    Q = torch.zeros((1, 2, 10, 64), dtype=torch.bfloat16, device="cuda")
    st = pkg.anchor_attn_backward_ptr(Q.data_ptr(), U.data_ptr(), Q.data_ptr(), Q.data_ptr(), Q.data_ptr(),
                                      dU.data_ptr(), Q.data_ptr() + 16 * 64, 1, 2, 10, 4, 64, 0.125, 0)
    assert st == 3, "an output over an input is rejected"


@pytest.mark.parametrize("shape", [(2, 3, 197, 30, 64), (1, 2, 700, 64, 64), (2, 2, 900, 128, 128)])
def test_backward_dependent_calls_back_to_back(env, shape):
    """The backward's two kernels (and the next call's) start while the kernel before them in
    the stream finishes and wait for it before touching global memory: calls that each take the
    previous call's dQ as their upstream gradient give the same bits queued back to back as
    with a synchronisation between them."""
    pkg, torch, _ = env
    B, heads, n, m, d = shape
    w = gen.WORKLOADS["vit14_f32"].with_(name="bwd_chain", B=B, heads=heads, n=n, m=m, d=d, dtype="bf16")
    x = gen.make_inputs(w, seed=81)
    t = {k: to_device(x[k], "bf16", torch) for k in "QUV"}
    dH0 = to_device(gen.make_inputs(w.with_(name="bwd_dh"), seed=82)["V"], "bf16", torch)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def chain(sync):
        dh, outs = dH0, []
        for _ in range(3):
            with torch.cuda.stream(stream):
                dQ, dU, dV = pkg.backward(t["Q"], t["U"], t["V"], dh, scale=w.scale)
            if sync:
                torch.cuda.synchronize()
            outs += [dQ, dU, dV]
            dh = dQ
        torch.cuda.synchronize()
        return outs

    for a, b in zip(chain(False), chain(True)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert pkg.device_error() == 0
