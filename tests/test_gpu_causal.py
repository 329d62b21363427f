"""GPU: the masked (causal) variant through the C ABI against the oracle's, element by element,
plus the properties that hold at any size: the last row equals the unmasked forward's, the
first row is its own value, and changing later tokens leaves earlier rows unchanged.  bf16 runs
on the tensor cores (the 64-anchor kernel for d = 64, m <= 64; the 128-anchor kernel for
d = 128, m <= 128 and d = 64, 64 < m <= 128); the rest, and fp32, on CUDA cores."""
import os
from concurrent.futures import ThreadPoolExecutor

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


# tensor-core path: one token; exactly one tile; a second tile of one token; a long slice; one
# anchor; a scale of either sign
_TC_SHAPES = [(3, 2, 1, 5, 64, None), (2, 2, 128, 64, 64, None), (1, 2, 129, 33, 64, None), (1, 1, 2000, 64, 64, None),
              (2, 2, 300, 1, 64, None), (1, 2, 250, 40, 64, -0.2), (2, 1, 400, 64, 64, 0.0)]


@pytest.mark.parametrize("shape", _TC_SHAPES)
def test_causal_tensor_core_shapes(env, shape):
    pkg, torch, orc = env
    *dims, scale = shape
    w = _w("bf16", *dims)
    sc = w.scale if scale is None else scale
    x = gen.make_inputs(w, seed=sum(dims) + 3)
    t = {k: to_device(x[k], "bf16", torch) for k in "QUV"}
    H = pkg.causal_forward(t["Q"], t["U"], t["V"], scale=sc)
    torch.cuda.synchronize()
    xx = widen(x, "bf16")
    assert_parity(to_host64(H), orc.causal(xx["Q"], xx["U"], xx["V"], sc), "bf16", f"causal {shape}")
    assert pkg.device_error() == 0


@pytest.mark.parametrize("name", ["deit_base", "det_800x1344"])
def test_causal_workload_every_slice(env, name):
    """Full size, every slice against the oracle (one slice per host core), and bit-stable."""
    pkg, torch, orc = env
    w = gen.WORKLOADS[name]
    x = gen.make_inputs(w, seed=0)
    t = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
    H = pkg.causal_forward(t["Q"], t["U"], t["V"], scale=w.scale)
    H2 = pkg.causal_forward(t["Q"], t["U"], t["V"], scale=w.scale)
    torch.cuda.synchronize()
    assert pkg.device_error() == 0
    assert torch.equal(H.view(torch.int16), H2.view(torch.int16))
    Hh = to_host64(H)
    U = gen.to_float64(x["U"], w.dtype)

    def one(s):
        b, h = divmod(s, w.heads)
        q = gen.to_float64(x["Q"][b, h], w.dtype)[None, None]
        v = gen.to_float64(x["V"][b, h], w.dtype)[None, None]
        return s, orc.causal(q, U[h:h + 1], v, w.scale)[0, 0]

    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        for s, ref in ex.map(one, range(w.slices)):
            b, h = divmod(s, w.heads)
            assert_parity(Hh[b, h], ref, w.dtype, f"{name} causal slice ({b},{h})")


# 128-anchor tensor-core path (d = 128, or d = 64 with m > 64): the same edge cases
_WIDE_SHAPES = [(3, 2, 1, 5, 128, None), (2, 2, 128, 128, 128, None), (1, 2, 129, 33, 128, None),
                (1, 1, 2000, 128, 128, None), (2, 2, 300, 1, 128, None), (1, 2, 250, 40, 128, -0.2),
                (2, 1, 400, 128, 128, 0.0), (2, 2, 300, 65, 64, None), (1, 2, 513, 128, 64, None)]


@pytest.mark.parametrize("shape", _WIDE_SHAPES)
def test_causal_wide_shapes(env, shape):
    pkg, torch, orc = env
    *dims, scale = shape
    w = _w("bf16", *dims)
    sc = w.scale if scale is None else scale
    x = gen.make_inputs(w, seed=sum(dims) + 5)
    t = {k: to_device(x[k], "bf16", torch) for k in "QUV"}
    H = pkg.causal_forward(t["Q"], t["U"], t["V"], scale=sc)
    torch.cuda.synchronize()
    xx = widen(x, "bf16")
    assert_parity(to_host64(H), orc.causal(xx["Q"], xx["U"], xx["V"], sc), "bf16", f"causal {shape}")
    assert pkg.device_error() == 0


def test_causal_wide_ignores_later_tokens(env):
    pkg, torch, _ = env
    w = _w("bf16", 1, 2, 1000, 128, 128)
    x = gen.make_inputs(w, seed=23)
    t = {k: to_device(x[k], "bf16", torch) for k in "QUV"}
    H1 = pkg.causal_forward(t["Q"], t["U"], t["V"], scale=w.scale)
    Q2, V2 = t["Q"].clone(), t["V"].clone()
    Q2[:, :, 700:] += 1.0
    V2[:, :, 700:] -= 1.0
    H2 = pkg.causal_forward(Q2, t["U"], V2, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(H1[:, :, :700].view(torch.int16), H2[:, :, :700].view(torch.int16))
    assert not torch.equal(H1[:, :, 700:], H2[:, :, 700:])


def test_causal_long_16k_sampled_slices(env):
    """long_16k at full size (the 128-anchor kernel): 16 of the 64 slices against the oracle,
    and bit-stable from run to run."""
    pkg, torch, orc = env
    w = gen.WORKLOADS["long_16k"]
    x = gen.make_inputs(w, seed=0)
    t = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
    H = pkg.causal_forward(t["Q"], t["U"], t["V"], scale=w.scale)
    H2 = pkg.causal_forward(t["Q"], t["U"], t["V"], scale=w.scale)
    torch.cuda.synchronize()
    assert pkg.device_error() == 0
    assert torch.equal(H.view(torch.int16), H2.view(torch.int16))
    Hh = to_host64(H)
    U = gen.to_float64(x["U"], w.dtype)

    def one(s):
        b, h = divmod(s, w.heads)
        q = gen.to_float64(x["Q"][b, h], w.dtype)[None, None]
        v = gen.to_float64(x["V"][b, h], w.dtype)[None, None]
        return s, orc.causal(q, U[h:h + 1], v, w.scale)[0, 0]

    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        for s, ref in ex.map(one, range(0, w.slices, 4)):
            b, h = divmod(s, w.heads)
            assert_parity(Hh[b, h], ref, w.dtype, f"long_16k causal slice ({b},{h})")


def test_causal_wide_chunks_do_not_change_bits(env):
    """With few slices the 128-anchor kernel cuts each slice's tokens over up to four CTAs (each
    first sums the tiles before its chunk); with many slices one CTA takes a slice whole.  The
    same slice gives the same bits either way."""
    pkg, torch, _ = env
    w = _w("bf16", 80, 1, 2000, 128, 128)  # 80 slices: one CTA per slice
    x = gen.make_inputs(w, seed=31)
    t = {k: to_device(x[k], "bf16", torch) for k in "QUV"}
    Hall = pkg.causal_forward(t["Q"], t["U"], t["V"], scale=w.scale)
    for b in (0, 37, 79):  # alone: four chunks of four tiles
        H1 = pkg.causal_forward(t["Q"][b:b + 1].contiguous(), t["U"], t["V"][b:b + 1].contiguous(), scale=w.scale)
        torch.cuda.synchronize()
        assert torch.equal(H1[0].view(torch.int16), Hall[b].view(torch.int16)), f"slice {b}"
    assert pkg.device_error() == 0


@pytest.mark.parametrize("shape", [(2, 3, 700, 49, 64), (1, 2, 2100, 100, 128)])
def test_causal_dependent_calls_back_to_back(env, shape):
    """The masked kernels start while the previous kernel in the stream finishes and wait for
    it before touching global memory: a chain of calls that each read the previous output
    gives the same bits queued back to back as with a synchronisation between them."""
    pkg, torch, _ = env
    w = _w("bf16", *shape)
    x = gen.make_inputs(w, seed=71)
    t = {k: to_device(x[k], "bf16", torch) for k in "QUV"}
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def chain(sync):
        q, v, outs = t["Q"], t["V"], []
        for _ in range(4):
            with torch.cuda.stream(stream):
                h = pkg.causal_forward(q, t["U"], v, scale=w.scale)
            if sync:
                torch.cuda.synchronize()
            outs.append(h)
            q, v = h, h
        torch.cuda.synchronize()
        return outs

    for a, b in zip(chain(False), chain(True)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert pkg.device_error() == 0
