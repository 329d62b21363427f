"""GPU: the forward from host buffers (anchor_attn_forward_host) gives the bits of the device
entry on the same inputs, chunked or not, pinned or pageable, bf16 or fp32, and orders its
copies on the caller's stream."""
import numpy as np
import pytest

import gen
from tests.conftest import gpu_available
from tests.gpu_util import to_device

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def env():
    import torch
    import linear_complexity_anchor_gb300 as pkg
    pkg.load()
    return pkg, torch


def _host(x, dtype, torch, pinned):
    t = torch.from_numpy(x if dtype == "f32" else x.view(np.int16))
    t = t if dtype == "f32" else t.view(torch.bfloat16)
    return t.pin_memory() if pinned else t.clone()


@pytest.mark.parametrize("name,pinned", [("deit_small", True), ("det_800x1344", True), ("det_800x1344", False),
                                         ("vit14_f32", True), ("deit_base", True)])
def test_host_entry_matches_device_entry(env, name, pinned):
    pkg, torch = env
    w = gen.WORKLOADS[name]
    x = gen.make_inputs(w, seed=51)
    h = {k: _host(x[k], w.dtype, torch, pinned) for k in "QUV"}
    d = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
    stream = torch.cuda.Stream()
    Hh = pkg.forward_host(h["Q"], h["U"], h["V"], scale=w.scale, stream=stream)
    stream.synchronize()
    Hd = pkg.forward(d["Q"], d["U"], d["V"], scale=w.scale)
    torch.cuda.synchronize()
    view = torch.float32 if w.dtype == "f32" else torch.int16
    assert torch.equal(Hh.view(view), Hd.cpu().view(view)), name
    assert pkg.device_error() == 0


def test_host_entry_head_chunks_persistent_plan(env):
    """One batch entry of 8 heads of 16384 tokens at d = m = 128 (100 MB of Q, V and H): two
    chunks of four heads each; the persistent tensor-core plan of each chunk follows the whole
    problem's slice count, so the bits are the device entry's."""
    pkg, torch = env
    w = gen.WORKLOADS["long_16k"].with_(name="host_heads", B=1, heads=8)
    x = gen.make_inputs(w, seed=53)
    h = {k: _host(x[k], w.dtype, torch, True) for k in "QUV"}
    d = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
    Hh = pkg.forward_host(h["Q"], h["U"], h["V"], scale=w.scale)
    torch.cuda.current_stream().synchronize()
    Hd = pkg.forward(d["Q"], d["U"], d["V"], scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(Hh.view(torch.int16), Hd.cpu().view(torch.int16))
    assert pkg.device_error() == 0


def test_host_entry_head_chunks_keep_the_cluster_plan(env):
    """One batch entry of 16 heads of 16384 tokens at d = m = 64: the device entry runs the
    slice-streaming kernel in clusters of 6 CTAs per slice (8 slices alone would take 8); the
    host entry cuts the heads into two chunks of 8 and runs each with clusters of 6, so the bits
    are the device entry's."""
    pkg, torch = env
    w = gen.WORKLOADS["det_800x1344"].with_(name="host_cluster", B=1, heads=16, n=16384, m=64, d=64)
    assert pkg.query_plan("bf16", 1, 16, 16384, 64, 64)["splits"] == 6
    assert pkg.query_plan("bf16", 1, 8, 16384, 64, 64)["splits"] == 8
    x = gen.make_inputs(w, seed=57)
    h = {k: _host(x[k], w.dtype, torch, True) for k in "QUV"}
    d = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
    Hh = pkg.forward_host(h["Q"], h["U"], h["V"], scale=w.scale)
    torch.cuda.current_stream().synchronize()
    Hd = pkg.forward(d["Q"], d["U"], d["V"], scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(Hh.view(torch.int16), Hd.cpu().view(torch.int16))
    assert pkg.device_error() == 0


def test_host_entry_more_large_entries_than_chunks(env):
    """17 batch entries of 72 MB of Q, V and H each (6 heads of 16384 tokens at d = m = 128):
    more entries than the 16 chunks a call overlaps, each larger than a chunk's aim; the
    chunks stay whole-entry groups (16 of them) and the bits are the device entry's."""
    pkg, torch = env
    w = gen.WORKLOADS["long_16k"].with_(name="host_many", B=17, heads=6)
    x = gen.make_inputs(w, seed=59)
    h = {k: _host(x[k], w.dtype, torch, True) for k in "QUV"}
    del x
    Hh = pkg.forward_host(h["Q"], h["U"], h["V"], scale=w.scale)
    torch.cuda.current_stream().synchronize()
    d = {k: h[k].to("cuda") for k in "QUV"}
    Hd = pkg.forward(d["Q"], d["U"], d["V"], scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(Hh.view(torch.int16), Hd.cpu().view(torch.int16))
    assert pkg.device_error() == 0


def test_host_entry_chunks_of_a_large_batch(env):
    """B = 5 entries, 184 MB of Q, V and H: three chunks (1, 2 and 2 entries) over two buffer
    sets; every entry against the device entry."""
    pkg, torch = env
    w = gen.WORKLOADS["det_800x1344"].with_(name="host_chunks", B=5, heads=12, n=8000, m=64, d=64)
    x = gen.make_inputs(w, seed=52)
    h = {k: _host(x[k], w.dtype, torch, True) for k in "QUV"}
    d = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
    Hh = pkg.forward_host(h["Q"], h["U"], h["V"], scale=w.scale)
    torch.cuda.current_stream().synchronize()
    Hd = pkg.forward(d["Q"], d["U"], d["V"], scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(Hh.view(torch.int16), Hd.cpu().view(torch.int16))
    assert pkg.device_error() == 0


def test_host_entry_reuses_its_buffers_across_calls(env):
    """Back-to-back calls into the same host output, each ordered after the last on the
    caller's stream: the last call's H wins, whole."""
    pkg, torch = env
    w = gen.WORKLOADS["det_800x1344"]
    xs = [gen.make_inputs(w, seed=53 + i) for i in range(3)]
    H = torch.empty((w.B, w.heads, w.n, w.d), dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.Stream()
    keep = []  # the host inputs stay alive until the copies that read them have run
    for x in xs:
        h = {k: _host(x[k], w.dtype, torch, True) for k in "QUV"}
        keep.append(h)
        pkg.forward_host(h["Q"], h["U"], h["V"], H=H, scale=w.scale, stream=stream)
    stream.synchronize()
    d = {k: to_device(xs[-1][k], w.dtype, torch) for k in "QUV"}
    Hd = pkg.forward(d["Q"], d["U"], d["V"], scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(H.view(torch.int16), Hd.cpu().view(torch.int16))
