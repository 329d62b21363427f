"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by element,
on the same seeded inputs."""
import math

import numpy as np
import pytest

import gen
from tests.conftest import gpu_available
from tests.gpu_util import assert_parity, assert_slices, oracle_slices, to_device, to_host64, widen

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch
    import linear_complexity_anchor_gb300 as pkg
    pkg.load()
    return pkg, torch, oracle_mod


def _run(env, w: gen.Workload, x: dict, scale=None, stream=None):
    pkg, torch, _ = env
    t = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
    H = pkg.forward(t["Q"], t["U"], t["V"], scale=w.scale if scale is None else scale, stream=stream)
    torch.cuda.synchronize()
    return H


def _check_full(env, w, seed=0, x=None, scale=None):
    pkg, torch, orc = env
    x = gen.make_inputs(w, seed=seed) if x is None else x
    H = _run(env, w, x, scale)
    xx = widen(x, w.dtype)
    ref = orc.forward(xx["Q"], xx["U"], xx["V"], w.scale if scale is None else scale)
    return assert_parity(to_host64(H), ref, w.dtype, f"{w.name} {w.B}x{w.heads}x{w.n} m={w.m} d={w.d}")


# ------------------------------------------------------------------ the five workloads

EXPECTED_VARIANT = {"vit14_f32": "simt_slice", "deit_small": "simt_slice", "deit_base": "short_tc",
                    "det_800x1344": "stream", "long_16k": "umma"}


@pytest.mark.parametrize("name", sorted(EXPECTED_VARIANT))
def test_workload_variant(env, name):
    pkg, _, _ = env
    w = gen.WORKLOADS[name]
    assert pkg.query_plan(w.dtype, w.B, w.heads, w.n, w.m, w.d)["variant"] == EXPECTED_VARIANT[name]


@pytest.mark.parametrize("name", ["vit14_f32", "deit_small"])
def test_workload_full(env, name):
    _check_full(env, gen.WORKLOADS[name])


@pytest.mark.parametrize("name", ["deit_base", "det_800x1344", "long_16k"])
def test_workload_every_slice(env, name):
    """Full-size launch (the bench's configuration), every slice checked against the oracle
    element by element (the oracle runs one slice per host core, 32 slices at a time); and a
    size-independent property on top: each column of H sums to the same column of V (S_t is
    doubly stochastic)."""
    pkg, torch, orc = env
    w = gen.WORKLOADS[name]
    x = gen.make_inputs(w, seed=0)
    H = _run(env, w, x)
    assert pkg.device_error() == 0
    Hc = H.cpu()
    for s0 in range(0, w.slices, 32):
        refs = oracle_slices(orc, w, x, range(s0, min(w.slices, s0 + 32)))
        assert_slices(Hc, w, refs, name)
    Hs = H.double().sum(dim=2)
    Vt = to_device(x["V"], w.dtype, torch).double()
    tol = 1e-3 * Vt.abs().sum(dim=2) + 1e-2
    assert ((Hs - Vt.sum(dim=2)).abs() <= tol).all(), "column sums of H differ from those of V"
    assert pkg.device_error() == 0


# The tensor-core plans recompute A in pass 2 when all slices' copies of A would not fit
# the 64 MB kept for them; each shared-memory layout stages the pass-2 H tiles differently
# (in the Q ring slot with two A buffers, in the A buffer with one), so each gets a case.
_RECOMPUTE = {
    "d64_mp64": dict(B=16, heads=12, n=4200, m=64, d=64),     # 103 MB of A, two A buffers
    "d128_mp64": dict(B=4, heads=16, n=8300, m=49, d=128),    # 68 MB of A, one A buffer, masked anchors
    "d64_mp128": dict(B=8, heads=12, n=4200, m=100, d=64),    # 103 MB of A, one A buffer, masked anchors
}


@pytest.mark.parametrize("case", sorted(_RECOMPUTE))
def test_recompute_plans(env, case):
    pkg, torch, orc = env
    w = gen.WORKLOADS["det_800x1344"].with_(name=case, **_RECOMPUTE[case])
    assert 2 * w.slices * w.n * (64 if w.m <= 64 else 128) > 64 * 1024 * 1024
    x = gen.make_inputs(w, seed=7)
    if pkg.query_plan(w.dtype, w.B, w.heads, w.n, w.m, w.d)["variant"] == "umma":
        H = _run(env, w, x)
    else:  # the persistent variant through the test entry (no held slice, the default wait limit)
        t = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
        H = torch.empty_like(t["Q"])
        assert pkg.anchor_attn_test_forward_ptr(t["Q"].data_ptr(), t["U"].data_ptr(), t["V"].data_ptr(), H.data_ptr(),
                                                w.B, w.heads, w.n, w.m, w.d, w.scale, -1, 2_000_000_000, False,
                                                0) == 0
        torch.cuda.synchronize()
    U = gen.to_float64(x["U"], w.dtype)
    for s in (0, w.slices // 2, w.slices - 1):
        b, h = divmod(s, w.heads)
        ref = orc.slice_forward(gen.to_float64(x["Q"][b, h], w.dtype), U[h], gen.to_float64(x["V"][b, h], w.dtype),
                                w.scale)["H"]
        assert_parity(to_host64(H[b, h]), ref, w.dtype, f"{case} slice ({b},{h})")
    Hs = H.double().sum(dim=2)
    Vt = to_device(x["V"], w.dtype, torch).double()
    assert ((Hs - Vt.sum(dim=2)).abs() <= 1e-3 * Vt.abs().sum(dim=2) + 1e-2).all()
    assert pkg.device_error() == 0


# ------------------------------------------------------------------ edge shapes

_MD = [(1, 16), (2, 64), (15, 32), (16, 64), (30, 64), (31, 16), (32, 64), (33, 64), (49, 64), (64, 64),
       (64, 128), (100, 128), (128, 64), (128, 128), (256, 64), (200, 32),
       (1, 128), (15, 128), (31, 128), (33, 128), (49, 128), (1024, 16), (512, 32)]
_N = [1, 2, 7, 8, 127, 128, 129, 197, 513, 1100]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("m,d", _MD)
def test_edge_shapes(env, dtype, m, d):
    for i, n in enumerate(_N):
        B, heads = (2, 3) if n <= 129 else (1, 2)
        w = gen.WORKLOADS["vit14_f32"].with_(name="edge", B=B, heads=heads, n=n, m=m, d=d, dtype=dtype)
        _check_full(env, w, seed=1000 + 17 * i + m + d)


# ------------------------------------------------------------------ degenerate cases

def _small(dtype, **kw):
    base = dict(name="degenerate", B=2, heads=2, n=300, m=40, d=64, dtype=dtype)
    base.update(kw)
    return gen.WORKLOADS["vit14_f32"].with_(**base)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("m,n", [(40, 300), (20, 2000), (64, 700)])
def test_constant_value_is_fixed(env, dtype, m, n):
    """S_t 1 = 1: a V with constant columns comes back unchanged."""
    w = _small(dtype, m=m, n=n)
    x = gen.make_inputs(w, seed=5)
    col = x["V"][:, :, :1, :]
    x["V"] = np.ascontiguousarray(np.broadcast_to(col, x["V"].shape))
    H = _run(env, w, x)
    assert_parity(to_host64(H), gen.to_float64(x["V"], dtype), dtype, "constant V")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", ["m1", "zero_q", "zero_scale", "identical_anchors"])
def test_degenerate_means(env, dtype, case):
    """One anchor, Q = 0, scale = 0 or identical anchors: every H row is the mean of V."""
    w = _small(dtype, m=1 if case == "m1" else 40)
    x = gen.make_inputs(w, seed=6)
    if case == "zero_q":
        x["Q"] = np.zeros_like(x["Q"])
    if case == "identical_anchors":
        x["U"] = np.ascontiguousarray(np.broadcast_to(x["U"][:, :1, :], x["U"].shape))
    H = _run(env, w, x, scale=0.0 if case == "zero_scale" else None)
    V = gen.to_float64(x["V"], dtype)
    ref = np.broadcast_to(V.mean(axis=2, keepdims=True), V.shape)
    assert_parity(to_host64(H), ref, dtype, case)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_unreached_anchor_drops_out(env, dtype):
    """An anchor whose scores underflow for every token (Delta_j = 0) contributes nothing."""
    w = _small(dtype, m=33)
    x = gen.make_inputs(w, seed=7)
    Q = gen.to_float64(x["Q"], dtype)
    U = gen.to_float64(x["U"], dtype)
    # anchor 5 of every head: score = -2000 * q_0 * scale <= -250 while the others stay
    # within a few units, so its A column underflows to exactly 0 in fp32
    U[:, 5, :] = 0.0
    U[:, 5, 0] = -2000.0
    x["Q"] = np.where(np.arange(w.d) == 0, np.abs(Q) + 1.0, Q)
    x["Q"] = x["Q"].astype(np.float32) if dtype == "f32" else gen.round_bf16(x["Q"])
    x["U"] = U.astype(np.float32) if dtype == "f32" else gen.round_bf16(U)
    _check_full(env, w, x=x)


# ------------------------------------------------------------------ run-time properties

@pytest.mark.parametrize("shape", [(1, 1, 196, 16, 64, "f32"), (2, 3, 2000, 20, 64, "bf16"), (2, 3, 2000, 64, 64, "bf16"),
                                   (4, 6, 197, 30, 64, "bf16"), (2, 4, 700, 64, 64, "bf16"),
                                   (1, 4, 1500, 128, 128, "bf16")])
def test_bit_stable(env, shape):
    pkg, torch, _ = env
    B, heads, n, m, d, dtype = shape
    w = _small(dtype, B=B, heads=heads, n=n, m=m, d=d)
    x = gen.make_inputs(w, seed=8)
    H1 = _run(env, w, x)
    H2 = _run(env, w, x)
    assert torch.equal(H1.view(torch.int16) if dtype == "bf16" else H1.view(torch.int32),
                       H2.view(torch.int16) if dtype == "bf16" else H2.view(torch.int32))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n,m,d", [(197, 30, 64), (1100, 20, 64), (700, 64, 64), (333, 128, 128)])
def test_guard_bands_untouched(env, dtype, n, m, d):
    """Sentinels before and after H stay intact (no write outside the output)."""
    pkg, torch, orc = env
    w = _small(dtype, B=2, heads=2, n=n, m=m, d=d)
    x = gen.make_inputs(w, seed=9)
    t = {k: to_device(x[k], dtype, torch) for k in "QUV"}
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    pad = 4096
    buf = torch.full((pad + t["Q"].numel() + pad,), -4096.0, dtype=tdt, device="cuda")
    H = buf[pad:pad + t["Q"].numel()].view(t["Q"].shape)
    pkg.forward(t["Q"], t["U"], t["V"], H=H, scale=w.scale)
    torch.cuda.synchronize()
    assert (buf[:pad] == -4096.0).all() and (buf[-pad:] == -4096.0).all()
    xx = widen(x, dtype)
    assert_parity(to_host64(H), orc.forward(xx["Q"], xx["U"], xx["V"], w.scale), dtype, "guarded")


def test_valid_call_after_rejected_calls(env):
    """A rejected call leaves nothing behind: the next valid call on the same thread succeeds."""
    pkg, torch, orc = env
    w = _small("bf16", n=1100, m=20)
    x = gen.make_inputs(w, seed=11)
    t = {k: to_device(x[k], "bf16", torch) for k in "QUV"}
    H = torch.empty_like(t["Q"])
    args = (t["Q"].data_ptr(), t["U"].data_ptr(), t["V"].data_ptr())
    # H aliasing Q, and an unsupported head dimension
    assert pkg.anchor_attn_forward_ptr(*args[:3], t["Q"].data_ptr(), w.B, w.heads, w.n, w.m, w.d, w.scale, 0) == 3
    assert pkg.anchor_attn_forward_ptr(*args, H.data_ptr(), w.B, w.heads, w.n, w.m, 48, w.scale, 0) == 2
    assert pkg.anchor_attn_forward_ptr(*args, H.data_ptr(), w.B, w.heads, w.n, w.m, w.d, w.scale, 0) == 0
    torch.cuda.synchronize()
    xx = widen(x, "bf16")
    assert_parity(to_host64(H), orc.forward(xx["Q"], xx["U"], xx["V"], w.scale), "bf16", "after rejected calls")


def test_no_device_error_after_runs(env):
    pkg, _, _ = env
    assert pkg.device_error() == 0


def test_empty_problems_are_noops(env):
    pkg, torch, _ = env
    for shape in [(0, 2, 10, 4, 64), (2, 0, 10, 4, 64), (2, 2, 0, 4, 64)]:
        B, heads, n, m, d = shape
        Q = torch.zeros((B, heads, n, d), dtype=torch.bfloat16, device="cuda")
        U = torch.zeros((heads, m, d), dtype=torch.bfloat16, device="cuda")
        H = pkg.forward(Q, U, Q.clone())
        assert H.shape == Q.shape


def test_runs_on_the_given_stream(env):
    pkg, torch, orc = env
    w = _small("bf16", n=900, m=48)
    x = gen.make_inputs(w, seed=10)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        H = _run(env, w, x, stream=s)
    s.synchronize()
    xx = widen(x, "bf16")
    assert_parity(to_host64(H), orc.forward(xx["Q"], xx["U"], xx["V"], w.scale), "bf16", "side stream")


# More slices than 152: the tile list cut over 152 resident CTAs (slices shared by two or
# more CTAs, partials summed in part order by the last arriver).
@pytest.mark.parametrize("shape", [(16, 12, 700, 64, 64), (40, 4, 1000, 40, 64), (2, 80, 600, 33, 64)])
def test_split_tiles_every_slice(env, shape):
    pkg, torch, orc = env
    B, heads, n, m, d = shape
    w = gen.WORKLOADS["det_800x1344"].with_(name="split", B=B, heads=heads, n=n, m=m, d=d)
    assert pkg.query_plan("bf16", B, heads, n, m, d)["variant"] == "split_tc"
    x = gen.make_inputs(w, seed=sum(shape))
    H = _run(env, w, x)
    H2 = _run(env, w, x)
    assert pkg.device_error() == 0
    assert torch.equal(H.view(torch.int16), H2.view(torch.int16))
    Hc = H.cpu()
    for s0 in range(0, w.slices, 64):
        assert_slices(Hc, w, oracle_slices(orc, w, x, range(s0, min(w.slices, s0 + 64))), "split")


# A few slices of many tiles: a cluster of c CTAs per slice, the c partial sums added over
# distributed shared memory in rank order.  (B, heads, n, m, d, CTAs per slice): ragged
# tails, padded anchors, clusters of 4, 6 and 8.
@pytest.mark.parametrize("shape", [(1, 1, 4200, 64, 64, 8), (2, 3, 8000, 50, 64, 8), (1, 8, 16384, 64, 64, 8),
                                   (4, 8, 8000, 33, 64, 4), (1, 16, 16384, 40, 64, 6)])
def test_stream_clusters_every_slice(env, shape):
    pkg, torch, orc = env
    B, heads, n, m, d, per_slice = shape
    w = gen.WORKLOADS["det_800x1344"].with_(name="clusters", B=B, heads=heads, n=n, m=m, d=d)
    plan = pkg.query_plan("bf16", B, heads, n, m, d)
    assert plan["variant"] == "stream" and plan["splits"] == per_slice
    x = gen.make_inputs(w, seed=sum(shape))
    H = _run(env, w, x)
    H2 = _run(env, w, x)
    assert pkg.device_error() == 0
    assert torch.equal(H.view(torch.int16), H2.view(torch.int16))
    Hc = H.cpu()
    for s0 in range(0, w.slices, 64):
        assert_slices(Hc, w, oracle_slices(orc, w, x, range(s0, min(w.slices, s0 + 64))), "clusters")


@pytest.mark.parametrize("name", ["det_800x1344", "deit_base", "deit_small"])
def test_dependent_calls_back_to_back(env, name):
    """Kernels launched with programmatic stream serialization start while the previous kernel
    in the stream finishes; each waits for it before touching global memory.  A chain of calls
    that each read the previous call's output (H as the next Q and V), queued back to back on
    one stream, gives the same bits as the same calls with a full synchronisation between them."""
    pkg, torch, _ = env
    w = gen.WORKLOADS[name]
    x = gen.make_inputs(w, seed=41)
    t = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def chain(sync):
        q, v = t["Q"], t["V"]
        outs = []
        for _ in range(4):
            h = pkg.forward(q, t["U"], v, scale=w.scale, stream=stream)
            if sync:
                torch.cuda.synchronize()
            outs.append(h)
            q, v = h, h
        torch.cuda.synchronize()
        return outs

    queued, synced = chain(False), chain(True)
    for i, (a, b) in enumerate(zip(queued, synced)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{name}: call {i} differs"
    assert pkg.device_error() == 0


@pytest.mark.parametrize("name", ["det_800x1344", "deit_base", "deit_small", "long_16k"])
def test_graph_capture_replays_the_same_bits(env, name):
    """The forward calls can be captured in a CUDA graph (the stream-ordered workspace becomes
    graph allocation nodes, programmatic launches become programmatic edges) and replayed:
    every replay gives the bits of the eager call."""
    pkg, torch, _ = env
    w = gen.WORKLOADS[name]
    x = gen.make_inputs(w, seed=61)
    t = {k: to_device(x[k], w.dtype, torch) for k in "QUV"}
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    ref = pkg.forward(t["Q"], t["U"], t["V"], scale=w.scale, stream=stream)
    ref2 = pkg.forward(ref, t["U"], ref, scale=w.scale, stream=stream)
    torch.cuda.synchronize()
    H1, H2 = torch.empty_like(ref), torch.empty_like(ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        pkg.forward(t["Q"], t["U"], t["V"], H=H1, scale=w.scale, stream=stream)
        pkg.forward(H1, t["U"], H1, H=H2, scale=w.scale, stream=stream)
    for _ in range(3):
        H1.zero_()
        H2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(H1.view(torch.int16), ref.view(torch.int16)), name
        assert torch.equal(H2.view(torch.int16), ref2.view(torch.int16)), name
    assert pkg.device_error() == 0
