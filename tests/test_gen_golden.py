"""The seeded input generator and the stored oracle fixture."""
import json
import os

import numpy as np
import pytest

import gen

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_splitmix64_published_sequence():
    # splitmix64 started from state 0 (Steele, Lea, Flood 2014; the sequence printed with
    # the public reference implementation).
    got = [int(v) for v in gen.splitmix64(np.uint64(0), 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_uniform_and_normal_moments():
    key = gen._key(0, 99)
    u = gen.uniform(key, 0, 200000)
    assert 0.0 < u.min() and u.max() < 1.0 and abs(u.mean() - 0.5) < 0.005
    z = gen.normal(key, 0, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    # counter-based: any window equals the same window of a longer draw
    np.testing.assert_array_equal(gen.normal(key, 12345, 777), z[12345:12345 + 777])


def test_bf16_rounding_is_nearest_even():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(50000).astype(np.float32) * 7,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, -0.0], np.float32)])
    ours = gen.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(gen.bf16_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("name", ["vit14_f32", "deit_small", "deit_base"])
def test_workload_inputs(name):
    w = gen.WORKLOADS[name]
    x = gen.make_inputs(w, seed=0)
    assert x["Q"].shape == (w.B, w.heads, w.n, w.d) and x["V"].shape == x["Q"].shape
    assert x["U"].shape == (w.heads, w.m, w.d)
    y = gen.slice_inputs(w, w.B - 1, w.heads - 1, seed=0)
    np.testing.assert_array_equal(y["Q"], x["Q"][-1, -1])
    np.testing.assert_array_equal(y["V"], x["V"][-1, -1])
    U = gen.to_float64(x["U"], w.dtype)
    if w.recipe == "u_half":
        assert abs(U.std() - 2 ** -0.5) < 0.02
    if w.recipe == "u_from_k":
        # 49 distinct rows per head, each a key row plus N(0, 0.1^2) noise
        assert all(len({tuple(np.round(r, 1)) for r in U[h]}) == w.m for h in range(w.heads))


def test_golden_fixture_reproduces(oracle_mod):
    with open(os.path.join(GOLDEN, "vit14_f32_seed0.json")) as f:
        g = json.load(f)
    w = gen.WORKLOADS[g["workload"]]
    x = gen.make_inputs(w, seed=g["seed"])
    Q, U, V = (gen.to_float64(x[k], w.dtype) for k in "QUV")
    fp = g["input_fingerprint"]
    assert Q.reshape(-1)[:4].tolist() == fp["Q_first"] and V.reshape(-1)[-4:].tolist() == fp["V_last"]
    assert abs(Q.sum() - fp["Q_sum"]) < 1e-9 and abs(V.sum() - fp["V_sum"]) < 1e-9
    H = oracle_mod.forward(Q, U, V, g["scale"])
    np.testing.assert_allclose(H[0, 0, g["rows"]], np.array(g["H_rows"]), rtol=0, atol=1e-13)
    assert abs(H.sum() - g["H_sum"]) < 1e-10
