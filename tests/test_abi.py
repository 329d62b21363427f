"""The C ABI library without a GPU: it loads, exports what include/anchor_attn.h declares,
and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkg():
    from linear_complexity_anchor_gb300 import _build
    _build.build()
    import linear_complexity_anchor_gb300 as p
    p.load()
    return p


def _declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^ANCHOR_ATTN_API[^;(]*?\b(\w+)\s*\(", text, flags=re.M)
    return names


def test_exports_every_declared_symbol(pkg):
    names = _declared_symbols()
    assert "anchor_attn_forward" in names and "anchor_attn_forward_f32" in names
    lib = ctypes.CDLL(pkg.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


A = 1 << 20  # a 16-byte aligned fake address; never dereferenced by the rejected calls


def _call(pkg, f32=False, Q=A, U=2 * A, V=3 * A, H=4 * A, B=1, heads=1, n=8, m=4, d=16, scale=0.25):
    f = pkg.anchor_attn_forward_f32_ptr if f32 else pkg.anchor_attn_forward_ptr
    return f(Q, U, V, H, B, heads, n, m, d, scale, 0)


@pytest.mark.parametrize("f32", [False, True])
def test_argument_validation(pkg, f32):
    c = lambda **kw: _call(pkg, f32=f32, **kw)
    INVALID, UNSUP, ALIAS = 1, 2, 3
    assert c(Q=0) == INVALID
    assert c(H=0) == INVALID
    assert c(V=3 * A + 4) == INVALID                       # misaligned
    assert c(B=-1) == INVALID
    assert c(n=-5) == INVALID
    assert c(m=0) == INVALID
    assert c(scale=float("nan")) == INVALID
    assert c(scale=float("inf")) == INVALID
    assert c(d=48) == UNSUP
    assert c(d=128, m=129) == UNSUP                        # m * d > 16384
    assert c(d=64, m=257) == UNSUP
    assert c(H=A + 64) == ALIAS                            # H inside Q
    assert c(H=3 * A - 16) == ALIAS                        # H runs into V
    assert c(U=4 * A + 32, B=2) == ALIAS                   # U inside H
    # empty problems are valid no-ops and accept NULL pointers
    assert c(B=0, Q=0, U=0, V=0, H=0) == 0
    assert c(n=0, Q=0, U=0, V=0, H=0) == 0
    assert c(heads=0, Q=0, U=0, V=0, H=0) == 0


def test_status_strings(pkg):
    for code in range(7):
        assert pkg.status_string(code) != "unknown status"
    assert pkg.status_string(99) == "unknown status"


def test_plans(pkg):
    p = pkg.query_plan("f32", 1, 1, 196, 16, 64)
    assert p["variant"] == "simt_slice" and p["kernels_per_call"] == 1 and p["workspace_bytes"] == 0
    p = pkg.query_plan("bf16", 1, 2, 1100, 20, 64)
    assert p["variant"] == "simt_split" and p["splits"] == 3 and p["workspace_bytes"] > 0
    assert p["kernels_per_call"] == 1
    # the largest anchor count per head dimension still fits the chunked kernel's tiles
    assert pkg.query_plan("f32", 2, 2, 100000, 1024, 16)["variant"] == "simt_split"
    assert pkg.query_plan("f32", 2, 2, 20000, 512, 32)["variant"] == "simt_split"
    assert pkg.query_plan("bf16", 64, 6, 197, 30, 64)["variant"] == "simt_slice"
    assert pkg.query_plan("bf16", 0, 2, 100, 20, 64)["variant"] == "empty"
    # slice-streaming tensor-core variants: bf16, d = 64, 32 <= m <= 64, n > 512; one CTA per
    # slice up to 152 slices (workspace: the A tiles of pass 1), the tile list cut over 152
    # CTAs beyond (the A tiles first, then counters, partials and W' images)
    # (CTAs per slice: 96 slices of 33 tiles: one; 1 slice of 33 tiles: a cluster of 8; 16
    # slices of 128 tiles: clusters of 6; 40 slices of 5 tiles: one)
    p = pkg.query_plan("bf16", 8, 12, 4200, 64, 64)
    assert p["variant"] == "stream" and p["kernels_per_call"] == 1 and p["stored_a"] and p["splits"] == 1
    assert p["workspace_bytes"] == 8 * 12 * 4200 * 64 * 2
    assert pkg.query_plan("bf16", 1, 1, 4200, 64, 64)["splits"] == 8
    assert pkg.query_plan("bf16", 1, 16, 16384, 64, 64)["splits"] == 6
    # clusters up to 38 slices (38 of 128 tiles: 3 CTAs; 39: one CTA per slice) and only with
    # four tiles or more per CTA (1 slice of 5 tiles: one CTA)
    assert pkg.query_plan("bf16", 1, 38, 16384, 64, 64)["splits"] == 3
    assert pkg.query_plan("bf16", 1, 39, 16384, 64, 64)["splits"] == 1
    assert pkg.query_plan("bf16", 1, 1, 600, 64, 64)["splits"] == 1
    assert pkg.query_plan("bf16", 4, 10, 600, 40, 64)["splits"] == 1
    p = pkg.query_plan("bf16", 16, 12, 4200, 64, 64)
    assert p["variant"] == "split_tc" and p["stored_a"] and p["workspace_bytes"] > 16 * 12 * 4200 * 64 * 2
    assert pkg.query_plan("bf16", 8, 12, 512, 64, 64)["variant"] == "umma"
    # persistent tensor-core variant: d in {64, 128}, 32 <= m <= 128, bf16 only
    # 33 tiles of 128 tokens in chunks of at most 16: 3 chunks x 96 slices is at least 1.5
    # items per SM of a 152-SM GPU (the count assumed without a device)
    p = pkg.query_plan("bf16", 8, 12, 4200, 100, 64)
    assert p["variant"] == "umma" and p["kernels_per_call"] == 1 and p["splits"] == 3
    p = pkg.query_plan("bf16", 256, 12, 197, 49, 64)   # short slices, d = 64: one CTA per slice
    assert p["variant"] == "short_tc" and p["splits"] == 1 and p["workspace_bytes"] == 0
    p = pkg.query_plan("bf16", 256, 12, 197, 49, 128)  # d = 128: the persistent variant, whole slices
    assert p["variant"] == "umma" and p["splits"] == 1 and p["workspace_bytes"] == 256
    assert pkg.query_plan("f32", 8, 12, 4200, 64, 64)["variant"] == "simt_split"
    assert pkg.query_plan("bf16", 1, 1, 4200, 31, 64)["variant"] == "simt_split"
    assert pkg.query_plan("bf16", 1, 1, 4200, 64, 32)["variant"] == "simt_split"
    with pytest.raises(pkg.AnchorAttnError):
        pkg.query_plan("bf16", 1, 1, 10, 4, 48)


def test_alloc_failure_is_reported(pkg, monkeypatch):
    """Host-side fault injection: the workspace allocation reports failure."""
    monkeypatch.setenv("ANCHOR_ATTN_TEST_FAIL_ALLOC", "1")
    assert pkg.query_plan("bf16", 1, 1, 2000, 20, 64)["workspace_bytes"] > 0
    assert _call(pkg, n=2000, m=20, d=64) == 4     # CUDA-core split variant
    assert _call(pkg, n=2000, m=64, d=64) == 4     # tensor-core variant


def test_missing_library_fails_loudly(tmp_path):
    import linear_complexity_anchor_gb300 as p
    with pytest.raises(RuntimeError, match="not built"):
        p.load(str(tmp_path / "nope.so"))


def test_block_argument_validation(pkg):
    """The block front end rejects bad arguments before touching the device."""
    def c(X=A, Wq=2 * A, Wv=3 * A, U=4 * A, H=5 * A, B=2, heads=3, n=197, m=49, d=64, dm=768, scale=0.125):
        return pkg.anchor_attn_block_forward_ptr(X, Wq, Wv, U, H, B, heads, n, m, d, dm, scale, 0)
    INVALID, UNSUP, ALIAS = 1, 2, 3
    assert c(X=0) == INVALID
    assert c(U=4 * A + 8) == INVALID
    assert c(m=0) == INVALID
    assert c(dm=0) == INVALID
    assert c(B=-1) == INVALID
    assert c(scale=float("nan")) == INVALID
    assert c(d=32) == UNSUP
    assert c(m=65) == UNSUP
    assert c(n=257) == UNSUP
    assert c(dm=96) == UNSUP                    # not a multiple of 64
    assert c(H=A + 64) == ALIAS                 # overlaps X
    assert c(H=2 * A) == ALIAS                  # overlaps Wq
    assert c(B=0) == 0 and c(heads=0) == 0 and c(n=0) == 0   # no-ops (no device access)
    assert c(B=0, X=0, H=0) == 0


def test_forward_host_validates_before_any_device_call(pkg):
    """The host-buffer entry checks its arguments as the device entry does, before it touches
    a device (so these run without one)."""
    lib = pkg.load()
    buf = (ctypes.c_uint16 * 1024)()
    p = ctypes.addressof(buf)
    assert lib.anchor_attn_forward_host(p, p, p, p, -1, 2, 100, 20, 64, 0.125, None) == 1   # negative B
    assert lib.anchor_attn_forward_host(p, p, p, p, 1, 1, 10, 4, 48, 0.125, None) == 2      # d = 48
    assert lib.anchor_attn_forward_host(p, p, p, p, 0, 2, 100, 20, 64, 0.125, None) == 0    # empty: a no-op
    assert lib.anchor_attn_forward_host(None, p, p, p, 1, 2, 100, 20, 64, 0.125, None) == 1  # null Q
    assert lib.anchor_attn_forward_host_f32(p, p, p, p, 1, 1, 10, 4, 64, float("nan"), None) == 1
