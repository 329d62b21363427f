"""CPU oracle for the anchor-attention forward H = A Delta^{-1} A^T V (AnchorFormer), its
backward (the gradients with respect to Q, U and V of a loss with upstream gradient dH), the
masked variant, full softmax attention for the approximation-error diagnostic, and the block
front end (Q and V projected from the token embeddings, then the forward).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` are the only callers.  The arithmetic lives in ``anchor_oracle.c`` (plain C,
double precision, one thread); this module compiles it with gcc and marshals numpy arrays.
It shares no code with the CUDA path and imports nothing from it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "anchor_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None  # the default Oracle instance


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library next to its source (no -ffast-math: the C
    compiler keeps the written evaluation order)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                        "-ffp-contract=off", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


class Oracle:
    """Bound to one compiled oracle library (the default one, or a variant the tests build)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        D = ctypes.POINTER(ctypes.c_double)
        L = ctypes.c_long
        lib.oracle_anchor_forward.argtypes = [D, D, D, D, L, L, L, L, L, ctypes.c_double]
        lib.oracle_anchor_slice.argtypes = [D, D, D, L, L, L, ctypes.c_double, D, D, D, D, D]
        lib.oracle_anchor_slice_rows.argtypes = [D, D, D, L, L, L, ctypes.c_double,
                                                 ctypes.POINTER(ctypes.c_long), L, D]
        lib.oracle_anchor_backward.argtypes = [D, D, D, D, D, D, D, L, L, L, L, L, ctypes.c_double]
        lib.oracle_full_attention.argtypes = [D, D, D, D, L, L, L, L, ctypes.c_double]
        lib.oracle_anchor_causal.argtypes = [D, D, D, D, L, L, L, L, L, ctypes.c_double]
        lib.oracle_anchor_causal.restype = ctypes.c_int
        lib.oracle_full_attention.restype = ctypes.c_int
        lib.oracle_anchor_slice_backward.argtypes = [D, D, D, D, L, L, L, ctypes.c_double, D, D, D]
        lib.oracle_anchor_block.argtypes = [D, D, D, D, D, L, L, L, L, L, L, ctypes.c_double]
        lib.oracle_anchor_block.restype = ctypes.c_int
        lib.oracle_anchor_block_slice.argtypes = [D, D, D, D, L, L, L, L, ctypes.c_double, D]
        lib.oracle_anchor_block_slice.restype = ctypes.c_int
        for f in (lib.oracle_anchor_forward, lib.oracle_anchor_slice, lib.oracle_anchor_slice_rows,
                  lib.oracle_anchor_backward, lib.oracle_anchor_slice_backward):
            f.restype = ctypes.c_int
        self._lib = lib

    def forward(self, Q, U, V, scale: float) -> np.ndarray:
        """H for Q, V [B][heads][n][d] and U [heads][m][d] (float64)."""
        Q, U, V = _f64(Q), _f64(U), _f64(V)
        B, heads, n, d = Q.shape
        m = U.shape[1]
        assert U.shape == (heads, m, d) and V.shape == Q.shape
        H = np.empty_like(Q)
        _check(self._lib.oracle_anchor_forward(_dp(Q), _dp(U), _dp(V), _dp(H), B, heads, n, m, d,
                                               float(scale)))
        return H

    def slice_forward(self, Q, U, V, scale: float) -> dict:
        """One slice (Q, V [n][d], U [m][d]) with its intermediates A, delta, W = A^T V,
        Wp = Delta^{-1} W and H."""
        Q, U, V = _f64(Q), _f64(U), _f64(V)
        n, d = Q.shape
        m = U.shape[0]
        out = {"A": np.empty((n, m)), "delta": np.empty(m), "W": np.empty((m, d)),
               "Wp": np.empty((m, d)), "H": np.empty((n, d))}
        _check(self._lib.oracle_anchor_slice(_dp(Q), _dp(U), _dp(V), n, m, d, float(scale),
                                             _dp(out["A"]), _dp(out["delta"]), _dp(out["W"]),
                                             _dp(out["Wp"]), _dp(out["H"])))
        return out

    def backward(self, Q, U, V, dH, scale: float) -> tuple:
        """(dQ, dU, dV) for Q, V, dH [B][heads][n][d] and U [heads][m][d]; dU sums the batch."""
        Q, U, V, dH = _f64(Q), _f64(U), _f64(V), _f64(dH)
        B, heads, n, d = Q.shape
        m = U.shape[1]
        assert U.shape == (heads, m, d) and V.shape == Q.shape and dH.shape == Q.shape
        dQ, dU, dV = np.empty_like(Q), np.empty_like(U), np.empty_like(V)
        _check(self._lib.oracle_anchor_backward(_dp(Q), _dp(U), _dp(V), _dp(dH), _dp(dQ), _dp(dU), _dp(dV),
                                                B, heads, n, m, d, float(scale)))
        return dQ, dU, dV

    def slice_backward(self, Q, U, V, dH, scale: float) -> tuple:
        """(dQ, dU, dV) of one slice (Q, V, dH [n][d], U [m][d]); dU is this slice's share."""
        Q, U, V, dH = _f64(Q), _f64(U), _f64(V), _f64(dH)
        n, d = Q.shape
        m = U.shape[0]
        dQ, dV, dU = np.empty((n, d)), np.empty((n, d)), np.zeros((m, d))
        _check(self._lib.oracle_anchor_slice_backward(_dp(Q), _dp(U), _dp(V), _dp(dH), n, m, d, float(scale),
                                                      _dp(dQ), _dp(dU), _dp(dV)))
        return dQ, dU, dV

    def full_attention(self, Q, K, V, scale: float) -> np.ndarray:
        """softmax(scale Q K^T) V for Q, V [B][heads][n][d] and K [heads][n][d] (float64)."""
        Q, K, V = _f64(Q), _f64(K), _f64(V)
        B, heads, n, d = Q.shape
        assert K.shape == (heads, n, d) and V.shape == Q.shape
        H = np.empty_like(Q)
        _check(self._lib.oracle_full_attention(_dp(Q), _dp(K), _dp(V), _dp(H), B, heads, n, d, float(scale)))
        return H

    def causal(self, Q, U, V, scale: float) -> np.ndarray:
        """The masked (causal) variant: token i's anchor summaries use tokens j <= i only."""
        Q, U, V = _f64(Q), _f64(U), _f64(V)
        B, heads, n, d = Q.shape
        m = U.shape[1]
        assert U.shape == (heads, m, d) and V.shape == Q.shape
        H = np.empty_like(Q)
        _check(self._lib.oracle_anchor_causal(_dp(Q), _dp(U), _dp(V), _dp(H), B, heads, n, m, d, float(scale)))
        return H

    def block(self, X, Wq, Wv, U, scale: float) -> np.ndarray:
        """The block front end: Q = X Wq^T and V = X Wv^T per head, then the forward.
        X [B][n][dm]; Wq, Wv [heads][d][dm]; U [heads][m][d]; returns H [B][heads][n][d]."""
        X, Wq, Wv, U = _f64(X), _f64(Wq), _f64(Wv), _f64(U)
        B, n, dm = X.shape
        heads, m, d = U.shape
        assert Wq.shape == (heads, d, dm) and Wv.shape == Wq.shape
        H = np.empty((B, heads, n, d))
        _check(self._lib.oracle_anchor_block(_dp(X), _dp(Wq), _dp(Wv), _dp(U), _dp(H), B, heads, n, m, d, dm,
                                             float(scale)))
        return H

    def block_slice(self, X, Wq, Wv, U, scale: float) -> np.ndarray:
        """One slice of the block front end: X [n][dm], Wq, Wv [d][dm], U [m][d] -> H [n][d]."""
        X, Wq, Wv, U = _f64(X), _f64(Wq), _f64(Wv), _f64(U)
        n, dm = X.shape
        m, d = U.shape
        assert Wq.shape == (d, dm) and Wv.shape == Wq.shape
        H = np.empty((n, d))
        _check(self._lib.oracle_anchor_block_slice(_dp(X), _dp(Wq), _dp(Wv), _dp(U), n, m, d, dm, float(scale),
                                                   _dp(H)))
        return H

    @staticmethod
    def relative_frobenius(Href, H) -> np.ndarray:
        """Per (batch, head) slice: ||Href - H||_F / ||Href||_F, in float64 (the approximation
        error of the anchor construction against full attention)."""
        a = np.asarray(Href, dtype=np.float64)
        b = np.asarray(H, dtype=np.float64)
        num = np.sqrt(((a - b) ** 2).sum(axis=(-2, -1)))
        den = np.sqrt((a ** 2).sum(axis=(-2, -1)))
        return num / den

    def slice_rows(self, Q, U, V, scale: float, rows) -> np.ndarray:
        """H rows ``rows`` of one slice (Q, V [n][d], U [m][d])."""
        Q, U, V = _f64(Q), _f64(U), _f64(V)
        n, d = Q.shape
        m = U.shape[0]
        r = np.ascontiguousarray(rows, dtype=np.int64).astype(np.dtype("l"))
        Hr = np.empty((len(r), d))
        _check(self._lib.oracle_anchor_slice_rows(_dp(Q), _dp(U), _dp(V), n, m, d, float(scale),
                                                  r.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
                                                  len(r), _dp(Hr)))
        return Hr


def _dp(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _check(rc: int) -> None:
    if rc == 1:
        raise ValueError("oracle: bad argument")
    if rc == 2:
        raise MemoryError("oracle: out of memory")


def _default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def forward(Q, U, V, scale: float) -> np.ndarray:
    return _default().forward(Q, U, V, scale)


def slice_forward(Q, U, V, scale: float) -> dict:
    return _default().slice_forward(Q, U, V, scale)


def slice_rows(Q, U, V, scale: float, rows) -> np.ndarray:
    return _default().slice_rows(Q, U, V, scale, rows)


def causal(Q, U, V, scale: float) -> np.ndarray:
    return _default().causal(Q, U, V, scale)


def full_attention(Q, K, V, scale: float) -> np.ndarray:
    return _default().full_attention(Q, K, V, scale)


def relative_frobenius(Href, H) -> np.ndarray:
    return Oracle.relative_frobenius(Href, H)


def block(X, Wq, Wv, U, scale: float) -> np.ndarray:
    return _default().block(X, Wq, Wv, U, scale)


def block_slice(X, Wq, Wv, U, scale: float) -> np.ndarray:
    return _default().block_slice(X, Wq, Wv, U, scale)


def backward(Q, U, V, dH, scale: float) -> tuple:
    return _default().backward(Q, U, V, dH, scale)


def slice_backward(Q, U, V, dH, scale: float) -> tuple:
    return _default().slice_backward(Q, U, V, dH, scale)


def compile_variant(source_text: str, out_path: str) -> Oracle:
    """Compile a modified copy of the oracle source (used by the tests that plant a mistake
    in the oracle to show that the pins catch it)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                    "-ffp-contract=off", "-o", out_path, src, "-lm"], check=True)
    return Oracle(out_path)


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()
