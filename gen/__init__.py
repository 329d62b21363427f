"""Seeded synthetic inputs for the anchor-attention forward (shared by tests and bench).

This module holds no arithmetic of the method: it only draws Q, U and V.

Generator
---------
Counter-based, so that any element (or any slice of a tensor) can be drawn on its own:

* ``splitmix64`` (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): output k of a stream with state ``key`` is
  ``mix(key + (k + 1) * 0x9E3779B97F4A7C15)`` with the published 64-bit finaliser ``mix``.
* Stream key for (seed, stream id): ``mix(mix(seed + G) + stream * G)``, G the golden-ratio
  constant above.  Stream ids: Q=1, V=2, U=3, K=4, row choice=5, noise=6; for the block
  front end X=7, Wq=8, Wv=9.
* Uniform in (0, 1): ``((x >> 11) + 0.5) * 2**-53``.
* Normal: Box-Muller on the pair (2p, 2p+1) of uniforms: element 2p takes the cosine
  branch and element 2p+1 the sine branch.
* Rounding: float64 -> float32 (round to nearest even), and for bf16 a further
  round-to-nearest-even on the float32 bit pattern.  bf16 tensors are returned as uint16
  bit patterns.

Workloads
---------
The ViT-shaped shapes and value distributions the anchor-attention forward is measured on
(AnchorFormer, arXiv 2505.16463: DeiT classification at 197 tokens, COCO detection at
800x1344 with 16-pixel patches = 50x84 = 4200 tokens, and a long-sequence stress case).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "splitmix64", "uniform", "normal", "round_bf16", "bf16_to_f32",
    "make_inputs", "slice_inputs", "make_keys", "BlockWorkload", "BLOCK_WORKLOADS", "make_block_inputs",
]

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_Q, STREAM_V, STREAM_U, STREAM_K, STREAM_ROWS, STREAM_NOISE = 1, 2, 3, 4, 5, 6
STREAM_X, STREAM_WQ, STREAM_WV = 7, 8, 9

_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        a = _mix(np.array([seed], dtype=np.uint64) + _G)
        return _mix(a + np.uint64(stream) * _G)[0]


def splitmix64(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the splitmix64 stream whose state is ``key``."""
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + k * _G)


def uniform(key: np.uint64, start: int, count: int) -> np.ndarray:
    x = splitmix64(key, start, count)
    return ((x >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Standard normals for element indices start .. start+count-1 (float64)."""
    out = np.empty(count, dtype=np.float64)
    pos = 0
    while pos < count:
        c = min(_CHUNK, count - pos)
        k0 = start + pos
        p0 = k0 // 2
        p1 = (k0 + c - 1) // 2
        npair = p1 - p0 + 1
        u = uniform(key, 2 * p0, 2 * npair).reshape(npair, 2)
        r = np.sqrt(-2.0 * np.log(u[:, 0]))
        t = 2.0 * math.pi * u[:, 1]
        z = np.empty((npair, 2), dtype=np.float64)
        z[:, 0] = r * np.cos(t)
        z[:, 1] = r * np.sin(t)
        z = z.reshape(-1)
        off = k0 - 2 * p0
        out[pos:pos + c] = z[off:off + c]
        pos += c
    return out


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64/float32 -> bf16 bit patterns (uint16), round to nearest even via float32."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    heads: int
    n: int
    m: int
    d: int
    dtype: str          # "f32" or "bf16"
    recipe: str         # value distribution, see _draw_u / make_inputs
    about: str

    @property
    def slices(self) -> int:
        return self.B * self.heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def algorithmic_bytes(self) -> int:
        """Q, V and H once each plus U once (the roofline traffic of one forward)."""
        return (3 * self.slices * self.n * self.d + self.heads * self.m * self.d) * self.elem_bytes

    @property
    def flops(self) -> int:
        """Q.U^T, A^T.V and A.W' once each: 6 n m d per slice."""
        return 6 * self.slices * self.n * self.m * self.d

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS: dict[str, Workload] = {w.name: w for w in [
    Workload("vit14_f32", 1, 1, 196, 16, 64, "f32", "normal",
             "smallest case: one 14x14 patch grid, fp32, Q,V,U ~ N(0,1)"),
    Workload("deit_small", 64, 6, 197, 30, 64, "bf16", "u_half",
             "DeiT-Small shaped: 196 patches + cls, 30 anchors/head, U ~ N(0,1)/sqrt(2)"),
    Workload("deit_base", 256, 12, 197, 49, 64, "bf16", "u_from_k",
             "DeiT-Base shaped: 49 anchors taken from rows of a N(0,1) key matrix + N(0,0.1^2) noise"),
    Workload("det_800x1344", 8, 12, 4200, 64, 64, "bf16", "normal",
             "detection grid 800x1344 / patch 16 = 50x84 tokens, 64 anchors"),
    Workload("long_16k", 4, 16, 16384, 128, 128, "bf16", "q_peaked",
             "long-sequence stress: 16384 tokens, 128 anchors, d=128, Q = 4*N(0,1)"),
]}


def _draw_u(w: Workload, seed: int) -> np.ndarray:
    """U [heads][m][d] as float64 before rounding."""
    cnt = w.heads * w.m * w.d
    if w.recipe == "u_half":
        return (normal(_key(seed, STREAM_U), 0, cnt) / math.sqrt(2.0)).reshape(w.heads, w.m, w.d)
    if w.recipe == "u_from_k":
        # per head: a N(0,1) key matrix K [n][d]; m distinct rows chosen by a seeded
        # Fisher-Yates shuffle; plus N(0, 0.1^2) noise.
        K = normal(_key(seed, STREAM_K), 0, w.heads * w.n * w.d).reshape(w.heads, w.n, w.d)
        noise = normal(_key(seed, STREAM_NOISE), 0, cnt).reshape(w.heads, w.m, w.d)
        rk = _key(seed, STREAM_ROWS)
        U = np.empty((w.heads, w.m, w.d), dtype=np.float64)
        for h in range(w.heads):
            perm = list(range(w.n))
            u = uniform(rk, h * w.n, w.n)
            for i in range(w.n - 1, 0, -1):
                j = int(u[i] * (i + 1))
                perm[i], perm[j] = perm[j], perm[i]
            U[h] = K[h, perm[:w.m]] + 0.1 * noise[h]
        return U
    return normal(_key(seed, STREAM_U), 0, cnt).reshape(w.heads, w.m, w.d)


def make_keys(w: Workload, seed: int = 0) -> np.ndarray:
    """The per-head key matrix K [heads][n][d] of the workload, in its dtype: for the recipe
    that draws the anchors from the rows of K ("u_from_k") it is that same K, so that full
    softmax attention over K and anchor attention over U can be compared; for the others an
    independent N(0, 1) draw on the same stream."""
    K = normal(_key(seed, STREAM_K), 0, w.heads * w.n * w.d).reshape(w.heads, w.n, w.d)
    return _round(K, w.dtype)


def _round(x: np.ndarray, dtype: str) -> np.ndarray:
    return x.astype(np.float32) if dtype == "f32" else round_bf16(x)


def _draw_big(w: Workload, seed: int, stream: int, mult: float, start: int, count: int) -> np.ndarray:
    """Chunks are independent (counter-based), so they are drawn on a thread pool;
    numpy releases the GIL inside its ufuncs.  The result does not depend on the
    number of threads."""
    key = _key(seed, stream)
    out = np.empty(count, dtype=np.float32 if w.dtype == "f32" else np.uint16)

    def work(pos: int) -> None:
        c = min(_CHUNK, count - pos)
        z = normal(key, start + pos, c)
        if mult != 1.0:
            z *= mult
        out[pos:pos + c] = _round(z, w.dtype)

    starts = range(0, count, _CHUNK)
    if count <= _CHUNK:
        for p in starts:
            work(p)
    else:
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    return out


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Q, V [B][heads][n][d] and U [heads][m][d] in the workload's dtype.

    f32 -> float32 arrays; bf16 -> uint16 bit patterns.
    """
    qmult = 4.0 if w.recipe == "q_peaked" else 1.0
    cnt = w.slices * w.n * w.d
    Q = _draw_big(w, seed, STREAM_Q, qmult, 0, cnt).reshape(w.B, w.heads, w.n, w.d)
    V = _draw_big(w, seed, STREAM_V, 1.0, 0, cnt).reshape(w.B, w.heads, w.n, w.d)
    U = _round(_draw_u(w, seed), w.dtype).reshape(w.heads, w.m, w.d)
    return {"Q": Q, "U": U, "V": V}


def slice_inputs(w: Workload, b: int, h: int, seed: int = 0) -> dict:
    """The Q and V rows of one (batch, head) slice, identical to make_inputs()[..][b, h]."""
    qmult = 4.0 if w.recipe == "q_peaked" else 1.0
    per = w.n * w.d
    start = (b * w.heads + h) * per
    Q = _draw_big(w, seed, STREAM_Q, qmult, start, per).reshape(w.n, w.d)
    V = _draw_big(w, seed, STREAM_V, 1.0, start, per).reshape(w.n, w.d)
    return {"Q": Q, "V": V}


def to_float64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Widen stored inputs (float32 or bf16 bits) exactly to float64."""
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    return bf16_to_f32(x).astype(np.float64)


@dataclass(frozen=True)
class BlockWorkload:
    """The block front end: token embeddings X [B][n][dm] projected per head to Q and V by
    Wq, Wv [heads][d][dm], then the forward with the anchors of ``base`` (same B, heads, n,
    m, d).  X ~ N(0, 1) and W ~ N(0, 1/dm), so that Q and V are about N(0, 1) as in the
    forward's workloads."""
    name: str
    base: Workload      # the forward workload whose shape, dtype and anchor recipe this block uses
    dm: int
    about: str

    @property
    def w(self) -> Workload:
        return self.base

    @property
    def algorithmic_bytes(self) -> int:
        """X, the two projection matrices and U read once, H written once."""
        w = self.w
        return (w.B * w.n * self.dm + 2 * w.heads * w.d * self.dm + w.heads * w.m * w.d
                + w.slices * w.n * w.d) * w.elem_bytes

    @property
    def flops(self) -> int:
        """The two projections (2 n dm d flop each per slice) plus the forward's 6 n m d."""
        w = self.w
        return w.slices * w.n * (4 * self.dm * w.d + 6 * w.m * w.d)


BLOCK_WORKLOADS: dict[str, BlockWorkload] = {b.name: b for b in [
    BlockWorkload("deit_base_block", WORKLOADS["deit_base"], 768,
                  "DeiT-Base block: 197 tokens of width 768 projected to 12 heads of 64"),
    BlockWorkload("deit_small_block", WORKLOADS["deit_small"], 384,
                  "DeiT-Small block: 197 tokens of width 384 projected to 6 heads of 64"),
]}


def make_block_inputs(bw: BlockWorkload, seed: int = 0) -> dict:
    """X [B][n][dm], Wq, Wv [heads][d][dm] and U [heads][m][d] in the base workload's dtype."""
    w = bw.w
    X = _draw_big(w, seed, STREAM_X, 1.0, 0, w.B * w.n * bw.dm).reshape(w.B, w.n, bw.dm)
    wmult = 1.0 / math.sqrt(bw.dm)
    Wq = _draw_big(w, seed, STREAM_WQ, wmult, 0, w.heads * w.d * bw.dm).reshape(w.heads, w.d, bw.dm)
    Wv = _draw_big(w, seed, STREAM_WV, wmult, 0, w.heads * w.d * bw.dm).reshape(w.heads, w.d, bw.dm)
    U = _round(_draw_u(w, seed), w.dtype).reshape(w.heads, w.m, w.d)
    return {"X": X, "Wq": Wq, "Wv": Wv, "U": U}
