"""Seeded synthetic inputs for the matmul tests and the benchmark.

This module only draws numbers and lays them out in memory; it holds none of
the matmul or tuning arithmetic, so both the CUDA path and the CPU oracle can
consume its output without sharing any of the method's code.

Generator: splitmix64 used as a counter-based generator (value i of a stream
is splitmix64's output for state seed + (i+1)*0x9E3779B97F4A7C15), its top 53
bits as a uniform double in [0, 1).  Normals use the Box-Muller transform on
consecutive pairs.  Values are then stored in the operand dtype: float32 by
IEEE round-to-nearest-even (numpy's cast), bfloat16 by a further
round-to-nearest-even of that float32 to its top 16 bits, float16 by numpy's
cast.  Whatever the rounding, the stored bits ARE the input: both sides read
the same bits.

Strided operands are generated as one flat buffer of the whole span; elements
that the logical matrix does not cover (row padding beyond the logical
columns, gaps between batch items) are filled with NaN so that a kernel that
reads them poisons its result.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

BF16, F16, F32 = 0, 1, 2
DTYPE_NAMES = {BF16: "bf16", F16: "f16", F32: "f32"}
DTYPE_BYTES = {BF16: 2, F16: 2, F32: 4}


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n consecutive outputs of a splitmix64 stream, starting at counter offset."""
    i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, n: int) -> np.ndarray:
    return (splitmix64(seed, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def draw(seed: int, n: int, dist: str) -> np.ndarray:
    """n float64 draws of a named distribution.

    dist: "u11" uniform [-1,1); "int4" integers uniform in {-4..4};
    "normal" N(0,1); "normal:<sigma>" N(0, sigma^2).
    """
    if dist == "u11":
        return uniform01(seed, n) * 2.0 - 1.0
    if dist == "int4":
        return (splitmix64(seed, n) % np.uint64(9)).astype(np.int64).astype(np.float64) - 4.0
    if dist.startswith("normal"):
        sigma = float(dist.split(":", 1)[1]) if ":" in dist else 1.0
        m = (n + 1) // 2
        u = uniform01(seed, 2 * m)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))
        t = 2.0 * math.pi * u2
        z = np.empty(2 * m, dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        return z[:n] * sigma
    raise ValueError(f"unknown distribution {dist!r}")


def to_storage(x: np.ndarray, dtype: int) -> np.ndarray:
    """Store float64 values in the operand dtype; returns the raw element array.

    bf16 is returned as uint16 bit patterns, f16 as float16, f32 as float32.
    """
    if dtype == F32:
        return x.astype(np.float32)
    if dtype == F16:
        return x.astype(np.float16)
    if dtype == BF16:
        f = x.astype(np.float32)
        bits = f.view(np.uint32).astype(np.uint64)
        nan = np.isnan(f)
        lsb = (bits >> np.uint64(16)) & np.uint64(1)
        r = ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
        r[nan] = np.uint16(0x7FC0)
        return r
    raise ValueError(dtype)


def storage_nan(dtype: int):
    if dtype == BF16:
        return np.uint16(0x7FC0)
    if dtype == F16:
        return np.float16("nan")
    return np.float32("nan")


@dataclass
class Operand:
    """A logical rows x cols matrix (optionally batched) in a flat buffer.

    trans=False: element (b, r, c) at b*bstride + r*ld + c   (row-major, "N")
    trans=True:  element (b, r, c) at b*bstride + c*ld + r   (column-major, "T")
    """

    buf: np.ndarray          # flat storage array (uint16 for bf16)
    dtype: int
    rows: int
    cols: int
    ld: int
    trans: bool
    batch: int
    bstride: int

    def index(self, b, r, c):
        if self.trans:
            return b * self.bstride + c * self.ld + r
        return b * self.bstride + r * self.ld + c


def span(rows: int, cols: int, ld: int, trans: bool, batch: int = 1, bstride: int = 0) -> int:
    """Elements from the first to one past the last addressed element."""
    if rows == 0 or cols == 0 or batch == 0:
        return 0
    outer, inner = (cols, rows) if trans else (rows, cols)
    one = (outer - 1) * ld + inner
    return (batch - 1) * bstride + one if batch > 1 else one


def make_operand(seed: int, dtype: int, rows: int, cols: int, *, ld: int | None = None,
                 trans: bool = False, batch: int = 1, bstride: int | None = None,
                 dist: str = "u11") -> Operand:
    """Draw a (batch x) rows x cols operand; values in logical row-major order.

    The logical values of item b are draws [b*rows*cols, (b+1)*rows*cols) of
    the stream, laid out row-major, whatever the storage layout.
    """
    inner = rows if trans else cols
    outer = cols if trans else rows
    if ld is None:
        ld = max(inner, 1)
    one = span(rows, cols, ld, trans)
    if bstride is None:
        bstride = one if batch > 1 else 0
    total = span(rows, cols, ld, trans, batch, bstride)
    buf = np.full(total, storage_nan(dtype), dtype=to_storage(np.zeros(1), dtype).dtype)
    vals = to_storage(draw(seed, batch * rows * cols, dist), dtype).reshape(batch, rows, cols)
    for b in range(batch):
        base = b * bstride
        if rows == 0 or cols == 0:
            continue
        v = vals[b].T if trans else vals[b]      # shape (outer, inner)
        idx = base + (np.arange(outer)[:, None] * ld + np.arange(inner)[None, :])
        buf[idx] = v
    return Operand(buf=buf, dtype=dtype, rows=rows, cols=cols, ld=ld, trans=trans,
                   batch=batch, bstride=bstride)


def output_buffer(dtype: int, rows: int, cols: int, ld: int | None = None,
                  batch: int = 1, bstride: int | None = None) -> Operand:
    """A NaN-filled row-major output operand (C is always stored row-major)."""
    if ld is None:
        ld = max(cols, 1)
    one = span(rows, cols, ld, False)
    if bstride is None:
        bstride = one if batch > 1 else 0
    total = span(rows, cols, ld, False, batch, bstride)
    buf = np.full(total, storage_nan(dtype), dtype=to_storage(np.zeros(1), dtype).dtype)
    return Operand(buf=buf, dtype=dtype, rows=rows, cols=cols, ld=ld, trans=False,
                   batch=batch, bstride=bstride)
