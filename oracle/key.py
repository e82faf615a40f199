"""Tuning-key oracle (test infrastructure only).

Restates the matmul tuning key of the burn "autotune" page (rustineverything.app
.../06-cubecl/autotune), section "tuning key: shape bucketing", field by field:

* m, n, k are anchored: Balanced rounds up to a power of two (base 2);
  Minimal uses base 2.5 (wider buckets), Extensive base 1.5, Full does not
  bucket.  Read here as: the smallest power of the base that is >= x,
  rounded up to an integer.
* the vectorisation (pow2) factor of an operand is the number of trailing
  zero bits of the anchored size of its contiguous dimension, at most 4.
  (The page says "of k or n"; read as: lhs -> k when stored row-major, m when
  stored transposed; rhs -> n when row-major, k when transposed.)
* the stride factor of an operand is the largest power of two (exponent, at
  most 10) dividing every stride in BYTES other than the unit one, using the
  real, un-anchored strides.  The strides counted are the leading dimension
  and, for a batch of more than one matrix, the batch stride.  A zero stride
  is divisible by every power of two.
* the layout is Contiguous, MildlyPermuted{transposed, batch_swap} or
  HighlyPermuted.  transposed = the operand is stored column-major;
  batch_swap = batch > 1 and the batch stride is smaller than the span of one
  matrix.  Our strides (one unit-stride dimension per matrix) cannot express
  HighlyPermuted.
* scale: every anchored dimension < 512 -> Small, every one < 2048 ->
  Medium, else Large.
* kind (names only on the page): first match of m=n=1 InnerProduct,
  k=1&m=1 ScalarVec, k=1&n=1 VecScalar, k=1 OuterProduct, m=1 VecMat,
  n=1 MatVec, else General -- on anchored sizes.
* the anchored batch count is part of the key.
"""
from __future__ import annotations

import math

LEVELS = {"minimal": 2.5, "balanced": 2.0, "extensive": 1.5, "full": None}
DTYPE_NAME = {0: "bf16", 1: "f16", 2: "f32"}
DTYPE_BYTES = {0: 2, 1: 2, 2: 4}


def anchor(x: int, level: str = "balanced") -> int:
    base = LEVELS[level]
    if base is None or x <= 1:
        return int(x)
    p = 1.0
    while p < x:
        p *= base
    return int(math.ceil(p))


def trailing_zeros(v: int, cap: int) -> int:
    if v == 0:
        return cap
    n = 0
    while v % 2 == 0 and n < cap:
        v //= 2
        n += 1
    return n


def pow2_factor(anchored: int) -> int:
    return trailing_zeros(anchored, 4)


def stride_factor(strides_bytes) -> int:
    f = 10
    for s in strides_bytes:
        f = min(f, trailing_zeros(abs(int(s)), 10))
    return f


def span(rows, cols, ld, trans):
    if rows == 0 or cols == 0:
        return 0
    outer, inner = (cols, rows) if trans else (rows, cols)
    return (outer - 1) * ld + inner


def layout_name(trans: bool, batch_swap: bool) -> str:
    if not trans and not batch_swap:
        return "Contiguous"
    return "MildlyPermuted{transposed:%s,batch_swap:%s}" % (
        "true" if trans else "false", "true" if batch_swap else "false")


def scale(m, n, k) -> str:
    if m < 512 and n < 512 and k < 512:
        return "Small"
    if m < 2048 and n < 2048 and k < 2048:
        return "Medium"
    return "Large"


def kind(m, n, k) -> str:
    if m == 1 and n == 1:
        return "InnerProduct"
    if k == 1 and m == 1:
        return "ScalarVec"
    if k == 1 and n == 1:
        return "VecScalar"
    if k == 1:
        return "OuterProduct"
    if m == 1:
        return "VecMat"
    if n == 1:
        return "MatVec"
    return "General"


def make_key(M, N, K, lda, ldb, dt_a, dt_b, dt_c, a_trans=False, b_trans=False,
             batch=1, stride_a=0, stride_b=0, level="balanced") -> dict:
    """The key as an ordered dict of field -> value."""
    m, n, k = anchor(M, level), anchor(N, level), anchor(K, level)
    ea, eb = DTYPE_BYTES[dt_a], DTYPE_BYTES[dt_b]
    a_strides = [lda * ea] + ([stride_a * ea] if batch > 1 else [])
    b_strides = [ldb * eb] + ([stride_b * eb] if batch > 1 else [])
    a_swap = batch > 1 and stride_a < span(M, K, lda, a_trans)
    b_swap = batch > 1 and stride_b < span(K, N, ldb, b_trans)
    return {
        "m": m, "n": n, "k": k, "batch": anchor(batch, level),
        "lhs_pow2": pow2_factor(m if a_trans else k),
        "lhs_stride": stride_factor(a_strides),
        "rhs_pow2": pow2_factor(k if b_trans else n),
        "rhs_stride": stride_factor(b_strides),
        "elem_lhs": DTYPE_NAME[dt_a], "elem_rhs": DTYPE_NAME[dt_b], "elem_out": DTYPE_NAME[dt_c],
        "layout_lhs": layout_name(a_trans, a_swap),
        "layout_rhs": layout_name(b_trans, b_swap),
        "scale": scale(m, n, k),
        "kind": kind(m, n, k),
    }


def key_text(fields: dict) -> str:
    return " ".join(f"{k}={v}" for k, v in fields.items())


def parse_key_text(text: str) -> dict:
    out = {}
    for tok in text.split():
        k, v = tok.split("=", 1)
        out[k] = int(v) if v.lstrip("-").isdigit() else v
    return out
