"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: the pages' worked
example, closed forms (identity, permutation, rank-1), brute force in plain
Python on tiny shapes, exhaustive decoding against numpy's IEEE types, and
rounding against numpy's correctly rounded casts and an exhaustive
nearest-value search.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
import synth
from synth import BF16, F16, F32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            out[k] = v
    return out


class Op:
    """Minimal operand record for hand-built matrices."""

    def __init__(self, buf, dtype, ld, trans=False, bstride=0):
        self.buf, self.dtype, self.ld, self.trans, self.bstride = buf, dtype, ld, trans, bstride


def _f32(a):
    return Op(np.ascontiguousarray(np.asarray(a, dtype=np.float32).ravel()), F32,
              np.asarray(a).shape[1])


def test_worked_example_transposed_view():
    """d . d^T with the rhs read through the strided view, as printed."""
    g = _golden("transposed_rhs.txt")
    d = np.array([float(x) for x in g["d"]], dtype=np.float32)
    A = Op(d, F32, 3)                          # 2x3 row-major
    s0, s1 = (int(x) for x in g["t_strides"])  # t[r][c] at r*1 + c*3
    assert (s0, s1) == (1, 3)
    B = Op(d, F32, 3, trans=True)              # 3x2 logical, column-major view of d
    # the view's logical values are the ones the page prints for into_data(t)
    t_logical = [d[r * s0 + c * s1] for r in range(3) for c in range(2)]
    assert t_logical == [float(x) for x in g["t_logical"]]
    C = oracle.gemm_f64(A, B, 2, 2, 3)
    assert C.ravel().tolist() == [float(x) for x in g["dt"]]
    assert 21 ** 2 + 42 ** 2 + 63 ** 2 == 6174


@pytest.mark.parametrize("M,N,K", [(5, 7, 3), (16, 9, 33), (1, 1, 1)])
def test_identity(M, N, K):
    rng = np.random.default_rng(1)
    A = rng.integers(-50, 50, (M, K)).astype(np.float32)
    B = rng.integers(-50, 50, (K, N)).astype(np.float32)
    I_K = np.eye(K, dtype=np.float32)
    np.testing.assert_array_equal(oracle.gemm_f64(_f32(A), _f32(I_K), M, K, K)[0], A)
    np.testing.assert_array_equal(oracle.gemm_f64(_f32(I_K), _f32(B), K, N, K)[0], B)
    R = np.eye(K, N, dtype=np.float32)  # rectangular identity: keeps the first min(K,N) cols
    expect = np.zeros((M, N))
    expect[:, :min(K, N)] = A[:, :min(K, N)]
    np.testing.assert_array_equal(oracle.gemm_f64(_f32(A), _f32(R), M, N, K)[0], expect)


def test_permutation_rows_and_cols():
    rng = np.random.default_rng(2)
    M, K, N = 9, 9, 6
    B = rng.standard_normal((K, N)).astype(np.float32)
    perm = rng.permutation(K)
    P = np.zeros((M, K), dtype=np.float32)
    P[np.arange(M), perm] = 1.0
    C = oracle.gemm_f64(_f32(P), _f32(B), M, N, K)[0]
    np.testing.assert_array_equal(C, B[perm].astype(np.float64))
    # column permutation from the right: A . Q permutes columns
    A = rng.standard_normal((4, K)).astype(np.float32)
    Q = np.zeros((K, K), dtype=np.float32)
    Q[perm, np.arange(K)] = 1.0
    C2 = oracle.gemm_f64(_f32(A), _f32(Q), 4, K, K)[0]
    np.testing.assert_array_equal(C2, A[:, perm].astype(np.float64))


def test_rank1_closed_form():
    """A = u 1^T, B = 1 v^T  =>  C = K u v^T exactly (integers)."""
    M, N, K = 7, 5, 11
    u = np.arange(1, M + 1, dtype=np.float32) * np.array([(-1) ** i for i in range(M)])
    v = np.arange(2, N + 2, dtype=np.float32) * 3
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[None, :], K, axis=0)
    C = oracle.gemm_f64(_f32(A), _f32(B), M, N, K)[0]
    np.testing.assert_array_equal(C, K * np.outer(u, v))


def _brute(Aop, Bop, M, N, K, batch):
    """Independent plain-Python double loop over the same bits."""
    a = oracle_free_decode(Aop)
    b = oracle_free_decode(Bop)
    out = []
    for bi in range(batch):
        for i in range(M):
            for j in range(N):
                s = 0.0
                for k in range(K):
                    s += a[Aop.index(bi, i, k)] * b[Bop.index(bi, k, j)]
                out.append(s)
    return np.array(out).reshape(batch, M, N)


def oracle_free_decode(op):
    """numpy's own IEEE types decode the storage (not the oracle's routine)."""
    if op.dtype == F32:
        return [float(x) for x in op.buf]
    if op.dtype == F16:
        return [float(x) for x in op.buf.astype(np.float16)]
    bits = op.buf.astype(np.uint32) << np.uint32(16)
    return [float(x) for x in bits.view(np.float32)]


@pytest.mark.parametrize("dt", [BF16, F16, F32])
@pytest.mark.parametrize("at,bt", list(itertools.product([False, True], repeat=2)))
@pytest.mark.parametrize("M,N,K,batch", [(1, 1, 1, 1), (3, 5, 7, 1), (7, 9, 11, 3), (2, 4, 1, 2)])
def test_brute_force_tiny(dt, at, bt, M, N, K, batch):
    A = synth.make_operand(11, dt, M, K, trans=at, batch=batch, dist="normal",
                           ld=(M if at else K) + 2)
    B = synth.make_operand(12, dt, K, N, trans=bt, batch=batch, dist="normal",
                           ld=(K if bt else N) + 1,
                           bstride=None if batch == 1 else synth.span(K, N, (K if bt else N) + 1, bt) + 5)
    C = oracle.gemm_f64(A, B, M, N, K, batch)
    R = _brute(A, B, M, N, K, batch)
    # same k order, same binary64 arithmetic: identical
    np.testing.assert_array_equal(C, R)
    # NaN padding is never read
    assert np.isfinite(C).all()


def test_points_match_full():
    A = synth.make_operand(3, BF16, 13, 40, dist="normal")
    B = synth.make_operand(4, BF16, 40, 17, trans=True, dist="normal")
    C = oracle.gemm_f64(A, B, 13, 17, 40)
    pts = np.array([[0, i, j] for i in range(13) for j in range(17)])
    P = oracle.gemm_points(A, B, 40, pts)
    np.testing.assert_array_equal(P, C.reshape(-1))


def test_thread_count_changes_nothing():
    """Each output is one fixed-order fp64 sum, so the oracle's value cannot
    depend on how many threads share the outputs (one core is timed beside
    all of them)."""
    A = synth.make_operand(5, BF16, 37, 300, dist="normal")
    B = synth.make_operand(6, BF16, 300, 29, dist="normal")
    full = oracle.num_threads()
    C = oracle.gemm_f64(A, B, 37, 29, 300)
    pts = np.array([[0, i, j] for i in range(37) for j in range(29)])
    P = oracle.gemm_points(A, B, 300, pts)
    oracle.set_num_threads(1)
    try:
        assert oracle.num_threads() == 1 or full == 1
        C1 = oracle.gemm_f64(A, B, 37, 29, 300)
        P1 = oracle.gemm_points(A, B, 300, pts)
    finally:
        oracle.set_num_threads(full)
    assert oracle.num_threads() == full
    np.testing.assert_array_equal(C1, C)
    np.testing.assert_array_equal(P1, P)


def _decode_via_gemm(bits, dtype):
    """Expose the oracle's input decoding through the public gemm: C = A . [1]."""
    A = Op(bits, dtype, 1)
    one = Op(np.array([1.0], dtype=np.float32), F32, 1)
    return oracle.gemm_f64(A, one, bits.size, 1, 1)[0, :, 0]


def test_decode_bf16_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = _decode_via_gemm(bits, BF16)
    ref = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_decode_f16_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = _decode_via_gemm(bits, F16)
    ref = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def _bf16_values():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return bits, v


def test_round_bf16_special_values():
    cases = {
        1.0: 0x3F80, -1.0: 0xBF80, 0.0: 0x0000,
        1.0 + 2 ** -8: 0x3F80,            # tie between 1 and 1+2^-7 -> even (1)
        1.0 + 3 * 2 ** -8: 0x3F82,        # tie between 1+2^-7 and 1+2^-6 -> even
        1.0 + 2 ** -8 + 2 ** -30: 0x3F81,  # just above the tie -> up
        2.0 ** 127 * (2 - 2 ** -7): 0x7F7F,  # max finite
        2.0 ** 128: 0x7F80,               # overflow -> inf
        2.0 ** 127 * (2 - 2 ** -8): 0x7F80,  # tie at the top rounds to even = 2^128 -> inf
        2.0 ** -133: 0x0001,              # smallest subnormal
        2.0 ** -134: 0x0000,              # tie with 0 -> even (0)
        3 * 2.0 ** -134: 0x0002,          # tie between 1 and 2 quanta -> even
        -(2.0 ** -126): 0x8080,           # smallest normal, negative
    }
    x = np.array(list(cases), dtype=np.float64)
    got = oracle.round_out(x, BF16)
    assert [int(g) for g in got] == list(cases.values())


def test_round_bf16_nearest_search():
    """Random doubles: the result is the nearest bf16 value, ties to even bits."""
    bits, vals = _bf16_values()
    fin = np.isfinite(vals) & (bits < 0x8000)
    pos_bits, pos_vals = bits[fin], vals[fin]
    order = np.argsort(pos_vals, kind="stable")
    pos_bits, pos_vals = pos_bits[order], pos_vals[order]
    # drop the duplicate +0 / -0 (only +0 is in the non-negative set already)
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-40, 38, 4000),
        rng.standard_normal(500) * 1e-39,
    ])
    got = oracle.round_out(x, BF16)
    for xv, g in zip(x, got):
        ax = abs(xv)
        i = np.searchsorted(pos_vals, ax)
        cand = []
        for j in (i - 1, i):
            if 0 <= j < len(pos_vals):
                cand.append((abs(pos_vals[j] - ax), int(pos_bits[j] & 1), int(pos_bits[j])))
        cand.sort()
        best = cand[0]
        if len(cand) > 1 and cand[1][0] == best[0]:   # tie -> even significand bit
            best = min(cand, key=lambda c: (c[0], c[1]))
        want = best[2] | (0x8000 if xv < 0 else 0)
        assert int(g) == want, (xv, hex(int(g)), hex(want))


def test_round_f16_matches_numpy():
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
                        [65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -25,
                         -0.0, 1e10, -1e10]])
    got = oracle.round_out(x, F16)
    ref = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_round_f32_matches_numpy():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(10000) * 10.0 ** rng.integers(-40, 38, 10000)
    np.testing.assert_array_equal(oracle.round_out(x, F32), x.astype(np.float32))


def test_integer_inputs_exact_at_K4096():
    """Integers in {-4..4}, K = 4096: |partial sums| <= 16*4096 < 2^24, so the
    fp64 result is an exact integer representable in fp32 and bf16 rounding of
    it is a single rounding."""
    M, N, K = 3, 5, 4096
    A = synth.make_operand(21, BF16, M, K, dist="int4")
    B = synth.make_operand(22, BF16, K, N, dist="int4")
    C = oracle.gemm_f64(A, B, M, N, K)
    assert np.array_equal(C, np.round(C))
    assert np.abs(C).max() <= 16 * K
    a = oracle.decode(A.buf, BF16).reshape(M, K).astype(np.int64)
    b = oracle.decode(B.buf, BF16).reshape(K, N).astype(np.int64)
    np.testing.assert_array_equal(C[0], (a @ b).astype(np.float64))  # integer matmul
