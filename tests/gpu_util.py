"""Helpers shared by the GPU tests: move synth operands to the device, run a
candidate or the tuner through the C ABI, compare with the oracle."""
from __future__ import annotations

import numpy as np

import oracle
import synth

BF16, F16, F32 = synth.BF16, synth.F16, synth.F32
TOL_REL_FRO = 2e-3   # relative Frobenius error bound for real-valued inputs


def torch():
    import torch as t
    return t


def to_device(op, offset_bytes: int = 0):
    """Copy an operand's flat buffer to a device byte tensor; returns (tensor, ptr).

    offset_bytes shifts the data inside the allocation (to test misaligned
    base pointers)."""
    t = torch()
    raw = op.buf.view(np.uint8)
    dev = t.zeros(raw.size + offset_bytes + 256, dtype=t.uint8, device="cuda")
    dev[offset_bytes:offset_bytes + raw.size].copy_(t.from_numpy(raw.copy()))
    return dev, dev.data_ptr() + offset_bytes


def from_device(dev, op, offset_bytes: int = 0) -> np.ndarray:
    n = op.buf.view(np.uint8).size
    raw = dev[offset_bytes:offset_bytes + n].cpu().numpy()
    return raw.view(op.buf.dtype)


def logical_out(op, flat: np.ndarray) -> np.ndarray:
    """The batch x rows x cols logical outputs of a row-major output operand."""
    out = np.empty((op.batch, op.rows, op.cols), dtype=flat.dtype)
    for b in range(op.batch):
        for r in range(op.rows):
            base = b * op.bstride + r * op.ld
            out[b, r] = flat[base:base + op.cols]
    return out


def padding_untouched(op, flat: np.ndarray) -> bool:
    """Every element outside the logical output still holds the NaN sentinel."""
    mask = np.ones(flat.size, dtype=bool)
    for b in range(op.batch):
        for r in range(op.rows):
            base = b * op.bstride + r * op.ld
            mask[base:base + op.cols] = False
    rest = flat[mask]
    if rest.size == 0:
        return True
    if op.dtype == BF16:
        return bool(np.all(rest == 0x7FC0))
    return bool(np.all(np.isnan(rest.astype(np.float32))))


def decode(vals: np.ndarray, dtype: int) -> np.ndarray:
    return oracle.decode(vals, dtype)


class Case:
    """One problem: operands on host and device, oracle result."""

    def __init__(self, M, N, K, layout="NN", dt=(BF16, BF16, F32), dist="u11", batch=1,
                 pad=(0, 0, 0), seed=1000, a_off=0, b_off=0, c_off=0, dist_b=None,
                 bstride_extra=(0, 0, 0)):
        self.M, self.N, self.K = M, N, K
        self.layout, self.dt, self.batch = layout, dt, batch
        at, bt = layout[0] == "T", layout[1] == "T"
        lda = (M if at else K) + pad[0]
        ldb = (K if bt else N) + pad[1]
        ldc = N + pad[2]
        lda, ldb, ldc = max(lda, 1), max(ldb, 1), max(ldc, 1)
        sa = synth.span(M, K, lda, at) + bstride_extra[0] if batch > 1 else None
        sb = synth.span(K, N, ldb, bt) + bstride_extra[1] if batch > 1 else None
        sc = synth.span(M, N, ldc, False) + bstride_extra[2] if batch > 1 else None
        self.A = synth.make_operand(seed, dt[0], M, K, ld=lda, trans=at, batch=batch,
                                    bstride=sa, dist=dist)
        self.B = synth.make_operand(seed + 1, dt[1], K, N, ld=ldb, trans=bt, batch=batch,
                                    bstride=sb, dist=dist_b or dist)
        self.C = synth.output_buffer(dt[2], M, N, ld=ldc, batch=batch, bstride=sc)
        self.offs = (a_off, b_off, c_off)
        self._c64 = None

    @property
    def c64(self):
        if self._c64 is None:
            self._c64 = oracle.gemm_f64(self.A, self.B, self.M, self.N, self.K, self.batch)
        return self._c64

    def device(self):
        self.dA, self.pA = to_device(self.A, self.offs[0])
        self.dB, self.pB = to_device(self.B, self.offs[1])
        self.dC, self.pC = to_device(self.C, self.offs[2])
        return self

    def args(self):
        b = None
        if self.batch != 1:
            b = (self.batch, self.A.bstride, self.B.bstride, self.C.bstride)
        return (self.pA, self.pB, self.pC, self.M, self.N, self.K, self.A.ld, self.B.ld,
                self.C.ld, self.dt, self.layout, b)

    def result(self) -> np.ndarray:
        torch().cuda.synchronize()
        return from_device(self.dC, self.C, self.offs[2])

    def check(self, exact: bool, tol: float = TOL_REL_FRO):
        flat = self.result()
        assert padding_untouched(self.C, flat), "output padding was written"
        got = logical_out(self.C, flat)
        if exact:
            want = oracle.round_out(self.c64, self.dt[2])
            if not np.array_equal(got.view(np.uint8), want.view(np.uint8)):
                g = decode(got, self.dt[2])
                w = decode(want, self.dt[2])
                bad = np.argwhere(g != w)
                raise AssertionError(f"{len(bad)} mismatches, first at {bad[0].tolist()}: "
                                     f"got {g[tuple(bad[0])]} want {w[tuple(bad[0])]}")
            return 0.0
        g = decode(got, self.dt[2])
        ref = self.c64
        num = np.linalg.norm((g - ref).ravel())
        den = np.linalg.norm(ref.ravel())
        err = num / den if den > 0 else num
        assert np.isfinite(g).all(), "non-finite output"
        assert err <= tol, f"relative Frobenius error {err:.3e} > {tol}"
        return err
