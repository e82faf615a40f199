"""The split-K GEMM entry point that allocates nothing (GPU).

It exists for callers that may not call cudaMalloc/cudaFree (a server that
reserves all device memory at start-up, a plugin inside a framework that owns
the allocator, a loop that cannot take an allocation's implicit device
synchronisation).  It must give the same product as the regular entry point,
call after call, while the device's free memory stays put.  This file is
collected last so a failure here cannot hide the rest of the GPU suite.
"""
import numpy as np
import pytest

import matmul_selection_gb300 as mm
import oracle
from gpu_util import BF16, F32, Case, logical_out, padding_untouched

pytestmark = pytest.mark.gpu


def _noalloc(c):
    st = mm.mm_splitk_gemm_noalloc(c.pA, c.pB, c.pC, c.M, c.N, c.K, c.A.ld, c.B.ld, c.C.ld,
                                   c.dt, c.layout)
    if st == mm.MM_OK:  # no kernel of the call gave up a bounded wait
        st = mm.mm_splitk_gemm_noalloc_status()
    return st


def _regular(c):
    return mm.mm_autotune_execute(*c.args())


@pytest.mark.parametrize("layout", ["NN", "NT", "TN"])
def test_noalloc_matches_regular_entry_point_twice(layout):
    import torch
    ref = Case(256, 192, 8192, layout=layout, dt=(BF16, BF16, F32), dist="normal",
               seed=31).device()
    mm.check(_regular(ref))
    want = logical_out(ref.C, ref.result()).astype(np.float64)
    ref.check(exact=False)                       # the regular path against the oracle

    c = Case(256, 192, 8192, layout=layout, dt=(BF16, BF16, F32), dist="normal",
             seed=31).device()
    mm.check(_noalloc(c))                        # first call on the device: set-up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    outs = []
    for _ in range(2):
        c.dC[:].fill_(0xFF)                      # NaN pattern: stale output cannot pass
        mm.check(_noalloc(c))
        flat = c.result()
        assert padding_untouched(c.C, flat) or c.C.ld == c.N
        outs.append(logical_out(c.C, flat).astype(np.float64))
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "device memory changed across calls"
    for got in outs:
        assert np.isfinite(got).all()
        err = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert err <= 2e-3, f"relative Frobenius difference {err:.2e}"
    assert np.array_equal(outs[0], outs[1]), "two calls in a row differ"
    c.check(exact=False)                         # and against the oracle


def test_noalloc_integer_inputs_exact():
    c = Case(128, 128, 4096, dt=(BF16, BF16, BF16), dist="int4", seed=32).device()
    for _ in range(2):
        mm.check(_noalloc(c))
        c.check(exact=True)


def test_noalloc_largest_output_that_fits():
    """1024 x 2040 outputs: two fp32 K slices fill all but 31 KB of the
    workspace.  Sampled outputs bit-exact (integer inputs, K = 16384: every
    partial sum is an integer below 2^24)."""
    c = Case(1024, 2040, 16384, dt=(BF16, BF16, F32), dist="int4", seed=34).device()
    rng = np.random.default_rng(34)
    pts = np.stack([np.zeros(3000, np.int64), rng.integers(0, 1024, 3000),
                    rng.integers(0, 2040, 3000)], 1)
    pts = np.concatenate([pts, [[0, 0, 0], [0, 1023, 2039], [0, 1023, 0], [0, 0, 2039]]])
    want = oracle.round_out(oracle.gemm_points(c.A, c.B, c.K, pts), F32)
    for _ in range(2):
        c.dC.fill_(0xFF)
        mm.check(_noalloc(c))
        flat = c.result().view(np.float32)
        assert np.isfinite(flat[:1024 * 2040]).all(), "an output was never written"
        got = flat[pts[:, 1] * c.C.ld + pts[:, 2]]
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_noalloc_rejects_sizes_beyond_the_workspace():
    c = Case(2048, 1024, 64, dt=(BF16, BF16, F32), dist="int4", seed=33)
    st = mm.mm_splitk_gemm_noalloc(16, 16, 16, 2048, 1024, 64, 64, 1024, 1024, c.dt, "NN")
    assert st == mm.MM_ERR_INVALID_ARG
    assert "workspace" in mm.mm_last_error() and "2097120" in mm.mm_last_error()
    # one output past the limit (2,097,121 = 1 x 2,097,121)
    st = mm.mm_splitk_gemm_noalloc(16, 16, 16, 1, 2097121, 256, 256, 2097121, 2097121, c.dt,
                                   "NN")
    assert st == mm.MM_ERR_INVALID_ARG and "2097120" in mm.mm_last_error()


def test_noalloc_k_rules():
    """K = 0 is rejected (nothing to split), and so is a K that fits in one
    128-byte block (K <= 64 for bf16); a K of two blocks runs."""
    c = Case(128, 128, 64, dt=(BF16, BF16, F32), dist="int4", seed=35).device()
    st = mm.mm_splitk_gemm_noalloc(c.pA, c.pB, c.pC, 128, 128, 0, 64, 128, 128, c.dt, "NN")
    assert st == mm.MM_ERR_INVALID_ARG
    st = mm.mm_splitk_gemm_noalloc(c.pA, c.pB, c.pC, 128, 128, 64, 64, 128, 128, c.dt, "NN")
    assert st == mm.MM_ERR_UNSUPPORTED and "two K" in mm.mm_last_error()
    c = Case(128, 128, 72, dt=(BF16, BF16, F32), dist="int4", seed=35).device()
    mm.check(_noalloc(c))
    c.check(exact=True)
