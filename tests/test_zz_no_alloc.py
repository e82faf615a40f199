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
from gpu_util import BF16, F32, Case, logical_out, padding_untouched

pytestmark = pytest.mark.gpu


def _noalloc(c):
    return mm.mm_splitk_gemm_noalloc(c.pA, c.pB, c.pC, c.M, c.N, c.K, c.A.ld, c.B.ld, c.C.ld,
                                     c.dt, c.layout)


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


def test_noalloc_rejects_sizes_beyond_the_workspace():
    c = Case(2048, 1024, 64, dt=(BF16, BF16, F32), dist="int4", seed=33)
    st = mm.mm_splitk_gemm_noalloc(16, 16, 16, 2048, 1024, 64, 64, 1024, 1024, c.dt, "NN")
    assert st == mm.MM_ERR_INVALID_ARG
    assert "workspace" in mm.mm_last_error() and "2097120" in mm.mm_last_error()
