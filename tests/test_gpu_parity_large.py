"""Large-shape parity (GPU): every tensor-core candidate on full-size output
grids, checked against the oracle on sampled outputs (the oracle computes
each sampled element on its own).  4096 x 4096 outputs make the 2-SM kernels
split their last partial wave into half-width units; the samples include
every tile of that tail."""
import numpy as np
import pytest

import matmul_selection_gb300 as mm
import oracle
from gpu_util import BF16, F32, Case

pytestmark = pytest.mark.gpu

NAMES = mm.candidate_names()
TC = [i for i, n in enumerate(NAMES) if n.startswith("tc")]


def sample_points(M, N, rng, n=6000, batch=1):
    pts = [np.stack([rng.integers(0, batch, n), rng.integers(0, M, n), rng.integers(0, N, n)], 1)]
    # every 256 x 256 tile of the last two tile columns, four points each
    for tm in range(0, M, 256):
        for tn in range(max(0, N - 512), N, 64):
            r = rng.integers(tm, min(M, tm + 256), 4)
            c = rng.integers(tn, min(N, tn + 64), 4)
            pts.append(np.stack([np.zeros(4, np.int64), r, c], 1))
    # corners
    pts.append(np.array([[0, 0, 0], [0, M - 1, N - 1], [0, 0, N - 1], [0, M - 1, 0]]))
    return np.concatenate(pts).astype(np.int64)


@pytest.fixture(scope="module")
def big_cases():
    out = {}
    for lay in ("NN", "NT"):
        c = Case(4096, 4096, 512, layout=lay, dt=(BF16, BF16, F32), dist="int4", seed=41)
        c.device()
        out[lay] = c
    return out


@pytest.mark.parametrize("cand", TC, ids=[NAMES[i] for i in TC])
@pytest.mark.parametrize("layout", ["NN", "NT"])
def test_full_grid_sampled_exact(big_cases, cand, layout):
    c = big_cases[layout]
    c.dC.fill_(0xFF)
    st = mm.mm_execute_candidate(cand, *c.args())
    if st == mm.MM_ERR_UNSUPPORTED:
        pytest.skip(mm.mm_last_error())
    assert st == 0, mm.mm_last_error()
    flat = c.result().view(np.float32)
    rng = np.random.default_rng(cand)
    pts = sample_points(4096, 4096, rng)
    want = oracle.round_out(oracle.gemm_points(c.A, c.B, 512, pts), F32)
    got = flat[pts[:, 1] * c.C.ld + pts[:, 2]]
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {pts[bad[0]].tolist()}"
    assert np.isfinite(flat[:4096 * 4096]).all(), "an output was never written"


def test_tuned_square_real_valued_sampled():
    """The benchmark's own workload (4096^3 bf16, N(0,1)) through the tuner:
    relative Frobenius error of sampled outputs <= 2e-3."""
    c = Case(4096, 4096, 4096, dt=(BF16, BF16, BF16), dist="normal", seed=1002).device()
    mm.check(mm.mm_autotune_execute(*c.args()))
    flat = c.result()
    rng = np.random.default_rng(3)
    pts = sample_points(4096, 4096, rng, n=3000)
    ref = oracle.gemm_points(c.A, c.B, 4096, pts)
    got = oracle.decode(flat[pts[:, 1] * c.C.ld + pts[:, 2]], BF16)
    err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= 2e-3, err


SPLITK = [i for i, n in enumerate(NAMES) if "splitk" in n]


@pytest.fixture(scope="module")
def splitk_case():
    c = Case(128, 128, 65536, layout="NN", dt=(BF16, BF16, F32), dist="int4", seed=43)
    c.device()
    return c


@pytest.mark.parametrize("cand", SPLITK, ids=[NAMES[i] for i in SPLITK])
def test_splitk_full_size_exact(splitk_case, cand):
    """The split-K workload at full size (128 x 128 x 65536): dozens of K
    slices a tile, so several threads share each output in the reduction.
    Entries in {-4..4} keep every partial sum below 2^24 in magnitude, exact
    in fp32 in any order."""
    c = splitk_case
    c.dC.fill_(0xFF)
    st = mm.mm_execute_candidate(cand, *c.args())
    if st == mm.MM_ERR_UNSUPPORTED:
        pytest.skip(mm.mm_last_error())
    assert st == 0, mm.mm_last_error()
    c.check(exact=True)


@pytest.mark.parametrize("cand", SPLITK, ids=[NAMES[i] for i in SPLITK])
def test_splitk_full_size_real_repeatable(cand):
    """Real-valued inputs at the same size: within the Frobenius bound, and
    two launches give the same bytes (the slice sums are added in a fixed
    order)."""
    c = Case(128, 128, 65536, layout="NN", dt=(BF16, BF16, BF16), dist="normal", seed=44).device()
    st = mm.mm_execute_candidate(cand, *c.args())
    if st == mm.MM_ERR_UNSUPPORTED:
        pytest.skip(mm.mm_last_error())
    assert st == 0, mm.mm_last_error()
    c.check(exact=False)
    first = c.result().copy()
    assert mm.mm_execute_candidate(cand, *c.args()) == 0
    assert np.array_equal(first.view(np.uint8), c.result().view(np.uint8))
