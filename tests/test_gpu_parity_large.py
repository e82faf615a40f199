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


# (layout, lda padding): the padded cases give A rows of 1032 bytes, which no
# TMA map can describe, so only the candidates that copy A to aligned rows
# first (and the CUDA-core ones) run there
BIG = {"NN": ("NN", 0), "NT": ("NT", 0), "NN_lda+4": ("NN", 4), "TN_lda+4": ("TN", 4)}


@pytest.fixture(scope="module")
def big_cases():
    out = {}
    for name, (lay, pad) in BIG.items():
        c = Case(4096, 4096, 512, layout=lay, dt=(BF16, BF16, F32), dist="int4", seed=41,
                 pad=(pad, 0, 0))
        c.device()
        out[name] = c
    return out


@pytest.mark.parametrize("cand", TC, ids=[NAMES[i] for i in TC])
def test_full_grid_sampled_exact(big_cases, cand):
    """Every tensor-core candidate on a 4096 x 4096 output grid (K = 512) in
    every case it supports: aligned NN and NT, and A with a leading dimension
    of K + 4 (the copying candidates).  Each candidate must run on at least
    one case."""
    ran = []
    for name, c in big_cases.items():
        c.dC.fill_(0xFF)
        st = mm.mm_execute_candidate(cand, *c.args())
        if st == mm.MM_ERR_UNSUPPORTED:
            continue
        assert st == 0, f"{name}: {mm.mm_last_error()}"
        flat = c.result().view(np.float32)
        rng = np.random.default_rng(cand)
        pts = sample_points(4096, 4096, rng)
        want = oracle.round_out(oracle.gemm_points(c.A, c.B, 512, pts), F32)
        got = flat[pts[:, 1] * c.C.ld + pts[:, 2]]
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, f"{name}: {bad.size} mismatches, first at {pts[bad[0]].tolist()}"
        assert np.isfinite(flat[:4096 * 4096]).all(), f"{name}: an output was never written"
        ran.append(name)
    assert ran, f"{NAMES[cand]} ran on none of {list(big_cases)}"


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


# ---------------------------------------------------------------- skinny f32 and batched
def _sampled_check(c, pts, exact, tol=2e-3):
    """Compare the outputs at pts = [(b, i, j)] with the oracle's; the whole
    logical output must be finite (every element written)."""
    import torch
    torch.cuda.synchronize()
    dt = c.dt[2]
    ebytes = 4 if dt == F32 else 2
    n = c.C.buf.view(np.uint8).size // ebytes
    dev = c.dC[:n * ebytes]
    vals = dev.view(torch.float32) if dt == F32 else dev.view(torch.bfloat16).float()
    assert bool(torch.isfinite(vals).all()), "an output was never written"
    idx = pts[:, 0] * c.C.bstride + pts[:, 1] * c.C.ld + pts[:, 2]
    flat = vals.cpu().numpy() if dt == F32 else c.result()
    got = flat[idx]
    ref = oracle.gemm_points(c.A, c.B, c.K, pts)
    if exact:
        want = oracle.round_out(ref, dt)
        bits = np.uint32 if dt == F32 else np.uint16
        bad = np.nonzero(got.view(bits) != want.view(bits))[0]
        assert bad.size == 0, f"{bad.size} mismatches, first at {pts[bad[0]].tolist()}"
        return 0.0
    g = oracle.decode(got, dt)
    err = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    assert err <= tol, f"relative Frobenius error {err:.3e}"
    return err


def _points(M, N, batch, rng, n=20000):
    pts = np.stack([rng.integers(0, batch, n), rng.integers(0, M, n), rng.integers(0, N, n)], 1)
    corners = [[b, i, j] for b in {0, batch - 1} for i in (0, M - 1) for j in (0, N - 1)]
    return np.concatenate([pts, np.array(corners)]).astype(np.int64)


SKINNY = [(25088, 4096, 64), (4096, 4096, 64)]


@pytest.mark.parametrize("shape", SKINNY, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dist", ["u11", "int4"])
def test_skinny_f32_nt_full_size_every_candidate(shape, dist):
    """The skinny f32 NT workloads at full size (25088 x 4096 x 64 and
    4096 x 4096 x 64, inputs uniform in [-1, 1]; the tensor-core candidates
    multiply them as tf32): every candidate that supports the problem, on
    sampled outputs, within 2e-3 relative Frobenius error; with integer
    inputs in {-4..4} (exact in tf32) bit-exact."""
    M, N, K = shape
    c = Case(M, N, K, layout="NT", dt=(F32, F32, F32), dist=dist, seed=1003).device()
    pts = _points(M, N, 1, np.random.default_rng(M))
    ran = []
    for i, n in enumerate(NAMES):
        c.dC.fill_(0xFF)
        st = mm.mm_execute_candidate(i, *c.args())
        if st == mm.MM_ERR_UNSUPPORTED:
            continue
        assert st == 0, f"{n}: {mm.mm_last_error()}"
        _sampled_check(c, pts, exact=dist == "int4")
        ran.append(n)
    assert "naive" in ran and any(n.startswith("tc") for n in ran), ran


@pytest.mark.parametrize("dist", ["normal", "int4"])
def test_batched_32x512_full_size_every_candidate(dist):
    """Batch 32 of 512 x 512 x 512 bf16 -> f32 (N(0,1) inputs; integer
    inputs bit-exact): every candidate that supports batched problems."""
    c = Case(512, 512, 512, layout="NN", dt=(BF16, BF16, F32), dist=dist, batch=32,
             seed=1004).device()
    pts = _points(512, 512, 32, np.random.default_rng(32))
    ran = []
    for i, n in enumerate(NAMES):
        c.dC.fill_(0xFF)
        st = mm.mm_execute_candidate(i, *c.args())
        if st == mm.MM_ERR_UNSUPPORTED:
            continue
        assert st == 0, f"{n}: {mm.mm_last_error()}"
        _sampled_check(c, pts, exact=dist == "int4")
        ran.append(n)
    assert "naive" in ran and sum(n.startswith("tc") for n in ran) >= 3, ran


# ---------------------------------------------------------------- small-M rows, full size
SMALL_M_EXPECT = {  # candidates that must be among those run
    (1, "NN"): {"gemv_n", "gemv_n_stream", "gemv_n_cluster", "gemv_swap_tc_splitk_128x64_s8"},
    (1, "NT"): {"gemv_t", "gemv_t_stream", "gemv_t_rows", "gemv_swap_tc_splitk_128x64_s8"},
    (8, "NN"): {"gemv_n", "gemv_n_cluster", "gemv_n_mma", "gemv_swap_tc_splitk_128x64_s8",
                "gemv_swap_tc_128x64_s8"},
    (8, "NT"): {"gemv_t", "gemv_t_rows", "gemv_t_mma", "gemv_swap_tc_splitk_128x64_s8",
                "gemv_swap_tc_128x64_s8"},
    (16, "NN"): {"gemv_n", "gemv_n_mma", "gemv_swap_tc_splitk_128x64_s8", "gemv_swap_tc_128x64_s8"},
    (16, "NT"): {"gemv_t", "gemv_t_mma", "gemv_swap_tc_splitk_128x64_s8",
                 "gemv_swap_tc_128x64_s8"},
}


@pytest.mark.parametrize("M,layout", sorted(SMALL_M_EXPECT), ids=lambda x: str(x))
def test_gemv_workload_real_every_candidate(M, layout):
    """The GEMV workload's own distribution (A ~ N(0,1), B ~ N(0, 0.02),
    bf16 out) at full size, N = K = 4096: every candidate that supports it,
    the streaming M = 1 kernels, the clustered and row-per-warp M <= 8
    kernels and the swapped tensor-core forms included, within 2e-3 relative
    Frobenius error of the oracle."""
    c = Case(M, 4096, 4096, layout=layout, dt=(BF16, BF16, BF16), dist="normal",
             dist_b="normal:0.02", seed=1001).device()
    ran = set()
    for i, n in enumerate(NAMES):
        c.device()
        st = mm.mm_execute_candidate(i, *c.args())
        if st == mm.MM_ERR_UNSUPPORTED:
            continue
        assert st == 0, f"{n}: {mm.mm_last_error()}"
        c.check(exact=False)
        ran.add(n)
    missing = SMALL_M_EXPECT[(M, layout)] - ran
    assert not missing, f"not run: {sorted(missing)}"


@pytest.mark.parametrize("M", [1, 16, 127])
@pytest.mark.parametrize("rhs", ["N", "T"])
def test_bucket_rows_lda4100_every_candidate(M, rhs):
    """The key-bucketing rows with lda = 4100 (A rows of 8200 bytes, no TMA
    map can describe them) and N = K = 4096, rhs stored N or T, N(0,1)
    inputs, bf16 out: every candidate that supports the problem within
    2e-3 relative Frobenius error (whole output)."""
    c = Case(M, 4096, 4096, layout="N" + rhs, dt=(BF16, BF16, BF16), dist="normal",
             pad=(4, 0, 0), seed=1004).device()
    ran = []
    for i, n in enumerate(NAMES):
        c.device()
        st = mm.mm_execute_candidate(i, *c.args())
        if st == mm.MM_ERR_UNSUPPORTED:
            continue
        assert st == 0, f"{n}: {mm.mm_last_error()}"
        c.check(exact=False)
        ran.append(n)
    assert any("repack" in n for n in ran), ran


@pytest.mark.parametrize("M", [1000, 4097])
def test_bucket_rows_lda4100_large_sampled(M):
    """M = 1000 and 4097 with lda = 4100: every candidate that supports the
    problem, on sampled outputs (the 4097th row is a lone partial tile)."""
    c = Case(M, 4096, 4096, layout="NN", dt=(BF16, BF16, BF16), dist="normal", pad=(4, 0, 0),
             seed=1004).device()
    pts = _points(M, 4096, 1, np.random.default_rng(M), n=8000)
    pts = np.concatenate([pts, np.array([[0, M - 1, j] for j in range(0, 4096, 97)])])
    ran = []
    for i, n in enumerate(NAMES):
        c.dC.fill_(0xFF)
        st = mm.mm_execute_candidate(i, *c.args())
        if st == mm.MM_ERR_UNSUPPORTED:
            continue
        assert st == 0, f"{n}: {mm.mm_last_error()}"
        _sampled_check(c, pts, exact=False)
        ran.append(n)
    assert "tc2_repack_256x256" in ran, ran
