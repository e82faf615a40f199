"""Every candidate against the CPU oracle, through the C ABI (GPU).

Bar (from the method's correctness target): integer-valued inputs in
{-4..4} with K <= 4096 must match the oracle bit-exactly (every partial sum
is an integer below 2^24, exact in fp32 in any order; the single rounding to
the output type is round-to-nearest-even on both sides); real-valued inputs
must reach a relative Frobenius error <= 2e-3.  Every candidate, not only the
tuner's choice, is held to it.  Output padding must never be written.
"""
import numpy as np
import pytest

import matmul_selection_gb300 as mm
import oracle
from gpu_util import BF16, F16, F32, Case

pytestmark = pytest.mark.gpu

NAMES = mm.candidate_names()
CANDS = list(range(len(NAMES)))
LAYOUTS = ["NN", "NT", "TN", "TT"]


def run(cand, case):
    return mm.mm_execute_candidate(cand, *case.args())


def _expect_supported_or_skip(st, cand, case):
    if st == mm.MM_ERR_UNSUPPORTED:
        return False
    assert st == mm.MM_OK, f"{NAMES[cand]}: {mm.mm_last_error()}"
    return True


SMALL = [(256, 256, 256), (17, 33, 65), (3, 5, 7), (1, 1, 1), (130, 260, 200),
         (16, 72, 1000), (8, 1000, 1001), (200, 136, 64)]


@pytest.mark.parametrize("cand", CANDS, ids=NAMES)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_integer_exact_bf16_to_f32(cand, layout, shape):
    c = Case(*shape, layout=layout, dt=(BF16, BF16, F32), dist="int4").device()
    if _expect_supported_or_skip(run(cand, c), cand, c):
        c.check(exact=True)


@pytest.mark.parametrize("cand", CANDS, ids=NAMES)
@pytest.mark.parametrize("dt", [(BF16, BF16, BF16), (F16, F16, F32), (F16, F16, F16),
                                (F32, F32, F32), (F32, F32, BF16)],
                         ids=["bf16-bf16", "f16-f32", "f16-f16", "f32-f32", "f32-bf16"])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_integer_exact_dtypes(cand, dt, layout):
    c = Case(16, 264, 520, layout=layout, dt=dt, dist="int4", seed=7).device()
    if _expect_supported_or_skip(run(cand, c), cand, c):
        c.check(exact=True)
    c = Case(140, 96, 300, layout=layout, dt=dt, dist="int4", seed=8).device()
    if _expect_supported_or_skip(run(cand, c), cand, c):
        c.check(exact=True)


@pytest.mark.parametrize("cand", CANDS, ids=NAMES)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("dt", [(BF16, BF16, F32), (BF16, BF16, BF16), (F32, F32, F32)],
                         ids=["bf16-f32", "bf16-bf16", "f32-f32"])
def test_real_valued_frobenius(cand, layout, dt):
    for shape in [(256, 256, 256), (16, 520, 777), (129, 200, 3000)]:
        c = Case(*shape, layout=layout, dt=dt, dist="normal", seed=11).device()
        if _expect_supported_or_skip(run(cand, c), cand, c):
            c.check(exact=False)


@pytest.mark.parametrize("cand", CANDS, ids=NAMES)
def test_batched_with_gaps(cand):
    # batch strides leave NaN-filled gaps between items; C items too
    for layout in LAYOUTS:
        c = Case(12, 40, 72, layout=layout, dt=(BF16, BF16, F32), dist="int4", batch=3,
                 bstride_extra=(8, 16, 8), pad=(8, 8, 4)).device()
        if _expect_supported_or_skip(run(cand, c), cand, c):
            c.check(exact=True)


@pytest.mark.parametrize("cand", CANDS, ids=NAMES)
def test_padded_and_misaligned_lda(cand):
    # lda = K + 4 (bf16: 8-byte aligned rows), ldc padded
    c = Case(16, 256, 512, layout="NN", dt=(BF16, BF16, F32), dist="int4", pad=(4, 0, 3)).device()
    if _expect_supported_or_skip(run(cand, c), cand, c):
        c.check(exact=True)
    # base pointers offset by 2 bytes
    c = Case(8, 128, 96, layout="NN", dt=(BF16, BF16, F32), dist="int4", a_off=2, c_off=4).device()
    if _expect_supported_or_skip(run(cand, c), cand, c):
        c.check(exact=True)


def test_every_candidate_runs_somewhere():
    """Coverage guard: each candidate is supported on at least one home case."""
    home = {
        "naive": Case(33, 17, 9, dist="int4"),
        "gemv_n": Case(4, 256, 512, layout="NN", dist="int4"),
        "gemv_t": Case(4, 256, 512, layout="NT", dist="int4"),
        "gemv_n_cluster": Case(4, 1000, 520, layout="NN", dist="int4"),
        "gemv_t_rows": Case(3, 300, 1000, layout="NT", dist="int4"),
        "gemv_n_stream": Case(1, 1000, 700, layout="NN", dist="int4"),
        "gemv_t_stream": Case(1, 1000, 704, layout="NT", dist="int4"),
        "gemv_n_mma": Case(16, 1000, 520, layout="NN", dt=(BF16, BF16, F32), dist="int4"),
        "gemv_t_mma": Case(16, 1000, 520, layout="NT", dt=(BF16, BF16, F32), dist="int4"),
        "tc2_repack_256x256": Case(300, 264, 200, layout="NN", dist="int4", pad=(4, 0, 0)),
        "tc2_repack_256x224": Case(300, 264, 200, layout="NN", dist="int4", pad=(4, 0, 0)),
        "tc2_cpasync_256x256_s7": Case(300, 264, 200, layout="NN", dist="int4", pad=(4, 0, 0)),
        "tc_repack_128x128": Case(300, 264, 200, layout="TN", dist="int4", pad=(3, 0, 0)),
        "tc_repack_128x64": Case(130, 72, 136, layout="NT", dist="int4", pad=(0, 5, 0)),
        "gemv_swap_tc_repack_splitk_128x64": Case(16, 264, 200, layout="NN", dist="int4",
                                                  pad=(4, 0, 0)),
        "tc_repack_splitk_128x128": Case(200, 264, 520, layout="NN", dist="int4", pad=(4, 0, 0)),
        "tc_repack_splitk_128x64": Case(130, 72, 600, layout="TN", dist="int4", pad=(3, 0, 0)),
    }
    for i, n in enumerate(NAMES):
        c = home.get(n) or Case(256, 256, 256, layout="NN", dist="int4")
        c.device()
        st = run(i, c)
        assert st == mm.MM_OK, f"{n} unsupported on its home case: {mm.mm_last_error()}"
        c.check(exact=True)


def test_empty_and_zero_k():
    for i in CANDS:
        c = Case(0, 8, 8).device()
        assert run(i, c) in (mm.MM_OK, mm.MM_ERR_UNSUPPORTED)
    c = Case(5, 7, 0, dt=(BF16, BF16, F32)).device()
    assert run(0, c) == mm.MM_OK
    got = c.result().view(np.float32)[:35]
    assert np.all(got == 0.0)


def test_transposed_view_worked_example():
    """d . d^T with the rhs a transposed view of d (strides [1, 3]); one launch."""
    import torch
    d = torch.tensor([[21., 42., 63.], [84., 105., 126.]], device="cuda")
    out = torch.empty(2, 2, device="cuda")
    for i in CANDS:
        out.fill_(float("nan"))
        st = mm.mm_execute_candidate(i, d, d, out, 2, 2, 3, 3, 3, 2, (F32, F32, F32), "NT")
        if st == mm.MM_ERR_UNSUPPORTED:
            continue
        assert st == 0, mm.mm_last_error()
        torch.cuda.synchronize()
        assert out.cpu().tolist() == [[6174.0, 14112.0], [14112.0, 33957.0]], NAMES[i]


def test_results_deterministic():
    for i in CANDS:
        c = Case(16, 512, 2048, layout="NN", dt=(BF16, BF16, F32), dist="normal").device()
        if run(i, c) != mm.MM_OK:
            continue
        r1 = c.result().copy()
        assert run(i, c) == mm.MM_OK
        assert np.array_equal(r1.view(np.uint8), c.result().view(np.uint8)), NAMES[i]


def test_gemv_n_stream_interleaved_shapes():
    """Shapes that change the number of column groups, splits and batch items
    from call to call on one stream, which share one scratch buffer and one
    set of arrival counters: every result must match the oracle."""
    import torch
    i = NAMES.index("gemv_n_stream")
    cases = [Case(1, 4096, 4096, layout="NN", dist="int4", seed=21),
             Case(1, 1000, 700, layout="NN", dist="int4", seed=22),
             Case(1, 296, 900, layout="NN", dist="int4", seed=23, batch=3, pad=(8, 8, 4),
                  bstride_extra=(8, 16, 8)),
             Case(1, 8, 20000, layout="NN", dist="int4", seed=24)]
    for k in [0, 1, 0, 2, 3, 0, 1, 2, 3, 3, 0]:
        c = cases[k].device()
        assert run(i, c) == mm.MM_OK, mm.mm_last_error()
        c.check(exact=True)
    s = torch.cuda.Stream()
    c = cases[0].device()
    assert mm.mm_execute_candidate(i, *c.args(), stream=s) == mm.MM_OK, mm.mm_last_error()
    s.synchronize()
    c.check(exact=True)


def test_gemv_n_stream_graph_replay():
    """A captured call replayed with new inputs each time: the arrival
    counters live in device memory and are back at zero after every call,
    so every replay must be exact."""
    import torch
    i = NAMES.index("gemv_n_stream")
    c = Case(1, 4096, 4096, layout="NN", dist="int4", seed=30).device()
    s = torch.cuda.Stream()
    assert mm.mm_execute_candidate(i, *c.args(), stream=s) == mm.MM_OK, mm.mm_last_error()
    s.synchronize()
    c.check(exact=True)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st = mm.mm_execute_candidate(i, *c.args(), stream=s)
    assert st == mm.MM_OK, mm.mm_last_error()
    for rep in range(3):
        n = Case(1, 4096, 4096, layout="NN", dist="int4", seed=31 + rep)
        for dst, op in ((c.dA, n.A), (c.dB, n.B), (c.dC, n.C)):
            raw = op.buf.view(np.uint8)
            dst[:raw.size].copy_(torch.from_numpy(raw.copy()))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        n.dA, n.dB, n.dC = c.dA, c.dB, c.dC
        n.check(exact=True)


@pytest.mark.parametrize("shape_pad", [((1, 4096, 4096), 0), ((1, 1000, 700), 4), ((1, 5, 20000), 0),
                                       ((1, 70000, 24), 0), ((1, 300, 4100), 4), ((1, 77, 3), 5)],
                         ids=lambda s: "x".join(map(str, s[0])) + f"+{s[1]}")
@pytest.mark.parametrize("dt", [(BF16, BF16, F32), (F16, F16, F16), (F32, F32, F32)],
                         ids=["bf16-f32", "f16-f16", "f32-f32"])
def test_gemv_t_stream_rows(shape_pad, dt):
    """The transposed-B M=1 GEMV that gives each CTA whole rows of B: fewer
    rows than CTAs, many row blocks a CTA (wide N), K not a multiple of the
    16-byte piece with NaN-filled row padding right after it (elements past K
    must not reach the sums), three launches in a row over a fresh output;
    A read as packed 16-byte pieces (contiguous, aligned, K a whole number of
    pieces) and element by element (K ragged, batch strides off 16 bytes, A
    transposed)."""
    shape, pad = shape_pad
    i = NAMES.index("gemv_t_stream")
    c = Case(*shape, layout="NT", dt=dt, dist="int4", pad=(0, pad, 0), seed=sum(shape)).device()
    for _ in range(3):
        c.device()
        assert run(i, c) == mm.MM_OK, mm.mm_last_error()
        c.check(exact=True)
    # batch gaps that keep every B item 16-byte aligned
    cb = Case(1, 296, 900, layout="NT", dt=dt, dist="int4", batch=3, bstride_extra=(8, 20, 8),
              pad=(8, 4, 4)).device()
    assert run(i, cb) == mm.MM_OK, mm.mm_last_error()
    cb.check(exact=True)
    cr = Case(1, 4096, 4096, layout="NT", dt=dt, dist="normal", seed=5).device()
    assert run(i, cr) == mm.MM_OK, mm.mm_last_error()
    cr.check(exact=False)
    # A stored transposed (its K elements lda apart): A's elements one by one,
    # at a K that would otherwise take the packed 16-byte pieces of A
    ct = Case(1, 1000, 704, layout="TT", dt=dt, dist="int4", pad=(3, 0, 0), seed=6).device()
    assert run(i, ct) == mm.MM_OK, mm.mm_last_error()
    ct.check(exact=True)
    # A's base one element off a 16-byte boundary: element by element too
    ea = 4 if dt[0] == F32 else 2
    co = Case(1, 1000, 704, layout="NT", dt=dt, dist="int4", a_off=ea, seed=7).device()
    assert run(i, co) == mm.MM_OK, mm.mm_last_error()
    co.check(exact=True)


@pytest.mark.parametrize("shape", [(1, 4096, 4096), (1, 1000, 700), (1, 136, 5000), (1, 64, 33),
                                   (1, 8, 20000), (1, 81920, 40), (1, 4104, 3)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dt", [(BF16, BF16, F32), (F16, F16, F16), (F32, F32, F32)],
                         ids=["bf16-f32", "f16-f16", "f32-f32"])
def test_gemv_n_stream_splits(shape, dt):
    """The split-K GEMV whose split sums the last-arriving CTA of each column
    group adds: one split (wide N), as many splits as K rows, the split cap
    (narrow N, long K), a ragged last column group, and three launches in a
    row over a fresh output each time (the arrival counters must be back at
    zero after every call)."""
    i = NAMES.index("gemv_n_stream")
    c = Case(*shape, layout="NN", dt=dt, dist="int4", seed=sum(shape)).device()
    for _ in range(3):
        c.device()  # a fresh output each time: a launch that skipped a column would show
        assert run(i, c) == mm.MM_OK, mm.mm_last_error()
        c.check(exact=True)
    # batched with gaps; B rows of 304 elements keep the 16-byte row alignment
    cb = Case(1, 296, 900, layout="NN", dt=dt, dist="int4", batch=3, bstride_extra=(8, 16, 8),
              pad=(8, 8, 4)).device()
    assert run(i, cb) == mm.MM_OK, mm.mm_last_error()
    cb.check(exact=True)


@pytest.mark.parametrize("shape_pad", [((16, 4096, 4096), (0, 0)), ((8, 4096, 4096), (4, 0)),
                                       ((2, 1000, 700), (0, 0)), ((5, 70, 4100), (0, 2)),
                                       ((16, 8, 20000), (0, 0)), ((13, 4104, 24), (4, 0)),
                                       ((16, 264, 1000), (4, 0)), ((3, 1, 17), (3, 7))],
                         ids=lambda s: "x".join(map(str, s[0])) + "+" + "_".join(map(str, s[1])))
@pytest.mark.parametrize("dt", [(BF16, BF16, F32), (F16, F16, F16), (BF16, BF16, BF16)],
                         ids=["bf16-f32", "f16-f16", "bf16-bf16"])
def test_gemv_n_mma_shapes(shape_pad, dt):
    """The warp-MMA small-M GEMV: M from 2 to 16 (rows past M zero in the
    MMA), N ragged against the 64-column groups (including a single column),
    K ragged against the 16-row chunks and the splits (zero-filled past K),
    A's leading dimension padded so that its rows are only 8-byte aligned
    (copied in 8-byte pieces; NaN padding must not reach the sums), B rows
    padded to 16 bytes, three
    launches in a row over a fresh output (the arrival counters back at
    zero), a batch with gaps, and a real-valued case."""
    shape, (pa, pb) = shape_pad
    i = NAMES.index("gemv_n_mma")
    c = Case(*shape, layout="NN", dt=dt, dist="int4", pad=(pa, pb, 0), seed=sum(shape)).device()
    for _ in range(3):
        c.device()
        assert run(i, c) == mm.MM_OK, mm.mm_last_error()
        c.check(exact=True)
    cb = Case(7, 296, 900, layout="NN", dt=dt, dist="int4", batch=3, bstride_extra=(8, 16, 8),
              pad=(4, 8, 4)).device()
    assert run(i, cb) == mm.MM_OK, mm.mm_last_error()
    cb.check(exact=True)
    cr = Case(16, 4096, 4096, layout="NN", dt=dt, dist="normal", seed=9).device()
    assert run(i, cr) == mm.MM_OK, mm.mm_last_error()
    cr.check(exact=False)


@pytest.mark.parametrize("shape_pad", [((16, 4096, 4096), (0, 0)), ((8, 4096, 4096), (4, 0)),
                                       ((2, 1000, 700), (0, 4)), ((5, 70, 4100), (0, 4)),
                                       ((16, 8, 20000), (0, 0)), ((13, 4104, 24), (4, 0)),
                                       ((16, 264, 1000), (4, 0)), ((3, 1, 17), (3, 7))],
                         ids=lambda s: "x".join(map(str, s[0])) + "+" + "_".join(map(str, s[1])))
@pytest.mark.parametrize("dt", [(BF16, BF16, F32), (F16, F16, F16), (BF16, BF16, BF16)],
                         ids=["bf16-f32", "f16-f16", "bf16-bf16"])
def test_gemv_t_mma_shapes(shape_pad, dt):
    """The warp-MMA small-M GEMV with B transposed (rows of n, k contiguous):
    N ragged against the 64-row groups (down to one row), K ragged against
    the 16-k chunks (zero-filled past K), B's rows padded to a multiple of
    16 bytes, A padded to 8-byte rows, three launches in a row, a batch with
    gaps, and a real-valued case."""
    shape, (pa, pb) = shape_pad
    i = NAMES.index("gemv_t_mma")
    c = Case(*shape, layout="NT", dt=dt, dist="int4", pad=(pa, pb, 0), seed=sum(shape) + 1).device()
    for _ in range(3):
        c.device()
        assert run(i, c) == mm.MM_OK, mm.mm_last_error()
        c.check(exact=True)
    # B's batch stride (295 * 904 + 896 + 16 elements) keeps 16-byte rows
    cb = Case(7, 296, 896, layout="NT", dt=dt, dist="int4", batch=3, bstride_extra=(8, 16, 8),
              pad=(4, 8, 4)).device()
    assert run(i, cb) == mm.MM_OK, mm.mm_last_error()
    cb.check(exact=True)
    cr = Case(16, 4096, 4096, layout="NT", dt=dt, dist="normal", seed=19).device()
    assert run(i, cr) == mm.MM_OK, mm.mm_last_error()
    cr.check(exact=False)


@pytest.mark.parametrize("shape_pad_batch", [((4, 128, 4096), (0, 0), 1), ((6, 1216, 8192), (4, 8), 1),
                                             ((3, 8192, 4096), (0, 0), 1), ((5, 256, 4096), (4, 0), 2)],
                         ids=lambda s: "x".join(map(str, s[0])) + "+" + "_".join(map(str, s[1])) +
                         f"+b{s[2]}")
@pytest.mark.parametrize("dt", [(BF16, BF16, F32), (F16, F16, F16)], ids=["bf16-f32", "f16-f16"])
@pytest.mark.parametrize("cand,layout", [("gemv_n_mma", "NN"), ("gemv_t_mma", "NT")],
                         ids=["n", "t"])
def test_gemv_mma_even_splits(shape_pad_batch, dt, cand, layout):
    """Shapes whose K splits give every warp the same whole number of 16-row
    chunks and whose N is a whole number of 64-column groups, so the kernel
    runs its unchecked instance: with 152 SMs these take 2, 4, 16 and (with a
    batch of two) 2 chunks a warp; A padded to 8-byte rows in two of them;
    B row-major and transposed."""
    shape, (pa, pb), batch = shape_pad_batch
    i = NAMES.index(cand)
    extra = (8, 16, 8) if batch > 1 else (0, 0, 0)
    c = Case(*shape, layout=layout, dt=dt, dist="int4", pad=(pa, pb, 0), batch=batch,
             bstride_extra=extra, seed=sum(shape) + batch).device()
    for _ in range(2):
        c.device()
        assert run(i, c) == mm.MM_OK, mm.mm_last_error()
        c.check(exact=True)


@pytest.mark.parametrize("shape", [(1, 4096, 4096), (3, 37, 4104), (8, 64, 2056), (2, 20, 104),
                                   (1, 17, 8)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dt", [(BF16, BF16, BF16), (F32, F32, F32)], ids=["bf16", "f32"])
def test_gemv_t_rows_chunks(shape, dt):
    """The row-per-warp GEMV walks each row in 512-byte chunks from a
    starting chunk of its own, wrapping at the row's end: whole and ragged
    last chunks, rows shorter than one chunk, and a partial last CTA."""
    i = NAMES.index("gemv_t_rows")
    c = Case(*shape, layout="NT", dt=dt, dist="int4", seed=sum(shape)).device()
    assert run(i, c) == mm.MM_OK, mm.mm_last_error()
    c.check(exact=True)


TC1 = [i for i, n in enumerate(NAMES) if n.startswith("tc_") and "repack" not in n]


@pytest.mark.parametrize("cand", TC1, ids=[NAMES[i] for i in TC1])
@pytest.mark.parametrize("shape,dt", [((256, 160, 512), (BF16, BF16, F32)),
                                      ((256, 320, 512), (BF16, BF16, BF16)),
                                      ((256, 192, 4096), (BF16, BF16, F32))],
                         ids=["f32-one-box-in-last-tile", "bf16-one-box-in-last-tile",
                              "splitk-last-box"])
def test_ragged_n_bulk_store_boxes_repeat(cand, shape, dt):
    """The epilogue stages output boxes in two alternating buffers and reuses
    one once its previous bulk store has read it.  Tiles whose last columns
    fall past N stage fewer boxes; ten launches in a row, each over a fresh
    NaN-filled output, catch a box refilled while its store still reads it."""
    c = Case(*shape, layout="NN", dt=dt, dist="int4", seed=sum(shape)).device()
    for _ in range(10):
        c.device()
        st = run(cand, c)
        if st == mm.MM_ERR_UNSUPPORTED:
            pytest.skip(mm.mm_last_error())
        assert st == mm.MM_OK, mm.mm_last_error()
        c.check(exact=True)


@pytest.mark.parametrize("shape,pad,batch", [((4, 42, 3000), (0, 6, 0), 1),
                                             ((3, 42, 2000), (0, 6, 0), 2),
                                             ((4, 136, 3000), (0, 0, 5), 1),
                                             ((5, 33, 1500), (0, 7, 0), 1)],
                         ids=["groups-cross-rows", "groups-cross-batch", "ldc-padded", "odd-total"])
def test_splitk_reduce_groups(shape, pad, batch):
    """The split-K reduction takes four consecutive outputs of the flattened
    grid a thread when it can: groups that run across a row or a batch item,
    padded C rows, and an output count that is not a multiple of four (one
    output a thread).  Every split-K candidate, swapped ones included."""
    c = Case(*shape, layout="NN", dt=(BF16, BF16, F32), dist="int4", pad=pad, batch=batch,
             seed=sum(shape)).device()
    ran = 0
    for i, n in enumerate(NAMES):
        if "splitk" not in n:
            continue
        c.device()  # a fresh output (and padding) for each candidate
        st = run(i, c)
        if st == mm.MM_ERR_UNSUPPORTED:
            continue
        assert st == mm.MM_OK, f"{n}: {mm.mm_last_error()}"
        c.check(exact=True)
        ran += 1
    assert ran >= 2


@pytest.mark.parametrize("shape,pad,batch", [((40, 72, 5000), (4, 0, 0), 1),
                                             ((16, 136, 2056), (2, 0, 0), 3),
                                             ((300, 64, 520), (1, 0, 0), 2)],
                         ids=["rows-of-two-blocks", "4-byte-pieces-batched", "2-byte-pieces-batched"])
def test_repack_rows(shape, pad, batch):
    """A with rows that TMA cannot address is copied to aligned rows first:
    rows longer than one block's share of pieces, 8-, 4- and 2-byte pieces,
    several batch items."""
    i = NAMES.index("tc_repack_128x64")
    c = Case(*shape, layout="NN", dt=(BF16, BF16, F32), dist="int4", pad=pad, batch=batch,
             seed=sum(shape)).device()
    assert run(i, c) == mm.MM_OK, mm.mm_last_error()
    c.check(exact=True)


# ---------------------------------------------------------------- full sizes
@pytest.mark.parametrize("M", [1, 8, 16])
@pytest.mark.parametrize("layout", ["NN", "NT"])
def test_gemv_full_size_exact(M, layout):
    """The GEMV workload at full size (N = K = 4096), every GEMV candidate."""
    c = Case(M, 4096, 4096, layout=layout, dt=(BF16, BF16, BF16), dist="int4").device()
    ran = 0
    for i, n in enumerate(NAMES):
        if not n.startswith("gemv"):
            continue
        if run(i, c) == mm.MM_OK:
            c.check(exact=True)
            ran += 1
    assert ran >= 1


@pytest.mark.parametrize("M", [1, 8, 16])
def test_gemv_full_size_real(M):
    c = Case(M, 4096, 4096, layout="NN", dt=(BF16, BF16, BF16), dist="normal",
             dist_b="normal:0.02").device()
    i = NAMES.index("gemv_n")
    assert run(i, c) == mm.MM_OK
    c.check(exact=False)
