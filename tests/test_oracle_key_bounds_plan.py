"""Pins for the key, bound and plan oracles against the pages' printed values."""
import os

import pytest

from oracle import bounds, key, plan

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = 2


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.split() for l in f if l.strip() and not l.startswith("#")]


def _square_key(tok):
    n = int(tok.rstrip("T"))
    trans = tok.endswith("T")
    return key.make_key(n, n, n, n, n, F32, F32, F32, a_trans=False, b_trans=trans)


@pytest.mark.parametrize("row", _rows("key_rows.txt"), ids=lambda r: r[0])
def test_key_golden_rows(row):
    shape, m, n, k, lp, ls, rp, rs, layout_rhs, scale, kind = row
    got = _square_key(shape)
    assert (got["m"], got["n"], got["k"]) == (int(m), int(n), int(k))
    assert (got["lhs_pow2"], got["lhs_stride"]) == (int(lp), int(ls))
    assert (got["rhs_pow2"], got["rhs_stride"]) == (int(rp), int(rs))
    assert got["layout_rhs"] == layout_rhs
    assert got["layout_lhs"] == "Contiguous"
    assert got["scale"] == scale and got["kind"] == kind


def test_key_equalities_printed():
    assert _square_key("768") == _square_key("1024")
    assert _square_key("1000") != _square_key("1024")
    assert _square_key("1024T") != _square_key("1024")


def test_anchor_levels():
    assert [key.anchor(x) for x in (1, 2, 3, 4, 5, 127, 128, 129, 4097)] == \
        [1, 2, 4, 4, 8, 128, 128, 256, 8192]
    assert key.anchor(1000, "full") == 1000
    # wider buckets at Minimal, narrower at Extensive
    assert key.anchor(1000, "minimal") == 1526     # 2.5^8 = 1525.88...
    assert key.anchor(1000, "extensive") == 1478   # 1.5^17 = 985.3 < 1000 <= 1.5^18 = 1477.9
    assert key.anchor(0) == 0


def test_stride_factor_examples_from_text():
    # the page's explanations: 768*4 = 3072 B and 4096 B both cap at 10;
    # 1000*4 = 4000 = 2^5 * 125 -> 5
    assert key.stride_factor([768 * 4]) == 10
    assert key.stride_factor([1024 * 4]) == 10
    assert key.stride_factor([1000 * 4]) == 5
    assert key.stride_factor([1025 * 4]) == 2
    assert key.stride_factor([4100 * 2]) == 3          # bf16 lda 4100
    assert key.stride_factor([]) == 10
    assert key.stride_factor([0]) == 10


def test_key_buckets_4097_and_8192_share():
    k1 = key.make_key(4097, 4096, 4096, 4100, 4096, 0, 0, 0)
    k2 = key.make_key(8192, 4096, 4096, 4100, 4096, 0, 0, 0)
    assert k1 == k2
    assert k1["m"] == 8192 and k1["lhs_stride"] == 3


def test_key_batch_swap_and_text_roundtrip():
    k = key.make_key(512, 512, 512, 512, 512, 0, 0, 2, batch=32,
                     stride_a=512 * 512, stride_b=512 * 512)
    assert k["layout_lhs"] == "Contiguous" and k["batch"] == 32
    k2 = key.make_key(4, 4, 4, 32 * 4, 4, 0, 0, 2, batch=32, stride_a=4, stride_b=16)
    assert k2["layout_lhs"].startswith("MildlyPermuted") and "batch_swap:true" in k2["layout_lhs"]
    assert key.parse_key_text(key.key_text(k)) == k


def test_bounds_worked_example():
    g = {r[0]: r[1] for r in _rows("roofline_limit.txt")}
    ops = bounds.compute_ops(1024, 1024, 1024)
    assert ops == int(g["ops"])
    assert bounds.bytes_moved(1024, 1024, 1024, 4, 4, 4) == int(g["bytes"])
    lim = bounds.time_limit_s(ops, float(g["peak_ops_per_s"]), int(g["bytes"]),
                              float(g["peak_bytes_per_s"]), float(g["threshold"]),
                              int(g["launch_overhead_ns"]) * 1e-9)
    assert int(lim * 1e9) == int(g["limit_ns"])
    assert round(lim * 1e9) == int(g["limit_ns"])


def test_plan_wgsl_demotion_story():
    """All candidates of the first group unsupported: they are demoted to the
    minimum tier, still form the first round, and the group's priority still
    puts it first; the next group is the backup."""
    cands = [dict(index=0, group="naive", group_prio=0, prio=0, supported=True)]
    cands += [dict(index=1 + i, group="accel", group_prio=2, prio=2, supported=False) for i in range(20)]
    cands += [dict(index=21, group="unit", group_prio=1, prio=1, supported=True)]
    p = plan.make_plan(cands)
    assert [g for g, _ in p] == ["accel", "unit", "naive"]
    assert p[0][1] == [list(range(1, 21))]


def test_plan_tiers_and_skip():
    cands = [
        dict(index=0, group="naive", group_prio=0, prio=0, supported=True),
        dict(index=1, group="tc", group_prio=2, prio=2, supported=True),
        dict(index=2, group="tc", group_prio=2, prio=1, supported=True),
        dict(index=3, group="tc", group_prio=2, prio=2, supported=False),
        dict(index=4, group="tc", group_prio=2, prio=-1, supported=True),
        dict(index=5, group="gemv", group_prio=-1, prio=3, supported=True),
    ]
    p = plan.make_plan(cands)
    assert p == [("tc", [[1], [2], [3]]), ("naive", [[0]])]
