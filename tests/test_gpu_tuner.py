"""The tuner through the C ABI (GPU): table hits and misses, the result file
and its validators, the plan, host-side fault injection, the numerical
check, the decision log and the host-buffer entry point."""
import json
import os
import threading

import numpy as np
import pytest

import matmul_selection_gb300 as mm
import oracle
import synth
from gpu_util import BF16, F32, Case, logical_out, padding_untouched
from oracle import plan as oplan

pytestmark = pytest.mark.gpu

NAMES = mm.candidate_names()
DEFAULTS = {"tuning": "1", "autotune_cache": "1", "fault": "", "numerical_check": "",
            "decisions": "", "cache_file": "", "max_tuning_iterations": "100",
            "max_tuning_duration_ms": "30", "l2_flush": "0", "rotating_buffer_mb": "-1",
            "record_untuned": "", "pending_wait_ms": "120000", "wait_limit_us": "2000000",
            "wait_stall": "0"}


@pytest.fixture(autouse=True)
def fresh_table():
    import torch
    torch.cuda.init()
    for k, v in DEFAULTS.items():
        mm.check(mm.mm_set_option(k, v))
    mm.check(mm.mm_cache_clear())
    mm.mm_reset_stats()
    yield
    for k, v in DEFAULTS.items():
        mm.mm_set_option(k, v)
    mm.mm_cache_clear()


def execute(c):
    return mm.mm_autotune_execute(*c.args())


def test_tune_then_hit_one_launch():
    c = Case(256, 256, 256, dist="int4").device()
    mm.check(execute(c))
    c.check(exact=True)
    s = mm.mm_get_stats()
    assert s["misses"] == 1 and s["tunes"] == 1 and s["hits"] == 0
    launches = s["launches"]
    for _ in range(5):
        mm.check(execute(c))
    c.check(exact=True)
    s = mm.mm_get_stats()
    assert s["hits"] == 5
    assert s["launches"] == launches + 5  # a warm call is exactly one launch


def test_bucket_sharing_story():
    """f32 squares 1024, 768, 1000, 2048 in one process: 768 reuses 1024's
    entry (one launch), 1000 has stride factor 5 and re-tunes, the table ends
    with three entries."""
    f32 = (F32, F32, F32)
    for n, expect_hit in [(1024, False), (768, True), (1000, False), (2048, False)]:
        c = Case(n, n, n, dt=f32, dist="int4", seed=n).device()
        before = mm.mm_get_stats()
        mm.check(execute(c))
        after = mm.mm_get_stats()
        assert (after["hits"] - before["hits"] == 1) == expect_hit, n
        if expect_hit:
            assert after["launches"] - before["launches"] == 1
        c.check(exact=True)
    assert mm.mm_cache_size() == 3


def test_lookup_and_key():
    c = Case(64, 64, 64, dist="int4").device()
    mm.check(execute(c))
    st, kb, _ = mm.mm_tune_key(64, 64, 64, 64, 64, 64, (BF16, BF16, F32), "NN")
    st, idx = mm.mm_lookup(kb)
    assert st == 0 and 0 <= idx < len(NAMES)
    st, kb2, _ = mm.mm_tune_key(64, 64, 65, 65, 64, 64, (BF16, BF16, F32), "NN")
    assert mm.mm_lookup(kb2) == (mm.MM_ERR_NOT_FOUND, -1)


def test_result_file_roundtrip(tmp_path):
    cases = [Case(256, 256, 256, dist="int4"), Case(1, 4096, 4096, dist="int4"),
             Case(8, 512, 512, layout="NT", dist="int4")]
    winners = {}
    for c in cases:
        c.device()
        mm.check(execute(c))
        st, kb, _ = mm.mm_tune_key(*c.args()[3:11])
        winners[kb] = mm.mm_lookup(kb)[1]
    path = str(tmp_path / "results.csv")
    mm.check(mm.mm_cache_save(path))
    lines = open(path).read().splitlines()
    vals = {l.split(",")[1] for l in lines if l.startswith("Validator,")}
    assert vals == {"MM_VERSION", "CANDIDATE_CHECKSUM", "DEVICE", "CUDA_VERSION"}
    assert sum(l.startswith("MatmulKey,") for l in lines) == 3
    mm.check(mm.mm_cache_clear())
    assert mm.mm_cache_size() == 0
    mm.check(mm.mm_cache_load(path))
    assert mm.mm_cache_size() == 3
    for kb, w in winners.items():
        assert mm.mm_lookup(kb)[1] == w
    # loaded entries are hits: no tuning
    before = mm.mm_get_stats()
    for c in cases:
        mm.check(execute(c))
        c.check(exact=True)
    after = mm.mm_get_stats()
    assert after["tunes"] == before["tunes"] and after["hits"] - before["hits"] == 3


@pytest.mark.parametrize("field", ["MM_VERSION", "CANDIDATE_CHECKSUM", "DEVICE", "CUDA_VERSION"])
def test_validator_mismatch_rejects_whole_file(tmp_path, field):
    c = Case(64, 64, 64, dist="int4").device()
    mm.check(execute(c))
    path = str(tmp_path / "r.csv")
    mm.check(mm.mm_cache_save(path))
    text = open(path).read().splitlines()
    text = [l + "x" if l.startswith(f"Validator,{field},") else l for l in text]
    open(path, "w").write("\n".join(text) + "\n")
    mm.check(mm.mm_cache_clear())
    assert mm.mm_cache_load(path) == mm.MM_ERR_CACHE_VALIDATION
    assert field in mm.mm_last_error()
    assert mm.mm_cache_size() == 0


def test_hand_edits_default_and_unknown_name(tmp_path):
    ca = Case(64, 64, 64, dist="int4").device()
    cb = Case(128, 64, 64, dist="int4").device()
    mm.check(execute(ca))
    mm.check(execute(cb))
    path = str(tmp_path / "r.csv")
    mm.check(mm.mm_cache_save(path))
    lines = open(path).read().splitlines()
    keys = [l for l in lines if l.startswith("MatmulKey,")]
    out = []
    for l in lines:
        if l == keys[0]:
            f = l.split(",")
            f[2] = "Default"
            f = f[:4]
            l = ",".join(f)
        elif l == keys[1]:
            f = l.split(",")
            f[2] = "no_such_kernel"
            l = ",".join(f)
        out.append(l)
    open(path, "w").write("\n".join(out) + "\n")
    mm.check(mm.mm_cache_clear())
    mm.check(mm.mm_cache_load(path))
    assert mm.mm_cache_size() == 1  # the unknown-name row was skipped
    k0 = keys[0].split(",")[1]
    st, kb, _ = mm.mm_tune_key(64, 64, 64, 64, 64, 64, (BF16, BF16, F32), "NN")
    which = mm.mm_lookup(kb)[1]
    st, kb2, _ = mm.mm_tune_key(128, 64, 64, 64, 64, 64, (BF16, BF16, F32), "NN")
    which2 = mm.mm_lookup(kb2)[1]
    assert 0 in (which, which2) and -1 in (which, which2)
    assert k0


def test_tuning_disabled_runs_default():
    """With tuning off a miss runs the default candidate (the shape-class
    heuristic's choice), records nothing and measures nothing."""
    mm.check(mm.mm_set_option("tuning", "0"))
    for shape in [(96, 80, 200), (1, 512, 512), (4096, 256, 64), (8, 1024, 1024)]:
        c = Case(*shape, dist="int4").device()
        first = mm.mm_default_candidate(*shape, shape[2], shape[1], shape[1], c.dt, "NN")
        assert first >= 0
        n0 = mm.mm_candidate_launches(first)
        mm.check(execute(c))
        c.check(exact=True)
        assert mm.mm_candidate_launches(first) == n0 + 1, NAMES[first]
    assert mm.mm_cache_size() == 0 and mm.mm_get_stats()["tunes"] == 0


@pytest.mark.parametrize("shape,layout,pad,dt,batch,want", [
    ((1, 4096, 4096), "NN", 0, (BF16, BF16, BF16), None, "gemv_n_stream"),
    ((1, 4096, 4096), "NT", 0, (BF16, BF16, BF16), None, "gemv_t_stream"),
    ((16, 4096, 4096), "NN", 0, (BF16, BF16, BF16), None, "gemv_n_mma"),
    ((16, 4096, 4096), "NN", 4, (BF16, BF16, BF16), None, "gemv_n_mma"),
    ((8, 4096, 4096), "NN", 0, (BF16, BF16, BF16), None, "gemv_n_mma"),
    ((8, 4096, 4096), "NT", 0, (BF16, BF16, BF16), None, "gemv_swap_tc_splitk_128x64_s8"),
    ((16, 4096, 4096), "NT", 4, (BF16, BF16, BF16), None, "gemv_t_mma"),
    ((128, 128, 65536), "NN", 0, (BF16, BF16, BF16), None, "tc_splitk_128x128_s7"),
    ((4096, 4096, 4096), "NN", 0, (BF16, BF16, BF16), None, "tc2_256x256_s7"),
    ((8192, 4096, 4096), "NN", 4, (BF16, BF16, BF16), None, "tc2_repack_256x256"),
    ((25088, 4096, 64), "NT", 0, (F32, F32, F32), None, "tc_128x256_s4"),
    ((256, 256, 256), "NN", 0, (BF16, BF16, F32), None, "tc_128x64_s8"),
    ((512, 512, 512), "NN", 0, (BF16, BF16, F32), (32, 512 * 512, 512 * 512, 512 * 512),
     "tc_128x256_s4"),
])
def test_default_heuristic_matches_tuned_winners(shape, layout, pad, dt, batch, want):
    """The default for an untuned key is the candidate that won that shape
    class in the committed GB300 table."""
    M, N, K = shape
    lda = (M if layout[0] == "T" else K) + pad
    ldb = K if layout[1] == "T" else N
    got = mm.mm_default_candidate(M, N, K, lda, ldb, N, dt, layout, batch)
    assert NAMES[got] == want


@pytest.mark.parametrize("mode", ["error", "nan"])
def test_fault_injected_candidate_is_excluded(mode):
    mm.check(mm.mm_set_option("fault", f"gemv_n:{mode}"))
    c = Case(1, 512, 512, dist="int4").device()
    mm.check(execute(c))
    c.check(exact=True)
    st, kb, _ = mm.mm_tune_key(1, 512, 512, 512, 512, 512, (BF16, BF16, F32), "NN")
    assert NAMES[mm.mm_lookup(kb)[1]] != "gemv_n"


def test_numerical_check_excludes_wrong_candidate():
    mm.check(mm.mm_set_option("numerical_check", "1e-3_1e-3"))
    mm.check(mm.mm_set_option("fault", "gemv_n:wrong"))
    c = Case(1, 512, 512, dist="int4").device()
    mm.check(execute(c))
    c.check(exact=True)
    st, kb, _ = mm.mm_tune_key(1, 512, 512, 512, 512, 512, (BF16, BF16, F32), "NN")
    assert NAMES[mm.mm_lookup(kb)[1]] != "gemv_n"


def test_numerical_check_keeps_correct_candidates(tmp_path):
    path = str(tmp_path / "d.jsonl")
    mm.check(mm.mm_set_option("numerical_check", "1e-3_1e-3"))
    mm.check(mm.mm_set_option("decisions", path))
    c = Case(1, 512, 512, dist="int4").device()
    mm.check(execute(c))
    st, kb, _ = mm.mm_tune_key(1, 512, 512, 512, 512, 512, (BF16, BF16, F32), "NN")
    assert NAMES[mm.mm_lookup(kb)[1]].startswith("gemv")
    rec = json.loads(open(path).read().splitlines()[-1])
    assert not [x for x in rec["candidates"] if x["state"] == "numeric"]


def test_decision_log(tmp_path):
    path = str(tmp_path / "decisions.jsonl")
    mm.check(mm.mm_set_option("decisions", path))
    c = Case(256, 256, 256, dist="int4").device()
    mm.check(execute(c))
    rec = json.loads(open(path).read().splitlines()[-1])
    assert rec["fastest"] == NAMES[rec["fastest_index"]]
    assert "m=256 n=256 k=256" in rec["key"]
    assert rec["limit_ns"] > 0 and rec["bounds"]["compute"]["amount"] == 256 * 256 * 511
    measured = [x for x in rec["candidates"] if x["state"] == "ok"]
    assert measured and all(x["n"] >= 1 for x in measured)
    # re-timed finalists: the recorded choice is the finalist with the lowest
    # re-timed median, and only candidates near the first winner were re-timed
    fin = [x for x in rec["candidates"] if "final_ms" in x]
    if fin:
        assert len(fin) >= 2 and len(fin) <= 3
        best = min(fin, key=lambda x: (x["final_ms"], x["index"]))
        assert rec["fastest_index"] == best["index"]
        lead = min(x["median_ms"] for x in measured)
        assert all(x["median_ms"] <= 1.10 * lead + 1e-9 for x in fin)


def test_record_untuned_then_tune_file(tmp_path):
    """Offline tuning: misses with tuning off are recorded once per key;
    mm_tune_file tunes them on synthetic operands; later calls hit."""
    path = str(tmp_path / "untuned.csv")
    mm.check(mm.mm_set_option("tuning", "0"))
    mm.check(mm.mm_set_option("record_untuned", path))
    c1 = Case(96, 80, 200, dist="int4").device()
    c2 = Case(1, 512, 512, layout="NT", dist="int4").device()
    c3 = Case(12, 40, 72, layout="TN", dt=(BF16, BF16, F32), dist="int4", batch=3,
              bstride_extra=(8, 16, 8), pad=(8, 8, 4)).device()
    for c in (c1, c2, c3, c1):  # the repeated key is recorded once
        mm.check(execute(c))
        c.check(exact=True)
    rows = [r for r in open(path).read().splitlines() if r.startswith("Untuned,")]
    assert len(rows) == 3
    assert mm.mm_cache_size() == 0 and mm.mm_get_stats()["tunes"] == 0
    st, n = mm.mm_tune_file(path)
    assert st == 0 and n == 3, mm.mm_last_error()
    assert mm.mm_cache_size() == 3
    before = mm.mm_get_stats()["hits"]
    for c in (c1, c2, c3):
        c.device()
        mm.check(execute(c))
        c.check(exact=True)
    assert mm.mm_get_stats()["hits"] == before + 3
    st, n = mm.mm_tune_file(path)  # nothing left to tune
    assert st == 0 and n == 0
    st, n = mm.mm_tune_file(str(tmp_path / "absent.csv"))
    assert st == mm.MM_ERR_IO


def test_finalists_are_retimed(tmp_path):
    """Two configurations of nearly equal speed (forced on the same shape)
    give a close call; the log then carries their re-timed medians."""
    path = str(tmp_path / "fin.jsonl")
    mm.check(mm.mm_set_option("decisions", path))
    c = Case(1024, 1024, 1024, dt=(BF16, BF16, BF16), dist="int4").device()
    mm.check(execute(c))
    c.check(exact=True)
    rec = json.loads(open(path).read().splitlines()[-1])
    ok = sorted((x for x in rec["candidates"] if x["state"] == "ok"), key=lambda x: x["median_ms"])
    close = [x for x in ok if x["median_ms"] <= 1.10 * ok[0]["median_ms"]]
    short = any(x.get("short_circuit") for x in ok)
    if len(close) >= 2 and not short:
        assert sum("final_ms" in x for x in rec["candidates"]) == min(3, len(close))


def test_host_buffers_entry_point():
    c = Case(37, 45, 130, layout="TN", dt=(BF16, BF16, F32), dist="int4", pad=(3, 0, 5))
    out = c.C.buf.copy()
    st = mm.mm_autotune_execute_host(c.A.buf, c.B.buf, out, 37, 45, 130, c.A.ld, c.B.ld, c.C.ld,
                                     c.dt, "TN")
    mm.check(st)
    assert padding_untouched(c.C, out)
    got = logical_out(c.C, out)
    want = oracle.round_out(c.c64, F32)
    assert np.array_equal(got, want)


def test_plan_matches_oracle_and_has_naive_last():
    probs = [(1, 4096, 4096, "NN"), (16, 4096, 4096, "NT"), (256, 256, 256, "NN"),
             (4097, 4096, 4096, "NN"), (128, 128, 65536, "NN"), (3, 5, 7, "TT")]
    for M, N, K, lay in probs:
        at, bt = lay[0] == "T", lay[1] == "T"
        lda, ldb = (M if at else K), (K if bt else N)
        items = mm.mm_plan(M, N, K, lda, ldb, N, (BF16, BF16, F32), lay)
        cands = [dict(index=it["cand"], group=mm.mm_group_name(it["group"]),
                      group_prio=it["group_prio"], prio=it["prio"],
                      supported=bool(it["supported"])) for it in items]
        want = oplan.make_plan(sorted(cands, key=lambda d: d["index"]))
        got = []
        for it in items:
            g = mm.mm_group_name(it["group"])
            if not got or got[-1][0] != g:
                got.append((g, []))
            tiers = got[-1][1]
            while len(tiers) <= it["tier"]:
                tiers.append([])
            tiers[it["tier"]].append(it["cand"])
        assert got == want, (M, N, K, lay)
        assert items[-1]["cand"] == 0  # the default closes every plan
    # lda = 4100 bf16 (stride factor 3): gemv still supported for M <= 16
    items = mm.mm_plan(16, 4096, 4096, 4100, 4096, 4096, (BF16, BF16, F32), "NN")
    first = items[0]
    assert mm.mm_group_name(first["group"]) == "gemv" and first["supported"]


def test_concurrent_callers_tune_once():
    cs = [Case(200, 136, 512, dist="int4", seed=5).device() for _ in range(4)]
    errs = []

    def work(c):
        import torch
        torch.cuda.set_device(0)
        st = mm.mm_autotune_execute(*c.args())
        if st != 0:
            errs.append(mm.mm_last_error())

    ts = [threading.Thread(target=work, args=(c,)) for c in cs]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs
    for c in cs:
        c.check(exact=True)
    assert mm.mm_get_stats()["tunes"] == 1


def test_large_gemv_workload_selects_gemv():
    c = Case(1, 4096, 4096, dt=(BF16, BF16, BF16), dist="int4").device()
    mm.check(execute(c))
    c.check(exact=True)
    st, kb, _ = mm.mm_tune_key(1, 4096, 4096, 4096, 4096, 4096, (BF16, BF16, BF16), "NN")
    assert NAMES[mm.mm_lookup(kb)[1]].startswith("gemv")


def test_misaligned_lda_workload_key_sharing():
    """lda = 4100 (stride factor 3); M = 4097 and 8192 share one key, so the
    second call is a hit."""
    c1 = Case(4097, 4096, 4096, dt=(BF16, BF16, F32), dist="int4", pad=(4, 0, 0))
    c2 = Case(8192, 4096, 4096, dt=(BF16, BF16, F32), dist="int4", pad=(4, 0, 0))
    st, k1, _ = mm.mm_tune_key(4097, 4096, 4096, 4100, 4096, 4096, (BF16, BF16, F32), "NN")
    st, k2, _ = mm.mm_tune_key(8192, 4096, 4096, 4100, 4096, 4096, (BF16, BF16, F32), "NN")
    assert k1 == k2
    mm.check(mm.mm_set_option("max_tuning_iterations", "3"))
    c1.device()
    mm.check(execute(c1))
    del c1
    c2.device()
    before = mm.mm_get_stats()["hits"]
    mm.check(execute(c2))
    assert mm.mm_get_stats()["hits"] == before + 1
    # sampled outputs against the oracle (full oracle would take minutes)
    import torch
    torch.cuda.synchronize()
    flat = c2.result()
    rng = np.random.default_rng(0)
    pts = np.stack([np.zeros(400, dtype=np.int64), rng.integers(0, 8192, 400),
                    rng.integers(0, 4096, 400)], axis=1)
    want = oracle.round_out(oracle.gemm_points(c2.A, c2.B, 4096, pts), F32)
    got = flat[pts[:, 1] * c2.C.ld + pts[:, 2]]
    assert np.array_equal(got, want)


def test_graph_capture_miss_uses_default():
    import torch
    c = Case(48, 40, 72, dist="int4").device()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    n0 = mm.mm_candidate_launches(0)
    with torch.cuda.graph(g, stream=s):
        st = mm.mm_autotune_execute(*c.args(), stream=s)
    assert st == 0, mm.mm_last_error()
    g.replay()
    torch.cuda.synchronize()
    c.check(exact=True)
    assert mm.mm_get_stats()["tunes"] == 0
    assert mm.mm_candidate_launches(0) == n0 + 1


def test_graph_capture_hit_whose_winner_needs_new_scratch():
    """A table hit captured on a stream that never ran the recorded winner:
    split-K needs a workspace on that stream, which cannot be allocated
    while the stream is captured.  The call must still be captured (the
    winner declines and the next candidate of the ranking that needs no new
    scratch runs), and the replayed graph must compute the product."""
    import torch
    c = Case(128, 128, 8192, dt=(BF16, BF16, F32), dist="int4", seed=77).device()
    mm.check(mm.mm_autotune_execute(*c.args()))  # tuned on the default stream
    torch.cuda.synchronize()
    _, key, _ = mm.mm_tune_key(128, 128, 8192, c.A.ld, c.B.ld, c.C.ld, (BF16, BF16, F32), "NN")
    winner = mm.mm_candidate_name(mm.mm_lookup(key)[1])
    assert "splitk" in winner, f"the case needs a split-K winner, got {winner}"
    c.dC.fill_(0xFF)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st = mm.mm_autotune_execute(*c.args(), stream=s)
    assert st == 0, mm.mm_last_error()
    g.replay()
    torch.cuda.synchronize()
    c.check(exact=True)


# ---------------------------------------------------------------- harness paths
def _last_decision(path):
    return json.loads(open(path).read().splitlines()[-1])


def test_l2_flush_times_every_call(tmp_path):
    """With the L2 flush on, a flush kernel runs before every timed call, so
    each call is timed on its own (one sample per call) and the finalists are
    not re-timed; the tuned result is still the product."""
    path = str(tmp_path / "flush.jsonl")
    mm.check(mm.mm_set_option("l2_flush", "1"))
    mm.check(mm.mm_set_option("decisions", path))
    c = Case(256, 256, 256, dist="int4").device()
    mm.check(execute(c))
    c.check(exact=True)
    rec = _last_decision(path)
    assert rec["l2_flush"] is True
    ok = [x for x in rec["candidates"] if x["state"] == "ok"]
    assert ok and all(x["samples"] == x["n"] for x in ok), ok
    assert not any("final_ms" in x for x in rec["candidates"])
    for _ in range(3):  # warm calls
        mm.check(execute(c))
    c.check(exact=True)


@pytest.mark.parametrize("mb,expect", [("0", 1), ("-1", None)])
def test_rotating_buffer_size(tmp_path, mb, expect):
    """rotating_buffer_mb = 0 turns the rotation off (one private output, the
    caller's inputs read in place); the default (-1) rotates over enough sets
    to cover twice the L2.  Either way the caller's output is only written by
    the final launch and holds the product."""
    path = str(tmp_path / "rot.jsonl")
    mm.check(mm.mm_set_option("rotating_buffer_mb", mb))
    mm.check(mm.mm_set_option("decisions", path))
    c = Case(1, 4096, 4096, dt=(BF16, BF16, F32), dist="int4").device()
    mm.check(execute(c))
    c.check(exact=True)
    rec = _last_decision(path)
    if expect is not None:
        assert rec["rotating_sets"] == expect
    else:
        import torch
        l2 = torch.cuda.get_device_properties(0).L2_cache_size
        set_bytes = (4096 + 4096 * 4096) * 2 + 4096 * 4
        assert rec["rotating_sets"] * set_bytes >= 2 * l2


def test_shutdown_saves_table_and_library_is_usable_again(tmp_path):
    """mm_shutdown with a cache file set writes the device's table (file name
    with the device ordinal) and frees the library's state; the next call on
    the same key loads that file lazily and runs the recorded kernel without
    tuning."""
    base = str(tmp_path / "table.csv")
    mm.check(mm.mm_set_option("cache_file", base))
    c = Case(200, 136, 512, dist="int4", seed=9).device()
    mm.check(execute(c))
    c.check(exact=True)
    tunes = mm.mm_get_stats()["tunes"]
    assert tunes == 1
    mm.mm_shutdown()
    saved = str(tmp_path / "table0.csv")
    assert os.path.exists(saved)
    assert sum(l.startswith("MatmulKey,") for l in open(saved)) == 1
    c.device()
    mm.check(execute(c))
    c.check(exact=True)
    assert mm.mm_get_stats()["tunes"] == tunes, "the saved entry was not used"
    assert mm.mm_cache_size() == 1


def test_cache_file_loaded_lazily_on_first_miss(tmp_path):
    """A table saved earlier is read when the first miss of a fresh library
    state meets the cache_file option: both keys become hits, no tuning."""
    ca = Case(64, 64, 64, dist="int4").device()
    cb = Case(1, 512, 512, layout="NT", dist="int4").device()
    mm.check(execute(ca))
    mm.check(execute(cb))
    mm.check(mm.mm_cache_save(str(tmp_path / "lazy0.csv")))
    mm.mm_shutdown()
    mm.mm_reset_stats()
    mm.check(mm.mm_set_option("cache_file", str(tmp_path / "lazy.csv")))
    for c in (ca, cb):
        c.device()
        mm.check(execute(c))
        c.check(exact=True)
    s = mm.mm_get_stats()
    assert s["tunes"] == 0 and mm.mm_cache_size() == 2
    assert s["hits"] == 1  # the second key found the table already loaded


def test_pending_key_wait_runs_out_and_default_runs():
    """A second caller missing on a key that another thread is still tuning
    waits pending_wait_ms, then runs the default candidate instead of
    waiting for the tuner; both results are the product and the key is tuned
    once."""
    import time
    import torch
    mm.check(mm.mm_set_option("fault", "gemv_n:stall"))  # the tuner sleeps 1.5 s on the host
    mm.check(mm.mm_set_option("pending_wait_ms", "100"))
    c1 = Case(1, 512, 512, dist="int4", seed=3).device()
    c2 = Case(1, 512, 512, dist="int4", seed=4).device()
    errs = []

    def tuner():
        torch.cuda.set_device(0)
        st = mm.mm_autotune_execute(*c1.args())
        if st != 0:
            errs.append(mm.mm_last_error())

    t = threading.Thread(target=tuner)
    t.start()
    time.sleep(0.4)  # the tuner holds the key (it sleeps inside its first benchmark)
    t0 = time.perf_counter()
    mm.check(execute(c2))
    waited = time.perf_counter() - t0
    c2.check(exact=True)
    still_tuning = t.is_alive()
    t.join()
    assert not errs, errs
    c1.check(exact=True)
    assert still_tuning and waited < 1.0, (still_tuning, waited)
    assert mm.mm_get_stats()["tunes"] == 1


def test_wait_limit_timeout_is_reported(tmp_path):
    """A 1-SM tensor-core kernel whose wait runs out (the test hook makes its
    MMA warp first wait on a barrier nothing arrives on, limit 1 ms) records
    a code in its error word, stops its other roles, lets its copies land
    and returns.  The tuner marks those candidates `timeout` and picks
    another; the no-allocation split-K call reports MM_ERR_TIMEOUT through its
    status query.  Without the hook both give the exact product again."""
    one_sm = {n for n in NAMES if n.startswith("tc_") and "repack" not in n}
    path = str(tmp_path / "timeout.jsonl")
    mm.mm_shutdown()  # fresh peaks: the next options take effect
    try:
        # peaks so high that no candidate lands inside the time limit: the
        # round is not cut short before the 1-SM candidates are measured
        mm.check(mm.mm_set_option("peak_tflops", "1e9"))
        mm.check(mm.mm_set_option("peak_gbs", "1e9"))
        mm.check(mm.mm_set_option("decisions", path))
        mm.check(mm.mm_set_option("wait_limit_us", "1000"))
        mm.check(mm.mm_set_option("wait_stall", "1"))
        c = Case(256, 256, 512, dist="int4", seed=12).device()
        mm.check(execute(c))
        c.check(exact=True)
        rec = _last_decision(path)
        states = {x["name"]: x["state"] for x in rec["candidates"]}
        measured = {n for n in one_sm if states.get(n) not in (None, "skipped", "unsupported")}
        assert measured and all(states[n] == "timeout" for n in measured), states
        assert rec["fastest"] not in one_sm, rec["fastest"]
        s = Case(128, 128, 4096, dt=(BF16, BF16, F32), dist="int4", seed=13).device()
        st = mm.mm_splitk_gemm_noalloc(s.pA, s.pB, s.pC, 128, 128, 4096, s.A.ld, s.B.ld, s.C.ld,
                                       s.dt, "NN")
        assert st == mm.MM_OK, mm.mm_last_error()
        assert mm.mm_splitk_gemm_noalloc_status() == mm.MM_ERR_TIMEOUT
        assert "gave up" in mm.mm_last_error()
        mm.check(mm.mm_set_option("wait_stall", "0"))
        mm.check(mm.mm_set_option("wait_limit_us", "2000000"))
        for _ in range(2):
            s.device()
            mm.check(mm.mm_splitk_gemm_noalloc(s.pA, s.pB, s.pC, 128, 128, 4096, s.A.ld, s.B.ld,
                                               s.C.ld, s.dt, "NN"))
            assert mm.mm_splitk_gemm_noalloc_status() == mm.MM_OK
            s.check(exact=True)
        i = NAMES.index("tc_128x128_s6")
        c.device()
        mm.check(mm.mm_execute_candidate(i, *c.args()))
        c.check(exact=True)
    finally:
        for k in ("peak_tflops", "peak_gbs"):
            mm.mm_set_option(k, "0")
        mm.mm_set_option("wait_stall", "0")
        mm.mm_set_option("wait_limit_us", "2000000")
        mm.mm_shutdown()  # drop the inflated peaks


def test_device_peaks_probed_once_and_cached():
    """The roofline peaks (autotune page: probes run once per device): the
    first query runs or returns the probes, later queries return the same
    cached values, all positive and plausible for one GB300 (a launch costs
    well under 100 us; memory and tensor rates above 1 TB/s and 100 TFLOP/s)."""
    st, ops, bw, launch = mm.mm_device_peaks()
    assert st == mm.MM_OK, mm.mm_last_error()
    assert ops > 1e14 and bw > 1e12 and 0 < launch < 1e5
    again = mm.mm_device_peaks()
    assert again == (st, ops, bw, launch)

