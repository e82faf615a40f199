"""The committed GB300 tuning table on the GPU: it loads (its validators
match this device and runtime), every recorded problem then runs without
tuning and gives the product.  With MM_TUNED_GATE=1 it is also a performance
gate: each committed winner must run within 15 % of the winner of a fresh
tune of the same problem (the offline table must not have gone stale)."""
import csv
import os

import numpy as np
import pytest

import matmul_selection_gb300 as mm

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TUNED = os.path.join(ROOT, "matmul_selection_gb300", "tuned")
TABLE = os.path.join(TUNED, "gb300.csv")
PROBLEMS = os.path.join(TUNED, "problems.csv")
CODE = {"bf16": 0, "f16": 1, "f32": 2}
EB = {"bf16": 2, "f16": 2, "f32": 4}


def _problems():
    with open(PROBLEMS, newline="") as f:
        return [r for r in csv.reader(f) if r and r[0] == "Untuned"]


class Buffers:
    """Device operands of a recorded problem (integer values in {-2..2}, so
    every output is exact in any summation order)."""

    def __init__(self, p, seed):
        import torch
        self.M, self.N, self.K, self.lda, self.ldb, self.ldc = (int(x) for x in p[2:8])
        self.dt = tuple(CODE[x] for x in p[8:11])
        self.layout = p[11]
        self.batch, sa, sb, sc = (int(x) for x in p[12:16])
        at, bt = self.layout[0] == "T", self.layout[1] == "T"
        span_a = (self.K if at else self.M) * self.lda
        span_b = (self.N if bt else self.K) * self.ldb
        span_c = self.M * self.ldc
        self.b = None if self.batch == 1 else (self.batch, sa, sb, sc)
        na = span_a if self.batch == 1 else sa * self.batch
        nb = span_b if self.batch == 1 else sb * self.batch
        nc = span_c if self.batch == 1 else sc * self.batch
        g = torch.Generator(device="cuda").manual_seed(seed)
        tdt = {0: torch.bfloat16, 1: torch.float16, 2: torch.float32}
        self.A = torch.randint(-2, 3, (na,), generator=g, device="cuda").to(tdt[self.dt[0]])
        self.B = torch.randint(-2, 3, (nb,), generator=g, device="cuda").to(tdt[self.dt[1]])
        self.C = torch.empty(nc, dtype=tdt[self.dt[2]], device="cuda")

    def args(self):
        return (self.A, self.B, self.C, self.M, self.N, self.K, self.lda, self.ldb, self.ldc,
                self.dt, self.layout, self.b)

    def key(self):
        st, kb, _ = mm.mm_tune_key(self.M, self.N, self.K, self.lda, self.ldb, self.ldc, self.dt,
                                   self.layout, self.b)
        return kb


@pytest.fixture(autouse=True)
def clean_table():
    mm.check(mm.mm_set_option("tuning", "1"))
    mm.check(mm.mm_cache_clear())
    yield
    mm.check(mm.mm_cache_clear())


def test_committed_table_loads_and_serves_every_problem():
    mm.check(mm.mm_cache_load(TABLE))
    probs = _problems()
    assert mm.mm_cache_size() == len(probs)
    mm.mm_reset_stats()
    for i, p in enumerate(probs):
        if int(p[2]) * int(p[3]) > (1 << 26):  # the 8192^2 outputs: only the lookup
            continue
        buf = Buffers(p, i)
        mm.check(mm.mm_autotune_execute(*buf.args()))
        import torch
        torch.cuda.synchronize()
        assert mm.mm_lookup(buf.key())[0] == 0
    s = mm.mm_get_stats()
    assert s["tunes"] == 0 and s["hits"] == s["calls"]


def _time(cand, buf, reps=5, chunk=40):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    mm.check(mm.mm_execute_candidate(cand, *buf.args()))
    out = []
    for _ in range(reps):
        e0.record()
        for _ in range(chunk):
            mm.mm_execute_candidate(cand, *buf.args())
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) / chunk)
    return float(np.median(out))


@pytest.mark.skipif(os.environ.get("MM_TUNED_GATE") != "1", reason="set MM_TUNED_GATE=1")
def test_committed_winners_within_15_percent_of_a_fresh_tune():
    names = mm.candidate_names()
    report = []
    for i, p in enumerate(_problems()):
        buf = Buffers(p, i)
        mm.check(mm.mm_cache_clear())
        mm.check(mm.mm_cache_load(TABLE))
        committed = mm.mm_lookup(buf.key())[1]
        mm.check(mm.mm_cache_clear())
        mm.check(mm.mm_autotune_execute(*buf.args()))  # a fresh tune
        fresh = mm.mm_lookup(buf.key())[1]
        tc, tf = _time(committed, buf), _time(fresh, buf)
        report.append((p[2:5], p[11], names[committed], tc, names[fresh], tf))
        print(f"{'x'.join(p[2:5])} {p[11]} committed {names[committed]} {tc * 1e3:.2f} us, "
              f"fresh {names[fresh]} {tf * 1e3:.2f} us")
    slow = [r for r in report if r[3] > 1.15 * r[5]]
    assert not slow, slow
