"""The committed tuning table of the GB300 (the offline-tuning result file in
matmul_selection_gb300/tuned/), checked without a GPU: it parses, its four
validator rows hold what this build writes (library version, candidate
checksum) and the GB300's model and architecture, every row names registered
candidates, and every recorded problem's key has exactly one row.  A table
that no longer matches the candidate set or the version is rejected whole by
mm_cache_load, so this is the gate that tells it must be re-tuned."""
import csv
import os
import re

import matmul_selection_gb300 as mm
from oracle import key as okey

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TUNED = os.path.join(ROOT, "matmul_selection_gb300", "tuned")
TABLE = os.path.join(TUNED, "gb300.csv")
PROBLEMS = os.path.join(TUNED, "problems.csv")
CODE = {"bf16": 0, "f16": 1, "f32": 2}


def _rows(path):
    with open(path, newline="") as f:
        return [r for r in csv.reader(f) if r]


def _validators():
    return {r[1]: ",".join(r[2:]) for r in _rows(TABLE) if r[0] == "Validator"}


def _entries():
    return [r for r in _rows(TABLE) if r[0] == "MatmulKey"]


def test_validators_match_this_build():
    v = _validators()
    assert set(v) == {"MM_VERSION", "CANDIDATE_CHECKSUM", "DEVICE", "CUDA_VERSION"}
    assert v["MM_VERSION"] == mm.mm_version().split("+")[0]
    assert v["CANDIDATE_CHECKSUM"] == "%016x" % mm.mm_candidate_checksum()
    assert re.fullmatch(r"NVIDIA GB300[^|]*\|sm_103", v["DEVICE"]), v["DEVICE"]
    assert re.fullmatch(r"\d{5,}", v["CUDA_VERSION"]), v["CUDA_VERSION"]


def test_rows_name_registered_candidates():
    names = set(mm.candidate_names()) | {"Default"}
    entries = _entries()
    assert entries
    for r in entries:
        assert len(r) == 5, r
        okey.parse_key_text(r[1])  # a well-formed key
        assert r[2] in names, r[2]
        assert float(r[3]) > 0
        ranking = [tok.rsplit(":", 1)[0] for tok in r[4].split(";")]
        assert ranking[0] == r[2], "the winner heads its ranking"
        assert set(ranking) <= names, set(ranking) - names


def test_every_recorded_problem_has_one_row():
    keys = [r[1] for r in _entries()]
    assert len(keys) == len(set(keys)), "duplicate keys"
    problems = [r for r in _rows(PROBLEMS) if r[0] == "Untuned"]
    assert {p[1] for p in problems} == set(keys)
    for p in problems:  # the recorded key is the key of the recorded shape
        M, N, K, lda, ldb, ldc = (int(x) for x in p[2:8])
        dt = tuple(CODE[x] for x in p[8:11])
        batch, sa, sb, sc = (int(x) for x in p[12:16])
        b = None if batch == 1 else (batch, sa, sb, sc)
        st, _, text = mm.mm_tune_key(M, N, K, lda, ldb, ldc, dt, p[11], b)
        assert st == 0 and text == p[1], (text, p[1])
