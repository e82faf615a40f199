"""Write the committed tuning table of one GPU model (offline tuning).

    python matmul_selection_gb300/tuned/make_table.py problems   # no GPU needed
    python matmul_selection_gb300/tuned/make_table.py tune [OUT]  # on the GPU

``problems`` writes ``problems.csv``: one record per benchmark workload in
the format the library's ``record_untuned`` option writes (the PyTorch
TunableOp guide's record-then-tune workflow, sections 6-7).  ``tune`` runs
``mm_tune_file`` on it in a fresh process (empty table) and saves the result
with ``mm_cache_save`` as ``gb300.csv`` (or OUT), a result file whose
validators name the library version, the candidate set, the device model and
the CUDA runtime.  Load it with ``mm_cache_load`` (or point the
``cache_file`` option at a copy named for the device ordinal) to skip the
cold tune of these keys.
"""
from __future__ import annotations

import csv
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PROBLEMS = os.path.join(HERE, "problems.csv")
TABLE = os.path.join(HERE, "gb300.csv")

# (M, N, K, layout, (a, b, c), lda padding, batch): the benchmark workloads
BF16, F32 = "bf16", "f32"
WORKLOADS = [
    (256, 256, 256, "NN", (BF16, BF16, F32), 0, 1),
    (1, 4096, 4096, "NN", (BF16, BF16, BF16), 0, 1),
    (8, 4096, 4096, "NN", (BF16, BF16, BF16), 0, 1),
    (16, 4096, 4096, "NN", (BF16, BF16, BF16), 0, 1),
    (1, 4096, 4096, "NT", (BF16, BF16, BF16), 0, 1),
    (8, 4096, 4096, "NT", (BF16, BF16, BF16), 0, 1),
    (16, 4096, 4096, "NT", (BF16, BF16, BF16), 0, 1),
    (4096, 4096, 4096, "NN", (BF16, BF16, BF16), 0, 1),
    (4096, 4096, 4096, "NT", (BF16, BF16, BF16), 0, 1),
    (4096, 4096, 4096, "TN", (BF16, BF16, BF16), 0, 1),
    (4096, 4096, 4096, "TT", (BF16, BF16, BF16), 0, 1),
    (8192, 8192, 8192, "NN", (BF16, BF16, BF16), 0, 1),
    (25088, 4096, 64, "NT", (F32, F32, F32), 0, 1),
    (4096, 4096, 64, "NT", (F32, F32, F32), 0, 1),
    (128, 128, 65536, "NN", (BF16, BF16, BF16), 0, 1),
    (512, 512, 512, "NN", (BF16, BF16, F32), 0, 32),
] + [(m, 4096, 4096, "N" + t, (BF16, BF16, BF16), 4, 1)
     for m in (1, 16, 127, 1000, 4097, 8192) for t in "NT"]

CODE = {"bf16": 0, "f16": 1, "f32": 2}


def records():
    """The problems as record_untuned rows (key text from the library)."""
    import matmul_selection_gb300 as mm
    rows, seen = [], set()
    for M, N, K, lay, dts, pad, batch in WORKLOADS:
        at, bt = lay[0] == "T", lay[1] == "T"
        lda = (M if at else K) + pad
        ldb = K if bt else N
        ldc = N
        sa = (K if at else M) * lda
        sb = (N if bt else K) * ldb
        sc = M * ldc
        b = None if batch == 1 else (batch, sa, sb, sc)
        st, _, text = mm.mm_tune_key(M, N, K, lda, ldb, ldc, tuple(CODE[d] for d in dts), lay, b)
        mm.check(st)
        if text in seen:  # M = 4097 and 8192 share a key: one record
            continue
        seen.add(text)
        rows.append(["Untuned", text, M, N, K, lda, ldb, ldc, *dts, lay,
                     batch, sa if batch > 1 else 0, sb if batch > 1 else 0,
                     sc if batch > 1 else 0])
    return rows


def write_problems(path=PROBLEMS):
    with open(path, "w", newline="") as f:
        csv.writer(f, lineterminator="\n").writerows(records())
    return path


def tune(out=TABLE, problems=PROBLEMS):
    import matmul_selection_gb300 as mm
    mm.check(mm.mm_set_option("tuning", "1"))
    mm.check(mm.mm_cache_clear())
    st, n = mm.mm_tune_file(problems)
    mm.check(st)
    mm.check(mm.mm_cache_save(out))
    return n


if __name__ == "__main__":
    what = sys.argv[1] if len(sys.argv) > 1 else "problems"
    if what == "problems":
        print(write_problems())
    elif what == "tune":
        import torch
        torch.cuda.init()
        out = sys.argv[2] if len(sys.argv) > 2 else TABLE
        print(tune(out), "keys tuned ->", out)
    else:
        raise SystemExit(__doc__)
