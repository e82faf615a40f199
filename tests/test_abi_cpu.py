"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and its host-only logic (key, bound, options) agrees with
the oracle.  No call here launches device work."""
import ctypes
import itertools
import os
import re

import pytest

import matmul_selection_gb300 as mm
from oracle import key as okey

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mm.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mm_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(mm.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in mm.h but not exported"
    assert set(names) == set(mm.EXPORTED), "binding and header disagree"


def test_version_and_registry():
    assert mm.mm_version().startswith("0.2.0+")
    names = mm.candidate_names()
    assert names[0] == "naive"
    assert len(names) == len(set(names))
    assert "gemv_n" in names and "gemv_t" in names
    assert mm.mm_candidate_name(len(names)) is None


def test_roofline_limit_pin():
    ns = mm.mm_roofline_limit_ns(2146435072, 9044321293800.54, 12582912, 319882855399.6339,
                                 0.8, 3626)
    assert int(ns) == 300281


def _fields(text):
    return okey.parse_key_text(text)


DT = {0: "bf16", 1: "f16", 2: "f32"}


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 4096, 4096), (127, 4096, 4096),
                                   (1000, 1000, 1000), (4097, 4096, 4096), (8192, 4096, 4096),
                                   (768, 768, 768), (1025, 1025, 1025), (256, 256, 256),
                                   (3, 5, 7), (1, 1, 1), (25088, 4096, 64), (128, 128, 65536)])
@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("dt", [(0, 0, 0), (2, 2, 2), (0, 0, 2), (1, 1, 1)])
def test_key_matches_oracle(M, N, K, layout, dt):
    at, bt = layout[0] == "T", layout[1] == "T"
    for pad in (0, 4, 1):
        lda = (M if at else K) + pad
        ldb = (K if bt else N) + pad
        st, kb, text = mm.mm_tune_key(M, N, K, lda, ldb, N, dt, layout)
        assert st == 0, mm.mm_last_error()
        want = okey.make_key(M, N, K, lda, ldb, *dt, a_trans=at, b_trans=bt)
        assert _fields(text) == want


def test_key_golden_rows_through_abi():
    for n, ls in [(512, 10), (768, 10), (1000, 5), (1024, 10), (1025, 2), (2048, 10)]:
        st, kb, text = mm.mm_tune_key(n, n, n, n, n, n, (2, 2, 2), "NN")
        f = _fields(text)
        assert f["lhs_stride"] == ls and f["rhs_stride"] == ls and f["lhs_pow2"] == 4
    k768 = mm.mm_tune_key(768, 768, 768, 768, 768, 768, (2, 2, 2), "NN")[1]
    k1024 = mm.mm_tune_key(1024, 1024, 1024, 1024, 1024, 1024, (2, 2, 2), "NN")[1]
    k1000 = mm.mm_tune_key(1000, 1000, 1000, 1000, 1000, 1000, (2, 2, 2), "NN")[1]
    assert k768 == k1024 and k1000 != k1024
    _, _, t = mm.mm_tune_key(1024, 1024, 1024, 1024, 1024, 1024, (2, 2, 2), "NT")
    assert "layout_rhs=MildlyPermuted{transposed:true,batch_swap:false}" in t


def test_key_batched_matches_oracle():
    cases = [(512, 512, 512, 32, 512 * 512, 512 * 512), (4, 4, 4, 32, 4, 16),
             (64, 48, 32, 3, 64 * 32 + 8, 0)]
    for M, N, K, b, sa, sb in cases:
        st, _, text = mm.mm_tune_key(M, N, K, K, N, N, (0, 0, 2), "NN", batch=(b, sa, sb, M * N))
        assert st == 0, mm.mm_last_error()
        assert _fields(text) == okey.make_key(M, N, K, K, N, 0, 0, 2, batch=b, stride_a=sa,
                                              stride_b=sb)


def test_element_misaligned_pointers_rejected_before_any_launch():
    """An operand that does not start on a multiple of its element size is
    refused on the host (no kernel can read half an element); the pointers
    here are never dereferenced, so this runs without a GPU."""
    bf = (0, 0, 0)
    f32 = (2, 2, 2)
    for dt, bad in ((bf, (0x1001, 0x2000, 0x3000)), (bf, (0x1000, 0x2001, 0x3000)),
                    (bf, (0x1000, 0x2000, 0x3001)), (f32, (0x1002, 0x2000, 0x3000)),
                    (f32, (0x1000, 0x2000, 0x3006))):
        for call in (lambda: mm.mm_autotune_execute(*bad, 1, 64, 64, 64, 64, 64, dt, "NT"),
                     lambda: mm.mm_execute_candidate(0, *bad, 1, 64, 64, 64, 64, 64, dt, "NT")):
            assert call() == mm.MM_ERR_INVALID_ARG
            assert "element size" in mm.mm_last_error()


def test_key_invalid_arguments():
    assert mm.mm_tune_key(-1, 4, 4, 4, 4, 4, (0, 0, 0), "NN")[0] == mm.MM_ERR_INVALID_ARG
    assert mm.mm_tune_key(4, 4, 4, 3, 4, 4, (0, 0, 0), "NN")[0] == mm.MM_ERR_INVALID_ARG
    assert mm.mm_tune_key(4, 4, 4, 4, 4, 4, (0, 7, 0), "NN")[0] == mm.MM_ERR_INVALID_ARG
    assert mm.mm_tune_key(4, 4, 4, 4, 4, 4, (0, 0, 0), 9)[0] == mm.MM_ERR_INVALID_ARG
    mm.mm_tune_key(4, 4, 4, 3, 4, 4, (0, 0, 0), "NN")
    assert "leading dimension" in mm.mm_last_error()


def test_options_roundtrip_and_errors():
    st, v = mm.mm_get_option("max_tuning_iterations")
    assert st == 0 and v == "100"
    assert mm.mm_set_option("max_tuning_iterations", "7") == 0
    assert mm.mm_get_option("max_tuning_iterations")[1] == "7"
    assert mm.mm_set_option("max_tuning_iterations", "100") == 0
    assert mm.mm_set_option("no_such_option", "1") == mm.MM_ERR_NOT_FOUND
    assert mm.mm_set_option("autotune_level", "sideways") == mm.MM_ERR_INVALID_ARG
    assert mm.mm_set_option("numerical_check", "1e-5") == mm.MM_ERR_INVALID_ARG
    assert mm.mm_set_option("numerical_check", "1e-5_1e-5") == 0
    assert mm.mm_set_option("numerical_check", "") == 0


def test_level_option_changes_buckets():
    try:
        assert mm.mm_set_option("autotune_level", "full") == 0
        _, _, t = mm.mm_tune_key(1000, 1000, 1000, 1000, 1000, 1000, (2, 2, 2), "NN")
        assert _fields(t)["m"] == 1000
        assert mm.mm_set_option("autotune_level", "minimal") == 0
        _, _, t = mm.mm_tune_key(1000, 1000, 1000, 1000, 1000, 1000, (2, 2, 2), "NN")
        assert _fields(t)["m"] == okey.anchor(1000, "minimal")
    finally:
        mm.mm_set_option("autotune_level", "balanced")
