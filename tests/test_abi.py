"""The C-ABI library builds, loads and exports every symbol include/*.h declares (no GPU needed)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        names |= set(re.findall(r"SPMM_API\s+[^;(]*?\b(spmm_\w+)\s*\(", txt))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from sparse_dense_matrix_spmm_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("spmm_bcsr", "spmm_wcsr", "spmm_24", "spmm_tvw", "spmm_build_bcsr_count", "spmm_build_bcsr_fill",
              "spmm_build_wcsr_count", "spmm_build_wcsr_fill", "spmm_compress_24", "spmm_build_tvw"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_signatures_cover_the_header():
    from sparse_dense_matrix_spmm_gb300 import _lib
    assert sorted(_lib.SIGNATURES) == _declared()


def test_host_only_calls(lib):
    from sparse_dense_matrix_spmm_gb300 import _lib
    L = _lib.load()
    assert L.spmm_version() >= 100
    assert L.spmm_status_string(0) == b"ok"
    assert L.spmm_status_string(4) == b"invalid sparse format data"


def test_struct_layouts_match_c():
    # sizes of the format structs as laid out by the C compiler (x86-64 / aarch64 LP64)
    from sparse_dense_matrix_spmm_gb300 import _lib
    assert ctypes.sizeof(_lib.BcsrT) == 8 * 2 + 4 * 2 + 8 + 8 + 8 * 3
    assert ctypes.sizeof(_lib.T24) == 8 * 2 + 8 + 8 * 3
    assert ctypes.sizeof(_lib.TvwT) == 8 * 2 + 4 * 2 + 8 * 2 + 8 * 4
    assert ctypes.sizeof(_lib.WcsrT) == 8 * 3 + 4 * 3 + 4 + 8 * 3 + 8 * 9
    assert ctypes.sizeof(_lib.SlideT) == 8 * 2 + 4 * 2 + 8 * 2


def test_host_validation_rejects_bad_arguments_before_launch():
    from sparse_dense_matrix_spmm_gb300 import _lib
    L = _lib.load()
    a = _lib.BcsrT(256, 256, 16, 16, 64, 0, None, None, None)
    # null B / C -> SPMM_ERR_NULL
    assert L.spmm_bcsr(ctypes.byref(a), None, 64, None, 64, 64, None) == 1
    # M not divisible by bh -> SPMM_ERR_SHAPE (checked before any device work)
    b = _lib.BcsrT(250, 256, 16, 16, 64, 0, 16, 16, 16)
    assert L.spmm_bcsr(ctypes.byref(b), 16, 64, 16, 64, 64, None) == 2
    # int8 BCSR SpMM -> SPMM_ERR_DTYPE
    c = _lib.BcsrT(256, 256, 16, 16, 64, 2, 16, 16, 16)
    assert L.spmm_bcsr(ctypes.byref(c), 16, 64, 16, 64, 64, None) == 3
    # K % 8 for the 2:4 compressor -> SPMM_ERR_SHAPE
    assert L.spmm_compress_24(16, 4, 12, 12, 2, 16, 16, None) == 2
    # (2n-2):2n: n outside [2, 8], K not a multiple of 64 n (SpMM) or 4 n (builder) -> SPMM_ERR_SHAPE
    sl = _lib.SlideT(128, 256, 1, 1, 16, 16)
    assert L.spmm_slide(ctypes.byref(sl), 16, 64, 16, 64, 64, None, 0, None) == 2
    sl = _lib.SlideT(128, 320, 4, 1, 16, 16)
    assert L.spmm_slide(ctypes.byref(sl), 16, 64, 16, 64, 64, None, 0, None) == 2
    assert L.spmm_build_slide(16, 4, 40, 40, 1, 4, 16, 16, None) == 2
    assert L.spmm_build_slide(16, 4, 64, 64, 1, 9, 16, 16, None) == 2
    # permutation: M != K for the permuted product -> SPMM_ERR_SHAPE; bad CSR for RCM -> SPMM_ERR_FORMAT
    rect = _lib.BcsrT(128, 256, 16, 16, 0, 1, 16, 16, 16)
    assert L.spmm_bcsr_permuted(ctypes.byref(rect), 16, 16, 64, 16, 64, 64, 16, 1 << 30, None) == 2
    rp = (ctypes.c_int32 * 3)(0, 1, 2)
    col = (ctypes.c_int32 * 2)(0, 5)                      # column 5 outside [0, 2)
    perm = (ctypes.c_int32 * 2)()
    assert L.spmm_rcm_order(2, rp, col, perm) == 4
    assert L.spmm_permute_rows(16, 4, 16, 4, 4, 4, 3, 16, 0, None) == 3   # 3-byte elements -> SPMM_ERR_DTYPE


def test_host_rcm_equals_the_oracle():
    """The library's host RCM and the oracle's (written separately) give the same order."""
    from sparse_dense_matrix_spmm_gb300 import _lib
    import numpy as np
    import oracle
    import spmm_inputs as gen
    L = _lib.load()
    rng = np.random.default_rng(9)
    for n, dens in ((1, 0.5), (7, 0.2), (60, 0.05), (150, 0.02)):
        A = (rng.random((n, n)) < dens).astype(np.int8)
        A[n // 2, :] = 0                                   # isolated or nearly isolated nodes
        rp = np.concatenate([[0], np.cumsum((A != 0).sum(axis=1))]).astype(np.int32)
        col = np.nonzero(A)[1].astype(np.int32)
        perm = np.zeros(n, np.int32)
        assert L.spmm_rcm_order(n, rp.ctypes.data_as(ctypes.c_void_p), col.ctypes.data_as(ctypes.c_void_p),
                                perm.ctypes.data_as(ctypes.c_void_p)) == 0
        assert np.array_equal(perm, oracle.rcm(n, rp, col))
    p = gen.banded_scrambled_problem(300, 4, 1, seed=2, dtype="i8")
    rp = np.concatenate([[0], np.cumsum((p["A"] != 0).sum(axis=1))]).astype(np.int32)
    col = np.nonzero(p["A"])[1].astype(np.int32)
    perm = np.zeros(300, np.int32)
    L.spmm_rcm_order(300, rp.ctypes.data_as(ctypes.c_void_p), col.ctypes.data_as(ctypes.c_void_p),
                     perm.ctypes.data_as(ctypes.c_void_p))
    assert np.array_equal(perm, oracle.rcm_dense(p["A"]))


def test_sddmm_validation():
    from sparse_dense_matrix_spmm_gb300 import _lib
    L = _lib.load()
    S = _lib.CsrT(64, 64, 10, 1, 16, 16, 16)
    assert L.spmm_sddmm(ctypes.byref(S), 12, 16, 16, 16, 16, 16, None) == 2      # K % 8 != 0
    assert L.spmm_sddmm(ctypes.byref(S), 16, 16, 8, 16, 16, 16, None) == 2       # lda < K
    S8 = _lib.CsrT(64, 64, 10, 2, 16, 16, 16)                                    # int8: 16-element steps
    assert L.spmm_sddmm(ctypes.byref(S8), 8, 16, 8, 16, 8, 16, None) == 2        # K % 16 != 0
    assert L.spmm_sddmm(ctypes.byref(S8), 32, 16, 40, 16, 32, 16, None) == 2     # lda % 16 != 0
    assert L.spmm_sddmm(ctypes.byref(S8), 131072, 16, 131072, 16, 131072, 16, None) == 2  # K * 16384 >= 2^31
    SF = _lib.CsrT(64, 64, 10, 3, 16, 16, 16)
    assert L.spmm_sddmm(ctypes.byref(SF), 16, 16, 16, 16, 16, 16, None) == 3     # fp8 -> SPMM_ERR_DTYPE
    E = _lib.CsrT(64, 64, 0, 1, None, None, None)
    assert L.spmm_sddmm(ctypes.byref(E), 16, None, 16, None, 16, None, None) == 0  # no entries: nothing to do


def test_widened_values_validation():
    """spmm_widen_24 and a pre-widened vals16 are int8 only; a NULL destination or
    an unaligned vals16 is refused before any launch."""
    from sparse_dense_matrix_spmm_gb300 import _lib
    L = _lib.load()
    f16 = _lib.T24(128, 256, 1, 16, 16, None)
    assert L.spmm_widen_24(ctypes.byref(f16), 16, None) == 3                  # fp16 -> SPMM_ERR_DTYPE
    i8 = _lib.T24(128, 256, 2, 16, 16, None)
    assert L.spmm_widen_24(ctypes.byref(i8), None, None) == 1                 # no destination -> SPMM_ERR_NULL
    assert L.spmm_widen_24(ctypes.byref(i8), 8, None) == 2                    # unaligned -> SPMM_ERR_SHAPE
    f16w = _lib.T24(128, 256, 1, 16, 16, 32)
    n = ctypes.c_size_t(0)
    assert L.spmm_24_workspace_size(ctypes.byref(f16w), 64, ctypes.byref(n)) == 3  # vals16 on fp16 -> DTYPE
    i8w = _lib.T24(128, 256, 2, 16, 16, 32)
    assert L.spmm_24_workspace_size(ctypes.byref(i8w), 64, ctypes.byref(n)) == 0
    m = ctypes.c_size_t(0)
    assert L.spmm_24_workspace_size(ctypes.byref(i8), 64, ctypes.byref(m)) == 0
    assert m.value > n.value > 0                                              # only B is widened per call
