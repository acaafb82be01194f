"""ctypes view of the C ABI in include/spmm_gb300.h (argument marshalling only)."""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspmm_gb300.so")

SPMM_BF16, SPMM_F16, SPMM_I8, SPMM_E4M3, SPMM_E5M2 = 0, 1, 2, 3, 4
DEVERR_TIMEOUT, DEVERR_INDEX, DEVERR_FORMAT = 1, 2, 4
KERNEL_BCSR, KERNEL_SPARSE, KERNEL_WIDEN, KERNEL_WCSR, KERNEL_PRUNE, KERNEL_PERMUTE, KERNEL_SDDMM = 1, 2, 3, 4, 5, 6, 7
STATUS = {0: "SPMM_OK", 1: "SPMM_ERR_NULL", 2: "SPMM_ERR_SHAPE", 3: "SPMM_ERR_DTYPE", 4: "SPMM_ERR_FORMAT",
          5: "SPMM_ERR_WORKSPACE", 6: "SPMM_ERR_TIMEOUT", 7: "SPMM_ERR_CUDA", 8: "SPMM_ERR_UNSUPPORTED"}

P, I32, I64, SZ = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t


class SpmmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{fn} failed: {self.name}")


class BcsrT(C.Structure):
    _fields_ = [("M", I64), ("K", I64), ("bh", I32), ("bw", I32), ("nnzb", I64), ("dtype", I32),
                ("row_ptr", P), ("col_idx", P), ("vals", P)]


class CsrT(C.Structure):
    _fields_ = [("M", I64), ("K", I64), ("nnz", I64), ("dtype", I32), ("row_ptr", P), ("col", P), ("val", P)]


class WcsrT(C.Structure):
    _fields_ = [("M", I64), ("K", I64), ("nnz", I64), ("h", I32), ("S", I32), ("dtype", I32),
                ("n_windows", I64), ("n_wcols", I64), ("n_units", I64),
                ("wcol_ptr", P), ("wcols", P), ("wnz_ptr", P), ("unit_ptr", P), ("unit_win", P),
                ("unit_nz_ptr", P), ("lrow", P), ("slot", P), ("val", P)]


class T24(C.Structure):
    _fields_ = [("M", I64), ("K", I64), ("dtype", I32), ("vals", P), ("meta", P), ("vals16", P)]


class SlideT(C.Structure):
    _fields_ = [("M", I64), ("K", I64), ("n", I32), ("dtype", I32), ("vals", P), ("meta", P)]


class TvwT(C.Structure):
    _fields_ = [("M", I64), ("K", I64), ("tile_rows", I32), ("dtype", I32), ("n_tiles", I64), ("Kp", I64),
                ("tile_ptr", P), ("cols", P), ("vals", P), ("meta", P)]


# name -> (restype, argtypes); every function declared in include/spmm_gb300.h
SIGNATURES = {
    "spmm_status_string": (C.c_char_p, [I32]),
    "spmm_version": (C.c_int, []),
    "spmm_last_device_error": (I32, [C.POINTER(I32)]),
    "spmm_selftest_timeout": (I32, [C.c_uint64, P]),
    "spmm_trace_enable": (I32, [I32]),
    "spmm_trace_read": (I32, [I32, C.POINTER(I64), C.POINTER(C.c_double)]),
    "spmm_bcsr": (I32, [C.POINTER(BcsrT), P, I64, P, I64, I64, P]),
    "spmm_wcsr_workspace_size": (I32, [C.POINTER(WcsrT), I64, C.POINTER(SZ)]),
    "spmm_wcsr": (I32, [C.POINTER(WcsrT), P, I64, P, I64, I64, P, SZ, P]),
    "spmm_24_workspace_size": (I32, [C.POINTER(T24), I64, C.POINTER(SZ)]),
    "spmm_widen_24": (I32, [C.POINTER(T24), P, P]),
    "spmm_24": (I32, [C.POINTER(T24), P, I64, P, I64, I64, P, SZ, P]),
    "spmm_24_noalloc": (I32, [C.POINTER(T24), P, I64, P, I64, I64, P]),
    "spmm_tvw": (I32, [C.POINTER(TvwT), P, I64, P, I64, I64, P]),
    "spmm_slide_workspace_size": (I32, [C.POINTER(SlideT), I64, C.POINTER(SZ)]),
    "spmm_slide": (I32, [C.POINTER(SlideT), P, I64, P, I64, I64, P, SZ, P]),
    "spmm_build_bcsr_count": (I32, [P, I64, I64, I64, I32, I32, I32, P, C.POINTER(I64), P]),
    "spmm_build_bcsr_fill": (I32, [P, I64, I64, I64, I32, I32, I32, P, P, P, P]),
    "spmm_build_wcsr_workspace_size": (I32, [C.POINTER(CsrT), I32, C.POINTER(SZ)]),
    "spmm_build_wcsr_count": (I32, [C.POINTER(CsrT), I32, I32, P, SZ, C.POINTER(I64), C.POINTER(I64), P]),
    "spmm_build_wcsr_fill": (I32, [C.POINTER(CsrT), I32, I32, P, SZ, C.POINTER(WcsrT), P]),
    "spmm_compress_24": (I32, [P, I64, I64, I64, I32, P, P, P]),
    "spmm_prune_24": (I32, [P, I64, I64, I64, I32, P, P, P]),
    "spmm_build_tvw": (I32, [P, I64, I64, I64, I32, I32, P, P, I64, I64, P, P, P]),
    "spmm_prune_tvw": (I32, [P, I64, I64, I64, I32, I32, P, P, I64, I64, P, P, P]),
    "spmm_build_slide": (I32, [P, I64, I64, I64, I32, I32, P, P, P]),
    "spmm_rcm_order": (I32, [I64, P, P, P]),
    "spmm_sddmm": (I32, [C.POINTER(CsrT), I64, P, I64, P, I64, P, P]),
    "spmm_permute_sym": (I32, [P, I64, I64, I32, P, P, I64, P]),
    "spmm_permute_rows": (I32, [P, I64, P, I64, I64, I64, I32, P, I32, P]),
    "spmm_bcsr_permuted_workspace_size": (I32, [C.POINTER(BcsrT), I64, C.POINTER(SZ)]),
    "spmm_bcsr_permuted": (I32, [C.POINTER(BcsrT), P, P, I64, P, I64, I64, P, SZ, P]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load the compiled library.  There is no fallback: a missing library is an error."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                "(this package has no CPU fallback)")
        lib = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def call(name: str, *args) -> None:
    st = getattr(load(), name)(*args)
    if st != 0:
        raise SpmmError(name, st)
