"""CPU oracle for C = A_sparse * B_dense (fp64 / int64), via ctypes.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py``.  The product
package never imports it, and it never imports the product package.

The arithmetic lives in ``spmm_oracle.c`` (plain C, no CUDA headers).  This
wrapper only marshals numpy arrays.  Every SpMM returns the exact fp64 (or
int64) sums for rows [r0, r1) and the selected output columns.

Pins (what ties this oracle to something other than itself) are in
``tests/test_oracle_*.py``: exhaustive fp16/bf16 decoding against numpy,
brute-force dense GEMM on the densified operand (numpy / scipy), format
round trips, hand-worked fixtures under ``tests/golden/``, invariants, and
reductions to textbook routines (h = 1 row windows == scipy CSR SpMM; all
blocks present == dense GEMM).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spmm_oracle.c")
_LIB = os.path.join(_HERE, "libspmm_oracle.so")

DTYPES = {"bf16": 0, "f16": 1, "i8": 2, "e4m3": 3, "e5m2": 4}
FP8 = ("e4m3", "e5m2")
ERR_SHAPE, ERR_FORMAT = 2, 4


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over output rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        P, I64, I32 = C.c_void_p, C.c_int64, C.c_int
        L.orc_decode_bf16.restype = C.c_double
        L.orc_decode_bf16.argtypes = [C.c_uint16]
        L.orc_decode_f16.restype = C.c_double
        L.orc_decode_f16.argtypes = [C.c_uint16]
        L.orc_decode_e4m3.restype = C.c_double
        L.orc_decode_e4m3.argtypes = [C.c_uint8]
        L.orc_decode_e5m2.restype = C.c_double
        L.orc_decode_e5m2.argtypes = [C.c_uint8]
        L.orc_num_threads.restype = I32
        L.orc_bcsr_count.restype = I64
        L.orc_bcsr_count.argtypes = [P, I64, I64, I64, I32, I32, I32, P]
        L.orc_bcsr_fill.restype = I32
        L.orc_bcsr_fill.argtypes = [P, I64, I64, I64, I32, I32, I32, P, P, P]
        L.orc_bcsr_densify.argtypes = [I64, I64, I32, I32, I32, P, P, P, P]
        L.orc_bcsr_spmm.argtypes = [I64, I64, I32, I32, I32, P, P, P, P, I64, I64, I64, P, I64, P]
        L.orc_csr_check.restype = I32
        L.orc_csr_check.argtypes = [I64, I64, P, P]
        L.orc_csr_spmm.argtypes = [I64, I32, P, P, P, P, I64, I64, I64, P, I64, P]
        L.orc_wcsr_sizes.restype = I32
        L.orc_wcsr_sizes.argtypes = [I64, I64, P, P, I32, I32, P, P]
        L.orc_wcsr_fill.restype = I32
        L.orc_wcsr_fill.argtypes = [I64, I64, I32, P, P, P, I32, I32] + [P] * 9
        L.orc_wcsr_to_csr.argtypes = [I64, I32, I32, P, P, P, P, P, P, P, P, P]
        L.orc_wcsr_spmm.argtypes = [I64, I32, I32, P, P, P, P, P, P, P, I64, I64, I64, P, I64, P]
        L.orc_compress24.restype = I32
        L.orc_compress24.argtypes = [P, I64, I64, I64, I32, P, P]
        L.orc_densify24.argtypes = [I64, I64, I32, P, P, P]
        L.orc_prune24.restype = I32
        L.orc_prune24.argtypes = [P, I64, I64, I64, I32, P, P]
        L.orc_prune_tvw.restype = I32
        L.orc_prune_tvw.argtypes = [P, I64, I64, I64, I32, I32, P, P, I64, P, P]
        L.orc_slide_src.restype = I64
        L.orc_slide_src.argtypes = [I64, I64, I32]
        L.orc_slide_decompose.restype = I32
        L.orc_slide_decompose.argtypes = [P, I64, I64, I64, I32, I32, P]
        L.orc_rcm.restype = I32
        L.orc_rcm.argtypes = [I64, P, P, P]
        L.orc_permute_sym.argtypes = [I64, I64, I32, P, P, P]
        L.orc_sddmm.argtypes = [I64, I64, I32, P, P, P, P, P]
        L.orc_sddmm_i64.argtypes = [I64, I64, P, P, P, P, P]
        L.orc_spmm24_f64.argtypes = [I64, I64, I32, P, P, P, I64, I64, I64, P, I64, P]
        L.orc_spmm24_i64.argtypes = [I64, I64, P, P, P, I64, I64, I64, P, I64, P]
        L.orc_tvw_build.restype = I32
        L.orc_tvw_build.argtypes = [P, I64, I64, I64, I32, I32, P, P, I64, P, P]
        L.orc_tvw_densify.argtypes = [I64, I64, I32, I32, P, P, I64, P, P, P]
        L.orc_tvw_spmm.argtypes = [I64, I32, I32, P, P, I64, P, P, P, I64, I64, I64, P, I64, P]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype=None):
    a = np.asarray(a)
    return np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))


def _hold(F):
    """Contiguous copies of a format's arrays, kept alive for the whole call."""
    return {k: _c(v) for k, v in F.items() if isinstance(v, np.ndarray)}


def _sel(N, rows, cols):
    r0, r1 = (0, None) if rows is None else rows
    colarr = None if cols is None else _c(np.asarray(cols), np.int64)
    ncols = N if colarr is None else colarr.shape[0]
    return r0, r1, colarr, ncols


def num_threads() -> int:
    return int(lib().orc_num_threads())


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Element-wise decode of stored bf16/fp16/fp8 bits (or int8) to float64."""
    L = lib()
    f = {"bf16": L.orc_decode_bf16, "f16": L.orc_decode_f16, "e4m3": L.orc_decode_e4m3,
         "e5m2": L.orc_decode_e5m2}.get(dtype)
    if dtype == "i8":
        return bits.astype(np.float64)
    flat = bits.reshape(-1)
    out = np.empty(flat.shape[0], dtype=np.float64)
    for i, b in enumerate(flat.tolist()):
        out[i] = f(b)
    return out.reshape(bits.shape)


def _edt(dtype):
    if dtype == "i8":
        return np.int8
    return np.uint8 if dtype in FP8 else np.uint16


# ------------------------------------------------------------------ BCSR
def bcsr_build(A, bh, bw, dtype):
    """dense (bits) -> dict(row_ptr, col_idx, vals) per the BCSR reading."""
    A = _c(A, _edt(dtype))
    M, K = A.shape
    row_ptr = np.zeros(M // bh + 1 if bh and M % bh == 0 else 1, dtype=np.int32)
    n = lib().orc_bcsr_count(_p(A), M, K, K, bh, bw, DTYPES[dtype], _p(row_ptr))
    if n < 0:
        raise OracleError(f"bcsr shape error {-n}")
    col_idx = np.zeros(max(n, 1), dtype=np.int32)[:n]
    vals = np.zeros((n, bh, bw), dtype=_edt(dtype))
    rc = lib().orc_bcsr_fill(_p(A), M, K, K, bh, bw, DTYPES[dtype], _p(row_ptr), _p(col_idx), _p(vals))
    if rc:
        raise OracleError(f"bcsr fill error {rc}")
    return {"M": M, "K": K, "bh": bh, "bw": bw, "dtype": dtype, "nnzb": int(n),
            "row_ptr": row_ptr, "col_idx": col_idx, "vals": vals}


def bcsr_densify(F):
    H = _hold(F)
    D = np.zeros((F["M"], F["K"]), dtype=_edt(F["dtype"]))
    lib().orc_bcsr_densify(F["M"], F["K"], F["bh"], F["bw"], DTYPES[F["dtype"]], _p(H["row_ptr"]),
                           _p(H["col_idx"]), _p(H["vals"]), _p(D))
    return D


def bcsr_spmm(F, B, rows=None, cols=None):
    H = _hold(F)
    B = _c(B, _edt(F["dtype"]))
    r0, r1, colarr, ncols = _sel(B.shape[1], rows, cols)
    r1 = F["M"] if r1 is None else r1
    out = np.zeros((r1 - r0, ncols), dtype=np.float64)
    lib().orc_bcsr_spmm(F["M"], F["K"], F["bh"], F["bw"], DTYPES[F["dtype"]], _p(H["row_ptr"]),
                        _p(H["col_idx"]), _p(H["vals"]), _p(B), B.shape[1], r0, r1,
                        _p(colarr), ncols, _p(out))
    return out


# ------------------------------------------------------------------ CSR / WCSR
def csr_check(M, K, row_ptr, col):
    rp, cl = _c(row_ptr, np.int32), _c(col, np.int32)
    return int(lib().orc_csr_check(M, K, _p(rp), _p(cl)))


def csr_spmm(M, row_ptr, col, val, B, dtype, rows=None, cols=None):
    B = _c(B, _edt(dtype))
    r0, r1, colarr, ncols = _sel(B.shape[1], rows, cols)
    r1 = M if r1 is None else r1
    out = np.zeros((r1 - r0, ncols), dtype=np.float64)
    rp, cl, vl = _c(row_ptr, np.int32), _c(col, np.int32), _c(val, _edt(dtype))
    lib().orc_csr_spmm(M, DTYPES[dtype], _p(rp), _p(cl), _p(vl), _p(B), B.shape[1], r0, r1,
                       _p(colarr), ncols, _p(out))
    return out


def wcsr_build(M, K, row_ptr, col, val, dtype, h=16, S=32):
    """CSR -> row-window format (see spmm_oracle.c for the layout reading)."""
    row_ptr = _c(row_ptr, np.int32)
    col = _c(col, np.int32)
    val = _c(val, _edt(dtype))
    L = lib()
    tw, tu = C.c_int64(0), C.c_int64(0)
    rc = L.orc_wcsr_sizes(M, K, _p(row_ptr), _p(col), h, S, C.byref(tw), C.byref(tu))
    if rc:
        raise OracleError(f"wcsr error {rc}")
    nw = (M + h - 1) // h
    nnz = int(row_ptr[M])
    F = {"M": M, "K": K, "h": h, "S": S, "dtype": dtype, "nw": nw, "nnz": nnz,
         "n_wcols": tw.value, "n_units": tu.value,
         "wcol_ptr": np.zeros(nw + 1, np.int32), "wcols": np.zeros(max(tw.value, 1), np.int32),
         "wnz_ptr": np.zeros(nw + 1, np.int32), "unit_ptr": np.zeros(nw + 1, np.int32),
         "unit_win": np.zeros(max(tu.value, 1), np.int32), "unit_nz_ptr": np.zeros(tu.value + 1, np.int32),
         "lrow": np.zeros(max(nnz, 1), np.uint8), "slot": np.zeros(max(nnz, 1), np.int32),
         "val": np.zeros(max(nnz, 1), _edt(dtype))}
    rc = L.orc_wcsr_fill(M, K, DTYPES[dtype], _p(row_ptr), _p(col), _p(val), h, S,
                         _p(F["wcol_ptr"]), _p(F["wcols"]), _p(F["wnz_ptr"]), _p(F["unit_ptr"]),
                         _p(F["unit_win"]), _p(F["unit_nz_ptr"]), _p(F["lrow"]), _p(F["slot"]), _p(F["val"]))
    if rc:
        raise OracleError(f"wcsr fill error {rc}")
    for k, n in (("wcols", tw.value), ("unit_win", tu.value), ("lrow", nnz), ("slot", nnz), ("val", nnz)):
        F[k] = F[k][:n]
    return F


def wcsr_to_csr(F):
    H = _hold(F)
    M, nnz = F["M"], F["nnz"]
    row_ptr = np.zeros(M + 1, np.int32)
    col = np.zeros(max(nnz, 1), np.int32)
    val = np.zeros(max(nnz, 1), _edt(F["dtype"]))
    lib().orc_wcsr_to_csr(M, F["h"], DTYPES[F["dtype"]], _p(H["wcol_ptr"]), _p(H["wcols"]),
                          _p(H["wnz_ptr"]), _p(H["lrow"]), _p(H["slot"]), _p(H["val"]),
                          _p(row_ptr), _p(col), _p(val))
    return row_ptr, col[:nnz], val[:nnz]


def wcsr_spmm(F, B, rows=None, cols=None):
    H = _hold(F)
    B = _c(B, _edt(F["dtype"]))
    r0, r1, colarr, ncols = _sel(B.shape[1], rows, cols)
    r1 = F["M"] if r1 is None else r1
    out = np.zeros((r1 - r0, ncols), dtype=np.float64)
    lib().orc_wcsr_spmm(F["M"], F["h"], DTYPES[F["dtype"]], _p(H["wcol_ptr"]), _p(H["wcols"]),
                        _p(H["wnz_ptr"]), _p(H["lrow"]), _p(H["slot"]), _p(H["val"]),
                        _p(B), B.shape[1], r0, r1, _p(colarr), ncols, _p(out))
    return out


# ------------------------------------------------------------------ 2:4
def compress24(A, dtype):
    A = _c(A, _edt(dtype))
    M, K = A.shape
    vals = np.zeros((M, K // 2), dtype=_edt(dtype))
    meta = np.zeros((M, (K + 7) // 8), dtype=np.uint8)
    rc = lib().orc_compress24(_p(A), M, K, K, DTYPES[dtype], _p(vals), _p(meta))
    if rc:
        raise OracleError(f"compress24 error {rc}")
    return {"M": M, "K": K, "dtype": dtype, "vals": vals, "meta": meta}


def prune24(A, dtype):
    """Magnitude pruning of a dense matrix into the 2:4 format (the two largest
    magnitudes of every 4-group, ties to the lower index)."""
    A = _c(A, _edt(dtype))
    M, K = A.shape
    vals = np.zeros((M, K // 2), dtype=_edt(dtype))
    meta = np.zeros((M, (K + 7) // 8), dtype=np.uint8)
    rc = lib().orc_prune24(_p(A), M, K, K, DTYPES[dtype], _p(vals), _p(meta))
    if rc:
        raise OracleError(f"prune24 error {rc}")
    return {"M": M, "K": K, "dtype": dtype, "vals": vals, "meta": meta}


def densify24(F):
    H = _hold(F)
    D = np.zeros((F["M"], F["K"]), dtype=_edt(F["dtype"]))
    lib().orc_densify24(F["M"], F["K"], DTYPES[F["dtype"]], _p(H["vals"]), _p(H["meta"]), _p(D))
    return D


def spmm24(F, B, rows=None, cols=None):
    """int8 -> exact int64; bf16/fp16/fp8 -> fp64 (B of the operand's type)."""
    H = _hold(F)
    B = _c(B, _edt(F["dtype"]))
    r0, r1, colarr, ncols = _sel(B.shape[1], rows, cols)
    r1 = F["M"] if r1 is None else r1
    if F["dtype"] == "i8":
        out = np.zeros((r1 - r0, ncols), dtype=np.int64)
        lib().orc_spmm24_i64(F["M"], F["K"], _p(H["vals"]), _p(H["meta"]), _p(B), B.shape[1],
                             r0, r1, _p(colarr), ncols, _p(out))
    else:
        out = np.zeros((r1 - r0, ncols), dtype=np.float64)
        lib().orc_spmm24_f64(F["M"], F["K"], DTYPES[F["dtype"]], _p(H["vals"]), _p(H["meta"]),
                             _p(B), B.shape[1], r0, r1, _p(colarr), ncols, _p(out))
    return out


# ------------------------------------------------------------------ (2n-2):2n
def slide_lifted_k(K, n):
    """Lifted depth K' = 4 (n - 1) K / 2n: n - 1 windows of 4 per group of 2n."""
    return 4 * (n - 1) * (K // (2 * n))


def slide_src(K, n):
    """Original column (= row of B) read by every lifted column, window-plane order."""
    return np.array([lib().orc_slide_src(q, K, n) for q in range(slide_lifted_k(K, n))], dtype=np.int64)


def slide_decompose(A, n, dtype):
    """Dense (2n-2):2n matrix -> dense lifted matrix (M x K'), each nonzero in
    exactly one window and every window 2:4."""
    A = _c(A, _edt(dtype))
    M, K = A.shape
    L = np.zeros((M, slide_lifted_k(K, n)), dtype=_edt(dtype))
    rc = lib().orc_slide_decompose(_p(A), M, K, K, DTYPES[dtype], n, _p(L))
    if rc:
        raise OracleError(f"slide_decompose error {rc}")
    return L


def slide_build(A, n, dtype):
    """(2n-2):2n -> the lifted operand in the 2:4 format: vals[M][K'/2] and
    meta[M][K'/8], as compress24 of the lifted matrix.  "K" is the original depth."""
    M, K = np.shape(A)
    F = compress24(slide_decompose(A, n, dtype), dtype)
    return {"M": M, "K": K, "n": n, "dtype": dtype, "vals": F["vals"], "meta": F["meta"]}


def slide_lift_b(B, K, n):
    """Activation lifting: lifted row q of B is original row slide_src(K, n)[q]."""
    return np.ascontiguousarray(np.asarray(B)[slide_src(K, n)])


def slide_spmm(F, B, rows=None, cols=None):
    """C = A_lifted * lift(B), through the 2:4 SpMM of the lifted operand."""
    Kl = slide_lifted_k(F["K"], F["n"])
    G = {"M": F["M"], "K": Kl, "dtype": F["dtype"], "vals": F["vals"], "meta": F["meta"]}
    return spmm24(G, slide_lift_b(B, F["K"], F["n"]), rows, cols)


# ------------------------------------------------------------------ TVW
def tvw_build(A, tile_rows, tile_ptr, cols, dtype, Kp=None):
    A = _c(A, _edt(dtype))
    M, K = A.shape
    tile_ptr = _c(tile_ptr, np.int32)
    cols = _c(cols, np.int32)
    kt_max = int(np.max(np.diff(tile_ptr))) if tile_ptr.shape[0] > 1 else 0
    if Kp is None:
        Kp = max(8, -(-kt_max // 8) * 8)
    vals = np.zeros((M, Kp // 2), dtype=_edt(dtype))
    meta = np.zeros((M, Kp // 8), dtype=np.uint8)
    rc = lib().orc_tvw_build(_p(A), M, K, K, DTYPES[dtype], tile_rows, _p(tile_ptr), _p(cols), Kp,
                             _p(vals), _p(meta))
    if rc:
        raise OracleError(f"tvw error {rc}")
    return {"M": M, "K": K, "dtype": dtype, "tile_rows": tile_rows, "tile_ptr": tile_ptr,
            "cols": cols, "Kp": Kp, "vals": vals, "meta": meta}


def prune_tvw(A, tile_rows, tile_ptr, cols, dtype, Kp=None):
    """Magnitude pruning into TVW: entries outside each tile's kept columns dropped,
    2:4 by magnitude inside (ties to the lower index)."""
    A = _c(A, _edt(dtype))
    M, K = A.shape
    tile_ptr = _c(tile_ptr, np.int32)
    cols = _c(cols, np.int32)
    kt_max = int(np.max(np.diff(tile_ptr))) if tile_ptr.shape[0] > 1 else 0
    if Kp is None:
        Kp = max(8, -(-kt_max // 8) * 8)
    vals = np.zeros((M, Kp // 2), dtype=_edt(dtype))
    meta = np.zeros((M, Kp // 8), dtype=np.uint8)
    rc = lib().orc_prune_tvw(_p(A), M, K, K, DTYPES[dtype], tile_rows, _p(tile_ptr), _p(cols), Kp,
                             _p(vals), _p(meta))
    if rc:
        raise OracleError(f"prune_tvw error {rc}")
    return {"M": M, "K": K, "dtype": dtype, "tile_rows": tile_rows, "tile_ptr": tile_ptr,
            "cols": cols, "Kp": Kp, "vals": vals, "meta": meta}


def tvw_densify(F):
    H = _hold(F)
    D = np.zeros((F["M"], F["K"]), dtype=_edt(F["dtype"]))
    lib().orc_tvw_densify(F["M"], F["K"], DTYPES[F["dtype"]], F["tile_rows"], _p(H["tile_ptr"]),
                          _p(H["cols"]), F["Kp"], _p(H["vals"]), _p(H["meta"]), _p(D))
    return D


def tvw_spmm(F, B, rows=None, cols=None):
    H = _hold(F)
    B = _c(B, _edt(F["dtype"]))
    r0, r1, colarr, ncols = _sel(B.shape[1], rows, cols)
    r1 = F["M"] if r1 is None else r1
    out = np.zeros((r1 - r0, ncols), dtype=np.float64)
    lib().orc_tvw_spmm(F["M"], DTYPES[F["dtype"]], F["tile_rows"], _p(H["tile_ptr"]), _p(H["cols"]),
                       F["Kp"], _p(H["vals"]), _p(H["meta"]), _p(B), B.shape[1], r0, r1,
                       _p(colarr), ncols, _p(out))
    return out


# ------------------------------------------------------------------ permutation before BCSR
def rcm(n, row_ptr, col):
    """Reverse Cuthill-McKee order of the symmetrised pattern: perm[i] is the
    original index placed at position i."""
    row_ptr = _c(row_ptr, np.int32)
    col = _c(col, np.int32)
    perm = np.zeros(n, dtype=np.int32)
    rc = lib().orc_rcm(n, _p(row_ptr), _p(col), _p(perm))
    if rc:
        raise OracleError(f"rcm error {rc}")
    return perm


def rcm_dense(A):
    """RCM of the stored (nonzero) pattern of a dense square matrix of any encoding."""
    A = np.asarray(A)
    nz = (A & 0x7FFF) != 0 if A.dtype == np.uint16 else A != 0
    n = A.shape[0]
    row_ptr = np.concatenate([[0], np.cumsum(nz.sum(axis=1))]).astype(np.int32)
    col = np.nonzero(nz)[1].astype(np.int32)
    return rcm(n, row_ptr, col)


def permute_sym(A, perm, dtype):
    """A'[i][j] = A[perm[i]][perm[j]]."""
    A = _c(A, _edt(dtype))
    n = A.shape[0]
    out = np.zeros((n, n), dtype=_edt(dtype))
    lib().orc_permute_sym(n, A.shape[1], DTYPES[dtype], _p(A), _p(_c(perm, np.int32)), _p(out))
    return out


def bcsr_spmm_permuted(F, perm, B, rows=None, cols=None):
    """C = P^T (A' (P B)) for the BCSR F of A' = P A P^T: B's rows gathered by
    perm, the BCSR product, then C' row i written to row perm[i]."""
    perm = np.asarray(perm)
    Cp = bcsr_spmm(F, np.ascontiguousarray(np.asarray(B)[perm]), cols=cols)
    C = np.empty_like(Cp)
    C[perm] = Cp
    if rows is not None:
        C = C[rows[0]:rows[1]]
    return C


# ------------------------------------------------------------------ SDDMM
def sddmm(row_ptr, col, A, Bt, dtype):
    """out[e] = sum_k A[i][k] Bt[j][k] for every stored (i, j) of the CSR pattern (fp64)."""
    row_ptr = _c(row_ptr, np.int32)
    col = _c(col, np.int32)
    A = _c(A, _edt(dtype))
    Bt = _c(Bt, _edt(dtype))
    M, K = A.shape
    if Bt.shape[1] != K or row_ptr.shape[0] != M + 1:
        raise OracleError("sddmm shape error")
    out = np.zeros(int(row_ptr[-1]), dtype=np.float64)
    lib().orc_sddmm(M, K, DTYPES[dtype], _p(row_ptr), _p(col), _p(A), _p(Bt), _p(out))
    return out


def sddmm_i64(row_ptr, col, A, Bt):
    """int8 A, Bt: out[e] = sum_k A[i][k] Bt[j][k] for every stored (i, j), exact (int64)."""
    row_ptr = _c(row_ptr, np.int32)
    col = _c(col, np.int32)
    A = _c(A, np.int8)
    Bt = _c(Bt, np.int8)
    M, K = A.shape
    if Bt.shape[1] != K or row_ptr.shape[0] != M + 1:
        raise OracleError("sddmm shape error")
    out = np.zeros(int(row_ptr[-1]), dtype=np.int64)
    lib().orc_sddmm_i64(M, K, _p(row_ptr), _p(col), _p(A), _p(Bt), _p(out))
    return out
