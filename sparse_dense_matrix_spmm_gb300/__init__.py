"""GB300 (sm_103a) sparse x dense matrix multiply: C = A_sparse @ B_dense.

Thin Python binding over the C ABI of ``libspmm_gb300.so`` (declared in
``include/spmm_gb300.h``).  Every step of the computation runs in the CUDA
library; this module only allocates outputs with torch and passes pointers,
sizes and the current CUDA stream.  There is no CPU fallback: a missing
library raises.

Format containers hold device tensors:
  BCSR(M, K, bh, bw, nnzb, dtype, row_ptr, col_idx, vals)
  Mat24(M, K, dtype, vals, meta)
  Slide(M, K, n, dtype, vals, meta)   ((2n-2):2n lifted into 2:4 windows)
  TVW(M, K, tile_rows, dtype, n_tiles, Kp, tile_ptr, cols, vals, meta)
  CSR(M, K, nnz, dtype, row_ptr, col, val)
  WCSR(...)  (see include/spmm_gb300.h for the field meanings)

Beyond C = A B for those formats: spmm_slide ((2n-2):2n as overlapping 2:4
windows), spmm_bcsr_permuted (BCSR after a Reverse Cuthill-McKee order from
rcm_order), spmm_sddmm (A B sampled at a CSR pattern) and the pruning
builders spmm_prune_24 / spmm_prune_tvw.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass, field
from typing import Optional

import torch

from . import _lib
from ._lib import SpmmError

__all__ = ["BCSR", "Mat24", "Slide", "TVW", "CSR", "WCSR", "SpmmError", "spmm_bcsr", "spmm_build_bcsr_count",
           "spmm_build_bcsr_fill", "build_bcsr", "spmm_compress_24", "spmm_prune_24", "spmm_widen_24", "spmm_24", "spmm_24_workspace_size",
           "spmm_build_tvw", "spmm_prune_tvw", "spmm_tvw", "spmm_build_wcsr_workspace_size", "spmm_build_wcsr_count",
           "spmm_build_wcsr_fill", "build_wcsr", "spmm_wcsr", "spmm_wcsr_workspace_size",
           "spmm_build_slide", "spmm_slide", "spmm_slide_workspace_size",
           "spmm_sddmm", "rcm_order", "spmm_permute_sym", "spmm_permute_rows", "spmm_bcsr_permuted", "spmm_bcsr_permuted_workspace_size",
           "last_device_error", "selftest_timeout", "library_path", "trace_enable", "trace_read"]

_DT = {torch.bfloat16: _lib.SPMM_BF16, torch.float16: _lib.SPMM_F16, torch.int8: _lib.SPMM_I8,
       torch.float8_e4m3fn: _lib.SPMM_E4M3, torch.float8_e5m2: _lib.SPMM_E5M2}


def library_path() -> str:
    return _lib.LIB_PATH


def _code(dtype) -> int:
    if dtype not in _DT:
        raise TypeError(f"unsupported dtype {dtype}")
    return _DT[dtype]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None or t.numel() == 0 else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _check_dev(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all operands must be CUDA tensors (this library has no CPU path)")


# ------------------------------------------------------------------ formats
@dataclass
class BCSR:
    M: int
    K: int
    bh: int
    bw: int
    nnzb: int
    dtype: torch.dtype
    row_ptr: torch.Tensor
    col_idx: torch.Tensor
    vals: torch.Tensor

    def c(self) -> _lib.BcsrT:
        return _lib.BcsrT(self.M, self.K, self.bh, self.bw, self.nnzb, _code(self.dtype), _ptr(self.row_ptr),
                          _ptr(self.col_idx), _ptr(self.vals))


@dataclass
class Mat24:
    M: int
    K: int
    dtype: torch.dtype
    vals: torch.Tensor
    meta: torch.Tensor
    vals16: Optional[torch.Tensor] = None  # int8: vals widened to fp16 once (spmm_widen_24)

    def c(self) -> _lib.T24:
        return _lib.T24(self.M, self.K, _code(self.dtype), _ptr(self.vals), _ptr(self.meta), _ptr(self.vals16))


@dataclass
class Slide:
    """(2n-2):2n operand lifted into n - 1 overlapping 2:4 windows per group of 2n
    (window planes); K is the original depth, vals/meta span K' = 2 K (n-1) / n."""
    M: int
    K: int
    n: int
    dtype: torch.dtype
    vals: torch.Tensor
    meta: torch.Tensor

    @property
    def K_lifted(self) -> int:
        return 4 * (self.n - 1) * (self.K // (2 * self.n))

    def c(self) -> _lib.SlideT:
        return _lib.SlideT(self.M, self.K, self.n, _code(self.dtype), _ptr(self.vals), _ptr(self.meta))


@dataclass
class TVW:
    M: int
    K: int
    tile_rows: int
    dtype: torch.dtype
    n_tiles: int
    Kp: int
    tile_ptr: torch.Tensor
    cols: torch.Tensor
    vals: torch.Tensor
    meta: torch.Tensor

    def c(self) -> _lib.TvwT:
        return _lib.TvwT(self.M, self.K, self.tile_rows, _code(self.dtype), self.n_tiles, self.Kp,
                         _ptr(self.tile_ptr), _ptr(self.cols), _ptr(self.vals), _ptr(self.meta))


@dataclass
class CSR:
    M: int
    K: int
    nnz: int
    dtype: torch.dtype
    row_ptr: torch.Tensor
    col: torch.Tensor
    val: torch.Tensor

    def c(self) -> _lib.CsrT:
        return _lib.CsrT(self.M, self.K, self.nnz, _code(self.dtype), _ptr(self.row_ptr), _ptr(self.col),
                         _ptr(self.val))


@dataclass
class WCSR:
    M: int
    K: int
    nnz: int
    h: int
    S: int
    dtype: torch.dtype
    n_windows: int
    n_wcols: int
    n_units: int
    wcol_ptr: torch.Tensor
    wcols: torch.Tensor
    wnz_ptr: torch.Tensor
    unit_ptr: torch.Tensor
    unit_win: torch.Tensor
    unit_nz_ptr: torch.Tensor
    lrow: torch.Tensor
    slot: torch.Tensor
    val: torch.Tensor
    workspace: Optional[torch.Tensor] = field(default=None, repr=False)

    def c(self) -> _lib.WcsrT:
        return _lib.WcsrT(self.M, self.K, self.nnz, self.h, self.S, _code(self.dtype), self.n_windows,
                          self.n_wcols, self.n_units, _ptr(self.wcol_ptr), _ptr(self.wcols), _ptr(self.wnz_ptr),
                          _ptr(self.unit_ptr), _ptr(self.unit_win), _ptr(self.unit_nz_ptr), _ptr(self.lrow),
                          _ptr(self.slot), _ptr(self.val))


# ------------------------------------------------------------------ utilities
def last_device_error() -> int:
    """Read and clear the sticky device error word (SPMM_DEVERR_* bits)."""
    v = C.c_int32(0)
    _lib.call("spmm_last_device_error", C.byref(v))
    return v.value


def selftest_timeout(timeout_ns: int = 1_000_000, stream=None) -> None:
    _lib.call("spmm_selftest_timeout", C.c_uint64(timeout_ns), _stream(stream))


def trace_enable(on: bool = True) -> None:
    """Record CUDA events around every library kernel launch (see spmm_trace_read)."""
    _lib.call("spmm_trace_enable", 1 if on else 0)


def trace_read(kernel: int):
    """(launches, total_ms) of one kernel kind since tracing was enabled."""
    n, ms = C.c_int64(0), C.c_double(0.0)
    _lib.call("spmm_trace_read", kernel, C.byref(n), C.byref(ms))
    return n.value, ms.value


def _out(C_, M, N, dtype, device):
    if C_ is None:
        return torch.empty((M, N), dtype=dtype, device=device)
    return C_


# ------------------------------------------------------------------ BCSR
def spmm_build_bcsr_count(dense: torch.Tensor, bh: int, bw: int, stream=None):
    _check_dev(dense)
    M, K = dense.shape
    row_ptr = torch.empty(M // bh + 1 if bh > 0 else 1, dtype=torch.int32, device=dense.device)
    n = C.c_int64(0)
    _lib.call("spmm_build_bcsr_count", _ptr(dense), M, K, dense.stride(0), bh, bw, _code(dense.dtype),
              _ptr(row_ptr), C.byref(n), _stream(stream))
    return row_ptr, n.value


def spmm_build_bcsr_fill(dense: torch.Tensor, bh: int, bw: int, row_ptr: torch.Tensor, nnzb: int,
                         stream=None) -> BCSR:
    _check_dev(dense, row_ptr)
    M, K = dense.shape
    col_idx = torch.empty(max(nnzb, 1), dtype=torch.int32, device=dense.device)[:nnzb]
    vals = torch.empty((max(nnzb, 1), bh, bw), dtype=dense.dtype, device=dense.device)[:nnzb]
    _lib.call("spmm_build_bcsr_fill", _ptr(dense), M, K, dense.stride(0), bh, bw, _code(dense.dtype),
              _ptr(row_ptr), _ptr(col_idx), _ptr(vals), _stream(stream))
    return BCSR(M, K, bh, bw, nnzb, dense.dtype, row_ptr, col_idx, vals)


def build_bcsr(dense: torch.Tensor, bh: int, bw: int, stream=None) -> BCSR:
    row_ptr, n = spmm_build_bcsr_count(dense, bh, bw, stream)
    return spmm_build_bcsr_fill(dense, bh, bw, row_ptr, n, stream)


def spmm_bcsr(A: BCSR, B: torch.Tensor, C_: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    _check_dev(B, C_)
    N = B.shape[1]
    out = _out(C_, A.M, N, torch.float32, B.device)
    a = A.c()
    _lib.call("spmm_bcsr", C.byref(a), _ptr(B), B.stride(0), _ptr(out), out.stride(0), N, _stream(stream))
    return out


# ------------------------------------------------------------------ SDDMM
def spmm_sddmm(S: CSR, A: torch.Tensor, Bt: torch.Tensor, out: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """out[e] = A[i] . Bt[j] for every stored (i, j) of the CSR pattern S, in pattern
    order: fp32 for fp16/bf16 operands, exact int32 for int8 (S.dtype torch.int8)."""
    _check_dev(A, Bt, out)
    K = A.shape[1]
    if out is None:
        odt = torch.int32 if S.dtype == torch.int8 else torch.float32
        out = torch.empty(S.nnz, dtype=odt, device=A.device)
    s = S.c()
    _lib.call("spmm_sddmm", C.byref(s), K, _ptr(A), A.stride(0), _ptr(Bt), Bt.stride(0), _ptr(out), _stream(stream))
    return out


# ------------------------------------------------------------------ permutation before BCSR
def rcm_order(n: int, row_ptr, col) -> torch.Tensor:
    """Reverse Cuthill-McKee order (host) of an n x n CSR pattern given as host
    arrays (numpy or CPU tensors); returns perm as a CPU int32 tensor."""
    rp = torch.as_tensor(row_ptr, dtype=torch.int32).contiguous()
    cl = torch.as_tensor(col, dtype=torch.int32).contiguous()
    if rp.is_cuda or cl.is_cuda:
        raise ValueError("rcm_order takes host arrays")
    perm = torch.empty(n, dtype=torch.int32)
    _lib.call("spmm_rcm_order", n, _ptr(rp), _ptr(cl), _ptr(perm))
    return perm


def spmm_permute_sym(dense: torch.Tensor, perm: torch.Tensor, stream=None) -> torch.Tensor:
    """out[i][j] = dense[perm[i]][perm[j]] (P A P^T) on the device."""
    _check_dev(dense, perm)
    n = dense.shape[0]
    out = torch.empty((n, n), dtype=dense.dtype, device=dense.device)
    _lib.call("spmm_permute_sym", _ptr(dense), n, dense.stride(0), _code(dense.dtype), _ptr(perm), _ptr(out),
              out.stride(0), _stream(stream))
    return out


def spmm_permute_rows(src: torch.Tensor, perm: torch.Tensor, scatter: bool = False,
                      out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Row gather (out[i] = src[perm[i]]) or scatter (out[perm[i]] = src[i])."""
    _check_dev(src, perm, out)
    rows, cols = src.shape
    if out is None:
        out = torch.empty_like(src)
    _lib.call("spmm_permute_rows", _ptr(src), src.stride(0), _ptr(out), out.stride(0), rows, cols,
              src.element_size(), _ptr(perm), 1 if scatter else 0, _stream(stream))
    return out


def spmm_bcsr_permuted_workspace_size(A: BCSR, N: int) -> int:
    n = C.c_size_t(0)
    a = A.c()
    _lib.call("spmm_bcsr_permuted_workspace_size", C.byref(a), N, C.byref(n))
    return n.value


def spmm_bcsr_permuted(A: BCSR, perm: torch.Tensor, B: torch.Tensor, C_: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """C = A B where A is given as the BCSR of P A P^T and perm (device int32)."""
    _check_dev(perm, B, C_, workspace)
    N = B.shape[1]
    out = _out(C_, A.M, N, torch.float32, B.device)
    if workspace is None:
        workspace = torch.empty(spmm_bcsr_permuted_workspace_size(A, N), dtype=torch.uint8, device=B.device)
    a = A.c()
    _lib.call("spmm_bcsr_permuted", C.byref(a), _ptr(perm), _ptr(B), B.stride(0), _ptr(out), out.stride(0), N,
              _ptr(workspace), workspace.numel(), _stream(stream))
    return out


# ------------------------------------------------------------------ 2:4
def spmm_compress_24(dense: torch.Tensor, stream=None) -> Mat24:
    _check_dev(dense)
    M, K = dense.shape
    vals = torch.empty((M, K // 2), dtype=dense.dtype, device=dense.device)
    meta = torch.empty((M, K // 8), dtype=torch.uint8, device=dense.device)
    _lib.call("spmm_compress_24", _ptr(dense), M, K, dense.stride(0), _code(dense.dtype), _ptr(vals),
              _ptr(meta), _stream(stream))
    return Mat24(M, K, dense.dtype, vals, meta)


def spmm_prune_24(dense: torch.Tensor, stream=None) -> Mat24:
    """Magnitude-prune a dense (M x K) matrix into 2:4 (two largest |a| per group of 4)."""
    _check_dev(dense)
    M, K = dense.shape
    vals = torch.empty((M, K // 2), dtype=dense.dtype, device=dense.device)
    meta = torch.empty((M, K // 8), dtype=torch.uint8, device=dense.device)
    _lib.call("spmm_prune_24", _ptr(dense), M, K, dense.stride(0), _code(dense.dtype), _ptr(vals),
              _ptr(meta), _stream(stream))
    return Mat24(M, K, dense.dtype, vals, meta)


def spmm_24_workspace_size(A: Mat24, N: int) -> int:
    n = C.c_size_t(0)
    a = A.c()
    _lib.call("spmm_24_workspace_size", C.byref(a), N, C.byref(n))
    return n.value


def spmm_widen_24(A: Mat24, stream=None) -> Mat24:
    """int8 2:4 operand: the same operand with its values widened to fp16 once
    (vals16), so that spmm_24 widens only B on each call."""
    v16 = torch.empty((A.M, A.K // 2), dtype=torch.float16, device=A.vals.device)
    a = A.c()
    _lib.call("spmm_widen_24", C.byref(a), _ptr(v16), _stream(stream))
    return Mat24(A.M, A.K, A.dtype, A.vals, A.meta, v16)


def spmm_24(A: Mat24, B: torch.Tensor, C_: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    _check_dev(B, C_, workspace)
    N = B.shape[1]
    odt = torch.int32 if A.dtype == torch.int8 else torch.float32
    out = _out(C_, A.M, N, odt, B.device)
    need = spmm_24_workspace_size(A, N)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=B.device)
    a = A.c()
    _lib.call("spmm_24", C.byref(a), _ptr(B), B.stride(0), _ptr(out), out.stride(0), N, _ptr(workspace),
              0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream))
    return out


# ------------------------------------------------------------------ (2n-2):2n
def spmm_build_slide(dense: torch.Tensor, n: int, stream=None) -> Slide:
    """Decompose a dense (2n-2):2n matrix into its lifted 2:4 operand (n - 1
    overlapping windows per group of 2n, window-plane order)."""
    _check_dev(dense)
    M, K = dense.shape
    Kl = 4 * (n - 1) * (K // (2 * n)) if n > 0 else 0
    vals = torch.empty((M, Kl // 2), dtype=dense.dtype, device=dense.device)
    meta = torch.empty((M, Kl // 8), dtype=torch.uint8, device=dense.device)
    _lib.call("spmm_build_slide", _ptr(dense), M, K, dense.stride(0), _code(dense.dtype), n, _ptr(vals),
              _ptr(meta), _stream(stream))
    return Slide(M, K, n, dense.dtype, vals, meta)


def spmm_slide_workspace_size(A: Slide, N: int) -> int:
    n = C.c_size_t(0)
    a = A.c()
    _lib.call("spmm_slide_workspace_size", C.byref(a), N, C.byref(n))
    return n.value


def spmm_slide(A: Slide, B: torch.Tensor, C_: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """C = A @ B for a lifted (2n-2):2n operand; B holds the original K rows."""
    _check_dev(B, C_, workspace)
    N = B.shape[1]
    odt = torch.int32 if A.dtype == torch.int8 else torch.float32
    out = _out(C_, A.M, N, odt, B.device)
    need = spmm_slide_workspace_size(A, N)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=B.device)
    a = A.c()
    _lib.call("spmm_slide", C.byref(a), _ptr(B), B.stride(0), _ptr(out), out.stride(0), N, _ptr(workspace),
              0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream))
    return out


# ------------------------------------------------------------------ TVW
def spmm_build_tvw(dense: torch.Tensor, tile_rows: int, tile_ptr: torch.Tensor, cols: torch.Tensor,
                   Kp: Optional[int] = None, stream=None) -> TVW:
    _check_dev(dense, tile_ptr, cols)
    M, K = dense.shape
    n_tiles = (M + tile_rows - 1) // tile_rows
    if Kp is None:
        kt = int((tile_ptr[1:] - tile_ptr[:-1]).max().item()) if n_tiles else 0
        Kp = max(128, -(-kt // 128) * 128)
    vals = torch.empty((M, Kp // 2), dtype=dense.dtype, device=dense.device)
    meta = torch.empty((M, Kp // 8), dtype=torch.uint8, device=dense.device)
    _lib.call("spmm_build_tvw", _ptr(dense), M, K, dense.stride(0), _code(dense.dtype), tile_rows, _ptr(tile_ptr),
              _ptr(cols), n_tiles, Kp, _ptr(vals), _ptr(meta), _stream(stream))
    return TVW(M, K, tile_rows, dense.dtype, n_tiles, Kp, tile_ptr, cols, vals, meta)



def spmm_prune_tvw(dense: torch.Tensor, tile_rows: int, tile_ptr: torch.Tensor, cols: torch.Tensor,
                   Kp: Optional[int] = None, stream=None) -> TVW:
    """Magnitude-prune a dense matrix into TVW (kept columns given; 2:4 by magnitude inside)."""
    _check_dev(dense, tile_ptr, cols)
    M, K = dense.shape
    n_tiles = (M + tile_rows - 1) // tile_rows
    if Kp is None:
        kt = int((tile_ptr[1:] - tile_ptr[:-1]).max().item()) if n_tiles else 0
        Kp = max(128, -(-kt // 128) * 128)
    vals = torch.empty((M, Kp // 2), dtype=dense.dtype, device=dense.device)
    meta = torch.empty((M, Kp // 8), dtype=torch.uint8, device=dense.device)
    _lib.call("spmm_prune_tvw", _ptr(dense), M, K, dense.stride(0), _code(dense.dtype), tile_rows, _ptr(tile_ptr),
              _ptr(cols), n_tiles, Kp, _ptr(vals), _ptr(meta), _stream(stream))
    return TVW(M, K, tile_rows, dense.dtype, n_tiles, Kp, tile_ptr, cols, vals, meta)


def spmm_tvw(A: TVW, B: torch.Tensor, C_: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    _check_dev(B, C_)
    N = B.shape[1]
    out = _out(C_, A.M, N, torch.float32, B.device)
    a = A.c()
    _lib.call("spmm_tvw", C.byref(a), _ptr(B), B.stride(0), _ptr(out), out.stride(0), N, _stream(stream))
    return out


# ------------------------------------------------------------------ WCSR
def spmm_build_wcsr_workspace_size(A: CSR, h: int) -> int:
    n = C.c_size_t(0)
    a = A.c()
    _lib.call("spmm_build_wcsr_workspace_size", C.byref(a), h, C.byref(n))
    return n.value


def spmm_build_wcsr_count(A: CSR, h: int, S: int, workspace: torch.Tensor, stream=None):
    _check_dev(workspace)
    tw, tu = C.c_int64(0), C.c_int64(0)
    a = A.c()
    _lib.call("spmm_build_wcsr_count", C.byref(a), h, S, _ptr(workspace), workspace.numel(), C.byref(tw),
              C.byref(tu), _stream(stream))
    return tw.value, tu.value


def spmm_build_wcsr_fill(A: CSR, h: int, S: int, workspace: torch.Tensor, n_wcols: int, n_units: int,
                         stream=None) -> WCSR:
    dev = A.row_ptr.device
    nw = (A.M + h - 1) // h

    def i32(n):
        return torch.empty(n, dtype=torch.int32, device=dev)

    W = WCSR(A.M, A.K, A.nnz, h, S, A.dtype, nw, n_wcols, n_units, i32(nw + 1), i32(max(n_wcols, 1))[:n_wcols],
             i32(nw + 1), i32(nw + 1), i32(max(n_units, 1))[:n_units], i32(n_units + 1),
             torch.empty(max(A.nnz, 1), dtype=torch.uint8, device=dev)[:A.nnz], i32(max(A.nnz, 1))[:A.nnz],
             torch.empty(max(A.nnz, 1), dtype=A.dtype, device=dev)[:A.nnz])
    w = W.c()
    a = A.c()
    _lib.call("spmm_build_wcsr_fill", C.byref(a), h, S, _ptr(workspace), workspace.numel(), C.byref(w),
              _stream(stream))
    return W


def build_wcsr(A: CSR, h: int = 16, S: int = 32, stream=None) -> WCSR:
    ws = torch.empty(max(1, spmm_build_wcsr_workspace_size(A, h)), dtype=torch.uint8, device=A.row_ptr.device)
    tw, tu = spmm_build_wcsr_count(A, h, S, ws, stream)
    return spmm_build_wcsr_fill(A, h, S, ws, tw, tu, stream)


def spmm_wcsr_workspace_size(A: WCSR, N: int) -> int:
    n = C.c_size_t(0)
    a = A.c()
    _lib.call("spmm_wcsr_workspace_size", C.byref(a), N, C.byref(n))
    return n.value


def spmm_wcsr(A: WCSR, B: torch.Tensor, C_: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """C = A B for a row-window operand (tensor-core window products).  The
    workspace (kept on A when not given) needs no clearing between calls."""
    _check_dev(B, C_, workspace)
    N = B.shape[1]
    out = _out(C_, A.M, N, torch.float32, B.device)
    if workspace is None:
        need = spmm_wcsr_workspace_size(A, N)
        if A.workspace is None or A.workspace.numel() < need:
            A.workspace = torch.zeros(max(need, 1), dtype=torch.uint8, device=B.device)
        workspace = A.workspace
    a = A.c()
    _lib.call("spmm_wcsr", C.byref(a), _ptr(B), B.stride(0), _ptr(out), out.stride(0), N, _ptr(workspace),
              workspace.numel(), _stream(stream))
    return out
