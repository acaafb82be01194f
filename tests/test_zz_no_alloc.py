"""spmm_24_noalloc: the 2:4 entry point for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (a plugin that is handed only its input and
output buffers, a service that reserves all device memory up front, a latency-
critical path that cannot absorb cudaMalloc's synchronisation).  For them the
library keeps the int8 widening scratch in a fixed 32 MiB device array.  These
tests call the entry point through the C ABI and compare it with spmm_24, the
entry point that takes a caller-provided workspace, on two calls in a row, and
with the CPU oracle (bit-exact for int8, within tolerance for bf16, whose calls
need no scratch).  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests.gpu_util import assert_close, dev, dev_half, need_gpu

pytestmark = pytest.mark.gpu


def _call_noalloc(F, B, C, N):
    import torch
    from sparse_dense_matrix_spmm_gb300 import _lib
    a = F.c()
    return _lib.load().spmm_24_noalloc(ctypes.byref(a), ctypes.c_void_p(B.data_ptr()), B.stride(0),
                                       ctypes.c_void_p(C.data_ptr()), C.stride(0), N,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("M,K,N", [(512, 2048, 384), (200, 1024, 136)])
def test_noalloc_matches_spmm_24_on_two_calls(M, K, N):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.mask24_problem(M, K, N, seed=M + K)
    F = spmm.spmm_compress_24(dev(p["A"]))
    B1 = dev(p["B"])
    B2 = torch.flip(B1, dims=[0]).contiguous()          # a second, different right-hand side
    for B in (B1, B2):
        ref = spmm.spmm_24(F, B)                         # caller-provided workspace
        C = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
        assert _call_noalloc(F, B, C, N) == 0
        torch.cuda.synchronize()
        assert torch.equal(C, ref)                       # int8 results are exact: equality
    assert spmm.last_device_error() == 0


def test_noalloc_rejects_scratch_beyond_32_mib():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    from sparse_dense_matrix_spmm_gb300 import _lib
    M, K, N = 8192, 8192, 8                              # widened A alone is 64 MiB
    F = spmm.Mat24(M, K, torch.int8, torch.zeros((M, K // 2), dtype=torch.int8, device="cuda"),
                   torch.full((M, K // 8), 0x44, dtype=torch.uint8, device="cuda"))
    B = torch.zeros((K, N), dtype=torch.int8, device="cuda")
    C = torch.zeros((M, N), dtype=torch.int32, device="cuda")
    assert spmm.spmm_24_workspace_size(F, N) > 32 << 20
    assert _call_noalloc(F, B, C, N) == 5                # SPMM_ERR_WORKSPACE, nothing launched
    assert _lib.STATUS[5] == "SPMM_ERR_WORKSPACE"


def test_noalloc_ragged_n_after_a_larger_call_matches_oracle():
    """A ragged N (130: the widened B's padding columns live in the shared array)
    right after a larger call (N = 384) that left other data there: both results
    equal the oracle's int64 sums."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    M, K = 256, 1024
    for N, seed in ((384, 3), (130, 4)):
        p = gen.mask24_problem(M, K, N, seed=seed)
        F = spmm.spmm_compress_24(dev(p["A"]))
        C = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
        assert _call_noalloc(F, dev(p["B"]), C, N) == 0
        torch.cuda.synchronize()
        O = oracle.compress24(p["A"], "i8")
        assert np.array_equal(C.cpu().numpy().astype(np.int64), oracle.spmm24(O, p["B"]))
    assert spmm.last_device_error() == 0


def test_noalloc_bf16_needs_no_scratch():
    """bf16 operands go to the kernel as they are (no scratch pointer): the result
    equals spmm_24's and the oracle's within tolerance."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    M, K, N = 384, 1024, 200
    p = gen.mask24_float_problem(M, K, N, seed=12, dtype="bf16")
    F = spmm.spmm_compress_24(dev_half(p["A"], "bf16"))
    B = dev_half(p["B"], "bf16")
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    assert _call_noalloc(F, B, C, N) == 0
    torch.cuda.synchronize()
    assert torch.equal(C, spmm.spmm_24(F, B))
    O = oracle.compress24(p["A"], "bf16")
    assert_close(C.cpu().numpy(), oracle.spmm24(O, p["B"]), "noalloc bf16")
    assert spmm.last_device_error() == 0


def test_noalloc_with_prewidened_values():
    """With values widened beforehand the entry point needs scratch for B only, and
    its result equals the oracle's bit for bit."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    M, K, N = 256, 2048, 200
    p = gen.mask24_problem(M, K, N, seed=9)
    W = spmm.spmm_widen_24(spmm.spmm_compress_24(dev(p["A"])))
    C = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    assert _call_noalloc(W, dev(p["B"]), C, N) == 0
    torch.cuda.synchronize()
    O = oracle.compress24(p["A"], "i8")
    assert np.array_equal(C.cpu().numpy().astype(np.int64), oracle.spmm24(O, p["B"]))
    assert spmm.last_device_error() == 0
