"""SDDMM on the GPU vs the CPU oracle: out[e] = A[i] . Bt[j] at every stored
(i, j) of a CSR pattern, within tolerance for fp16/bf16 and bit-exact (int32
against the oracle's int64) for int8."""
import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests.gpu_util import assert_close, dev, dev_half, need_gpu

pytestmark = pytest.mark.gpu


def _csr(p, dtype):
    import torch
    import sparse_dense_matrix_spmm_gb300 as spmm
    if dtype == "i8":  # the pattern of an int8 SDDMM (values unused)
        return spmm.CSR(p["M"], p["K"], int(p["row_ptr"][-1]), torch.int8, dev(p["row_ptr"].astype(np.int32)),
                        dev(p["col"].astype(np.int32)), torch.zeros(max(1, int(p["row_ptr"][-1])), dtype=torch.int8,
                                                                    device="cuda"))
    dt = torch.bfloat16 if dtype == "bf16" else torch.float16
    return spmm.CSR(p["M"], p["K"], int(p["row_ptr"][-1]), dt, dev(p["row_ptr"].astype(np.int32)),
                    dev(p["col"].astype(np.int32)), dev_half(p["val"], dtype))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("K", [8, 64, 128, 136, 256, 520])
def test_sddmm_matches_oracle(dtype, K):
    """Lane groups of 8, 16 and 32, a ragged last K step (136, 520), and log-normal
    rows of 1 to 200 entries (the long ones span several warp slices)."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.csr_lognormal_problem(300, 200, 1, seed=K, mean=10.0, sigma=1.5, clip=200, dtype=dtype)
    rng = np.random.default_rng(K)
    A = gen.normal_bits(rng, (300, K), dtype)
    Bt = gen.normal_bits(rng, (200, K), dtype)
    out = spmm.spmm_sddmm(_csr(p, dtype), dev_half(A, dtype), dev_half(Bt, dtype))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert_close(out.cpu().numpy(), oracle.sddmm(p["row_ptr"], p["col"], A, Bt, dtype), f"sddmm {dtype} K={K}")


def test_sddmm_one_long_row_and_padded_pitches():
    """A single row holding every column (3000 entries over many warp slices) next to
    empty rows; A and Bt with row pitches larger than K."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    M, N, K = 40, 3000, 64
    rp = np.zeros(M + 1, np.int64)
    rp[18:] = N                                                  # row 17 holds all N columns
    p = {"M": M, "K": N, "row_ptr": rp, "col": np.arange(N), "val": np.ones(N, np.uint16) * 0x3C00}
    rng = np.random.default_rng(5)
    A = gen.normal_bits(rng, (M, K), "f16")
    Bt = gen.normal_bits(rng, (N, K), "f16")
    Ap = torch.zeros((M, K + 24), dtype=torch.float16, device="cuda")
    Ap[:, :K] = dev_half(A, "f16")
    Bp = torch.zeros((N, K + 8), dtype=torch.float16, device="cuda")
    Bp[:, :K] = dev_half(Bt, "f16")
    out = spmm.spmm_sddmm(_csr(p, "f16"), Ap[:, :K], Bp[:, :K])
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert_close(out.cpu().numpy(), oracle.sddmm(rp, p["col"], A, Bt, "f16"), "sddmm long row")


def test_sddmm_full_size():
    """The benchmarked launch: the 65536^2 log-normal pattern (about 1.05 M entries),
    A and Bt 65536 x 128 fp16; every output against the oracle."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem("sddmm_lognormal")
    out = spmm.spmm_sddmm(_csr(p, "f16"), dev_half(p["A"], "f16"), dev_half(p["Bt"], "f16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert_close(out.cpu().numpy(), oracle.sddmm(p["row_ptr"], p["col"], p["A"], p["Bt"], "f16"), "sddmm full size")


# ---------------------------------------------------------------- int8 (quantized) SDDMM
def _i8(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.mark.parametrize("K", [16, 128, 256, 272, 512, 528])
def test_sddmm_i8_exact(K):
    """Lane groups of 8, 16 and 32 (16 int8 per 16-byte load), ragged last K steps
    (272, 528), full-range operands and log-normal rows: every int32 output equals
    the oracle's int64 sum."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.csr_lognormal_problem(300, 200, 1, seed=K + 1, mean=10.0, sigma=1.5, clip=200, dtype="f16")
    rng = np.random.default_rng(K)
    A = rng.integers(-128, 128, size=(300, K), dtype=np.int8)
    Bt = rng.integers(-128, 128, size=(200, K), dtype=np.int8)
    out = spmm.spmm_sddmm(_csr(p, "i8"), _i8(A), _i8(Bt))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0 and out.dtype == torch.int32
    assert np.array_equal(out.cpu().numpy().astype(np.int64), oracle.sddmm_i64(p["row_ptr"], p["col"], A, Bt))


@pytest.mark.parametrize("a,b", [(-128, -128), (-128, 127)])
def test_sddmm_i8_largest_depth_extremes(a, b):
    """The largest accepted depth K = 131056 with constant extreme operands: every
    sum is K * a * b (2 147 221 504 for -128 * -128, just below 2^31), exact in
    int32; one more 16-element step is refused."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    K = 131056
    rp = np.array([0, 2, 2, 5, 6], np.int64)
    p = {"M": 4, "K": 7, "row_ptr": rp, "col": np.array([0, 6, 1, 3, 5, 2])}
    A = np.full((4, K), a, np.int8)
    Bt = np.full((7, K), b, np.int8)
    out = spmm.spmm_sddmm(_csr(p, "i8"), _i8(A), _i8(Bt))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert out.cpu().numpy().astype(np.int64).tolist() == [K * a * b] * 6
    assert oracle.sddmm_i64(rp, p["col"], A, Bt).tolist() == [K * a * b] * 6
    with pytest.raises(spmm.SpmmError):
        spmm.spmm_sddmm(_csr(p, "i8"), _i8(np.zeros((4, K + 16), np.int8)), _i8(np.zeros((7, K + 16), np.int8)))


def test_sddmm_i8_shape_rules():
    """int8 needs K and both pitches in multiples of 16 (one 16-byte load covers 16
    elements): K = 8 and a pitch of 40 are refused."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    rp = np.array([0, 1, 2], np.int64)
    p = {"M": 2, "K": 2, "row_ptr": rp, "col": np.array([1, 0]), "val": np.zeros(2, np.uint16)}
    with pytest.raises(spmm.SpmmError):
        spmm.spmm_sddmm(_csr(p, "i8"), _i8(np.ones((2, 8), np.int8)), _i8(np.ones((2, 8), np.int8)))
    Ap = torch.zeros((2, 40), dtype=torch.int8, device="cuda")
    with pytest.raises(spmm.SpmmError):  # pitch 40: not a multiple of 16
        spmm.spmm_sddmm(_csr(p, "i8"), Ap[:, :32], _i8(np.ones((2, 32), np.int8)))
    Ap = torch.ones((2, 48), dtype=torch.int8, device="cuda")
    out = spmm.spmm_sddmm(_csr(p, "i8"), Ap[:, :32], _i8(np.full((2, 32), 2, np.int8)))
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [64, 64]


def test_sddmm_i8_full_size():
    """The benchmarked launch: the 65536^2 log-normal pattern (about 1.05 M entries),
    A and Bt 65536 x 128 int8; every output bit-exact against the oracle."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem("sddmm_lognormal_i8")
    out = spmm.spmm_sddmm(_csr(p, "i8"), _i8(p["A"]), _i8(p["Bt"]))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert np.array_equal(out.cpu().numpy().astype(np.int64), oracle.sddmm_i64(p["row_ptr"], p["col"], p["A"], p["Bt"]))
