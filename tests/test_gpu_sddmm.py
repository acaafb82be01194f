"""SDDMM on the GPU vs the CPU oracle: out[e] = A[i] . Bt[j] at every stored
(i, j) of a CSR pattern, within tolerance."""
import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests.gpu_util import assert_close, dev, dev_half, need_gpu

pytestmark = pytest.mark.gpu


def _csr(p, dtype):
    import torch
    import sparse_dense_matrix_spmm_gb300 as spmm
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
