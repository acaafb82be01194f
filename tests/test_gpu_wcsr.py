"""Row-window CSR on the GPU vs the CPU oracle: builder bit-exact, SpMM within
tolerance and run-to-run identical (split windows are summed in a fixed order)."""
import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests.gpu_util import assert_close, dev, dev_half, host_bits, need_gpu, padded_b

pytestmark = pytest.mark.gpu

ARRAYS = ("wcol_ptr", "wcols", "wnz_ptr", "unit_ptr", "unit_win", "unit_nz_ptr", "lrow", "slot")


def _csr(p):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    dt = torch.float16 if p["dtype"] == "f16" else torch.bfloat16
    return spmm.CSR(p["M"], p["K"], int(p["row_ptr"][-1]), dt, dev(p["row_ptr"]), dev(p["col"]),
                    dev_half(p["val"], p["dtype"]))


def _build(p, h, S):
    import sparse_dense_matrix_spmm_gb300 as spmm
    W = spmm.build_wcsr(_csr(p), h, S)
    O = oracle.wcsr_build(p["M"], p["K"], p["row_ptr"], p["col"], p["val"], p["dtype"], h=h, S=S)
    assert (W.n_wcols, W.n_units) == (O["n_wcols"], O["n_units"])
    for k in ARRAYS:
        assert np.array_equal(getattr(W, k).cpu().numpy(), O[k]), k
    assert np.array_equal(host_bits(W.val), O["val"])
    return W, O


@pytest.mark.parametrize("M,K,N,h,S,sigma", [
    (300, 2000, 128, 16, 32, 1.5),    # ragged last window
    (256, 5000, 136, 16, 1, 2.0),     # S = 1: most windows split; N past one 128-column slab
    (97, 700, 64, 1, 2, 1.5),         # one-row windows
    (512, 30000, 200, 32, 4, 2.0),    # taller windows, power-law rows
])
def test_wcsr_parity(M, K, N, h, S, sigma):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.csr_lognormal_problem(M, K, N, seed=M + K, mean=12.0, sigma=sigma, clip=min(K, 2048))
    W, O = _build(p, h, S)
    B = padded_b(p["B"], "f16")
    C1 = spmm.spmm_wcsr(W, B)
    C2 = spmm.spmm_wcsr(W, B)
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert torch.equal(C1, C2)          # fixed summation order, workspace counters reset
    assert_close(C1.cpu().numpy(), oracle.wcsr_spmm(O, p["B"]), "wcsr")


def test_wcsr_empty_rows_and_windows():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    M, K, N = 70, 50, 40
    rows = [[] for _ in range(M)]
    rows[3] = [1, 7, 9]
    rows[40] = [0, 49]
    rows[41] = [7]
    rp = np.zeros(M + 1, np.int64)
    np.cumsum([len(r) for r in rows], out=rp[1:])
    col = np.array([c for r in rows for c in r], np.int32)
    rng = np.random.default_rng(0)
    p = {"M": M, "K": K, "N": N, "dtype": "f16", "row_ptr": rp.astype(np.int32), "col": col,
         "val": gen.normal_bits(rng, (len(col),), "f16"), "B": gen.normal_bits(rng, (K, N), "f16")}
    W, O = _build(p, 16, 32)
    C = torch.full((M, N), 5.0, device="cuda")
    spmm.spmm_wcsr(W, padded_b(p["B"], "f16"), C)
    torch.cuda.synchronize()
    assert_close(C.cpu().numpy(), oracle.wcsr_spmm(O, p["B"]), "wcsr empty rows")


def test_wcsr_builder_rejects_unsorted_columns():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = {"M": 2, "K": 5, "dtype": "f16", "row_ptr": np.array([0, 2, 3], np.int32),
         "col": np.array([2, 1, 4], np.int32), "val": np.zeros(3, np.uint16)}
    with pytest.raises(spmm.SpmmError) as e:
        spmm.build_wcsr(_csr(p), 16, 32)
    assert e.value.name == "SPMM_ERR_FORMAT"


def test_wcsr_full_size_sampled_rows():
    """A 65536 x 65536 with log-normal rows (mean 16, sigma 1.5, clipped to 4096),
    B 65536 x 128: builder bit-exact in full, SpMM checked on 4 seeded windows
    of rows plus the longest row."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem("wcsr_lognormal")
    W, O = _build(p, 16, 32)
    C = spmm.spmm_wcsr(W, dev_half(p["B"], "f16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    longest = int(np.argmax(np.diff(p["row_ptr"])))
    rng = np.random.default_rng(31)
    starts = sorted(set([int(w) * 16 for w in rng.choice(p["M"] // 16, 4, replace=False)] + [longest // 16 * 16]))
    for r0 in starts:
        got = C[r0:r0 + 16].cpu().numpy()
        assert_close(got, oracle.wcsr_spmm(O, p["B"], rows=(r0, r0 + 16)), f"wcsr rows {r0}..")
