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


def test_wcsr_full_size_every_row():
    """A 65536 x 65536 with log-normal rows (mean 16, sigma 1.5, clipped to 4096),
    B 65536 x 128: builder bit-exact in full, and every one of the 65536 x 128
    outputs of the SpMM (all work units, split windows and the longest row
    included) within tolerance of the oracle; a second call is bitwise equal."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem("wcsr_lognormal")
    W, O = _build(p, 16, 32)
    B = dev_half(p["B"], "f16")
    C = spmm.spmm_wcsr(W, B)
    C2 = spmm.spmm_wcsr(W, B)
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert torch.equal(C, C2)
    assert int(np.max(np.diff(O["unit_ptr"]))) > 1          # the workload has split windows
    assert_close(C.cpu().numpy(), oracle.wcsr_spmm(O, p["B"]), "wcsr full size")


def test_wcsr_workspace_needs_no_clearing():
    """The workspace's counters carry a per-call tag: a workspace full of arbitrary
    bytes (as a call that stopped early could leave it) gives the same, correct
    result, twice in a row."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.csr_lognormal_problem(400, 4000, 136, seed=17, mean=12.0, sigma=2.0, clip=2048)
    W, O = _build(p, 16, 1)                                  # S = 1: most windows split
    B = padded_b(p["B"], "f16")
    need = spmm.spmm_wcsr_workspace_size(W, 136)
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    ws = torch.randint(0, 256, (need,), generator=g, dtype=torch.uint8, device="cuda")
    C1 = spmm.spmm_wcsr(W, B, workspace=ws)
    ws[:4096] = torch.randint(0, 256, (4096,), generator=g, dtype=torch.uint8, device="cuda")
    C2 = spmm.spmm_wcsr(W, B, workspace=ws)
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert torch.equal(C1, C2)
    assert_close(C1.cpu().numpy(), oracle.wcsr_spmm(O, p["B"]), "wcsr arbitrary workspace")


@pytest.mark.parametrize("h", [8, 40, 64])
def test_wcsr_window_heights(h):
    """Window heights that are not a multiple of 16 (the MMA's N is h rounded up to
    16) and the largest supported one, with ragged N and split windows."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.csr_lognormal_problem(333, 6000, 72, seed=h, mean=10.0, sigma=1.8, clip=3000)
    W, O = _build(p, h, 2)
    C = spmm.spmm_wcsr(W, padded_b(p["B"], "f16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert_close(C.cpu().numpy(), oracle.wcsr_spmm(O, p["B"]), f"wcsr h={h}")


def test_wcsr_bf16():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.csr_lognormal_problem(520, 9000, 128, seed=9, mean=14.0, sigma=1.5, clip=4000, dtype="bf16")
    W, O = _build(p, 16, 4)
    C = spmm.spmm_wcsr(W, padded_b(p["B"], "bf16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert_close(C.cpu().numpy(), oracle.wcsr_spmm(O, p["B"]), "wcsr bf16")


# ---------------------------------------------------------------- tensor-core window products
# Operands whose windows reuse columns (at least 4 nonzeros per distinct window
# column) and whose work units carry at least 384 nonzeros on average run their
# window products on the tensor core.

def _tensor_core_path(W):
    return W.nnz >= 4 * W.n_wcols and W.nnz >= 384 * W.n_units

@pytest.mark.parametrize("M,K,N,h,S,pool,per_row", [
    (512, 4000, 128, 16, 32, 64, 32),      # whole windows, one slab
    (333, 5000, 72, 16, 2, 64, 56),        # ragged last window, ragged N, S = 2: every window split in two
    (500, 9000, 200, 32, 4, 96, 32),       # taller windows, two slabs (128 + 72 columns), splits
    (260, 3000, 136, 8, 4, 64, 56),        # h = 8 (MMA N rounded up to 16)
    (384, 6000, 200, 16, 4, 96, 56),       # 16-row windows (streaming kernel) over two slabs, every window split
    (200, 2500, 64, 48, 32, 200, 20),      # h = 48: several chunks of W tiles per unit
    (320, 4000, 128, 64, 4, 128, 40),      # h = 64, the largest window (MMA N = 64), split windows
])
def test_wcsr_tensor_core_parity(M, K, N, h, S, pool, per_row):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.csr_window_clustered_problem(M, K, N, seed=M + h, h=h, pool=pool, per_row=per_row)
    W, O = _build(p, h, S)
    assert _tensor_core_path(W)
    B = padded_b(p["B"], "f16")
    C1 = spmm.spmm_wcsr(W, B)
    C2 = spmm.spmm_wcsr(W, B)
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert torch.equal(C1, C2)
    assert_close(C1.cpu().numpy(), oracle.wcsr_spmm(O, p["B"]), "wcsr tensor core")


def test_wcsr_tensor_core_bf16_and_arbitrary_workspace():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.csr_window_clustered_problem(640, 7000, 128, seed=3, h=16, pool=64, per_row=56, dtype="bf16")
    W, O = _build(p, 16, 2)
    assert _tensor_core_path(W)
    need = spmm.spmm_wcsr_workspace_size(W, 128)
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    ws = torch.randint(0, 256, (need,), generator=g, dtype=torch.uint8, device="cuda")
    C = spmm.spmm_wcsr(W, padded_b(p["B"], "bf16"), workspace=ws)
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert_close(C.cpu().numpy(), oracle.wcsr_spmm(O, p["B"]), "wcsr tensor core bf16")


def test_wcsr_tensor_core_bad_slot_is_skipped_and_reported():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.csr_window_clustered_problem(256, 3000, 128, seed=5, h=16, pool=64, per_row=32)
    W, O = _build(p, 16, 32)
    assert _tensor_core_path(W)
    spmm.last_device_error()
    W.slot[0] = 1 << 30                    # first entry of window 0 points past its column list
    C = spmm.spmm_wcsr(W, padded_b(p["B"], "f16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() & 2
    got = C.cpu().numpy()
    assert np.isfinite(got).all()
    assert_close(got[16:], oracle.wcsr_spmm(O, p["B"])[16:], "wcsr tensor core other windows")


def test_wcsr_clustered_full_size_every_row():
    """The clustered workload at its benchmarked size (65536 x 65536, 16-row windows
    whose rows take 64 of 128 shared columns, B 65536 x 128): every output within
    tolerance, bitwise equal across two calls."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem("wcsr_clustered")
    W, O = _build(p, 16, 32)
    assert _tensor_core_path(W)
    B = dev_half(p["B"], "f16")
    C = spmm.spmm_wcsr(W, B)
    C2 = spmm.spmm_wcsr(W, B)
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert torch.equal(C, C2)
    assert_close(C.cpu().numpy(), oracle.wcsr_spmm(O, p["B"]), "wcsr clustered full size")
