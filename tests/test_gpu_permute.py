"""Permutation before BCSR on the GPU vs the CPU oracle: P A P^T and the row
gathers/scatters bit-exact, the permuted BCSR product within tolerance of the
plain product (and of the oracle's gather / BCSR / scatter)."""
import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests._helpers import bits_to_f64
from tests.gpu_util import assert_close, dev, dev_half, host_bits, need_gpu, padded_b

pytestmark = pytest.mark.gpu


def _pattern(A):
    nz = (A & 0x7FFF) != 0 if A.dtype == np.uint16 else A != 0
    rp = np.concatenate([[0], np.cumsum(nz.sum(axis=1))]).astype(np.int32)
    return rp, np.nonzero(nz)[1].astype(np.int32)


@pytest.mark.parametrize("dtype", ["i8", "f16"])
@pytest.mark.parametrize("n", [64, 77])
def test_permute_sym_bit_exact(dtype, n):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.banded_scrambled_problem(n, 3, 1, seed=n, dtype=dtype)
    perm = spmm.rcm_order(n, *_pattern(p["A"]))
    assert np.array_equal(perm.numpy(), oracle.rcm_dense(p["A"]))
    Ad = dev(p["A"]) if dtype == "i8" else dev_half(p["A"], dtype)
    out = spmm.spmm_permute_sym(Ad, perm.cuda())
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert np.array_equal(host_bits(out), oracle.permute_sym(p["A"], perm.numpy(), dtype))


@pytest.mark.parametrize("elem", [1, 2, 4])
@pytest.mark.parametrize("cols", [64, 37])
def test_permute_rows_gather_scatter(elem, cols):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    rng = np.random.default_rng(elem * cols)
    rows = 300
    dt = {1: np.int8, 2: np.int16, 4: np.int32}[elem]
    X = rng.integers(-100, 100, size=(rows, cols)).astype(dt)
    perm = rng.permutation(rows).astype(np.int32)
    Xd, pd = torch.from_numpy(X).cuda(), torch.from_numpy(perm).cuda()
    g = spmm.spmm_permute_rows(Xd, pd)
    s = spmm.spmm_permute_rows(Xd, pd, scatter=True)
    torch.cuda.synchronize()
    assert np.array_equal(g.cpu().numpy(), X[perm])
    ref = np.empty_like(X)
    ref[perm] = X
    assert np.array_equal(s.cpu().numpy(), ref)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("n,w,bh,N", [(512, 8, 16, 256), (512, 8, 64, 200), (384, 20, 32, 96)])
def test_bcsr_permuted_product(dtype, n, w, bh, N):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.banded_scrambled_problem(n, w, N, seed=n + w + N, dtype=dtype)
    perm = spmm.rcm_order(n, *_pattern(p["A"]))
    Ap_dev = spmm.spmm_permute_sym(dev_half(p["A"], dtype), perm.cuda())
    F = spmm.build_bcsr(Ap_dev, bh, bh)
    Ap = oracle.permute_sym(p["A"], perm.numpy(), dtype)
    O = oracle.bcsr_build(Ap, bh, bh, dtype)
    G = oracle.bcsr_build(p["A"], bh, bh, dtype)
    assert F.nnzb == O["nnzb"] < G["nnzb"]
    C = spmm.spmm_bcsr_permuted(F, perm.cuda(), padded_b(p["B"], dtype))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    got = C.cpu().numpy()
    assert_close(got, oracle.bcsr_spmm_permuted(O, perm.numpy(), p["B"]), f"permuted {dtype}")
    assert_close(got, bits_to_f64(p["A"], dtype) @ bits_to_f64(p["B"], dtype), f"permuted vs dense {dtype}")


def test_bcsr_permuted_full_size_sampled_rows():
    """Scrambled band 16384^2 (half-width 48), 64 x 64 blocks, B 16384 x 2048 fp16 (the
    benchmarked launch): RCM equals the oracle's, the block count falls from (nearly)
    all blocks to the band's, and 64 seeded rows of C equal the dense product rows."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem("bcsr_rcm")
    n = p["M"]
    perm = spmm.rcm_order(n, *_pattern(p["A"]))
    assert np.array_equal(perm.numpy(), oracle.rcm_dense(p["A"]))
    F = spmm.build_bcsr(spmm.spmm_permute_sym(dev_half(p["A"], "f16"), perm.cuda()), 64, 64)
    assert F.nnzb <= 5 * (n // 64)                        # bandwidth <= 2 w = 96: at most 5 blocks per block row
    C = spmm.spmm_bcsr_permuted(F, perm.cuda(), dev_half(p["B"], "f16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    rows = np.sort(np.random.default_rng(31).choice(n, size=64, replace=False))
    ref = bits_to_f64(p["A"][rows], "f16") @ bits_to_f64(p["B"], "f16")
    assert_close(C[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, "permuted full size")


@pytest.mark.parametrize("N", [130, 256])
def test_bcsr_permuted_fused_scatter_equals_two_pass(N):
    """64-row blocks with 16-byte aligned C rows take the epilogue scatter; an
    unaligned C pitch takes the gather / BCSR / scatter passes.  Both run the same
    products, so their results agree bit for bit (ragged N included)."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    n = 512
    p = gen.banded_scrambled_problem(n, 10, N, seed=N, dtype="f16")
    perm = spmm.rcm_order(n, *_pattern(p["A"]))
    F = spmm.build_bcsr(spmm.spmm_permute_sym(dev_half(p["A"], "f16"), perm.cuda()), 64, 64)
    B = padded_b(p["B"], "f16")
    pitch4 = -(-N // 4) * 4
    C1 = torch.full((n, pitch4), float("nan"), device="cuda")[:, :N]       # ldc % 4 == 0: fused
    C2 = torch.full((n, pitch4 + 1), float("nan"), device="cuda")[:, :N]   # ldc % 4 != 0: two passes
    spmm.spmm_bcsr_permuted(F, perm.cuda(), B, C1)
    spmm.spmm_bcsr_permuted(F, perm.cuda(), B, C2)
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    a, b = C1.cpu().numpy(), C2.cpu().numpy()
    assert not np.isnan(a).any() and np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert_close(a, bits_to_f64(p["A"], "f16") @ bits_to_f64(p["B"], "f16"), "fused scatter")


def test_permuted_degenerate_inputs():
    """An empty pattern: RCM visits every isolated node in index order, so perm is
    the reversed identity; the product (no blocks) is all zeros; N = 0 is a no-op."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    n = 128
    perm = spmm.rcm_order(n, np.zeros(n + 1, np.int32), np.zeros(0, np.int32))
    assert perm.tolist() == list(range(n - 1, -1, -1))
    assert np.array_equal(perm.numpy(), oracle.rcm(n, np.zeros(n + 1, np.int32), np.zeros(0, np.int32)))
    F = spmm.build_bcsr(torch.zeros((n, n), dtype=torch.float16, device="cuda"), 64, 64)
    assert F.nnzb == 0
    C = torch.full((n, 64), float("nan"), device="cuda")
    spmm.spmm_bcsr_permuted(F, perm.cuda(), torch.ones((n, 64), dtype=torch.float16, device="cuda"), C)
    torch.cuda.synchronize()
    assert not C.cpu().numpy().any()
    assert spmm.spmm_bcsr_permuted(F, perm.cuda(), torch.zeros((n, 0), dtype=torch.float16, device="cuda")).shape == (n, 0)
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
