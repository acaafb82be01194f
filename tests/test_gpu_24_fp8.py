"""fp8 (E4M3 / E5M2) 2:4 on the GPU vs the CPU oracle: compression and magnitude
pruning bit-exact, the SpMM (kind::f8f6f4 sparse tensor-core MMAs, fp32
accumulation) within |err| <= 1e-2 + 1e-2 |ref| of the oracle's fp64 sums."""
import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests.gpu_util import assert_close, dev_fp8, host_bits, need_gpu, padded_b8

pytestmark = pytest.mark.gpu


def _compress(A, dtype):
    import sparse_dense_matrix_spmm_gb300 as spmm
    F = spmm.spmm_compress_24(dev_fp8(A, dtype))
    O = oracle.compress24(A, dtype)
    assert np.array_equal(host_bits(F.vals), O["vals"])
    assert np.array_equal(F.meta.cpu().numpy(), O["meta"])
    return F, O


@pytest.mark.parametrize("dtype,M,K,N", [("e4m3", 256, 512, 256), ("e4m3", 200, 1024, 136), ("e4m3", 128, 256, 16),
                                         ("e4m3", 384, 2048, 520), ("e5m2", 264, 768, 200)])
def test_24_fp8_spmm(dtype, M, K, N):
    """Whole and ragged row tiles (M = 200, 264), ragged column tiles (N = 136, 200,
    520 with the row pitch padded to 16 bytes), one K step (K = 256), several."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.mask24_float_problem(M, K, N, seed=M + K + N, dtype=dtype)
    F, O = _compress(p["A"], dtype)
    C = spmm.spmm_24(F, padded_b8(p["B"], dtype))
    torch.cuda.synchronize()
    assert C.dtype == torch.float32 and tuple(C.shape) == (M, N)
    assert spmm.last_device_error() == 0
    assert_close(C.cpu().numpy(), oracle.spmm24(O, p["B"]), f"2:4 {dtype}")


def test_24_fp8_extreme_values():
    """Every product 448 * 448 (the largest E4M3 magnitude), signs mixed by row and
    column: sums of 2048 such products are exact in fp32, so the result must equal
    the oracle's exactly."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    M, K, N = 128, 4096, 128
    A = np.zeros((M, K), np.uint8)
    A[:, 1::4] = 0x7E
    A[:, 2::4] = 0x7E
    A[1::2, 1::4] = 0xFE          # odd rows: -448 in one of the pair
    B = np.full((K, N), 0x7E, np.uint8)
    B[:, 1::2] = 0xFE
    F, O = _compress(A, "e4m3")
    C = spmm.spmm_24(F, dev_fp8(B, "e4m3"))
    torch.cuda.synchronize()
    ref = oracle.spmm24(O, B)
    assert ref.max() == (K // 2) * 448.0 * 448.0
    assert np.array_equal(C.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("dtype", ["e4m3", "e5m2"])
def test_24_fp8_prune_bit_exact_and_spmm(dtype):
    """Magnitude pruning on the GPU equals the oracle's bit for bit (ties, -0, NaN
    and, for E5M2, infinities), and the pruned operand multiplies like any 2:4
    operand (rows free of NaN and infinities compared)."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    M, K = 96, 512
    rng = np.random.default_rng(5 + len(dtype))
    A = gen.normal_bits(rng, (M, K), dtype)
    A[rng.random((M, K)) < 0.15] = 0
    A[rng.random((M, K)) < 0.05] = 0x80                              # -0
    one = 0x38 if dtype == "e4m3" else 0x3C
    nan = 0x7F
    big = 0x7E if dtype == "e4m3" else 0x7C                          # 448 / +inf
    A[0, :8] = [nan, big, one, one, one | 0x80, one, one, 0]         # NaN above the rest; equal magnitudes
    F = spmm.spmm_prune_24(dev_fp8(A, dtype))
    O = oracle.prune24(A, dtype)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(F.vals), O["vals"])
    assert np.array_equal(F.meta.cpu().numpy(), O["meta"])
    B = gen.normal_bits(rng, (K, 96), dtype)
    C = spmm.spmm_24(F, padded_b8(B, dtype))
    torch.cuda.synchronize()
    assert_close(C[1:].cpu().numpy(), oracle.spmm24(O, B, rows=(1, M)), f"pruned 2:4 {dtype}")


def test_24_fp8_rejects_k_not_multiple_of_256():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    A = torch.zeros((128, 384), dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    F = spmm.spmm_compress_24(A)
    B = torch.zeros((384, 64), dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    with pytest.raises(spmm.SpmmError) as e:
        spmm.spmm_24(F, B)
    assert e.value.name == "SPMM_ERR_SHAPE"


def test_24_fp8_full_size_sampled_tiles():
    """The fp8 workload at its benchmarked size: A 8192 x 8192 E4M3 (2:4, N(0,1)
    values), B 8192 x 4096 E4M3, C fp32.  Eight seeded 128-row tiles (the last one
    among them: 1024 rows spread over the waves of persistent CTAs) against the
    oracle on 512 seeded columns."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem("mask24_e4m3")
    F, O = _compress(p["A"], "e4m3")
    C = spmm.spmm_24(F, dev_fp8(p["B"], "e4m3"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    rng = np.random.default_rng(71)
    tiles = sorted(set(int(t) for t in rng.choice(p["M"] // 128 - 1, 7, replace=False)) | {p["M"] // 128 - 1})
    cols = np.sort(rng.choice(p["N"], 512, replace=False))
    ct = torch.from_numpy(cols).cuda()
    for t in tiles:
        r0 = t * 128
        got = C[r0:r0 + 128][:, ct].cpu().numpy()
        assert_close(got, oracle.spmm24(O, p["B"], rows=(r0, r0 + 128), cols=cols), f"2:4 e4m3 rows {r0}..")
