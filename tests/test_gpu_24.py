"""2:4 on the GPU vs the CPU oracle: compression bit-exact, int8 SpMM exact,
fp16/bf16 SpMM within tolerance."""
import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests.gpu_util import assert_close, dev, dev_half, host_bits, need_gpu, padded_b

pytestmark = pytest.mark.gpu


def _compress(p, dtype):
    import sparse_dense_matrix_spmm_gb300 as spmm
    A = dev(p["A"]) if dtype == "i8" else dev_half(p["A"], dtype)
    F = spmm.spmm_compress_24(A)
    O = oracle.compress24(p["A"], dtype)
    assert np.array_equal(host_bits(F.vals), O["vals"])
    assert np.array_equal(F.meta.cpu().numpy(), O["meta"])
    return F, O


@pytest.mark.parametrize("M,K,N", [(256, 512, 256), (200, 1024, 300), (128, 128, 8), (384, 2048, 520)])
def test_24_int8_exact(M, K, N):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.mask24_problem(M, K, N, seed=M + K + N)
    F, O = _compress(p, "i8")
    C = spmm.spmm_24(F, dev(p["B"]))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    ref = oracle.spmm24(O, p["B"])
    assert np.array_equal(C.cpu().numpy().astype(np.int64), ref)


@pytest.mark.parametrize("M,K,N", [(384, 2048, 520), (200, 1024, 136)])
def test_24_int8_prewidened_values(M, K, N):
    """Values widened to fp16 once (spmm_widen_24) are the int8 values exactly, and
    spmm_24 with them (only B widened per call, a smaller workspace) equals the
    per-call path and the oracle bit for bit, on two different right-hand sides."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.mask24_problem(M, K, N, seed=M + 7)
    F, O = _compress(p, "i8")
    W = spmm.spmm_widen_24(F)
    torch.cuda.synchronize()
    assert torch.equal(W.vals16.float(), F.vals.float())
    assert spmm.spmm_24_workspace_size(W, N) < spmm.spmm_24_workspace_size(F, N)
    B1 = dev(p["B"])
    B2 = torch.flip(B1, dims=[1]).contiguous()
    for B, Bh in ((B1, p["B"]), (B2, np.ascontiguousarray(p["B"][:, ::-1]))):
        C = spmm.spmm_24(W, B)
        torch.cuda.synchronize()
        assert spmm.last_device_error() == 0
        assert torch.equal(C, spmm.spmm_24(F, B))
        assert np.array_equal(C.cpu().numpy().astype(np.int64), oracle.spmm24(O, Bh))


def _int8_b(B, ld):
    """int8 B on the device as a K x N view of rows ld bytes apart."""
    import torch
    K, N = B.shape
    full = torch.zeros((K, ld), dtype=torch.int8, device="cuda")
    full[:, :N] = dev(B)
    return full[:, :N]


@pytest.mark.parametrize("M,K,N", [(328, 1024, 200), (128, 512, 72), (256, 2048, 128)])
def test_24_int8_b_row_pitch(M, K, N):
    """int8 B with rows padded past N (pitch a multiple of 16 bytes) and with an odd
    pitch equals the oracle bit for bit: ragged N, a ragged last pair of row tiles,
    one row tile, with and without values widened beforehand."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.mask24_problem(M, K, N, seed=M + K + N + 1)
    F, O = _compress(p, "i8")
    W = spmm.spmm_widen_24(F)
    ref = oracle.spmm24(O, p["B"])
    ld16 = -(-N // 16) * 16 + 16          # rows on 16-byte boundaries, padded past N
    for B in (_int8_b(p["B"], ld16), _int8_b(p["B"], N + 1)):
        for A in (F, W):
            C = spmm.spmm_24(A, B)
            torch.cuda.synchronize()
            assert spmm.last_device_error() == 0
            assert np.array_equal(C.cpu().numpy().astype(np.int64), ref), (B.stride(0), A is W)


@pytest.mark.parametrize("M", [128, 256])  # one row tile, a pair of row tiles
def test_24_int8_extreme_values_stay_exact(M):
    """Every product 127*127 with equal signs: the kernel drains its fp32
    accumulator every 2048 dense K, so each chunk of 1024 products reaches the
    largest partial sum it can hold exactly (1024 * 16129 < 2^24), and any lost
    bit would show."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    K, N = 4096, 128
    A = np.zeros((M, K), np.int8)
    A[:, 0::4] = 127
    A[:, 3::4] = 127
    A[1::2, 0::4] = -127          # odd rows mix signs
    B = np.full((K, N), 127, np.int8)
    B[:, 1::2] = -127
    p = {"A": A, "B": B}
    F, O = _compress(p, "i8")
    C = spmm.spmm_24(F, dev(B))
    torch.cuda.synchronize()
    ref = oracle.spmm24(O, B)
    assert ref.max() == (K // 2) * 16129
    assert np.array_equal(C.cpu().numpy().astype(np.int64), ref)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,K,N", [(256, 512, 256), (136, 1024, 200)])
def test_24_float(dtype, M, K, N):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    rng = np.random.default_rng(M * K + N)
    mask = gen.mask24_problem(M, K, 1, seed=7)["A"] != 0
    Abits = gen.normal_bits(rng, (M, K), dtype)
    Abits[~mask] = 0
    Bbits = gen.normal_bits(rng, (K, N), dtype)
    F, O = _compress({"A": Abits}, dtype)
    C = spmm.spmm_24(F, padded_b(Bbits, dtype))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert_close(C.cpu().numpy(), oracle.spmm24(O, Bbits), f"2:4 {dtype}")


def test_24_compress_rejects_three_nonzeros():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    A = torch.zeros((16, 64), dtype=torch.int8, device="cuda")
    A[3, 8:11] = 1
    with pytest.raises(spmm.SpmmError) as e:
        spmm.spmm_compress_24(A)
    assert e.value.name == "SPMM_ERR_FORMAT"


def test_24_int8_full_size_sampled_rows():
    """A 8192 x 8192 int8 (2:4), B 8192 x 4096 int8: the oracle recomputes 96
    seeded rows and eight whole 128-row tiles (1024 rows) exactly, all 4096
    columns."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem("mask24_int8")
    F, O = _compress(p, "i8")
    C = spmm.spmm_24(F, dev(p["B"]))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    rows = np.sort(np.random.default_rng(21).choice(p["M"], size=96, replace=False))
    got = C[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.int64)
    ref = np.concatenate([oracle.spmm24(O, p["B"], rows=(int(r), int(r) + 1)) for r in rows])
    assert np.array_equal(got, ref)
    # eight whole 128-row tiles (1024 rows: the first, the last and six seeded ones)
    rng = np.random.default_rng(22)
    tiles = sorted(set([0, p["M"] // 128 - 1] + [int(t) for t in rng.choice(np.arange(1, p["M"] // 128 - 1), 6, replace=False)]))
    assert len(tiles) == 8
    for t in tiles:
        r0 = 128 * t
        assert np.array_equal(C[r0:r0 + 128].cpu().numpy().astype(np.int64), oracle.spmm24(O, p["B"], rows=(r0, r0 + 128)))


def test_24_f16_full_size_sampled_rows():
    """A 8192 x 8192 fp16 2:4 (N(0,1) values), B 8192 x 4096 fp16, C fp32: eight
    128-row tiles (1024 rows: the first, the last and six seeded ones) against
    the oracle."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem("mask24_f16")
    F, O = _compress(p, "f16")
    C = spmm.spmm_24(F, dev_half(p["B"], "f16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    rng = np.random.default_rng(61)
    tiles = sorted(set([0, p["M"] // 128 - 1] + [int(t) for t in rng.choice(np.arange(1, p["M"] // 128 - 1), 6, replace=False)]))
    assert len(tiles) == 8
    for r0 in [128 * t for t in tiles]:
        assert_close(C[r0:r0 + 128].cpu().numpy(), oracle.spmm24(O, p["B"], rows=(r0, r0 + 128)), f"2:4 f16 rows {r0}..")


@pytest.mark.parametrize("dtype", ["i8", "f16", "bf16"])
@pytest.mark.parametrize("M,K", [(64, 256), (37, 1024)])
def test_24_prune_bit_exact_and_spmm(dtype, M, K):
    """Magnitude pruning on the GPU equals the oracle's bit for bit (ties, signed
    zeros, int8 -128, NaN and infinities included), and the pruned operand
    multiplies like any 2:4 operand (rows without NaN or infinities compared)."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    rng = np.random.default_rng(M + K)
    if dtype == "i8":
        A = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
        small = rng.random((M, K)) < 0.3                            # many equal magnitudes
        A[small] = rng.integers(-2, 3, size=int(small.sum())).astype(np.int8)
        A[0, :4] = [-128, 127, -128, 5]
    else:
        A = gen.normal_bits(rng, (M, K), dtype)
        A[rng.random((M, K)) < 0.15] = 0
        A[rng.random((M, K)) < 0.05] = 0x8000                       # -0.0
        one, nan, inf = (0x3C00, 0x7E00, 0x7C00) if dtype == "f16" else (0x3F80, 0x7FC0, 0x7F80)
        A[0, :8] = [nan, inf, one, one, one | 0x8000, one, one, 0]  # NaN above inf; equal magnitudes
    Ad = dev(A) if dtype == "i8" else dev_half(A, dtype)
    F = spmm.spmm_prune_24(Ad)
    O = oracle.prune24(A, dtype)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(F.vals), O["vals"])
    assert np.array_equal(F.meta.cpu().numpy(), O["meta"])
    if dtype == "i8":
        B = rng.integers(-127, 128, size=(K, 96)).astype(np.int8)
        C = spmm.spmm_24(F, dev(B))
        torch.cuda.synchronize()
        assert np.array_equal(C.cpu().numpy(), oracle.spmm24(O, B))
    else:
        B = gen.normal_bits(rng, (K, 96), dtype)
        C = spmm.spmm_24(F, padded_b(B, dtype))
        torch.cuda.synchronize()
        assert_close(C[1:].cpu().numpy(), oracle.spmm24(O, B, rows=(1, M)), f"pruned 2:4 {dtype}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N", [384, 380])
def test_24_float_192_column_tiles(dtype, N):
    """M = 128 x (SM count) and N of three 128-column tiles: two waves of
    192-column tiles beat three of 128-column ones, so the kernel runs its
    192-column configuration (3-D B boxes at N = 384, per-chunk 2-D boxes and a
    ragged last chunk at N = 380).  Three 128-row tiles are checked."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, K = 128 * sms, 256
    rng = np.random.default_rng(N + len(dtype))
    mask = gen.mask24_problem(M, K, 1, seed=3)["A"] != 0
    Abits = gen.normal_bits(rng, (M, K), dtype)
    Abits[~mask] = 0
    Bbits = gen.normal_bits(rng, (K, N), dtype)
    F, O = _compress({"A": Abits}, dtype)
    C = spmm.spmm_24(F, padded_b(Bbits, dtype))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    for r0 in (0, 128 * (sms // 2), M - 128):
        assert_close(C[r0:r0 + 128].cpu().numpy(), oracle.spmm24(O, Bbits, rows=(r0, r0 + 128)), f"2:4 {dtype} wide {r0}")
