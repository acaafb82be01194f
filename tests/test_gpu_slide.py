"""(2n-2):2n through overlapping 2:4 windows on the GPU vs the CPU oracle: the
lifted operand bit-exact, int8 SpMM exact, fp16/bf16 SpMM within tolerance."""
import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests.gpu_util import assert_close, dev, dev_half, host_bits, need_gpu, padded_b

pytestmark = pytest.mark.gpu


def _on_dev(A, dtype):
    return dev(A) if dtype == "i8" else dev_half(A, dtype)


def _build(A, n, dtype):
    import sparse_dense_matrix_spmm_gb300 as spmm
    F = spmm.spmm_build_slide(_on_dev(A, dtype), n)
    O = oracle.slide_build(A, n, dtype)
    assert np.array_equal(host_bits(F.vals), O["vals"])
    assert np.array_equal(F.meta.cpu().numpy(), O["meta"])
    return F, O


@pytest.mark.parametrize("dtype", ["i8", "f16", "bf16"])
@pytest.mark.parametrize("n", [2, 3, 4, 5, 8])
def test_slide_build_bit_exact(dtype, n):
    """Random masks with 0 .. 2n-2 nonzeros per group (plus -0.0, NaN and infinities
    for 16-bit types): the GPU decomposition equals the oracle's bit for bit."""
    need_gpu()
    rng = np.random.default_rng(100 * n + len(dtype))
    M, K = 37, 4 * n * 24
    G = K // (2 * n)
    keep = np.zeros((M, G, 2 * n), bool)
    for i in range(M):
        for g in range(G):
            k = rng.integers(0, 2 * n - 1)
            keep[i, g, rng.choice(2 * n, size=k, replace=False)] = True
    keep = keep.reshape(M, K)
    if dtype == "i8":
        A = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
        A[A == 0] = 1
    else:
        A = gen.normal_bits(rng, (M, K), dtype)
        A[A & 0x7FFF == 0] = 0x3C00 if dtype == "f16" else 0x3F80
        nan, inf = (0x7E00, 0x7C00) if dtype == "f16" else (0x7FC0, 0x7F80)
        A[0, :3] = [nan, inf, inf | 0x8000]
    A[~keep] = 0
    if dtype != "i8":
        A[(~keep) & (rng.random((M, K)) < 0.3)] = 0x8000          # -0.0 counts as zero
    _build(A, n, dtype)


@pytest.mark.parametrize("n", [4, 3])
@pytest.mark.parametrize("M,N", [(256, 256), (200, 200), (128, 8)])
def test_slide_int8_exact(n, M, N):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    K = 64 * n * 2
    p = gen.slide_problem(M, K, N, n, seed=M + N + n, dtype="i8")
    F, O = _build(p["A"], n, "i8")
    C = spmm.spmm_slide(F, dev(p["B"]))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    ref = oracle.slide_spmm(O, p["B"])
    assert np.array_equal(ref, p["A"].astype(np.int64) @ p["B"].astype(np.int64))
    assert np.array_equal(C.cpu().numpy().astype(np.int64), ref)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("n,M,K,N", [(4, 256, 1024, 256), (4, 136, 512, 200), (5, 128, 640, 128),
                                     (2, 128, 256, 192), (8, 128, 1024, 64)])
def test_slide_float(dtype, n, M, K, N):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.slide_problem(M, K, N, n, seed=M * K + N + n, dtype=dtype)
    F, O = _build(p["A"], n, dtype)
    C = spmm.spmm_slide(F, padded_b(p["B"], dtype))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert_close(C.cpu().numpy(), oracle.slide_spmm(O, p["B"]), f"slide n={n} {dtype}")


def test_slide_build_rejects_too_many_nonzeros_and_bad_shapes():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    A = torch.zeros((16, 64), dtype=torch.int8, device="cuda")
    A[5, 8:15] = 1                                             # 7 nonzeros in a 6:8 group
    with pytest.raises(spmm.SpmmError) as e:
        spmm.spmm_build_slide(A, 4)
    assert e.value.name == "SPMM_ERR_FORMAT"
    F = spmm.spmm_build_slide(torch.zeros((16, 64), dtype=torch.float16, device="cuda"), 4)
    with pytest.raises(spmm.SpmmError) as e:                   # K = 64 is not a multiple of 64 n
        spmm.spmm_slide(F, torch.zeros((64, 8), dtype=torch.float16, device="cuda"))
    assert e.value.name == "SPMM_ERR_SHAPE"


def test_slide_f16_full_size_sampled_tiles():
    """6:8 A 18944 x 3584 fp16, B 3584 x 8192 fp16 (the benchmarked launch): the
    lifted operand bit-exact in full, and three seeded 128-row tiles of C (one of
    them the last) against the oracle."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem("slide68_f16")
    F, O = _build(p["A"], p["n"], "f16")
    C = spmm.spmm_slide(F, dev_half(p["B"], "f16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    rng = np.random.default_rng(71)
    M = p["M"]
    for r0 in sorted(set([int(t) * 128 for t in rng.choice(M // 128 - 1, 2, replace=False)] + [M - 128])):
        assert_close(C[r0:r0 + 128].cpu().numpy(), oracle.slide_spmm(O, p["B"], rows=(r0, r0 + 128)),
                     f"6:8 f16 rows {r0}..")


def test_slide_degenerate_inputs():
    """An all-zero operand (every window padded with (0, 1) and +0) multiplies to
    zeros; empty M or N returns without work."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    A = np.zeros((64, 512), np.int8)
    F, O = _build(A, 4, "i8")
    assert np.all(O["meta"] == 0x44) and not O["vals"].any()
    B = np.ones((512, 40), np.int8)
    C = spmm.spmm_slide(F, dev(B))
    torch.cuda.synchronize()
    assert not C.cpu().numpy().any()
    assert spmm.spmm_slide(F, torch.zeros((512, 0), dtype=torch.int8, device="cuda")).shape == (64, 0)
    E = spmm.spmm_build_slide(torch.zeros((0, 512), dtype=torch.float16, device="cuda"), 4)
    assert spmm.spmm_slide(E, torch.zeros((512, 16), dtype=torch.float16, device="cuda")).shape == (0, 16)
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0


@pytest.mark.parametrize("dtype,N", [("f16", 384), ("bf16", 380)])
def test_slide_many_row_tiles(dtype, N):
    """The lifted product at M = 128 x SM count (two 128-row tiles per CTA, many
    waves of output tiles) with three 128-column tiles of N: 4-D plane boxes at
    N = 384, per-chunk 3-D boxes at N = 380.  Three 128-row tiles are checked
    (the first, one in the middle, the last)."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, K = 128 * sms, 512
    p = gen.slide_problem(M, K, N, 4, seed=N, dtype=dtype)
    F = spmm.spmm_build_slide(_on_dev(p["A"], dtype), 4)
    O = oracle.slide_build(p["A"], 4, dtype)
    C = spmm.spmm_slide(F, padded_b(p["B"], dtype))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    for r0 in (0, 128 * (sms // 2), M - 128):
        assert_close(C[r0:r0 + 128].cpu().numpy(), oracle.slide_spmm(O, p["B"], rows=(r0, r0 + 128)),
                     f"slide {dtype} wide {r0}")
