"""BCSR on the GPU vs the CPU oracle: builder bit-exact, SpMM within tolerance."""
import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests.gpu_util import assert_close, dev_half, host_bits, need_gpu, padded_b

pytestmark = pytest.mark.gpu


def _run(p, dtype="bf16"):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    A = dev_half(p["A"], dtype)
    B = padded_b(p["B"], dtype)
    F = spmm.build_bcsr(A, p["bh"], p["bw"])
    O = oracle.bcsr_build(p["A"], p["bh"], p["bw"], dtype)
    assert F.nnzb == O["nnzb"]
    assert np.array_equal(F.row_ptr.cpu().numpy(), O["row_ptr"])
    assert np.array_equal(F.col_idx.cpu().numpy(), O["col_idx"])
    assert np.array_equal(host_bits(F.vals).reshape(O["vals"].shape), O["vals"])
    C = spmm.spmm_bcsr(F, B)
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    return F, O, C


def test_bcsr_tiny_config():
    p = gen.config_problem("bcsr_tiny")
    F, O, C = _run(p)
    assert_close(C.cpu().numpy(), oracle.bcsr_spmm(O, p["B"]), "bcsr_tiny")


@pytest.mark.parametrize("M,K,N,bh,bw,frac,dtype", [
    (512, 384, 200, 64, 64, 0.3, "bf16"),     # several tiles, ragged N tail
    (256, 512, 129, 32, 32, 0.25, "f16"),     # fp16, N = one tile + 1
    (384, 256, 300, 128, 16, 0.5, "bf16"),    # tall blocks, narrow K
    (512, 256, 64, 256, 64, 0.5, "f16"),      # bh = 256 (two accumulators)
    (128, 1024, 1000, 16, 64, 0.05, "bf16"),  # very sparse: empty block rows
    # 64-row blocks run the 64-row x 192-token kernel:
    (512, 256, 640, 64, 32, 0.3, "f16"),      # bw = 32, whole 64-token chunks, 3.3 token tiles
    (256, 256, 300, 64, 16, 0.4, "bf16"),     # bw = 16, ragged chunk (per-chunk loads)
    (1024, 512, 512, 64, 64, 0.02, "bf16"),   # very sparse: empty block rows write zeros
])
def test_bcsr_shapes(M, K, N, bh, bw, frac, dtype):
    nb = (M // bh) * (K // bw)
    p = gen.bcsr_problem(M, K, N, bh, bw, max(1, int(nb * frac)), seed=M + K + N, dtype=dtype)
    F, O, C = _run(p, dtype)
    assert_close(C.cpu().numpy(), oracle.bcsr_spmm(O, p["B"]), f"bcsr {M}x{K}x{N} {bh}x{bw}")


def test_bcsr_empty_matrix_writes_zeros():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    A = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    B = torch.randn((128, 40), dtype=torch.float32, device="cuda").to(torch.bfloat16)
    F = spmm.build_bcsr(A, 16, 16)
    assert F.nnzb == 0
    C = torch.full((128, 40), 7.0, device="cuda")
    spmm.spmm_bcsr(F, B, C)
    assert not C.any().item()


def test_bcsr_ldc_and_ldb_padding():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.bcsr_problem(128, 128, 100, 16, 16, 20, seed=3)
    A = dev_half(p["A"], "bf16")
    Bpad = torch.zeros((128, 104), dtype=torch.bfloat16, device="cuda")
    Bpad[:, :100] = dev_half(p["B"], "bf16")
    F = spmm.build_bcsr(A, 16, 16)
    Cpad = torch.full((128, 130), -1.0, device="cuda")
    out = spmm.spmm_bcsr(F, Bpad[:, :100], Cpad[:, :100])
    torch.cuda.synchronize()
    O = oracle.bcsr_build(p["A"], 16, 16, "bf16")
    assert_close(out.cpu().numpy(), oracle.bcsr_spmm(O, p["B"]), "padded")
    assert (Cpad[:, 100:] == -1.0).all().item()


def test_bcsr_llm_full_size_sampled_columns():
    """W 18944 x 3584 (64 x 64 blocks, 90% zero) times X 3584 x 65536: the oracle
    checks a seeded 512-column slice of the full result."""
    torch = need_gpu()
    p = gen.config_problem("bcsr_llm")
    F, O, C = _run(p)
    cols = np.sort(np.random.default_rng(41).choice(p["N"], size=512, replace=False))
    got = C[:, torch.from_numpy(cols).cuda()].cpu().numpy()
    del C
    assert_close(got, oracle.bcsr_spmm(O, p["B"], cols=cols), "bcsr_llm slice")


def test_bcsr_64_row_blocks_padded_strides():
    """64-row blocks with padded B and C rows (the 64-row x 192-token kernel): the
    padding columns of C stay untouched."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.bcsr_problem(384, 256, 320, 64, 64, 8, seed=11)
    A = dev_half(p["A"], "bf16")
    Bpad = torch.zeros((256, 336), dtype=torch.bfloat16, device="cuda")
    Bpad[:, :320] = dev_half(p["B"], "bf16")
    F = spmm.build_bcsr(A, 64, 64)
    Cpad = torch.full((384, 324), -1.0, device="cuda")
    out = spmm.spmm_bcsr(F, Bpad[:, :320], Cpad[:, :320])
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    O = oracle.bcsr_build(p["A"], 64, 64, "bf16")
    assert_close(out.cpu().numpy(), oracle.bcsr_spmm(O, p["B"]), "64-row blocks, padded")
    assert (Cpad[:, 320:] == -1.0).all().item()


@pytest.mark.parametrize("dtype,pad", [("bf16", 0), ("bf16", 4), ("i8", 0), ("i8", 3)])
def test_bcsr_builder_pitches(dtype, pad):
    """The builder's 16-byte path (aligned row pitch) and its element path (a pitch
    of K + 4 bf16 or K + 3 int8 elements) both give the oracle's row_ptr, col_idx
    and values bit for bit, for 16-bit and int8 operands (-0.0 and NaN included
    for bf16)."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    M, K, bh, bw = 256, 512, 32, 64
    p = gen.bcsr_problem(M, K, 8, bh, bw, 20, seed=31 + pad, dtype="bf16")
    if dtype == "i8":
        rng = np.random.default_rng(pad)
        A = np.where(p["A"] != 0, rng.integers(-128, 128, size=(M, K)), 0).astype(np.int8)
        Ad = torch.zeros((M, K + pad), dtype=torch.int8, device="cuda")
        Ad[:, :K] = torch.from_numpy(A).cuda()
    else:
        A = p["A"].copy()
        A[0, 0] = 0x8000                       # -0.0: zero, its block not stored unless other entries are
        A[5, 70] = 0x7FC0                      # NaN: nonzero
        Ad = torch.zeros((M, K + pad), dtype=torch.bfloat16, device="cuda")
        Ad[:, :K] = dev_half(A, "bf16")
    F = spmm.build_bcsr(Ad[:, :K], bh, bw)
    O = oracle.bcsr_build(A, bh, bw, dtype)
    assert F.nnzb == O["nnzb"]
    assert np.array_equal(F.row_ptr.cpu().numpy(), O["row_ptr"])
    assert np.array_equal(F.col_idx.cpu().numpy(), O["col_idx"])
    got = F.vals.cpu().numpy() if dtype == "i8" else host_bits(F.vals)
    assert np.array_equal(got.reshape(O["vals"].shape), O["vals"])
