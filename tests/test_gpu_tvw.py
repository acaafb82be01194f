"""Tile-vector-wise on the GPU vs the CPU oracle: builder bit-exact, SpMM within tolerance."""
import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests.gpu_util import assert_close, dev, dev_half, host_bits, need_gpu, padded_b

pytestmark = pytest.mark.gpu


def _build(p, Kp):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    A = dev_half(p["A"], p["dtype"])
    F = spmm.spmm_build_tvw(A, p["tile_rows"], dev(p["tile_ptr"]), dev(p["cols"]), Kp=Kp)
    O = oracle.tvw_build(p["A"], p["tile_rows"], p["tile_ptr"], p["cols"], p["dtype"], Kp=Kp)
    assert np.array_equal(host_bits(F.vals), O["vals"])
    assert np.array_equal(F.meta.cpu().numpy(), O["meta"])
    return F, O


@pytest.mark.parametrize("M,K,N,keep,dtype", [
    (256, 512, 256, 256, "f16"),
    (384, 1024, 200, [512, 100, 36], "f16"),   # ragged kept counts (100, 36: partial steps)
    (200, 768, 136, [384, 0], "bf16"),         # ragged M, an empty tile
])
def test_tvw_parity(M, K, N, keep, dtype):
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.tvw_problem(M, K, N, 128, keep, seed=M + K, dtype=dtype)
    kmax = max(np.diff(p["tile_ptr"]))
    Kp = max(128, -(-int(kmax) // 128) * 128)
    F, O = _build(p, Kp)
    C = spmm.spmm_tvw(F, padded_b(p["B"], dtype))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert_close(C.cpu().numpy(), oracle.tvw_spmm(O, p["B"]), "tvw")


def test_tvw_builder_rejects_nonzero_outside_kept():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.tvw_problem(128, 256, 8, 128, 64, seed=3)
    A = p["A"].copy()
    outside = np.setdiff1d(np.arange(256), p["cols"])[0]
    A[5, outside] = 0x3C00                              # 1.0 in fp16
    with pytest.raises(spmm.SpmmError) as e:
        spmm.spmm_build_tvw(dev_half(A, "f16"), 128, dev(p["tile_ptr"]), dev(p["cols"]), Kp=128)
    assert e.value.name == "SPMM_ERR_FORMAT"


def test_tvw_full_size_sampled_rows():
    """A 4096 x 4096 (32 tiles of 128 rows, 2048 kept columns each, 2:4 inside),
    B 4096 x 4096: the oracle recomputes 2 seeded rows of every tile and eight
    whole tiles (1024 rows)."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.config_problem("tvw")
    F, O = _build(p, 2048)
    C = spmm.spmm_tvw(F, dev_half(p["B"], "f16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    rng = np.random.default_rng(51)
    rows = np.sort(np.concatenate([t * 128 + rng.choice(128, 2, replace=False) for t in range(32)]))
    got = C[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref = np.concatenate([oracle.tvw_spmm(O, p["B"], rows=(int(r), int(r) + 1)) for r in rows])
    assert_close(got, ref, "tvw full-size rows")
    # eight whole tiles (1024 rows: the first, the last and six seeded ones)
    tiles = sorted(set([0, 31] + [int(t) for t in rng.choice(np.arange(1, 31), 6, replace=False)]))
    assert len(tiles) == 8
    for t in tiles:
        r0 = 128 * t
        assert_close(C[r0:r0 + 128].cpu().numpy(), oracle.tvw_spmm(O, p["B"], rows=(r0, r0 + 128)), f"tvw tile {t}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tvw_prune_bit_exact_and_spmm(dtype):
    """Magnitude pruning of a dense matrix into TVW on the GPU equals the oracle's bit
    for bit (ragged kept counts, an empty tile), and the pruned operand multiplies
    within tolerance."""
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    rng = np.random.default_rng(17)
    M, K, N = 300, 640, 136
    A = gen.normal_bits(rng, (M, K), dtype)
    A[rng.random((M, K)) < 0.1] = 0
    counts = [256, 100, 0]
    cols = np.concatenate([np.sort(rng.choice(K, c, replace=False)) for c in counts]).astype(np.int32)
    tp = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    F = spmm.spmm_prune_tvw(dev_half(A, dtype), 128, dev(tp), dev(cols), Kp=256)
    O = oracle.prune_tvw(A, 128, tp, cols, dtype, Kp=256)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(F.vals), O["vals"])
    assert np.array_equal(F.meta.cpu().numpy(), O["meta"])
    B = gen.normal_bits(rng, (K, N), dtype)
    C = spmm.spmm_tvw(F, padded_b(B, dtype))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    assert_close(C.cpu().numpy(), oracle.tvw_spmm(O, B), f"pruned tvw {dtype}")
