"""The seeded input generators produce the stated structure."""
import numpy as np

import spmm_inputs as gen


def test_bcsr_problem_exact_block_count_and_determinism():
    p = gen.bcsr_problem(256, 256, 64, 16, 16, 64, seed=1)
    blocks = (p["A"].reshape(16, 16, 16, 16) & 0x7FFF).any(axis=(1, 3))
    assert blocks.sum() == 64
    q = gen.bcsr_problem(256, 256, 64, 16, 16, 64, seed=1)
    assert np.array_equal(p["A"], q["A"]) and np.array_equal(p["B"], q["B"])


def test_mask24_problem_two_per_group():
    p = gen.mask24_problem(64, 256, 8, seed=2)
    g = p["A"].reshape(64, 64, 4)
    assert np.all((g != 0).sum(axis=2) == 2)
    assert p["A"].min() >= -127 and p["A"].max() <= 127
    assert p["B"].min() >= -127 and p["B"].max() <= 127


def test_csr_lognormal_rows_sorted_unique_and_mean():
    p = gen.csr_lognormal_problem(20000, 65536, 4, seed=3)
    rp, col = p["row_ptr"], p["col"]
    L = np.diff(rp)
    assert L.min() >= 1 and L.max() <= 4096
    assert 13.0 < L.mean() < 19.0
    rows = np.repeat(np.arange(20000), L)
    same = rows[1:] == rows[:-1]
    assert np.all(col[1:][same] > col[:-1][same])


def test_tvw_problem_structure():
    p = gen.tvw_problem(256, 512, 8, tile_rows=128, keep=256, seed=5)
    for t in range(2):
        kc = p["cols"][p["tile_ptr"][t]:p["tile_ptr"][t + 1]]
        assert len(kc) == 256 and np.all(np.diff(kc) > 0)
        rows = p["A"][t * 128:(t + 1) * 128]
        outside = np.setdiff1d(np.arange(512), kc)
        assert not (rows[:, outside] & 0x7FFF).any()
        g = (rows[:, kc] & 0x7FFF).reshape(128, 64, 4) != 0
        assert np.all(g.sum(axis=2) == 2)


def test_mask24_float_problem_two_kept_per_group():
    p = gen.mask24_float_problem(32, 128, 4, seed=6)
    nz = (p["A"] & 0x7FFF).reshape(32, 32, 4) != 0
    assert np.all(nz.sum(axis=2) <= 2) and nz.sum() >= 32 * 32 * 2 - 2
    q = gen.mask24_float_problem(32, 128, 4, seed=6)
    assert np.array_equal(p["A"], q["A"]) and np.array_equal(p["B"], q["B"])


def test_slide_problem_two_zeros_per_group():
    for n, dtype in ((4, gen.I8), (3, gen.I8), (4, gen.F16)):
        p = gen.slide_problem(12, 16 * n, 5, n, seed=3, dtype=dtype)
        nz = (p["A"].reshape(12, 8, 2 * n) != 0).sum(axis=2)
        assert nz.max() <= 2 * n - 2
        if dtype == gen.I8:
            assert np.all(nz == 2 * n - 2)
        q = gen.slide_problem(12, 16 * n, 5, n, seed=3, dtype=dtype)
        assert np.array_equal(p["A"], q["A"]) and np.array_equal(p["B"], q["B"])


def test_banded_scrambled_problem_is_a_permuted_band():
    p = gen.banded_scrambled_problem(64, 3, 5, seed=4, dtype=gen.I8)
    inv = np.argsort(p["q"])
    band = p["A"][np.ix_(inv, inv)]
    i = np.arange(64)
    assert np.all((band != 0) == (np.abs(i[:, None] - i[None, :]) <= 3))


def test_sddmm_config_shares_the_row_window_pattern():
    """The SDDMM workload samples the row-window workload's CSR pattern (same seed,
    rows sorted and unique) with dense A and Bt of the stated inner size."""
    c = dict(gen.CONFIGS["sddmm_lognormal"])
    q = gen.config_problem("sddmm_lognormal", M=512, K=512, inner=16)
    w = gen.config_problem("wcsr_lognormal", M=512, K=512, N=1)
    assert np.array_equal(q["row_ptr"], w["row_ptr"]) and np.array_equal(q["col"], w["col"])
    assert q["A"].shape == (512, 16) and q["Bt"].shape == (512, 16) and c["inner"] == 128
    assert "B" not in q


def test_sddmm_i8_config_shares_the_pattern_with_full_range_int8():
    """The quantized SDDMM workload has the fp16 workload's pattern and int8
    operands covering the whole range [-128, 127]."""
    q = gen.config_problem("sddmm_lognormal_i8", M=512, K=512, inner=64)
    f = gen.config_problem("sddmm_lognormal", M=512, K=512, inner=64)
    assert np.array_equal(q["row_ptr"], f["row_ptr"]) and np.array_equal(q["col"], f["col"])
    assert q["A"].dtype == np.int8 and q["Bt"].dtype == np.int8 and q["dtype"] == "i8"
    assert q["A"].min() == -128 and q["A"].max() == 127
