"""Pins for the CPU oracle: each check ties it to something other than itself.

* fp16 / bf16 decoding: exhaustive over all 65536 bit patterns, against numpy;
  fp8 (E4M3, E5M2) decoding: exhaustive over all 256 patterns, against torch's
  float8 types, plus the extreme codes of the format definition.
* hand-worked fixtures under tests/golden/ (each cites the passage it reads).
* brute-force dense GEMM (numpy) on the densified operand.
* format round trips, invariants, and reductions to textbook routines
  (scipy CSR SpMM for one-row windows; dense GEMM when every block is stored;
  dense GEMM on the even-compressed K when every nibble is (0, 1)).
"""
import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests._helpers import bits_to_f64, golden, to_bits


# ---------------------------------------------------------------- decoding
def test_decode_f16_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_bf16_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, "bf16")
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("dtype", ["e4m3", "e5m2"])
def test_decode_fp8_exhaustive(dtype):
    torch = pytest.importorskip("torch")
    bits = np.arange(256, dtype=np.uint16).astype(np.uint8)
    got = oracle.decode(bits, dtype)
    fd = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
    ref = torch.from_numpy(bits.copy()).view(fd).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_fp8_extreme_codes():
    # the format definitions' landmarks: largest finite, smallest subnormal, NaN, infinity
    e4 = oracle.decode(np.array([0x7E, 0x01, 0x08, 0x7F, 0xFF, 0x80, 0x38], np.uint8), "e4m3")
    assert e4[0] == 448.0 and e4[1] == 2.0 ** -9 and e4[2] == 2.0 ** -6 and e4[6] == 1.0
    assert np.isnan(e4[3]) and np.isnan(e4[4]) and e4[5] == 0.0 and np.signbit(e4[5])
    e5 = oracle.decode(np.array([0x7B, 0x01, 0x04, 0x7C, 0xFC, 0x7D, 0x3C], np.uint8), "e5m2")
    assert e5[0] == 57344.0 and e5[1] == 2.0 ** -16 and e5[2] == 2.0 ** -14 and e5[6] == 1.0
    assert e5[3] == np.inf and e5[4] == -np.inf and np.isnan(e5[5])


def test_bf16_rounding_is_rne():
    # the input generator's rounding: ties to even, checked on hand-picked values
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38], dtype=np.float32)
    b = gen.round_f32_to_bf16_bits(x)
    # 1 + 2^-8 is a tie between 1 and 1+2^-7 -> even (1.0);
    # 1 + 3*2^-8 is a tie between 1+2^-7 and 1+2^-6 -> even (1+2^-6)
    assert b.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x7F62]


# ---------------------------------------------------------------- BCSR
def test_bcsr_golden():
    g = golden("bcsr_bf16_4x6.json")
    A, B = to_bits(g["A"], "bf16"), to_bits(g["B"], "bf16")
    F = oracle.bcsr_build(A, g["bh"], g["bw"], "bf16")
    assert F["row_ptr"].tolist() == g["row_ptr"]
    assert F["col_idx"].tolist() == g["col_idx"]
    assert np.array_equal(F["vals"], to_bits(g["vals"], "bf16"))
    assert np.array_equal(oracle.bcsr_spmm(F, B), np.array(g["C"], dtype=np.float64))


def _dense_ref(A_bits, B_bits, dtype):
    return bits_to_f64(A_bits, dtype) @ bits_to_f64(B_bits, dtype)


@pytest.mark.parametrize("bh,bw", [(16, 16), (2, 4), (8, 8)])
def test_bcsr_vs_dense_gemm(bh, bw):
    p = gen.bcsr_problem(64, 96, 40, bh, bw, nnzb=(64 // bh) * (96 // bw) // 3, seed=7)
    F = oracle.bcsr_build(p["A"], bh, bw, "bf16")
    got = oracle.bcsr_spmm(F, p["B"])
    ref = _dense_ref(p["A"], p["B"], "bf16")
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # round trip and the exact block count
    assert np.array_equal(oracle.bcsr_densify(F), p["A"])
    blocks = (p["A"].reshape(64 // bh, bh, 96 // bw, bw) & 0x7FFF).any(axis=(1, 3))
    assert F["nnzb"] == int(blocks.sum()) == len(p["block_pos"])


def test_bcsr_all_blocks_is_dense_gemm_and_row_col_selection():
    rng = np.random.default_rng(3)
    A = gen.normal_bits(rng, (32, 48), "f16")
    B = gen.normal_bits(rng, (48, 20), "f16")
    F = oracle.bcsr_build(A, 8, 16, "f16")
    assert F["nnzb"] == (32 // 8) * (48 // 16)
    ref = _dense_ref(A, B, "f16")
    np.testing.assert_allclose(oracle.bcsr_spmm(F, B), ref, rtol=1e-12, atol=1e-12)
    cols = [19, 0, 7]
    np.testing.assert_allclose(oracle.bcsr_spmm(F, B, rows=(5, 17), cols=cols), ref[5:17][:, cols],
                               rtol=1e-12, atol=1e-12)


def test_bcsr_identity_blocks_copy_rows_and_zero():
    A = np.zeros((32, 32), dtype=np.float32)
    A[0:16, 16:32] = np.eye(16)            # block (0,1) = I
    A[16:32, 0:16] = np.eye(16)            # block (1,0) = I
    Ab = to_bits(A, "bf16")
    rng = np.random.default_rng(5)
    B = gen.normal_bits(rng, (32, 24), "bf16")
    F = oracle.bcsr_build(Ab, 16, 16, "bf16")
    out = oracle.bcsr_spmm(F, B)
    Bf = bits_to_f64(B, "bf16")
    assert np.array_equal(out[0:16], Bf[16:32]) and np.array_equal(out[16:32], Bf[0:16])
    Z = oracle.bcsr_build(np.zeros((32, 32), np.uint16), 16, 16, "bf16")
    assert Z["nnzb"] == 0 and not oracle.bcsr_spmm(Z, B).any()


def test_bcsr_nan_block_is_stored_and_shape_error():
    A = np.zeros((4, 4), dtype=np.uint16)
    A[3, 3] = 0x7FC0                      # NaN counts as nonzero
    A[0, 0] = 0x8000                      # -0.0 does not
    F = oracle.bcsr_build(A, 2, 2, "bf16")
    assert F["col_idx"].tolist() == [1] and F["row_ptr"].tolist() == [0, 0, 1]
    with pytest.raises(oracle.OracleError):
        oracle.bcsr_build(np.zeros((6, 4), np.uint16), 4, 4, "bf16")


# ---------------------------------------------------------------- WCSR
def test_wcsr_golden():
    g = golden("wcsr_f16_h2_s1.json")
    val = to_bits(g["csr_val"], "f16")
    F = oracle.wcsr_build(g["M"], g["K"], np.array(g["csr_row_ptr"]), np.array(g["csr_col"]), val,
                          "f16", h=g["h"], S=g["S"])
    for k in ("wcol_ptr", "wcols", "wnz_ptr", "unit_ptr", "unit_win", "unit_nz_ptr", "lrow", "slot"):
        assert F[k].tolist() == g[k], k
    assert np.array_equal(F["val"], to_bits(g["val"], "f16"))


def _small_csr(M=70, K=300, N=24, seed=11, sigma=1.5, mean=6.0, clip=200):
    return gen.csr_lognormal_problem(M, K, N, seed, mean=mean, sigma=sigma, clip=clip)


def _csr_dense(p):
    D = np.zeros((p["M"], p["K"]), dtype=np.float64)
    rows = np.repeat(np.arange(p["M"]), np.diff(p["row_ptr"]))
    D[rows, p["col"]] = bits_to_f64(p["val"], p["dtype"])
    return D


@pytest.mark.parametrize("h,S", [(16, 32), (4, 1), (1, 2), (7, 1)])
def test_wcsr_round_trip_invariants_and_dense(h, S):
    p = _small_csr()
    F = oracle.wcsr_build(p["M"], p["K"], p["row_ptr"], p["col"], p["val"], "f16", h=h, S=S)
    rp, col, val = oracle.wcsr_to_csr(F)
    assert np.array_equal(rp, p["row_ptr"]) and np.array_equal(col, p["col"])
    assert np.array_equal(val, p["val"])
    # units cover every window once, contiguous, in window order
    nw = F["nw"]
    assert F["unit_ptr"][0] == 0 and F["unit_ptr"][-1] == F["n_units"]
    for w in range(nw):
        us = range(F["unit_ptr"][w], F["unit_ptr"][w + 1])
        assert len(us) >= 1 and all(F["unit_win"][u] == w for u in us)
        assert F["unit_nz_ptr"][us[0]] == F["wnz_ptr"][w]
        assert F["unit_nz_ptr"][us[-1] + 1] == F["wnz_ptr"][w + 1]
        T = F["wcol_ptr"][w + 1] - F["wcol_ptr"][w]
        assert len(us) == max(1, -(-T // (16 * S)))
        # per-window nnz equals the CSR row-range nnz
        r1 = min(p["M"], (w + 1) * h)
        assert F["wnz_ptr"][w + 1] - F["wnz_ptr"][w] == p["row_ptr"][r1] - p["row_ptr"][w * h]
        wc = F["wcols"][F["wcol_ptr"][w]:F["wcol_ptr"][w + 1]]
        assert np.all(np.diff(wc) > 0)
    got = oracle.wcsr_spmm(F, p["B"])
    ref = _csr_dense(p) @ bits_to_f64(p["B"], "f16")
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_wcsr_h1_is_csr_spmm_scipy():
    sp = pytest.importorskip("scipy.sparse")
    p = _small_csr(M=50, K=120, N=9, seed=4)
    F = oracle.wcsr_build(p["M"], p["K"], p["row_ptr"], p["col"], p["val"], "f16", h=1, S=1)
    A = sp.csr_matrix((bits_to_f64(p["val"], "f16"), p["col"], p["row_ptr"]), shape=(p["M"], p["K"]))
    ref = A @ bits_to_f64(p["B"], "f16")
    np.testing.assert_allclose(oracle.wcsr_spmm(F, p["B"]), ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.csr_spmm(p["M"], p["row_ptr"], p["col"], p["val"], p["B"], "f16"),
                               ref, rtol=1e-12, atol=1e-12)


def test_csr_check_rejects_bad_input():
    assert oracle.csr_check(2, 5, [0, 2, 3], [1, 1, 4]) != 0       # duplicate column
    assert oracle.csr_check(2, 5, [0, 2, 3], [2, 1, 4]) != 0       # unsorted
    assert oracle.csr_check(2, 5, [0, 2, 1], [1, 2, 4]) != 0       # row_ptr not monotone
    assert oracle.csr_check(2, 5, [0, 2, 3], [1, 2, 5]) != 0       # out of range
    assert oracle.csr_check(2, 5, [0, 2, 3], [1, 2, 4]) == 0
    with pytest.raises(oracle.OracleError):
        oracle.wcsr_build(2, 5, np.array([0, 2, 3]), np.array([2, 1, 4]), np.zeros(3, np.uint16), "f16")


# ---------------------------------------------------------------- 2:4
def test_24_golden():
    g = golden("mask24_int8_2x8.json")
    A, B = np.array(g["A"], np.int8), np.array(g["B"], np.int8)
    F = oracle.compress24(A, "i8")
    assert F["vals"].tolist() == g["vals"] and F["meta"].tolist() == g["meta"]
    assert oracle.spmm24(F, B).tolist() == g["C"]


def test_24_fp8_golden():
    g = golden("mask24_e4m3_2x8.json")
    A, B = np.array(g["A"], np.uint8), np.array(g["B"], np.uint8)
    F = oracle.compress24(A, "e4m3")
    assert F["vals"].tolist() == g["vals"] and F["meta"].tolist() == g["meta"]
    assert oracle.spmm24(F, B).tolist() == g["C"]


@pytest.mark.parametrize("dtype", ["e4m3", "e5m2"])
def test_24_fp8_vs_dense_gemm_and_round_trip(dtype):
    """E4M3: every product and partial sum is exact in fp64, so the oracle equals a dense
    numpy GEMM on the densified operand (decoded by torch) bit for bit; E5M2 to 1e-12."""
    pytest.importorskip("torch")
    p = gen.mask24_float_problem(40, 256, 24, seed=12, dtype=dtype)
    F = oracle.compress24(p["A"], dtype)
    # the round trip holds up to the sign of zero (a value that rounded to -0 is not stored)
    A0 = np.where((p["A"] & 0x7F) == 0, 0, p["A"]).astype(np.uint8)
    assert F["vals"].dtype == np.uint8 and np.array_equal(oracle.densify24(F), A0)
    nib = np.stack([F["meta"] & 15, F["meta"] >> 4], axis=-1).reshape(40, 64)
    assert np.all((nib & 3) < (nib >> 2))
    ref = bits_to_f64(p["A"], dtype) @ bits_to_f64(p["B"], dtype)
    got = oracle.spmm24(F, p["B"])
    if dtype == "e4m3":
        assert np.array_equal(got, ref)
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # rows and columns selected on the way out are the same numbers
    sel = oracle.spmm24(F, p["B"], rows=(3, 9), cols=[5, 0, 23])
    assert np.array_equal(sel, got[3:9][:, [5, 0, 23]])


def test_24_fp8_negative_zero_is_zero_and_errors():
    A = np.zeros((1, 8), np.uint8)
    A[0, :4] = [0x80, 0x38, 0x80, 0x40]     # -0, 1, -0, 2: two nonzeros, -0 counts as zero
    F = oracle.compress24(A, "e4m3")
    assert F["vals"].tolist() == [[0x38, 0x40, 0, 0]] and F["meta"].tolist() == [[0x4D]]
    A[0, 4:7] = [0x38, 0x7F, 0x01]           # 1, NaN, 2^-9: three nonzeros (NaN is nonzero)
    with pytest.raises(oracle.OracleError):
        oracle.compress24(A, "e4m3")


def test_24_int8_exact_vs_int64_gemm_and_invariants():
    p = gen.mask24_problem(48, 128, 33, seed=9)
    nz = (p["A"].reshape(48, 32, 4) != 0).sum(axis=2)
    assert np.all(nz == 2)
    F = oracle.compress24(p["A"], "i8")
    assert np.array_equal(oracle.densify24(F), p["A"])
    nib = np.stack([F["meta"] & 15, F["meta"] >> 4], axis=-1).reshape(48, 32)
    assert np.all((nib & 3) < (nib >> 2))
    got = oracle.spmm24(F, p["B"])
    assert got.dtype == np.int64
    assert np.array_equal(got, p["A"].astype(np.int64) @ p["B"].astype(np.int64))


def test_24_linearity_and_zero():
    p = gen.mask24_problem(16, 64, 12, seed=10)
    F = oracle.compress24(p["A"], "i8")
    rng = np.random.default_rng(1)
    B1 = rng.integers(-60, 60, size=(64, 12)).astype(np.int8)
    B2 = rng.integers(-60, 60, size=(64, 12)).astype(np.int8)
    assert np.array_equal(oracle.spmm24(F, (B1 + B2).astype(np.int8)),
                          oracle.spmm24(F, B1) + oracle.spmm24(F, B2))
    Z = oracle.compress24(np.zeros((16, 64), np.int8), "i8")
    assert not oracle.spmm24(Z, B1).any()
    assert np.all(Z["meta"] == 0x44)


def test_24_meta01_is_dense_on_even_compressed_k():
    rng = np.random.default_rng(2)
    M, K, N = 8, 32, 5
    A = np.zeros((M, K), np.float32)
    A[:, 0::4] = rng.standard_normal((M, K // 4))
    A[:, 1::4] = rng.standard_normal((M, K // 4))
    Ab = to_bits(A, "bf16")
    F = oracle.compress24(Ab, "bf16")
    assert np.all(F["meta"] == 0x44)
    B = gen.normal_bits(rng, (K, N), "bf16")
    Bsel = bits_to_f64(B, "bf16").reshape(K // 4, 4, N)[:, :2, :].reshape(K // 2, N)
    ref = bits_to_f64(F["vals"], "bf16") @ Bsel
    np.testing.assert_allclose(oracle.spmm24(F, B), ref, rtol=1e-12, atol=1e-12)


def test_24_errors():
    A = np.zeros((2, 8), np.int8)
    A[1, 4:7] = 1                          # three nonzeros in a group
    with pytest.raises(oracle.OracleError):
        oracle.compress24(A, "i8")
    with pytest.raises(oracle.OracleError):
        oracle.compress24(np.zeros((2, 6), np.int8), "i8")


# ---------------------------------------------------------------- TVW
def test_tvw_golden():
    g = golden("tvw_f16_2x8.json")
    A, B = to_bits(g["A"], "f16"), to_bits(g["B"], "f16")
    F = oracle.tvw_build(A, g["tile_rows"], g["tile_ptr"], g["cols"], "f16", Kp=g["Kp"])
    assert np.array_equal(F["vals"], to_bits(g["vals"], "f16"))
    assert F["meta"].tolist() == g["meta"]
    assert np.array_equal(oracle.tvw_spmm(F, B), np.array(g["C"], np.float64))


def test_tvw_round_trip_and_dense():
    p = gen.tvw_problem(40, 64, 17, tile_rows=16, keep=32, seed=12)
    F = oracle.tvw_build(p["A"], 16, p["tile_ptr"], p["cols"], "f16")
    assert np.array_equal(oracle.tvw_densify(F), p["A"])
    for t in range(3):
        c = p["cols"][p["tile_ptr"][t]:p["tile_ptr"][t + 1]]
        assert np.all(np.diff(c) > 0)
    ref = _dense_ref(p["A"], p["B"], "f16")
    np.testing.assert_allclose(oracle.tvw_spmm(F, p["B"]), ref, rtol=1e-12, atol=1e-12)


def test_tvw_all_kept_reduces_to_24():
    p = gen.mask24_problem(16, 32, 6, seed=13)
    Ab = to_bits(p["A"].astype(np.float32), "f16")
    Bb = to_bits(p["B"].astype(np.float32), "f16")
    F = oracle.tvw_build(Ab, 16, [0, 32], np.arange(32), "f16")
    G = oracle.compress24(Ab, "f16")
    assert np.array_equal(F["vals"], G["vals"]) and np.array_equal(F["meta"], G["meta"])
    assert np.array_equal(oracle.tvw_spmm(F, Bb), oracle.spmm24(G, Bb))


def test_tvw_errors():
    g = golden("tvw_f16_2x8.json")
    A = to_bits(g["A"], "f16")
    A[0, 0] = to_bits([1.0], "f16")[0]     # nonzero outside the kept set
    with pytest.raises(oracle.OracleError):
        oracle.tvw_build(A, 2, g["tile_ptr"], g["cols"], "f16")
    with pytest.raises(oracle.OracleError):  # kept columns not ascending
        oracle.tvw_build(to_bits(g["A"], "f16"), 2, g["tile_ptr"], [2, 1, 5, 7], "f16")


def test_wcsr_windows_with_repeated_columns():
    # many rows share columns (K small): windows hold far fewer distinct columns
    # than nonzeros; the builder must still produce the exact layout
    p = gen.csr_lognormal_problem(200, 40, 8, seed=5, mean=10.0, sigma=1.0, clip=40)
    for h, S in ((32, 1), (16, 4), (7, 2)):
        F = oracle.wcsr_build(p["M"], p["K"], p["row_ptr"], p["col"], p["val"], "f16", h=h, S=S)
        rp, col, val = oracle.wcsr_to_csr(F)
        assert np.array_equal(rp, p["row_ptr"]) and np.array_equal(col, p["col"])
        assert F["n_wcols"] < p["row_ptr"][-1]
        np.testing.assert_allclose(oracle.wcsr_spmm(F, p["B"]), _csr_dense(p) @ bits_to_f64(p["B"], "f16"),
                                   rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- 2:4 magnitude pruning
def _prune_keys(A, dtype):
    if dtype == "i8":
        return np.abs(A.astype(np.int64))
    return (A.astype(np.int64) & (0x7F if dtype in ("e4m3", "e5m2") else 0x7FFF))


def test_prune24_hand_worked_groups():
    """Worked by hand: ties go to the lower index; -128 outranks 127; NaN outranks inf."""
    A = np.array([[3, -3, 3, 1, 0, 0, 0, 0, -128, 127, 5, -128, 0, 9, 0, -9]], dtype=np.int8)
    F = oracle.prune24(A, "i8")
    assert F["vals"].tolist() == [[3, -3, 0, 0, -128, -128, 9, -9]]
    # groups: (0,1) -> 0x4, (0,1) -> 0x4 | (0,3) -> 0xC, (1,3) -> 0xD
    assert F["meta"].tolist() == [[0x44, 0xDC]]
    h = np.array([[0x7E00, 0x7C00, 0x8000, 0x3C00, 0x8000, 0x0000, 0x0000, 0x0000]], dtype=np.uint16)
    Fh = oracle.prune24(h, "f16")
    assert Fh["vals"].tolist() == [[0x7E00, 0x7C00, 0x8000, 0x0000]]
    assert Fh["meta"].tolist() == [[0x44]]


@pytest.mark.parametrize("dtype", ["i8", "f16", "bf16", "e4m3"])
def test_prune24_keeps_the_largest_magnitudes(dtype):
    """Properties any correct magnitude pruning has: exactly two positions per group,
    kept values copied bit for bit, every dropped magnitude at most the smaller kept
    one (and on a tie the dropped index is the higher), the kept pair's magnitude sum
    the largest over all six pairs."""
    rng = np.random.default_rng(11)
    M, K = 24, 64
    if dtype == "i8":
        A = rng.integers(-4, 5, size=(M, K)).astype(np.int8)        # small range: many ties
    else:
        A = gen.normal_bits(rng, (M, K), dtype)
        A[rng.random((M, K)) < 0.3] = 0
        A[rng.random((M, K)) < 0.1] ^= A.dtype.type(0x80 if A.dtype == np.uint8 else 0x8000)  # sign flips
    F = oracle.prune24(A, dtype)
    D = oracle.densify24(F)
    keys = _prune_keys(A, dtype).reshape(M, K // 4, 4)
    nib = np.stack([F["meta"] & 15, F["meta"] >> 4], axis=2).reshape(M, K // 4)
    i0, i1 = nib & 3, nib >> 2
    assert np.all(i0 < i1)
    g = np.arange(K // 4)
    for r in range(M):
        kept = np.zeros((K // 4, 4), dtype=bool)
        kept[g, i0[r]] = True
        kept[g, i1[r]] = True
        dense_row = A[r].reshape(K // 4, 4)
        assert np.array_equal(D[r].reshape(K // 4, 4)[kept], dense_row[kept])
        assert not (D[r].reshape(K // 4, 4)[~kept].astype(np.int64) & (0xFFFF if A.dtype == np.uint16 else 0xFF)).any()
        kr = keys[r]
        kmin = np.minimum(kr[g, i0[r]], kr[g, i1[r]])
        lo_of_min = np.where(kr[g, i0[r]] <= kr[g, i1[r]], np.where(kr[g, i0[r]] == kr[g, i1[r]], i1[r], i0[r]), i1[r])
        for q in range(4):
            dropped = ~kept[:, q]
            assert np.all(kr[dropped, q] <= kmin[dropped])
            tie = dropped & (kr[:, q] == kmin)
            assert np.all(q > lo_of_min[tie])
        pair_sums = np.stack([kr[:, a] + kr[:, b] for a in range(4) for b in range(a + 1, 4)], axis=1)
        assert np.all(kr[g, i0[r]] + kr[g, i1[r]] == pair_sums.max(axis=1))


@pytest.mark.parametrize("dtype", ["i8", "f16", "e4m3"])
def test_prune24_of_a_24_matrix_is_its_compression(dtype):
    """A matrix that already has at most two nonzeros per group loses nothing: pruning
    equals plain 2:4 compression (padding with the lowest zero positions)."""
    if dtype == "i8":
        A = gen.mask24_problem(32, 256, 1, seed=4)["A"]
    else:
        A = gen.mask24_float_problem(32, 256, 1, seed=4, dtype=dtype)["A"]
    P, Cq = oracle.prune24(A, dtype), oracle.compress24(A, dtype)
    assert np.array_equal(P["vals"], Cq["vals"]) and np.array_equal(P["meta"], Cq["meta"])


def _kept_cols(rng, M, K, tile_rows, keep):
    n_tiles = -(-M // tile_rows)
    cols = np.concatenate([np.sort(rng.choice(K, keep, replace=False)) for _ in range(n_tiles)]).astype(np.int32)
    return np.arange(0, n_tiles * keep + 1, keep, dtype=np.int32), cols


@pytest.mark.parametrize("dtype", ["i8", "bf16"])
def test_prune_tvw_is_prune24_on_the_gathered_columns(dtype):
    """Pruning into TVW equals 2:4 pruning of each tile's kept columns gathered into a
    dense block, and drops everything outside them."""
    rng = np.random.default_rng(5)
    M, K, tr, keep = 40, 96, 16, 32
    A = rng.integers(-5, 6, size=(M, K)).astype(np.int8) if dtype == "i8" else gen.normal_bits(rng, (M, K), dtype)
    tp, cols = _kept_cols(rng, M, K, tr, keep)
    F = oracle.prune_tvw(A, tr, tp, cols, dtype, Kp=keep)
    for t in range(len(tp) - 1):
        kc = cols[tp[t]:tp[t + 1]]
        rows = slice(t * tr, min(M, (t + 1) * tr))
        P = oracle.prune24(np.ascontiguousarray(A[rows][:, kc]), dtype)
        assert np.array_equal(F["vals"][rows], P["vals"]) and np.array_equal(F["meta"][rows], P["meta"])
    D = oracle.tvw_densify(F)
    for t in range(len(tp) - 1):
        outside = np.setdiff1d(np.arange(K), cols[tp[t]:tp[t + 1]])
        assert not (D[t * tr:(t + 1) * tr][:, outside].astype(np.int64) & 0xFFFF).any()


def test_prune_tvw_of_a_tvw_matrix_is_its_build():
    p = gen.tvw_problem(256, 512, 8, tile_rows=128, keep=256, seed=9)
    P = oracle.prune_tvw(p["A"], 128, p["tile_ptr"], p["cols"], "f16")
    B = oracle.tvw_build(p["A"], 128, p["tile_ptr"], p["cols"], "f16")
    assert np.array_equal(P["vals"], B["vals"]) and np.array_equal(P["meta"], B["meta"])


# ---------------------------------------------------------------- (2n-2):2n sliding windows
def _fold_back(L, K, n):
    """Sum every lifted column into the original column it reads (numpy, int64/f64)."""
    src = oracle.slide_src(K, n)
    out = np.zeros((L.shape[0], K), dtype=L.dtype)
    np.add.at(out, (slice(None), src), L)
    return out


def test_slide_golden():
    g = golden("slide68_int8_2x16.json")
    A, B = np.array(g["A"], np.int8), np.array(g["B"], np.int8)
    assert oracle.slide_src(16, g["n"]).tolist() == g["src"]
    assert oracle.slide_decompose(A, g["n"], "i8").tolist() == g["L"]
    F = oracle.slide_build(A, g["n"], "i8")
    assert F["vals"].tolist() == g["vals"] and F["meta"].tolist() == g["meta"]
    assert oracle.slide_spmm(F, B).tolist() == g["C"]


def test_slide_window_map_covers_pairs():
    """Window j of group g reads the group's columns 2j .. 2j+3: pairs 0 and n-1 are
    read once, every inner pair twice (by windows j-1 and j), nothing else."""
    for n in (2, 3, 4, 5, 8):
        K = 2 * n * 3
        src = oracle.slide_src(K, n)
        assert src.shape[0] == 4 * (n - 1) * 3
        counts = np.bincount(src, minlength=K).reshape(3, n, 2)
        assert np.all(counts[:, 0] == 1) and np.all(counts[:, n - 1] == 1)
        assert np.all(counts[:, 1:n - 1] == 2)
        w = src.reshape(-1, 4)
        assert np.all(np.diff(w, axis=1) == 1) and np.all(w[:, 0] % 2 == 0)


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_slide_decompose_exhaustive_masks(n):
    """Every mask of at most 2n-2 nonzeros in a 2n-group decomposes: each window
    holds at most two nonzeros, and the lifted matrix folds back onto A exactly
    (every nonzero lands in exactly one window)."""
    import itertools
    masks = [m for k in range(2 * n - 1) for m in itertools.combinations(range(2 * n), k)]
    rng = np.random.default_rng(n)
    A = np.zeros((len(masks), 4 * n), np.int8)            # two groups per row
    for r, m in enumerate(masks):
        for h in range(2):
            for t in m:
                A[r, 2 * n * h + t] = rng.integers(1, 128) * rng.choice([-1, 1])
        A[r, 2 * n:] = np.roll(A[r, 2 * n:], r % (2 * n))  # second group: another mask
    L = oracle.slide_decompose(A, n, "i8")
    assert np.all((L.reshape(len(masks), -1, 4) != 0).sum(axis=2) <= 2)
    assert np.array_equal(_fold_back(L.astype(np.int64), 4 * n, n), A.astype(np.int64))
    assert np.count_nonzero(L) == np.count_nonzero(A)


def test_slide_int8_exact_vs_int64_gemm():
    """C = A B exactly (int64), whatever the decomposition, for 6:8 and 4:6."""
    for n in (4, 3):
        p = gen.slide_problem(40, 32 * n, 19, n, seed=12, dtype=gen.I8)
        F = oracle.slide_build(p["A"], n, "i8")
        assert np.array_equal(oracle.slide_spmm(F, p["B"]),
                              p["A"].astype(np.int64) @ p["B"].astype(np.int64))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_slide_float_vs_dense_gemm(dtype):
    p = gen.slide_problem(24, 64, 7, 4, seed=13, dtype=dtype)
    F = oracle.slide_build(p["A"], 4, dtype)
    ref = bits_to_f64(p["A"], dtype) @ bits_to_f64(p["B"], dtype)
    np.testing.assert_allclose(oracle.slide_spmm(F, p["B"]), ref, rtol=1e-12, atol=1e-12)
    # the lifted values are the original bit patterns (or +0 padding)
    L = oracle.slide_decompose(p["A"], 4, dtype)
    assert np.array_equal(_fold_back(L.astype(np.int64), 64, 4), p["A"].astype(np.int64) * (p["A"] & 0x7FFF != 0))


def test_slide_n2_is_24_and_ratio():
    """n = 2 is plain 2:4 (one window per group, the identity map); for 6:8 the
    tensor-core depth is K (n-1)/n, the N/(N-1) = 4/3 bound the abstract states."""
    p = gen.mask24_problem(16, 64, 3, seed=14)
    F, G = oracle.slide_build(p["A"], 2, "i8"), oracle.compress24(p["A"], "i8")
    assert np.array_equal(F["vals"], G["vals"]) and np.array_equal(F["meta"], G["meta"])
    assert oracle.slide_src(64, 2).tolist() == list(range(64))
    for K in (64, 3584, 8192):
        assert K / (oracle.slide_lifted_k(K, 4) // 2) == 4 / 3


def test_slide_errors():
    A = np.zeros((2, 16), np.int8)
    A[1, 8:15] = 3                                        # 7 nonzeros in a 6:8 group
    with pytest.raises(oracle.OracleError):
        oracle.slide_decompose(A, 4, "i8")
    with pytest.raises(oracle.OracleError):
        oracle.slide_decompose(np.zeros((2, 12), np.int8), 4, "i8")   # K % 8 != 0


# ---------------------------------------------------------------- permutation before BCSR (RCM)
def _bandwidth(A):
    r, c = np.nonzero(np.asarray(A) != 0)
    return int(np.max(np.abs(r - c))) if r.size else 0


def test_rcm_golden():
    g = golden("rcm_int8_7.json")
    A, B = np.array(g["A"], np.int8), np.array(g["B"], np.int8)
    perm = oracle.rcm_dense(A)
    assert perm.tolist() == g["perm"]
    F = oracle.bcsr_build(oracle.permute_sym(A, perm, "i8"), 1, 1, "i8")
    assert oracle.bcsr_spmm_permuted(F, perm, B).tolist() == g["C"]


def test_rcm_scrambled_path_and_band():
    """A scrambled path comes back as a path (bandwidth 1, a closed form of the
    breadth-first order from an end); a scrambled band of half-width w comes back
    within bandwidth 2w, every breadth-first level of a band being w wide."""
    rng = np.random.default_rng(3)
    n = 50
    q = rng.permutation(n)
    A = np.zeros((n, n), np.int8)
    for t in range(n - 1):
        A[q[t], q[t + 1]] = 1
    perm = oracle.rcm_dense(A)
    assert sorted(perm.tolist()) == list(range(n))
    assert _bandwidth(A[np.ix_(perm, perm)] | A[np.ix_(perm, perm)].T) == 1
    for w in (2, 5):
        p = gen.banded_scrambled_problem(96, w, 1, seed=w, dtype="i8")
        assert _bandwidth(p["A"]) > 4 * w
        perm = oracle.rcm_dense(p["A"])
        assert _bandwidth(p["A"][np.ix_(perm, perm)]) <= 2 * w


def test_rcm_components_isolated_nodes_and_asymmetric_pattern():
    rng = np.random.default_rng(5)
    n = 40
    A = (rng.random((n, n)) < 0.04).astype(np.int8)       # asymmetric, several components
    A[7, :] = 0
    A[:, 7] = 0                                            # an isolated node
    perm = oracle.rcm_dense(A)
    assert sorted(perm.tolist()) == list(range(n))
    # the order is the one of A + A^T: symmetrising the pattern changes nothing
    assert np.array_equal(oracle.rcm_dense(A | A.T), perm)


def test_permute_sym_and_permuted_spmm_equal_the_plain_product():
    """A' = P A P^T entrywise as numpy indexing gives it; gathering B, multiplying the
    BCSR of A' and scattering C equals A B (int8 exactly, bf16 to 1e-12)."""
    p = gen.banded_scrambled_problem(64, 3, 9, seed=8, dtype="i8")
    perm = oracle.rcm_dense(p["A"])
    Ap = oracle.permute_sym(p["A"], perm, "i8")
    assert np.array_equal(Ap, p["A"][np.ix_(perm, perm)])
    F = oracle.bcsr_build(Ap, 16, 16, "i8")
    G = oracle.bcsr_build(p["A"], 16, 16, "i8")
    assert F["nnzb"] <= 10 and G["nnzb"] >= 14             # the band's 4 + 2 * 3 blocks vs (nearly) all 16
    C = oracle.bcsr_spmm_permuted(F, perm, p["B"])
    assert np.array_equal(C, p["A"].astype(np.int64) @ p["B"].astype(np.int64))
    q = gen.banded_scrambled_problem(64, 3, 9, seed=8, dtype="bf16")
    perm = oracle.rcm_dense(q["A"])
    F = oracle.bcsr_build(oracle.permute_sym(q["A"], perm, "bf16"), 16, 16, "bf16")
    np.testing.assert_allclose(oracle.bcsr_spmm_permuted(F, perm, q["B"]),
                               bits_to_f64(q["A"], "bf16") @ bits_to_f64(q["B"], "bf16"), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- SDDMM
def test_sddmm_golden():
    g = golden("sddmm_int8_3x4.json")
    out = oracle.sddmm(np.array(g["row_ptr"]), np.array(g["col"]), np.array(g["A"], np.int8),
                       np.array(g["Bt"], np.int8), "i8")
    assert out.tolist() == g["out"]


def test_sddmm_i64_golden():
    """The exact int8 SDDMM on the hand-worked fixture (its operands are int8)."""
    g = golden("sddmm_int8_3x4.json")
    out = oracle.sddmm_i64(np.array(g["row_ptr"]), np.array(g["col"]), np.array(g["A"], np.int8),
                           np.array(g["Bt"], np.int8))
    assert out.dtype == np.int64 and out.tolist() == g["out"]


def test_sddmm_i64_is_the_integer_product_at_the_pattern():
    """Full-range int8 operands: every output equals the entry of the int64 product
    A Bt^T (numpy) at its position; an emptied row and a non-square pattern
    (M != N) catch a dropped row offset or a transposed operand."""
    q = gen.csr_lognormal_problem(70, 41, 1, seed=9, mean=6.0, sigma=1.0, clip=41, dtype="f16")
    rows = np.repeat(np.arange(70), np.diff(q["row_ptr"]))
    keep = rows != 11
    rp = np.concatenate([[0], np.cumsum(np.bincount(rows[keep], minlength=70))]).astype(np.int32)
    cl = q["col"][keep].astype(np.int32)
    rng = np.random.default_rng(2)
    A = rng.integers(-128, 128, size=(70, 48), dtype=np.int8)
    Bt = rng.integers(-128, 128, size=(41, 48), dtype=np.int8)
    D = A.astype(np.int64) @ Bt.astype(np.int64).T
    out = oracle.sddmm_i64(rp, cl, A, Bt)
    assert np.array_equal(out, D[rows[keep], cl])
    assert rp[11] == rp[12]


@pytest.mark.parametrize("a,b", [(-128, -128), (-128, 127), (127, 127)])
def test_sddmm_i64_extreme_values(a, b):
    """Constant operands give the closed form K * a * b at every entry (K = 4096:
    |sum| up to 2^26, well inside int64 and still exact in int32)."""
    K = 4096
    rp = np.array([0, 3, 3, 5], np.int32)
    cl = np.array([0, 2, 4, 1, 3], np.int32)
    A = np.full((3, K), a, np.int8)
    Bt = np.full((5, K), b, np.int8)
    assert oracle.sddmm_i64(rp, cl, A, Bt).tolist() == [K * a * b] * 5


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_sddmm_is_the_dense_product_at_the_pattern(dtype):
    """Every output equals the entry of the dense product A Bt^T (numpy, fp64) at its
    position (an emptied row included); a full pattern gives the whole product."""
    q = gen.csr_lognormal_problem(60, 45, 1, seed=4, mean=6.0, sigma=1.0, clip=45, dtype=dtype)
    rows = np.repeat(np.arange(60), np.diff(q["row_ptr"]))
    keep = rows != 7                                             # row 7 emptied
    rp = np.concatenate([[0], np.cumsum(np.bincount(rows[keep], minlength=60))]).astype(np.int32)
    cl = q["col"][keep].astype(np.int32)
    rng = np.random.default_rng(1)
    A = gen.normal_bits(rng, (60, 33), dtype)
    Bt = gen.normal_bits(rng, (45, 33), dtype)
    D = bits_to_f64(A, dtype) @ bits_to_f64(Bt, dtype).T
    out = oracle.sddmm(rp, cl, A, Bt, dtype)
    np.testing.assert_allclose(out, D[rows[keep], cl], rtol=1e-12, atol=1e-12)
    assert rp[7] == rp[8]
    full_rp = (np.arange(61) * 45).astype(np.int32)
    full_cl = np.tile(np.arange(45), 60).astype(np.int32)
    np.testing.assert_allclose(oracle.sddmm(full_rp, full_cl, A, Bt, dtype).reshape(60, 45), D, rtol=1e-12, atol=1e-12)
