"""Seeded synthetic inputs for the SpMM workloads.

This module only draws random numbers and lays them out as plain arrays
(dense matrices as raw 16-bit / 8-bit patterns, CSR arrays, kept-column
lists).  It holds none of the SpMM arithmetic and none of the format
builders: both the CPU oracle and the CUDA path receive exactly the arrays
produced here.

Every generator uses numpy's PCG64 (``numpy.random.default_rng(seed)``).
Floating-point values are drawn in fp32 from N(0, std) and rounded to
bf16 / fp16 / fp8 (E4M3, E5M2) with round-to-nearest-even; both sides read
the rounded bits.  The fp8 rounding is torch's fp32 -> float8 conversion.

Workload recipes (sizes follow the five configurations the library is
measured on):

* ``bcsr_problem``   block-sparse A: an exact number of bh x bw blocks,
  positions drawn uniformly without replacement, every entry of a drawn
  block N(0, std); dense B N(0, 1).
* ``mask24_problem`` 2:4 int8 A: in every group of 4 consecutive K entries
  exactly 2 positions (uniform among the 6 pairs) hold values uniform on
  {-127..-1, 1..127}; B uniform on [-127, 127].
* ``csr_lognormal_problem`` irregular CSR A: row lengths
  clip(round(LogNormal(ln(mean) - sigma^2/2, sigma)), 1, clip), columns
  uniform without duplicates per row (ascending), values N(0, 1); B N(0, 1).
* ``csr_window_clustered_problem`` CSR A with column reuse inside row windows:
  every window of h consecutive rows draws ``pool`` distinct columns uniform
  on [0, K) and each of its rows takes ``per_row`` of them (ascending), values
  N(0, 1); B N(0, 1).
* ``tvw_problem``    tile-vector-wise A: per tile of ``tile_rows`` rows a
  uniform random kept subset of K columns (ascending), then inside every
  group of 4 consecutive kept columns exactly 2 positions per row hold
  N(0, 1) values; B N(0, 1).
"""
from __future__ import annotations

import numpy as np

BF16, F16, I8, E4M3, E5M2 = "bf16", "f16", "i8", "e4m3", "e5m2"
FP8 = (E4M3, E5M2)

__all__ = [
    "BF16", "F16", "I8", "E4M3", "E5M2", "FP8", "round_f32_to_bf16_bits", "round_f32_to_fp8_bits",
    "normal_bits", "mask24_float_problem", "csr_window_clustered_problem",
    "bcsr_problem", "mask24_problem", "csr_lognormal_problem", "tvw_problem", "slide_problem", "banded_scrambled_problem",
    "CONFIGS", "config_problem",
]


def round_f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round-to-nearest-even (NaN kept quiet)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    r = ((u + bias) >> 16).astype(np.uint16)
    if nan.any():
        r[nan] = ((u[nan] >> 16) | 0x0040).astype(np.uint16)
    return r


def round_f32_to_fp8_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 -> fp8 (E4M3 or E5M2) bit patterns, round-to-nearest-even (torch's
    conversion; magnitudes beyond the largest finite value are not expected)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    fd = torch.float8_e4m3fn if dtype == E4M3 else torch.float8_e5m2
    return t.to(fd).view(torch.uint8).numpy().copy()


def normal_bits(rng: np.random.Generator, shape, dtype: str, std: float = 1.0) -> np.ndarray:
    """N(0, std) drawn in fp32, returned as uint16 (bf16/fp16) or uint8 (fp8) bit
    patterns of ``dtype``."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if dtype == BF16:
        return round_f32_to_bf16_bits(x)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype in FP8:
        return round_f32_to_fp8_bits(x, dtype)
    raise ValueError(dtype)


def bcsr_problem(M: int, K: int, N: int, bh: int, bw: int, nnzb: int, seed: int,
                 dtype: str = BF16, std: float = 1.0, b_std: float = 1.0) -> dict:
    """Dense A (bits, M x K) with exactly ``nnzb`` nonzero blocks, and B (K x N)."""
    rng = np.random.default_rng(seed)
    gm, gk = M // bh, K // bw
    nblocks = gm * gk
    pos = np.sort(rng.choice(nblocks, size=nnzb, replace=False)) if nnzb else np.zeros(0, np.int64)
    A = np.zeros((M, K), dtype=np.uint16)
    vals = normal_bits(rng, (nnzb, bh, bw), dtype, std)
    Ab = A.reshape(gm, bh, gk, bw)
    for t, p in enumerate(pos.tolist()):
        Ab[p // gk, :, p % gk, :] = vals[t]
    B = normal_bits(rng, (K, N), dtype, b_std)
    return {"A": A, "B": B, "M": M, "K": K, "N": N, "bh": bh, "bw": bw,
            "dtype": dtype, "block_pos": pos}


def mask24_problem(M: int, K: int, N: int, seed: int) -> dict:
    """int8 A with exactly 2 nonzeros in each group of 4 along K; int8 B."""
    assert K % 4 == 0
    rng = np.random.default_rng(seed)
    pairs = np.array([(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)], dtype=np.int64)
    G = K // 4
    A = np.zeros((M, K), dtype=np.int8)
    chunk = max(1, (1 << 24) // max(1, K))
    for r0 in range(0, M, chunk):
        r1 = min(M, r0 + chunk)
        sel = pairs[rng.integers(0, 6, size=(r1 - r0, G))]          # (rows, G, 2)
        mag = rng.integers(1, 128, size=(r1 - r0, G, 2), dtype=np.int16)
        sgn = rng.integers(0, 2, size=(r1 - r0, G, 2), dtype=np.int16) * 2 - 1
        v = (mag * sgn).astype(np.int8)
        cols = sel + (np.arange(G, dtype=np.int64) * 4)[None, :, None]
        rows = np.arange(r0, r1, dtype=np.int64)[:, None, None]
        A[np.broadcast_to(rows, cols.shape), cols] = v
    B = rng.integers(-127, 128, size=(K, N), dtype=np.int16).astype(np.int8)
    return {"A": A, "B": B, "M": M, "K": K, "N": N, "dtype": I8}


def mask24_float_problem(M: int, K: int, N: int, seed: int, dtype: str = F16) -> dict:
    """bf16 / fp16 / fp8 A keeping 2 of every 4 consecutive K-entries (positions uniform
    over the 6 pairs, values N(0,1); a kept value may round to zero), B (K x N) N(0,1) of
    the same type; all as raw bits."""
    assert K % 4 == 0
    rng = np.random.default_rng(seed)
    pairs = np.array([(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)], dtype=np.int64)
    G = K // 4
    A = normal_bits(rng, (M, K), dtype)
    keep = np.zeros((M, K), dtype=bool)
    sel = pairs[rng.integers(0, 6, size=(M, G))]                      # (M, G, 2)
    cols = sel + (np.arange(G, dtype=np.int64) * 4)[None, :, None]
    rows = np.broadcast_to(np.arange(M, dtype=np.int64)[:, None, None], cols.shape)
    keep[rows, cols] = True
    A[~keep] = 0
    B = normal_bits(rng, (K, N), dtype)
    return {"A": A, "B": B, "M": M, "K": K, "N": N, "dtype": dtype}


def slide_problem(M: int, K: int, N: int, n: int, seed: int, dtype: str = F16) -> dict:
    """(2n-2):2n A: in every group of 2n consecutive K-entries two positions, uniform
    over the pairs, are zero and the other 2n - 2 hold values (int8: nonzero, sign
    and magnitude uniform; 16-bit: N(0,1), which may round to zero); B (K x N) of the
    same type.  n = 4 is the 6:8 pattern (25% of the weights pruned)."""
    assert n >= 2 and K % (2 * n) == 0
    rng = np.random.default_rng(seed)
    G = K // (2 * n)
    if dtype == I8:
        mag = rng.integers(1, 128, size=(M, K), dtype=np.int16)
        sgn = rng.integers(0, 2, size=(M, K), dtype=np.int16) * 2 - 1
        A = (mag * sgn).astype(np.int8)
        B = rng.integers(-127, 128, size=(K, N), dtype=np.int16).astype(np.int8)
    else:
        A = normal_bits(rng, (M, K), dtype)
        B = None
    # two distinct zero positions per group: first uniform on 2n, second uniform on the rest
    z0 = rng.integers(0, 2 * n, size=(M, G))
    z1 = (z0 + 1 + rng.integers(0, 2 * n - 1, size=(M, G))) % (2 * n)
    base = (np.arange(G, dtype=np.int64) * 2 * n)[None, :]
    rows = np.broadcast_to(np.arange(M, dtype=np.int64)[:, None], (M, G))
    A[rows, base + z0] = 0
    A[rows, base + z1] = 0
    if B is None:
        B = normal_bits(rng, (K, N), dtype)
    return {"A": A, "B": B, "M": M, "K": K, "N": N, "n": n, "dtype": dtype}


def banded_scrambled_problem(n: int, w: int, N: int, seed: int, dtype: str = F16) -> dict:
    """A square band matrix (A[i][j] stored iff |i - j| <= w, values N(0,1); int8: nonzero
    uniform +-{1..127}) with its rows and columns scrambled by one uniform random
    permutation q (A = Q Band Q^T, i.e. A[i][j] = Band[q[i]][q[j]]); B (n x N)."""
    rng = np.random.default_rng(seed)
    q = rng.permutation(n)
    i = np.arange(n)
    band = np.abs(i[:, None] - i[None, :]) <= w
    if dtype == I8:
        v = (rng.integers(1, 128, size=(n, n)) * (rng.integers(0, 2, size=(n, n)) * 2 - 1)).astype(np.int8)
        B = rng.integers(-127, 128, size=(n, N), dtype=np.int16).astype(np.int8)
    else:
        v = normal_bits(rng, (n, n), dtype)
        B = normal_bits(rng, (n, N), dtype)
    v[~band] = 0
    A = np.ascontiguousarray(v[np.ix_(q, q)])
    return {"A": A, "B": B, "M": n, "K": n, "N": N, "w": w, "q": q, "dtype": dtype}


def _unique_sorted_rows(rng, lengths: np.ndarray, K: int):
    """Per row, ``lengths[r]`` distinct columns uniform on [0, K), ascending."""
    M = lengths.shape[0]
    row_ptr = np.zeros(M + 1, dtype=np.int64)
    np.cumsum(lengths, out=row_ptr[1:])
    nnz = int(row_ptr[-1])
    rows = np.repeat(np.arange(M, dtype=np.int64), lengths)
    cols = rng.integers(0, K, size=nnz, dtype=np.int64)
    while True:
        order = np.lexsort((cols, rows))
        rs, cs = rows[order], cols[order]
        dup = np.zeros(nnz, dtype=bool)
        if nnz > 1:
            dup[1:] = (rs[1:] == rs[:-1]) & (cs[1:] == cs[:-1])
        rows, cols = rs, cs
        nd = int(dup.sum())
        if nd == 0:
            break
        cols = cols.copy()
        cols[dup] = rng.integers(0, K, size=nd, dtype=np.int64)
    return row_ptr, cols


def csr_lognormal_problem(M: int, K: int, N: int, seed: int, mean: float = 16.0,
                          sigma: float = 1.5, clip: int = 4096, dtype: str = F16) -> dict:
    """CSR A with log-normal row lengths (mean ``mean``), values N(0,1); B (K x N)."""
    rng = np.random.default_rng(seed)
    mu = np.log(mean) - sigma * sigma / 2.0
    X = rng.lognormal(mean=mu, sigma=sigma, size=M)
    L = np.clip(np.rint(X), 1, min(clip, K)).astype(np.int64)
    row_ptr, cols = _unique_sorted_rows(rng, L, K)
    val = normal_bits(rng, (cols.shape[0],), dtype)
    B = normal_bits(rng, (K, N), dtype)
    return {"row_ptr": row_ptr.astype(np.int32), "col": cols.astype(np.int32), "val": val,
            "B": B, "M": M, "K": K, "N": N, "dtype": dtype}


def csr_window_clustered_problem(M: int, K: int, N: int, seed: int, h: int = 16, pool: int = 64,
                                 per_row: int = 16, dtype: str = F16) -> dict:
    """CSR A whose rows, h at a time, share a column pool: each window of h
    consecutive rows has ``pool`` distinct columns drawn uniformly from [0, K), and
    each row takes ``per_row`` distinct columns of its window's pool (ascending);
    values N(0,1), B (K x N) N(0,1).  A window's distinct columns then hold about
    h * per_row / pool nonzeros each (the column reuse of matrices with locality,
    such as meshes or graphs after a bandwidth-reducing reordering)."""
    assert per_row <= pool <= K
    rng = np.random.default_rng(seed)
    nw = (M + h - 1) // h
    cols = np.empty((M, per_row), dtype=np.int64)
    for w in range(nw):
        r0, r1 = w * h, min(M, (w + 1) * h)
        pw = rng.choice(K, size=pool, replace=False)
        pick = np.argsort(rng.random((r1 - r0, pool)), axis=1)[:, :per_row]
        cols[r0:r1] = np.sort(pw[pick], axis=1)
    row_ptr = np.arange(0, M * per_row + 1, per_row, dtype=np.int64)
    val = normal_bits(rng, (M * per_row,), dtype)
    B = normal_bits(rng, (K, N), dtype)
    return {"row_ptr": row_ptr.astype(np.int32), "col": cols.reshape(-1).astype(np.int32), "val": val,
            "B": B, "M": M, "K": K, "N": N, "dtype": dtype}


def tvw_problem(M: int, K: int, N: int, tile_rows: int, keep, seed: int,
                dtype: str = F16) -> dict:
    """Dense A (bits) in tile-vector-wise form plus the per-tile kept columns.

    ``keep`` is the kept-column count of every tile, or one count per tile."""
    rng = np.random.default_rng(seed)
    nt = (M + tile_rows - 1) // tile_rows
    keeps = [int(keep)] * nt if np.isscalar(keep) else [int(k) for k in keep]
    assert len(keeps) == nt and all(k % 4 == 0 and 0 <= k <= K for k in keeps)
    pairs = np.array([(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)], dtype=np.int64)
    tile_ptr = np.zeros(nt + 1, dtype=np.int64)
    np.cumsum(keeps, out=tile_ptr[1:])
    cols = np.zeros(int(tile_ptr[-1]), dtype=np.int64)
    A = np.zeros((M, K), dtype=np.uint16)
    for t in range(nt):
        keep = keeps[t]
        G = keep // 4
        kc = np.sort(rng.choice(K, size=keep, replace=False))
        cols[tile_ptr[t]:tile_ptr[t + 1]] = kc
        r0, r1 = t * tile_rows, min(M, (t + 1) * tile_rows)
        sel = pairs[rng.integers(0, 6, size=(r1 - r0, G))]
        kidx = sel + (np.arange(G, dtype=np.int64) * 4)[None, :, None]
        v = normal_bits(rng, (r1 - r0, G, 2), dtype)
        rows = np.arange(r0, r1, dtype=np.int64)[:, None, None]
        A[np.broadcast_to(rows, kidx.shape), kc[kidx]] = v
    B = normal_bits(rng, (K, N), dtype)
    return {"A": A, "B": B, "tile_ptr": tile_ptr.astype(np.int32), "cols": cols.astype(np.int32),
            "M": M, "K": K, "N": N, "tile_rows": tile_rows, "dtype": dtype}


# The five measured workloads.  ``nnzb`` for the block-sparse ones is the exact
# count round((1 - sparsity) * number_of_blocks).
CONFIGS = {
    "bcsr_tiny": dict(kind="bcsr", M=256, K=256, N=64, bh=16, bw=16, nnzb=64, seed=1,
                      dtype=BF16, std=1.0),
    "mask24_int8": dict(kind="24", M=8192, K=8192, N=4096, seed=2),
    "mask24_f16": dict(kind="24f", M=8192, K=8192, N=4096, seed=6, dtype=F16),
    # fp8 (E4M3) 2:4 at the same shape: A and B N(0,1) rounded to E4M3
    "mask24_e4m3": dict(kind="24f", M=8192, K=8192, N=4096, seed=11, dtype=E4M3),
    "prune24_f16": dict(kind="prune24", M=8192, K=8192, N=0, seed=7, dtype=F16),
    "prune_tvw_f16": dict(kind="prunetvw", M=4096, K=4096, N=0, tile_rows=128, keep=2048, seed=8, dtype=F16),
    "wcsr_lognormal": dict(kind="wcsr", M=65536, K=65536, N=128, seed=3, mean=16.0,
                           sigma=1.5, clip=4096, dtype=F16),
    # row windows with column reuse: every 16-row window's rows take 64 of a shared pool of 128 columns
    "wcsr_clustered": dict(kind="wcsrc", M=65536, K=65536, N=128, seed=12, h=16, pool=128, per_row=64, dtype=F16),
    "bcsr_llm": dict(kind="bcsr", M=18944, K=3584, N=65536, bh=64, bw=64, nnzb=1658, seed=4,
                     dtype=BF16, std=0.02),
    "tvw": dict(kind="tvw", M=4096, K=4096, N=4096, tile_rows=128, keep=2048, seed=5, dtype=F16),
    # SDDMM on the row-window workload's pattern: A, Bt 65536 x 128 (a sparse attention score)
    "sddmm_lognormal": dict(kind="sddmm", M=65536, K=65536, N=0, inner=128, seed=3, mean=16.0, sigma=1.5,
                            clip=4096, dtype=F16),
    # the same pattern with quantized operands: A, Bt 65536 x 128 int8, uniform over [-128, 127]
    "sddmm_lognormal_i8": dict(kind="sddmm", M=65536, K=65536, N=0, inner=128, seed=3, mean=16.0, sigma=1.5,
                               clip=4096, dtype=I8),
    # a scrambled band (half-width 48) before and after RCM, 64 x 64 blocks
    "bcsr_rcm": dict(kind="rcm", M=16384, K=16384, N=2048, w=48, bh=64, bw=64, seed=10, dtype=F16),
    # 6:8 on a Qwen2.5-7B-sized FFN projection (18944 x 3584), 8192 tokens
    "slide68_f16": dict(kind="slide", M=18944, K=3584, N=8192, n=4, seed=9, dtype=F16),
}


def config_problem(name: str, **overrides) -> dict:
    """Generate the named workload (keyword overrides shrink it for tests)."""
    c = dict(CONFIGS[name])
    c.update(overrides)
    kind = c.pop("kind")
    if kind == "bcsr":
        return bcsr_problem(c["M"], c["K"], c["N"], c["bh"], c["bw"], c["nnzb"], c["seed"],
                            c.get("dtype", BF16), c.get("std", 1.0))
    if kind == "24":
        return mask24_problem(c["M"], c["K"], c["N"], c["seed"])
    if kind == "24f":
        return mask24_float_problem(c["M"], c["K"], c["N"], c["seed"], c.get("dtype", F16))
    if kind == "wcsr":
        return csr_lognormal_problem(c["M"], c["K"], c["N"], c["seed"], c.get("mean", 16.0),
                                     c.get("sigma", 1.5), c.get("clip", 4096), c.get("dtype", F16))
    if kind == "wcsrc":
        return csr_window_clustered_problem(c["M"], c["K"], c["N"], c["seed"], c.get("h", 16), c.get("pool", 64),
                                            c.get("per_row", 16), c.get("dtype", F16))
    if kind == "tvw":
        return tvw_problem(c["M"], c["K"], c["N"], c["tile_rows"], c["keep"], c["seed"],
                           c.get("dtype", F16))
    if kind == "sddmm":  # the CSR pattern of csr_lognormal_problem, then A (M x inner) and Bt (K x inner)
        dt = c.get("dtype", F16)
        # int8 operands share the fp16 workload's pattern (same seed, same draws)
        p = csr_lognormal_problem(c["M"], c["K"], 1, c["seed"], c.get("mean", 16.0), c.get("sigma", 1.5),
                                  c.get("clip", 4096), F16 if dt == I8 else dt)
        rng = np.random.default_rng(c["seed"] + 1000)
        if dt == I8:
            p["A"] = rng.integers(-128, 128, size=(c["M"], c["inner"]), dtype=np.int8)
            p["Bt"] = rng.integers(-128, 128, size=(c["K"], c["inner"]), dtype=np.int8)
            p["dtype"] = I8
        else:
            p["A"] = normal_bits(rng, (c["M"], c["inner"]), dt)
            p["Bt"] = normal_bits(rng, (c["K"], c["inner"]), dt)
        del p["B"]
        return p
    if kind == "rcm":
        return banded_scrambled_problem(c["M"], c["w"], c["N"], c["seed"], c.get("dtype", F16))
    if kind == "slide":
        return slide_problem(c["M"], c["K"], c["N"], c["n"], c["seed"], c.get("dtype", F16))
    if kind in ("prune24", "prunetvw"):  # a dense matrix to prune (into 2:4, or into TVW given kept columns)
        rng = np.random.default_rng(c["seed"])
        return {"A": normal_bits(rng, (c["M"], c["K"]), c.get("dtype", F16)), "M": c["M"], "K": c["K"],
                "dtype": c.get("dtype", F16)}
    raise ValueError(kind)
