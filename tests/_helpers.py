"""Small shared helpers for the tests (no SpMM arithmetic here)."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def to_bits(x, dtype):
    """Exact small decimals -> bf16 / fp16 / fp8 bit patterns (or int8)."""
    from spmm_inputs import round_f32_to_bf16_bits, round_f32_to_fp8_bits
    a = np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return round_f32_to_bf16_bits(a)
    if dtype == "f16":
        return a.astype(np.float16).view(np.uint16)
    if dtype in ("e4m3", "e5m2"):
        return round_f32_to_fp8_bits(a, dtype)
    return a.astype(np.int8)


def bits_to_f64(bits, dtype):
    """Reference decode through numpy / torch (independent of the oracle's decoder)."""
    b = np.asarray(bits)
    if dtype == "bf16":
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "f16":
        return b.view(np.float16).astype(np.float64)
    if dtype in ("e4m3", "e5m2"):
        import torch
        fd = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
        t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(fd)
        return t.to(torch.float64).numpy()
    return b.astype(np.float64)
