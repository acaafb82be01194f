"""Helpers for the GPU parity tests (marshalling only; no SpMM arithmetic)."""
import numpy as np
import pytest

TOL_ABS, TOL_REL = 1e-2, 1e-2   # |gpu - oracle| <= 1e-2 + 1e-2 * |oracle| for bf16/fp16 inputs


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def dev(bits):
    import torch
    if bits.dtype == np.int8:
        return torch.from_numpy(np.ascontiguousarray(bits)).cuda()
    if bits.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(bits)).cuda()


def dev_half(bits, dtype):
    import torch
    t = dev(bits)
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


def dev_fp8(bits, dtype):
    """uint8 fp8 bit patterns -> a device tensor of torch's float8 type."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).cuda()
    return t.view(torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2)


def host_bits(t):
    """Device tensor -> numpy raw bits (uint16 for 16-bit types, uint8 for fp8)."""
    import torch
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return t.view(torch.uint8).cpu().numpy()
    return t.cpu().numpy()


def padded_b8(bits, dtype):
    """fp8 B on the device with its row pitch rounded up to 16 bytes, as a K x N view."""
    import torch
    K, N = bits.shape
    ld = -(-N // 16) * 16
    full = torch.zeros((K, ld), dtype=torch.uint8, device="cuda")
    full[:, :N] = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).cuda()
    full = full.view(torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2)
    return full[:, :N]


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {tuple(i)} "
                             f"gpu={got[tuple(i)]} oracle={ref[tuple(i)]}")


def padded_b(bits, dtype):
    """B on the device with its row pitch rounded up to 8 elements (16 bytes), as a K x N view."""
    import torch
    K, N = bits.shape
    ld = -(-N // 8) * 8
    full = torch.zeros((K, ld), dtype=torch.int16, device="cuda")
    full[:, :N] = dev(bits)
    full = full.view(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return full[:, :N]
