"""Failure detection on the GPU without a fault: a bounded wait gives up and
reports, and out-of-range indices in a format are skipped and reported by the
kernels' own bounds checks.  The context stays usable afterwards."""
import numpy as np
import pytest

import oracle
import spmm_inputs as gen
from tests.gpu_util import assert_close, dev, dev_half, need_gpu, padded_b

pytestmark = pytest.mark.gpu

TIMEOUT, INDEX = 1, 2  # SPMM_DEVERR_TIMEOUT, SPMM_DEVERR_INDEX


def test_bounded_wait_gives_up_and_reports():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    spmm.last_device_error()                        # start clean
    spmm.selftest_timeout(2_000_000)                # a 2 ms wait on a barrier nobody arrives on
    assert spmm.last_device_error() & TIMEOUT
    assert spmm.last_device_error() == 0            # reading clears the word
    # the context still runs kernels correctly
    p = gen.config_problem("bcsr_tiny")
    F = spmm.build_bcsr(dev_half(p["A"], "bf16"), 16, 16)
    C = spmm.spmm_bcsr(F, dev_half(p["B"], "bf16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() == 0
    ref = oracle.bcsr_spmm(oracle.bcsr_build(p["A"], 16, 16, "bf16"), p["B"])
    assert_close(C.cpu().numpy(), ref, "bcsr after timeout test")


def test_tvw_kept_column_out_of_range_is_skipped_and_reported():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.tvw_problem(256, 512, 136, 128, 256, seed=21, dtype="f16")
    F = spmm.spmm_build_tvw(dev_half(p["A"], "f16"), 128, dev(p["tile_ptr"]), dev(p["cols"]), Kp=256)
    O = oracle.tvw_build(p["A"], 128, p["tile_ptr"], p["cols"], "f16", Kp=256)
    spmm.last_device_error()
    F.cols[3] = p["K"] + 7                          # tile 0's fourth kept column points past B
    C = spmm.spmm_tvw(F, padded_b(p["B"], "f16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() & INDEX
    got = C.cpu().numpy()
    assert np.isfinite(got).all()
    # tile 1 does not use the bad index and is unaffected
    assert_close(got[128:], oracle.tvw_spmm(O, p["B"])[128:], "tvw other tile")


def test_wcsr_slot_out_of_range_is_skipped_and_reported():
    torch = need_gpu()
    import sparse_dense_matrix_spmm_gb300 as spmm
    p = gen.csr_lognormal_problem(256, 3000, 128, seed=22, mean=12.0, sigma=1.5, clip=1024)
    csr = spmm.CSR(p["M"], p["K"], int(p["row_ptr"][-1]), torch.float16, dev(p["row_ptr"]), dev(p["col"]),
                   dev_half(p["val"], "f16"))
    W = spmm.build_wcsr(csr, 16, 32)
    O = oracle.wcsr_build(p["M"], p["K"], p["row_ptr"], p["col"], p["val"], "f16", h=16, S=32)
    spmm.last_device_error()
    W.slot[0] = 1 << 30                             # first entry of window 0 points past its column list
    C = spmm.spmm_wcsr(W, padded_b(p["B"], "f16"))
    torch.cuda.synchronize()
    assert spmm.last_device_error() & INDEX
    got = C.cpu().numpy()
    assert np.isfinite(got).all()
    assert_close(got[16:], oracle.wcsr_spmm(O, p["B"])[16:], "wcsr other windows")
