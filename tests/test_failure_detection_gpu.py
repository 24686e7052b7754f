"""Device-side failure detection without a GPU fault.

Every barrier wait in the library is bounded.  bi_selftest_wait_timeout runs
the same wait routine on an mbarrier that nothing arrives on, with a short
limit: the wait must give up, the kernel must record BI_ERR_DEVICE_TIMEOUT and
exit normally, and the context must stay usable afterwards.
"""
import time

import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
import oracle
from invariant_bi_rmsnorm_gb300 import inputs
from tests._util import bits, ulp_distance

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    bi.get_device_error()  # start clean
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    bi.selftest_wait_timeout(20000)  # 20 ms
    with pytest.raises(bi.BiError, match="DEVICE_TIMEOUT"):
        bi.get_device_error()
    elapsed = time.perf_counter() - t0
    assert 0.015 <= elapsed < 2.0, elapsed
    # the word was cleared and the context still runs kernels correctly
    bi.get_device_error()
    x = inputs.rmsnorm_rows(4, 4096, seed=600)
    w = inputs.rmsnorm_weight(4096, seed=601)
    y = bits(bi.rmsnorm(x.cuda(), w.cuda(), 1e-6))
    assert ulp_distance(y, oracle.round_bf16(oracle.rmsnorm(x, w, 1e-6))).max() <= 2
    bi.get_device_error()


def test_selftest_rejects_bad_limits():
    for bad in (0, -5, 2000001):
        with pytest.raises(bi.BiError, match="INVALID_ARG"):
            bi.selftest_wait_timeout(bad)
