"""Failure detection without a GPU fault: a bounded in-kernel wait on a flag
that nothing sets gives up after its limit, the device error word reports
LBQ_ERR_TIMEOUT, and the context stays usable for the next GEMV."""
import time

import numpy as np
import pytest

from oracle import lbq_oracle as O

from gpu_util import assert_close, to_dev

torch = pytest.importorskip("torch")


def test_selftest_rejects_bad_limit_without_gpu(lbq):
    assert lbq.lib().lbq_selftest_wait_timeout(0, None) == 2          # LBQ_ERR_SHAPE, before any CUDA call
    assert lbq.lib().lbq_selftest_wait_timeout(5000001, None) == 2


@pytest.mark.gpu
def test_bounded_wait_times_out_and_context_survives(lbq):
    assert lbq.device_error() == 0
    t0 = time.perf_counter()
    lbq.selftest_wait_timeout(50000)                                  # 50 ms limit
    assert lbq.device_error() == 8                                    # LBQ_ERR_TIMEOUT
    dt = time.perf_counter() - t0
    assert 0.04 < dt < 5.0
    assert lbq.device_error() == 0                                    # cleared
    # the context is intact: a GEMV right after gives the oracle's answer
    rng = np.random.default_rng(3)
    W = (rng.standard_normal((40, 256)) * 0.02).astype(np.float32)
    x = rng.standard_normal(256).astype(np.float16)
    y = torch.empty(40, dtype=torch.float32, device="cuda:0")
    lbq.gemv_w4a16(to_dev(lbq.pack_w4(W)), 40, 256, 0, to_dev(x), y)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    assert_close(y.cpu().numpy(), O.gemv(O.pack_w4(W), x), what="after timeout")
