"""The failure path of the library's bounded waits, on the GPU without a
fault: a wait on an mbarrier that nothing completes expires after its
iteration limit, the kernel returns, W4A16_DEVERR_TIMEOUT is set in the
device error word (read and cleared through the C ABI), and the context
stays usable -- the next GEMV is checked against the oracle."""
import numpy as np
import pytest
import torch

from w4a16_int4_weight_gemv_gb300 import synth

from .test_gpu_parity import check_close, dense_dev, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_int4_weight_gemv_gb300 import build_ext
    build_ext.build()
    from w4a16_int4_weight_gemv_gb300 import binding
    binding.w4a16_device_error(clear=True)
    return binding


def test_completed_wait_raises_nothing(w):
    w.w4a16_wait_selftest(64, arrive=True)
    assert w.w4a16_device_error(clear=True) == 0


def test_expired_wait_sets_timeout_and_the_context_stays_usable(w, oracle):
    w.w4a16_wait_selftest(64, arrive=False)
    assert w.w4a16_device_error(clear=True) == w.DEVERR_TIMEOUT
    assert w.w4a16_device_error(clear=True) == 0  # cleared
    p = synth.dense_problem(1, 256, 1024, 128, "uniform6to10", seed=9900)
    y = w.w4a16_gemv(*dense_dev(p), 128, out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_close(host_f64(y), oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128), "after timeout")
    assert w.w4a16_device_error(clear=True) == 0


def test_wait_limit_is_validated(w):
    for bad in (0, 8193):
        with pytest.raises(w.W4A16Error) as ei:
            w.w4a16_wait_selftest(bad, arrive=True)
        assert ei.value.status == w.Status.ERR_SHAPE
