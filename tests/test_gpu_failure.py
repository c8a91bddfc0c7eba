"""Failure paths on the GPU, made without a fault: a pipeline wait that runs
out reports a status and leaves the context usable."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests.conftest import build_library
    build_library()
    from linear_cross_entropy_gb300 import _lib
    return _lib.load()


def test_bounded_wait_times_out_with_status(lib):
    import linear_cross_entropy_gb300 as cce
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = lib.cce_selftest_wait_timeout(ctypes.c_void_p(err.data_ptr()), 20000,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) & cce.DEVERR_TIMEOUT
    # the context is still usable
    E = torch.randn(64, 64, device="cuda").bfloat16()
    C = torch.randn(300, 64, device="cuda").bfloat16() * 0.1
    x = torch.randint(0, 300, (64,), device="cuda")
    loss, lse = cce.cce_forward(E, C, x)
    assert torch.isfinite(loss) and torch.isfinite(lse).all()


def test_selftest_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    assert lib.cce_selftest_wait_timeout(vp(0), 100, vp(0)) == 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.cce_selftest_wait_timeout(vp(err.data_ptr()), 0, vp(0)) == 4
