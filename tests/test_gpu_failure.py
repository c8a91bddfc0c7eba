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


def test_cta_pair_abort_ends_with_status(lib):
    """The CTA-pair handshake with one arrive held back: both CTAs' bounded
    waits run out, they meet at the final cluster barrier and the kernel
    returns with CCE_DEVERR_TIMEOUT; without the hold the handshake completes
    cleanly; afterwards a forward that runs as CTA pairs still matches the
    oracle."""
    import numpy as np

    import cce_workloads as W
    import linear_cross_entropy_gb300 as cce
    import oracle as O
    from tests.gpu_util import TOL_LSE, to_device
    vp = ctypes.c_void_p
    stream = vp(torch.cuda.current_stream().cuda_stream)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.cce_selftest_pair_timeout(vp(err.data_ptr()), 20000, 1, stream) == 0
    torch.cuda.synchronize()
    assert int(err.item()) & cce.DEVERR_TIMEOUT
    err.zero_()
    assert lib.cce_selftest_pair_timeout(vp(err.data_ptr()), 20000, 0, stream) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert lib.cce_selftest_pair_timeout(vp(err.data_ptr()), 20000, 2, stream) == 4
    assert lib.cce_selftest_pair_timeout(vp(0), 20000, 1, stream) == 1
    # the context is usable and the pair kernels still give the oracle's result
    w = W.small("pt", 3 * 128 + 5, 64, 2000)
    E_bits, C_bits, x = W.make_inputs(w)
    E, C, xt = to_device(E_bits, C_bits, x)
    loss, lse = cce.cce_forward(E, C, xt)
    Ef, Cf = O.from_bits(E_bits, C_bits)
    f = O.forward(Ef, Cf, x, reduction="mean")
    assert np.max(np.abs(lse.double().cpu().numpy() - f["lse"]) / np.abs(f["lse"])) <= TOL_LSE
    assert abs(loss.item() - f["loss"]) <= TOL_LSE * abs(f["loss"])
