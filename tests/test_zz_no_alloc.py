"""The forward entry point that allocates nothing (cce_forward_noalloc).

It serves callers that cannot allocate device memory where they need the
loss (inside a graph capture that must not allocate, or under a runtime that
owns all device memory through its own pool): it uses a fixed scratch array
the library declares in device memory instead of a caller workspace.  This
file is collected last so that, if it fails, a run stopping at the first
failure has already run every other test.  It passes alone in a fresh
process and after the other tests: nothing here depends on earlier state.
"""
import ctypes

import numpy as np
import pytest
import torch

import cce_workloads as W
import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests.conftest import build_library
    build_library()
    from linear_cross_entropy_gb300 import _lib
    return _lib.load()


def _noalloc(lib, E, C, x, reduction):
    N, D = E.shape
    V = C.shape[0]
    red = {"none": 0, "sum": 1, "mean": 2}[reduction]
    loss = torch.empty(N if red == 0 else 1, dtype=torch.float32, device="cuda")
    lse = torch.empty(N, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    vp = ctypes.c_void_p
    st = lib.cce_forward_noalloc(vp(E.data_ptr()), vp(C.data_ptr()), vp(x.data_ptr()), N, D, V, -100, red,
                                 vp(loss.data_ptr()), vp(lse.data_ptr()), vp(err.data_ptr()),
                                 vp(torch.cuda.current_stream().cuda_stream))
    return st, loss, lse, err


def test_noalloc_forward_matches_forward_on_two_calls_in_a_row(lib):
    import linear_cross_entropy_gb300 as cce
    from tests.gpu_util import TOL_LSE, to_device
    cases = [(W.small("na1", 1000, 256, 5000, reduction="mean"), "mean"),
             (W.small("na2", 300, 128, 3001, reduction="none"), "none")]
    for w, reduction in cases:  # two calls in a row, different sizes, sharing the scratch
        E, C, x = to_device(*W.make_inputs(w))
        st, loss, lse, err = _noalloc(lib, E, C, x, reduction)
        assert st == 0, lib.cce_status_string(st)
        ref_loss, ref_lse = cce.cce_forward(E, C, x, -100, reduction)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        lse_ref = ref_lse.double()
        assert float(((lse.double() - lse_ref).abs() / lse_ref.abs()).max()) <= TOL_LSE
        if reduction == "none":
            bound = TOL_LSE * lse_ref.abs()
            assert bool(((loss.double() - ref_loss.double()).abs() <= bound).all())
        else:
            assert abs(loss.item() - ref_loss.item()) <= TOL_LSE * abs(ref_loss.item())
        # and against the fp64 oracle directly
        E_bits, C_bits, xh = W.make_inputs(w)
        Ef, Cf = O.from_bits(E_bits, C_bits)
        f = O.forward(Ef, Cf, xh, reduction=reduction)
        got_lse = lse.double().cpu().numpy()
        assert np.max(np.abs(got_lse - f["lse"]) / np.abs(f["lse"])) <= TOL_LSE
        if reduction == "none":
            assert np.all(np.abs(loss.double().cpu().numpy() - f["loss_rows"]) <= TOL_LSE * np.abs(f["lse"]))
        else:
            assert abs(loss.item() - f["loss"]) <= TOL_LSE * abs(f["loss"])


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    import linear_cross_entropy_gb300 as cce
    E = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(8, dtype=torch.int64, device="cuda")
    # shapes whose workspace exceeds the fixed scratch are refused before any launch
    N, V = 1 << 22, 1 << 20
    assert cce.forward_workspace_bytes(N, 64, V) > 16 << 20
    vp = ctypes.c_void_p
    out = torch.zeros(N, dtype=torch.float32, device="cuda")
    st = lib.cce_forward_noalloc(vp(E.data_ptr()), vp(C.data_ptr()), vp(x.data_ptr()), N, 64, V, -100, 1,
                                 vp(out.data_ptr()), vp(out.data_ptr()), vp(0),
                                 vp(torch.cuda.current_stream().cuda_stream))
    assert st == 5  # CCE_ERR_WORKSPACE
    torch.cuda.synchronize()
