"""GPU parity at the edges of the shapes and for combinations of options.

Degenerate shapes: a one-entry vocabulary (every loss is 0 and every
gradient exactly 0: softmax = onehot), the smallest D the TMA row pitch
allows (8), D not a multiple of 32, a vocabulary smaller than one tile.
Both the two calls and the single call are checked against the fp64 oracle.

Combinations: vocabulary sorting with softcapping and with per-output
filtering; the single call with per-output filtering and with softcapping
under the filter; the forward that skips ignored rows feeding a sorted
backward.
"""
import numpy as np
import pytest
import torch

import cce_workloads as W
import oracle as O
from tests.gpu_util import TOL_GRAD, TOL_GRAD_FILTERED, TOL_LSE, bf16_to_f64, rel_fro, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests.conftest import build_library
    build_library()


def _loss_bound(lse, x, reduction):
    """The loss error allowed: each row's loss is LSE_i - target_i, so its
    rounding error scales with |LSE_i| (1e-5 relative), whatever the loss --
    a one-entry vocabulary makes every loss 0 by cancellation."""
    part = x != -100
    s = float(np.abs(lse[part]).sum())
    return TOL_LSE * (s / max(int(part.sum()), 1) if reduction == "mean" else s)


def _grads_ok(dE, dC, ref_dE, ref_dC, tol, zero_case=None):
    """Relative Frobenius error; when the exact gradient is 0 (a one-entry
    vocabulary), zero_case = (Ef, Cf, w, lse) bounds the absolute values
    instead: G = exp(a - LSE) - 1 is then only the LSE's rounding, at most
    1e-5 |LSE| per entry, carried through the two contractions."""
    gE, gC = bf16_to_f64(dE), bf16_to_f64(dC)
    if np.linalg.norm(ref_dE) == 0.0 and np.linalg.norm(ref_dC) == 0.0:
        Ef, Cf, w, lse = zero_case
        g_max = 2 * TOL_LSE * float(np.abs(lse).max())
        assert np.abs(gE).max() <= g_max * float(np.abs(w).max()) * float(np.abs(Cf).sum(axis=0).max())
        assert np.abs(gC).max() <= g_max * float((np.abs(w)[:, None] * np.abs(Ef)).sum(axis=0).max())
        return
    assert rel_fro(gE, ref_dE) <= tol and rel_fro(gC, ref_dC) <= tol, (rel_fro(gE, ref_dE), rel_fro(gC, ref_dC))


SHAPES = [(5, 8, 1), (300, 8, 3), (7, 40, 100), (260, 40, 1000), (129, 72, 200)]


@pytest.mark.parametrize("N,D,V", SHAPES)
def test_edge_shapes_two_calls(N, D, V):
    import linear_cross_entropy_gb300 as cce
    w = W.small("edge", N, D, V)
    E_bits, C_bits, x = W.make_inputs(w)
    E, C, xt = to_device(E_bits, C_bits, x)
    loss, lse = cce.cce_forward(E, C, xt, reduction="mean")
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    dE, dC = cce.cce_backward(E, C, xt, lse, g, reduction="mean", filter_eps=0.0)
    torch.cuda.synchronize()
    Ef, Cf = O.from_bits(E_bits, C_bits)
    f = O.forward(Ef, Cf, x, reduction="mean")
    err = np.abs(lse.double().cpu().numpy() - f["lse"]) / np.maximum(np.abs(f["lse"]), 1e-30)
    assert err.max() <= TOL_LSE
    r = float(f["loss"])
    assert abs(loss.item() - r) <= max(TOL_LSE * abs(r), _loss_bound(f["lse"], x, "mean"))
    wts = O.row_weights(x, -100, "mean", 1.0, f["count"])
    rdE, rdC = O.backward(Ef, Cf, x, f["lse"], wts)
    _grads_ok(dE, dC, rdE, rdC, TOL_GRAD, (Ef, Cf, wts, f["lse"]))


@pytest.mark.parametrize("N,D,V", SHAPES)
def test_edge_shapes_single_call(N, D, V):
    import linear_cross_entropy_gb300 as cce
    w = W.small("edge", N, D, V)
    E_bits, C_bits, x = W.make_inputs(w)
    E, C, xt = to_device(E_bits, C_bits, x)
    loss, lse, dE, dC = cce.cce_loss_and_grad(E, C, xt, reduction="sum", filter_eps=0.0)
    torch.cuda.synchronize()
    Ef, Cf = O.from_bits(E_bits, C_bits)
    ref = O.loss_and_grad(Ef, Cf, x, reduction="sum")
    part = x != -100
    got_lse = lse.double().cpu().numpy()
    assert np.all(np.abs(got_lse[part] - ref["lse"][part]) <= TOL_LSE * np.abs(ref["lse"][part]))
    assert abs(loss.item() - ref["loss"]) <= max(TOL_LSE * abs(ref["loss"]), _loss_bound(ref["lse"], x, "sum"))
    _grads_ok(dE, dC, ref["dE"], ref["dC"], TOL_GRAD, (Ef, Cf, O.row_weights(x, -100, "sum", 1.0), ref["lse"]))


def _freq(N=1024, D=128, V=9000, scatter=True):
    return W.frequent_token_inputs(N, D, V, n_freq=256, scatter=scatter, unigram=8.0 if scatter else 0.0)


def _sorted_oracle(E_bits, C_bits, x, softcap=0.0, filter_dE=True, filter_dC=True, reduction="mean"):
    Ef, Cf = O.from_bits(E_bits, C_bits)
    f = O.forward(Ef, Cf, x, reduction=reduction, softcap=softcap)
    w = O.row_weights(x, -100, reduction, 1.0, f["count"])
    perm = O.vocab_order(O.vocab_logit_sums(Ef, Cf, x)[0])
    dE, dC, keep = O.backward_filtered(Ef, Cf, x, f["lse"], w, 128, 128, O.FILTER_EPS, filter_dE=filter_dE,
                                       filter_dC=filter_dC, softcap=softcap, compact_ignored=True, vocab_perm=perm)
    return dE, dC, keep


def _two_calls(E_bits, C_bits, x, *, softcap=0.0, outputs="both", sort=True, skip=False, reduction="mean"):
    import linear_cross_entropy_gb300 as cce
    E, C, xt = to_device(E_bits, C_bits, x)
    loss, lse = cce.cce_forward(E, C, xt, reduction=reduction, softcap=softcap, skip_ignored=skip)
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    dE, dC, st = cce.cce_backward(E, C, xt, lse, g, reduction=reduction, softcap=softcap, filter_outputs=outputs,
                                  vocab_sort=sort, stats=True)
    torch.cuda.synchronize()
    return dE, dC, st


def test_sorted_with_softcap():
    E_bits, C_bits, x = _freq()
    dE, dC, st = _two_calls(E_bits, C_bits, x, softcap=20.0)
    rdE, rdC, keep = _sorted_oracle(E_bits, C_bits, x, softcap=20.0)
    _grads_ok(dE, dC, rdE, rdC, TOL_GRAD_FILTERED)
    assert abs(st["skipped"] - int((~keep).sum())) <= max(1, keep.size // 200)


@pytest.mark.parametrize("outputs,fde,fdc", [("dE", True, False), ("dC", False, True)])
def test_sorted_with_per_output_filtering(outputs, fde, fdc):
    E_bits, C_bits, x = _freq()
    dE, dC, st = _two_calls(E_bits, C_bits, x, outputs=outputs)
    rdE, rdC, keep = _sorted_oracle(E_bits, C_bits, x, filter_dE=fde, filter_dC=fdc)
    _grads_ok(dE, dC, rdE, rdC, TOL_GRAD_FILTERED)


def test_skipping_forward_feeds_a_sorted_backward():
    E_bits, C_bits, x = _freq()
    dE, dC, st = _two_calls(E_bits, C_bits, x, skip=True, reduction="sum")
    rdE, rdC, keep = _sorted_oracle(E_bits, C_bits, x, reduction="sum")
    _grads_ok(dE, dC, rdE, rdC, TOL_GRAD_FILTERED)


@pytest.mark.parametrize("outputs,fde,fdc,softcap", [("dE", True, False, 0.0), ("dC", False, True, 0.0),
                                                      ("both", True, True, 20.0)])
def test_single_call_filter_options(outputs, fde, fdc, softcap):
    import linear_cross_entropy_gb300 as cce
    E_bits, C_bits, x = _freq(scatter=False)
    E, C, xt = to_device(E_bits, C_bits, x)
    loss, lse, dE, dC, st = cce.cce_loss_and_grad(E, C, xt, reduction="mean", filter_outputs=outputs,
                                                  softcap=softcap, stats=True)
    torch.cuda.synchronize()
    Ef, Cf = O.from_bits(E_bits, C_bits)
    ref = O.loss_and_grad(Ef, Cf, x, reduction="mean", softcap=softcap, filter_eps=O.FILTER_EPS, filter_dE=fde,
                          filter_dC=fdc)
    assert abs(loss.item() - ref["loss"]) <= TOL_LSE * abs(ref["loss"])
    _grads_ok(dE, dC, ref["dE"], ref["dC"], TOL_GRAD_FILTERED)
    keep = ref["keep"]
    assert abs(st["skipped"] - int((~keep).sum())) <= max(1, keep.size // 200)


@pytest.mark.parametrize("softcap,sort", [(20.0, False), (0.0, True), (20.0, True)])
def test_many_blocks_cta_pairs_with_softcap_and_sorting(softcap, sort):
    """65 token blocks (an odd count): the forward and the recompute run as
    CTA pairs, here in their softcapped instantiations and over the sorted
    vocabulary, against the oracle's filtered gradients (sorted order when
    sorting)."""
    E_bits, C_bits, x = W.frequent_token_inputs(65 * 128, 64, 4000, n_freq=256, scatter=True, unigram=8.0)
    dE, dC, st = _two_calls(E_bits, C_bits, x, softcap=softcap, sort=sort)
    if sort:
        rdE, rdC, keep = _sorted_oracle(E_bits, C_bits, x, softcap=softcap)
    else:
        Ef, Cf = O.from_bits(E_bits, C_bits)
        f = O.forward(Ef, Cf, x, reduction="mean", softcap=softcap)
        w = O.row_weights(x, -100, "mean", 1.0, f["count"])
        rdE, rdC, keep = O.backward_filtered(Ef, Cf, x, f["lse"], w, 128, 128, O.FILTER_EPS, softcap=softcap,
                                             compact_ignored=True)
    _grads_ok(dE, dC, rdE, rdC, TOL_GRAD_FILTERED)
    assert abs(st["skipped"] - int((~keep).sum())) <= max(1, keep.size // 200)
