"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these checks re-types the oracle's own formulas: each compares it
with an independent fact -- a closed form, a finite difference of the loss,
a library routine for the same definition (torch cross_entropy on
materialised logits), an invariant (normalisation, G row sums, permutation)
or the pages' pigeonhole bound and threshold tie.  The last group plants
mistakes in a copy of the oracle and checks that some pin catches each.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _problem(rng, N, D, V, scale=1.0, ignore=()):
    E = rng.standard_normal((N, D))
    C = rng.standard_normal((V, D)) * scale
    x = rng.integers(0, V, size=N).astype(np.int64)
    for i in ignore:
        x[i] = O.IGNORE_INDEX
    return E, C, x


# ---------------------------------------------------------------- closed forms
def test_zero_classifier_gives_log_v(rng):
    """C = 0: every logit is 0, so LSE = loss = log V exactly and dE = 0."""
    N, D, V = 7, 5, 4096
    E = rng.standard_normal((N, D))
    C = np.zeros((V, D))
    x = rng.integers(0, V, size=N)
    f = O.forward(E, C, x, reduction="none")
    assert np.allclose(f["lse"], math.log(V), rtol=1e-15, atol=0)
    assert np.allclose(f["loss_rows"], math.log(V), rtol=1e-15, atol=0)
    w = O.row_weights(x, O.IGNORE_INDEX, "sum", 1.0)
    dE, dC = O.backward(E, C, x, f["lse"], w)
    assert np.all(dE == 0.0)
    # dC_v = sum_i (1/V - [v = x_i]) E_i (softmax of constant logits is 1/V)
    expect = np.tile(E.sum(0) / V, (V, 1))
    for i in range(N):
        expect[x[i]] -= E[i]
    assert np.allclose(dC, expect, rtol=1e-12, atol=1e-14)


def test_two_classes_is_softplus():
    """N = 1, V = 2: loss = log(1 + exp(a_o - a_t)) and dE = sigma(a_o - a_t)(C_o - C_t)."""
    E = np.array([[1.0, -2.0, 3.0]])
    C = np.array([[0.5, 1.0, -1.0], [2.0, 0.0, 0.25]])
    x = np.array([1])
    a_t = float(E[0] @ C[1])
    a_o = float(E[0] @ C[0])
    f = O.forward(E, C, x, reduction="sum")
    assert f["loss"] == pytest.approx(math.log1p(math.exp(a_o - a_t)), rel=1e-15)
    sig = 1.0 / (1.0 + math.exp(-(a_o - a_t)))
    dE, dC = O.backward(E, C, x, f["lse"], O.row_weights(x, -100, "sum", 1.0))
    assert np.allclose(dE[0], sig * (C[0] - C[1]), rtol=1e-14)
    assert np.allclose(dC[0], sig * E[0], rtol=1e-14)
    assert np.allclose(dC[1], -sig * E[0], rtol=1e-14)


def test_fully_masked_batch_is_zero(rng):
    """Kernel card 'Correctness': a fully masked batch gives zero loss and zero gradients."""
    E, C, x = _problem(rng, 6, 4, 9)
    x[:] = O.IGNORE_INDEX
    f = O.forward(E, C, x, reduction="mean")
    assert f["loss"] == 0.0 and f["count"] == 0
    w = O.row_weights(x, O.IGNORE_INDEX, "mean", 1.0, f["count"])
    dE, dC = O.backward(E, C, x, f["lse"], w)
    assert np.all(dE == 0.0) and np.all(dC == 0.0)


# ------------------------------------------------------- finite differences
def _loss_of(E, C, x, reduction):
    return O.forward(E, C, x, reduction=reduction)["loss"]


@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_finite_differences(rng, reduction):
    """Central differences of the fp64 loss match dE and dC entry by entry."""
    E, C, x = _problem(rng, 5, 6, 11, scale=0.7, ignore=(2,))
    f = O.forward(E, C, x, reduction=reduction)
    w = O.row_weights(x, O.IGNORE_INDEX, reduction, 1.0, f["count"])
    dE, dC = O.backward(E, C, x, f["lse"], w)
    h = 1e-6
    for M, dM in ((E, dE), (C, dC)):
        num = np.zeros_like(M)
        for idx in np.ndindex(*M.shape):
            old = M[idx]
            M[idx] = old + h
            lp = _loss_of(E, C, x, reduction)
            M[idx] = old - h
            lm = _loss_of(E, C, x, reduction)
            M[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        assert np.allclose(num, dM, rtol=1e-6, atol=1e-8), np.max(np.abs(num - dM))
    assert np.all(dE[2] == 0.0)  # ignored row: exactly zero


def test_none_reduction_weights_by_grad_out(rng):
    """reduction='none': the gradient of sum_i g_i loss_i, checked by differences."""
    E, C, x = _problem(rng, 4, 3, 6, ignore=(1,))
    g = rng.standard_normal(4)
    f = O.forward(E, C, x, reduction="none")
    w = O.row_weights(x, O.IGNORE_INDEX, "none", g)
    dE, dC = O.backward(E, C, x, f["lse"], w)
    h = 1e-6
    for M, dM in ((E, dE), (C, dC)):
        for idx in np.ndindex(*M.shape):
            old = M[idx]
            M[idx] = old + h
            lp = float(g @ O.forward(E, C, x, reduction="none")["loss_rows"])
            M[idx] = old - h
            lm = float(g @ O.forward(E, C, x, reduction="none")["loss_rows"])
            M[idx] = old
            assert (lp - lm) / (2 * h) == pytest.approx(dM[idx], rel=1e-6, abs=1e-8)


# ------------------------------------------------------ library cross-check
@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
def test_matches_torch_cross_entropy(rng, reduction):
    """torch.nn.functional.cross_entropy on materialised fp64 logits."""
    E, C, x = _problem(rng, 64, 32, 300, scale=0.5, ignore=(3, 17, 40))
    Et = torch.tensor(E, requires_grad=True)
    Ct = torch.tensor(C, requires_grad=True)
    ref = torch.nn.functional.cross_entropy(Et @ Ct.T, torch.tensor(x), ignore_index=-100,
                                            reduction=reduction)
    g = rng.standard_normal(64) if reduction == "none" else 1.0
    ref.backward(torch.tensor(g) if reduction == "none" else None)
    f = O.forward(E, C, x, reduction=reduction)
    w = O.row_weights(x, O.IGNORE_INDEX, reduction, g, f["count"])
    dE, dC = O.backward(E, C, x, f["lse"], w)
    assert np.allclose(f["loss"], ref.detach().numpy(), rtol=1e-13, atol=1e-13)
    assert np.allclose(dE, Et.grad.numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(dC, Ct.grad.numpy(), rtol=1e-12, atol=1e-14)


def test_row_subsets_match_full(rng):
    """The sampled-row entry points agree with the full computation."""
    E, C, x = _problem(rng, 40, 16, 100, ignore=(0, 9))
    f = O.forward(E, C, x, reduction="mean")
    w = O.row_weights(x, O.IGNORE_INDEX, "mean", 1.0, f["count"])
    dE, dC = O.backward(E, C, x, f["lse"], w)
    rows = np.array([0, 5, 9, 39])
    fr = O.forward(E, C, x, rows=rows)
    assert np.array_equal(fr["lse"], f["lse"][rows])
    assert np.allclose(O.backward_dE(E, C, x, f["lse"][rows], w[rows], rows), dE[rows], rtol=1e-13)
    vrows = np.array([0, 3, 77, 99])
    assert np.allclose(O.backward_dC(E, C, x, f["lse"], w, vrows), dC[vrows], rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------ invariants
def test_softmax_normalised_and_g_rows_sum_to_zero(rng):
    E, C, x = _problem(rng, 30, 8, 500, scale=2.0, ignore=(4,))
    f = O.forward(E, C, x, reduction="sum")
    G = O.grad_logits(E @ C.T, f["lse"], x)
    ok = x != O.IGNORE_INDEX
    assert np.allclose(G[ok].sum(1), 0.0, atol=1e-12)
    P = np.exp(E @ C.T - f["lse"][:, None])
    assert np.allclose(P.sum(1), 1.0, atol=1e-13)
    dE, dC = O.backward(E, C, x, f["lse"], O.row_weights(x, -100, "sum", 1.0))
    assert np.allclose(dC.sum(0), 0.0, atol=1e-11)


def test_vocab_permutation_invariance(rng):
    """Reordering the vocabulary (rows of C, relabelled targets) leaves loss and
    LSE unchanged and permutes dC ('Vocabulary Sorting' relies on this)."""
    E, C, x = _problem(rng, 20, 6, 50, ignore=(7,))
    perm = rng.permutation(50)            # new row j holds old row perm[j]
    inv = np.argsort(perm)
    x2 = np.where(x == O.IGNORE_INDEX, x, inv[np.maximum(x, 0)])
    f1 = O.forward(E, C, x, reduction="mean")
    f2 = O.forward(E, C[perm], x2, reduction="mean")
    assert np.allclose(f1["lse"], f2["lse"], rtol=1e-14)
    assert f1["loss"] == pytest.approx(f2["loss"], rel=1e-14)
    w = O.row_weights(x, -100, "mean", 1.0, f1["count"])
    dE1, dC1 = O.backward(E, C, x, f1["lse"], w)
    dE2, dC2 = O.backward(E, C[perm], x2, f2["lse"], w)
    assert np.allclose(dE1, dE2, rtol=1e-12, atol=1e-15)
    assert np.allclose(dC1[perm], dC2, rtol=1e-12, atol=1e-15)


def test_duplicated_row_under_sum(rng):
    E, C, x = _problem(rng, 6, 5, 13)
    f = O.forward(E, C, x, reduction="sum")
    E2, x2 = np.vstack([E, E[2:3]]), np.append(x, x[2])
    f2 = O.forward(E2, C, x2, reduction="sum")
    assert f2["loss"] == pytest.approx(f["loss"] + f["loss_rows"][2], rel=1e-14)


def test_pigeonhole_bound():
    """'Gradient filtering': at most 1/eps = 4096 entries per row can reach
    eps = 2^-12.  With V = 4096 and C = 0 every probability is 2^-12 (to fp64
    rounding): the bound is met with equality."""
    assert O.FILTER_EPS == 2.0 ** -7 / 32
    V, D = 4096, 3
    E = np.ones((2, D))
    C = np.zeros((V, D))
    x = np.array([5, 4000])
    f = O.forward(E, C, x, reduction="sum")
    P = np.exp(E @ C.T - f["lse"][:, None])
    assert np.allclose(P, 2.0 ** -12, rtol=1e-15, atol=0)
    assert np.all((P >= O.FILTER_EPS * (1 - 1e-12)).sum(1) == 4096)
    # A normalised row can never exceed the bound.
    rng = np.random.default_rng(0)
    for scale in (0.1, 1.0, 3.0):
        Cr = rng.standard_normal((20000, D)) * scale
        fr = O.forward(E, Cr, np.array([0, 1]), reduction="sum")
        Pr = np.exp(E @ Cr.T - fr["lse"][:, None])
        assert np.all((Pr >= O.FILTER_EPS).sum(1) <= 4096)


def test_filter_tie_semantics():
    """Skip iff all |G| < eps: an entry equal to eps keeps its tile."""
    eps = O.FILTER_EPS
    G = np.zeros((4, 6))
    G[1, 4] = -eps            # exactly eps in magnitude
    G[3, 0] = np.nextafter(eps, 0.0)
    keep = O.tile_keep(G, 2, 3, eps)
    assert keep.tolist() == [[False, True], [False, False]]


def test_filter_just_below_and_above_uniform_softmax(rng):
    """C = 0, V = 4096: non-target |G| = 2^-12.  A threshold a hair below keeps
    every tile; a hair above keeps exactly the tiles holding a target
    (|G| = 1 - 1/V there)."""
    V, D, N = 4096, 4, 300
    E = rng.standard_normal((N, D))
    C = np.zeros((V, D))
    x = rng.integers(0, V, size=N)
    f = O.forward(E, C, x, reduction="mean")
    keep = O.tile_survival(E, C, x, f["lse"], 128, 128, eps=2.0 ** -12 * (1 - 1e-9))
    assert keep.all()
    keep2 = O.tile_survival(E, C, x, f["lse"], 128, 128, eps=2.0 ** -12 * (1 + 1e-9))
    expect = np.zeros_like(keep2)
    for i in range(N):
        expect[i // 128, x[i] // 128] = True
    assert np.array_equal(keep2, expect)


def test_filtered_matches_unfiltered_at_eps_zero_and_bound(rng):
    E, C, x = _problem(rng, 200, 16, 700, scale=3.0, ignore=(1, 150))
    f = O.forward(E, C, x, reduction="mean")
    w = O.row_weights(x, -100, "mean", 1.0, f["count"])
    dE, dC = O.backward(E, C, x, f["lse"], w)
    dE0, dC0, keep0 = O.backward_filtered(E, C, x, f["lse"], w, 64, 64, eps=0.0)
    assert keep0.all() and np.allclose(dE0, dE) and np.allclose(dC0, dC)
    eps = 1e-3
    dEf, dCf, keep = O.backward_filtered(E, C, x, f["lse"], w, 16, 16, eps=eps)
    assert 0.05 < keep.mean() < 0.95
    # per-row bound: ||dE_f,i - dE_i|| <= sum_{dropped v} |w_i G_iv| ||C_v||
    G = O.grad_logits(E @ C.T, f["lse"], x)
    mask = np.repeat(np.repeat(keep, 16, 0), 16, 1)[:200, :700]
    dropped = np.where(mask, 0.0, np.abs(w[:, None] * G))
    assert np.all(dropped.max(1) <= eps * np.abs(w) + 1e-300)
    bound = dropped @ np.linalg.norm(C, axis=1)
    assert np.all(np.linalg.norm(dEf - dE, axis=1) <= bound * (1 + 1e-12) + 1e-18)


# ------------------------------------------------ planted mistakes are caught
def _pin_suite(mod, rng):
    """Runs a compact version of the pins against an oracle module; returns
    the names of the pins that failed."""
    failed = []
    E, C, x = _problem(rng, 5, 4, 9, scale=0.8, ignore=(1,))
    # finite differences (mean reduction)
    f = mod.forward(E, C, x, reduction="mean")
    w = mod.row_weights(x, -100, "mean", 1.0, f["count"])
    dE, dC = mod.backward(E, C, x, f["lse"], w)
    h = 1e-6
    ok = True
    for M, dM in ((E, dE), (C, dC)):
        for idx in np.ndindex(*M.shape):
            old = M[idx]
            M[idx] = old + h
            lp = mod.forward(E, C, x, reduction="mean")["loss"]
            M[idx] = old - h
            lm = mod.forward(E, C, x, reduction="mean")["loss"]
            M[idx] = old
            ok &= abs((lp - lm) / (2 * h) - dM[idx]) <= 1e-6 * max(1.0, abs(dM[idx]))
    if not ok:
        failed.append("finite_differences")
    # torch cross_entropy
    Et, Ct = torch.tensor(E, requires_grad=True), torch.tensor(C, requires_grad=True)
    ref = torch.nn.functional.cross_entropy(Et @ Ct.T, torch.tensor(x), reduction="mean")
    ref.backward()
    if not (np.allclose(f["loss"], ref.item(), rtol=1e-12)
            and np.allclose(dE, Et.grad.numpy(), rtol=1e-10, atol=1e-13)
            and np.allclose(dC, Ct.grad.numpy(), rtol=1e-10, atol=1e-13)):
        failed.append("torch_cross_entropy")
    # closed form C = 0
    Z = np.zeros((4096, 4))
    fz = mod.forward(E, Z, np.abs(x), reduction="none")
    if not np.allclose(fz["loss_rows"], math.log(4096), rtol=1e-14):
        failed.append("zero_classifier")
    return failed


def _mutant(**overrides):
    import types
    m = types.ModuleType("oracle_mutant")
    for k in dir(O):
        if not k.startswith("__"):
            setattr(m, k, getattr(O, k))
    for k, fn in overrides.items():
        setattr(m, k, fn)
    # rebind the module-level helpers the public functions call
    for name in ("forward", "backward", "grad_logits", "log_sum_exp", "row_weights", "logits"):
        f = getattr(m, name)
        if hasattr(f, "__globals__") and name not in overrides:
            g = dict(f.__globals__)
            g.update(overrides)
            setattr(m, name, type(f)(f.__code__, g, f.__name__, f.__defaults__, f.__closure__))
    return m


def test_true_oracle_passes_pin_suite(rng):
    assert _pin_suite(O, rng) == []


def _wrong_sign_onehot(A, lse, x_rows, v0=0, ignore_index=-100, softcap=0.0):
    G = np.exp(O.softcap_logits(A, softcap) - np.asarray(lse)[:, None])
    r = np.nonzero(x_rows != ignore_index)[0]
    G[r, x_rows[r] - v0] += 1.0
    G[x_rows == ignore_index] = 0.0
    return G


def _dropped_onehot(A, lse, x_rows, v0=0, ignore_index=-100, softcap=0.0):
    G = np.exp(O.softcap_logits(A, softcap) - np.asarray(lse)[:, None])
    G[x_rows == ignore_index] = 0.0
    return G


def _lse_without_max(A):
    return np.log(np.exp(A).sum(axis=1)) + A.max(axis=1) * 0.0 + 1e-3


def _mean_over_all_rows(x, ignore_index, reduction, grad_out, count=None):
    x = np.asarray(x)
    return np.where(x != ignore_index, 1.0 / len(x), 0.0)


def _transposed_logits(E, C):
    return (C @ E.T).T[:, ::-1].copy()


@pytest.mark.parametrize("name,overrides", [
    ("wrong sign of the one-hot", dict(grad_logits=_wrong_sign_onehot)),
    ("dropped one-hot term", dict(grad_logits=_dropped_onehot)),
    ("log-sum-exp off by a constant", dict(log_sum_exp=_lse_without_max)),
    ("mean over all rows instead of non-ignored", dict(row_weights=_mean_over_all_rows)),
    ("reversed vocabulary index", dict(logits=_transposed_logits)),
])
def test_planted_mistake_is_caught(rng, name, overrides):
    assert _pin_suite(_mutant(**overrides), rng) != [], name


def test_indexed_logits_match_gathered_torch_logits(rng):
    """Algorithm 1 (indexed matmul): o_i = C[x_i] . E_i equals the gathered
    entry of torch's materialised logit matrix; NaN on ignored rows."""
    E, C, x = _problem(rng, 40, 12, 90, ignore=(3, 7))
    o = O.indexed_logits(E, C, x)
    ok = x != O.IGNORE_INDEX
    full = (torch.tensor(E) @ torch.tensor(C).T).numpy()
    assert np.allclose(o[ok], full[np.nonzero(ok)[0], x[ok]], rtol=1e-14)
    assert np.all(np.isnan(o[~ok]))
    f = O.forward(E, C, x, reduction="none")
    assert np.allclose(f["target_logit"][ok], o[ok], rtol=1e-14)


def test_fwd_bwd_rows_is_the_sub_batch(rng):
    """The timed CPU sample (a standalone sub-batch) equals torch cross_entropy
    on that sub-batch's materialised logits."""
    E, C, x = _problem(rng, 30, 8, 70, ignore=(2,))
    rows = np.array([0, 2, 5, 11, 29])
    loss, dE, dC = O.fwd_bwd_rows(E, C, x, rows, reduction="mean")
    Et = torch.tensor(E[rows], requires_grad=True)
    Ct = torch.tensor(C, requires_grad=True)
    ref = torch.nn.functional.cross_entropy(Et @ Ct.T, torch.tensor(x[rows]), reduction="mean")
    ref.backward()
    assert loss == pytest.approx(ref.item(), rel=1e-13)
    assert np.allclose(dE, Et.grad.numpy(), rtol=1e-12, atol=1e-15)
    assert np.allclose(dC, Ct.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_widen_bf16_is_exact():
    """bf16 -> float64 widening: bit patterns of known values."""
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x3E80, 0x7F7F], dtype=np.uint16)
    assert O.widen_bf16(bits).tolist()[:5] == [1.0, -2.0, 0.0, -0.0, 0.25]
    assert O.widen_bf16(bits)[5] == float(np.float32(3.3895313892515355e38))


def test_per_output_filter_flags(rng):
    """FullC (filter dE only) leaves dC exactly unfiltered; FullE the reverse;
    both off equals the unfiltered backward."""
    E, C, x = _problem(rng, 200, 16, 700, scale=3.0, ignore=(1, 150))
    f = O.forward(E, C, x, reduction="mean")
    w = O.row_weights(x, -100, "mean", 1.0, f["count"])
    dE, dC = O.backward(E, C, x, f["lse"], w)
    dEf, dCf, keep = O.backward_filtered(E, C, x, f["lse"], w, 16, 16, eps=1e-3)
    assert 0.05 < keep.mean() < 0.95
    a_dE, a_dC, _ = O.backward_filtered(E, C, x, f["lse"], w, 16, 16, eps=1e-3, filter_dC=False)
    assert np.array_equal(a_dE, dEf) and np.allclose(a_dC, dC, rtol=1e-13, atol=1e-16)
    b_dE, b_dC, _ = O.backward_filtered(E, C, x, f["lse"], w, 16, 16, eps=1e-3, filter_dE=False)
    assert np.allclose(b_dE, dE, rtol=1e-13, atol=1e-16) and np.array_equal(b_dC, dCf)
    c_dE, c_dC, _ = O.backward_filtered(E, C, x, f["lse"], w, 16, 16, eps=1e-3, filter_dE=False,
                                        filter_dC=False)
    assert np.allclose(c_dE, dE, rtol=1e-13, atol=1e-16) and np.allclose(c_dC, dC, rtol=1e-13, atol=1e-16)


# ----------------------------------------------------------- softcapping
@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
def test_softcap_matches_torch(rng, reduction):
    """cap * tanh(logits / cap), cross-entropy and autograd in torch fp64."""
    cap = 5.0
    E, C, x = _problem(rng, 48, 16, 200, scale=2.0, ignore=(3, 9))
    Et = torch.tensor(E, requires_grad=True)
    Ct = torch.tensor(C, requires_grad=True)
    A = cap * torch.tanh((Et @ Ct.T) / cap)
    ref = torch.nn.functional.cross_entropy(A, torch.tensor(x), reduction=reduction)
    g = rng.standard_normal(48) if reduction == "none" else 1.0
    ref.backward(torch.tensor(g) if reduction == "none" else None)
    f = O.forward(E, C, x, reduction=reduction, softcap=cap)
    w = O.row_weights(x, -100, reduction, g, f["count"])
    dE, dC = O.backward(E, C, x, f["lse"], w, softcap=cap)
    assert np.allclose(f["loss"], ref.detach().numpy(), rtol=1e-13, atol=1e-13)
    assert np.allclose(dE, Et.grad.numpy(), rtol=1e-11, atol=1e-14)
    assert np.allclose(dC, Ct.grad.numpy(), rtol=1e-11, atol=1e-14)
    rows = np.array([0, 3, 20])
    assert np.allclose(O.backward_dE(E, C, x, f["lse"][rows], w[rows], rows, softcap=cap), dE[rows], rtol=1e-12)
    vr = np.array([1, 50, 199])
    assert np.allclose(O.backward_dC(E, C, x, f["lse"], w, vr, softcap=cap), dC[vr], rtol=1e-11, atol=1e-15)


def test_softcap_finite_differences(rng):
    cap = 3.0
    E, C, x = _problem(rng, 4, 5, 9, scale=2.0, ignore=(1,))
    f = O.forward(E, C, x, reduction="sum", softcap=cap)
    w = O.row_weights(x, -100, "sum", 1.0)
    dE, dC = O.backward(E, C, x, f["lse"], w, softcap=cap)
    h = 1e-6
    for M, dM in ((E, dE), (C, dC)):
        for idx in np.ndindex(*M.shape):
            old = M[idx]
            M[idx] = old + h
            lp = O.forward(E, C, x, reduction="sum", softcap=cap)["loss"]
            M[idx] = old - h
            lm = O.forward(E, C, x, reduction="sum", softcap=cap)["loss"]
            M[idx] = old
            assert (lp - lm) / (2 * h) == pytest.approx(dM[idx], rel=1e-6, abs=1e-8)


def test_softcap_bounds_the_logits(rng):
    """Every capped logit lies in (-cap, cap), so LSE <= cap + log V."""
    cap = 2.0
    E, C, x = _problem(rng, 10, 4, 50, scale=10.0)
    f = O.forward(E, C, x, reduction="none", softcap=cap)
    assert np.all(f["lse"] < cap + math.log(50))
    assert np.all(np.abs(f["target_logit"]) < cap)


def test_compacting_ignored_rows_changes_only_the_tiling(rng):
    """Unfiltered, removing ignored rows first changes nothing; filtered, it
    equals the filtered backward of the batch without those rows."""
    E, C, x = _problem(rng, 200, 16, 700, scale=3.0, ignore=tuple(range(0, 200, 3)))
    f = O.forward(E, C, x, reduction="mean")
    w = O.row_weights(x, -100, "mean", 1.0, f["count"])
    dE, dC = O.backward(E, C, x, f["lse"], w)
    a_dE, a_dC, _ = O.backward_filtered(E, C, x, f["lse"], w, 16, 16, eps=0.0, compact_ignored=True)
    assert np.allclose(a_dE, dE, rtol=1e-13, atol=1e-16) and np.allclose(a_dC, dC, rtol=1e-13, atol=1e-16)
    keep_rows = np.nonzero(x != -100)[0]
    b_dE, b_dC, keep = O.backward_filtered(E, C, x, f["lse"], w, 16, 16, eps=1e-3, compact_ignored=True)
    c_dE, c_dC, keep_c = O.backward_filtered(E[keep_rows], C, x[keep_rows], f["lse"][keep_rows], w[keep_rows],
                                             16, 16, eps=1e-3)
    assert np.array_equal(keep, keep_c) and np.array_equal(b_dC, c_dC)
    assert np.array_equal(b_dE[keep_rows], c_dE) and np.all(b_dE[x == -100] == 0.0)


# ------------------------------------------------------------- single call
@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_single_call_matches_torch_autograd(rng, reduction):
    """Unfiltered, the single call's loss and gradients are those of torch's
    cross_entropy on materialised fp64 logits (unit upstream gradient)."""
    E, C, x = _problem(rng, 40, 12, 70, scale=0.7, ignore=(3, 17))
    out = O.loss_and_grad(E, C, x, reduction=reduction)
    Et, Ct = torch.tensor(E, requires_grad=True), torch.tensor(C, requires_grad=True)
    ref = torch.nn.functional.cross_entropy(Et @ Ct.T, torch.tensor(x), ignore_index=-100, reduction=reduction)
    ref.backward()
    assert np.allclose(out["loss"], ref.item(), rtol=1e-12)
    assert np.allclose(out["dE"], Et.grad.numpy(), rtol=1e-10, atol=1e-14)
    assert np.allclose(out["dC"], Ct.grad.numpy(), rtol=1e-10, atol=1e-14)
    assert out["count"] == 38


def test_single_call_scales_linearly_with_the_upstream_gradient(rng):
    """What the single call's backward does -- multiply by the upstream
    gradient g -- is the gradient of g * loss (finite differences)."""
    E, C, x = _problem(rng, 6, 4, 9, scale=0.8, ignore=(2,))
    g = -1.7
    out = O.loss_and_grad(E, C, x, reduction="mean")
    h = 1e-6
    for idx in [(0, 1), (3, 2), (5, 0)]:
        E2 = E.copy()
        E2[idx] += h
        lp = O.loss_and_grad(E2, C, x, reduction="mean")["loss"]
        E2[idx] -= 2 * h
        lm = O.loss_and_grad(E2, C, x, reduction="mean")["loss"]
        assert abs(g * (lp - lm) / (2 * h) - g * out["dE"][idx]) <= 1e-6


def test_single_call_filter_tiles_are_over_the_rows_that_take_part(rng):
    """The single call removes the ignored rows first: with ignored rows
    between the others, its filtered gradient is the compacted tiling's, and
    equals the filtered backward of the batch without those rows."""
    E, C, x = _problem(rng, 96, 12, 300, scale=3.0, ignore=tuple(range(0, 96, 3)))
    out = O.loss_and_grad(E, C, x, reduction="sum", filter_eps=2e-2, BN=16, BV=16)
    f = O.forward(E, C, x, reduction="sum")
    w = O.row_weights(x, -100, "sum", 1.0, f["count"])
    a = O.backward_filtered(E, C, x, f["lse"], w, 16, 16, 2e-2)
    keep_rows = np.nonzero(x != -100)[0]
    b = O.backward_filtered(E[keep_rows], C, x[keep_rows], f["lse"][keep_rows], w[keep_rows], 16, 16, 2e-2)
    assert np.array_equal(out["keep"], b[2]) and np.array_equal(out["dC"], b[1])
    assert np.array_equal(out["dE"][keep_rows], b[0]) and np.all(out["dE"][x == -100] == 0.0)
    assert a[2].shape != b[2].shape
    with pytest.raises(ValueError):
        O.loss_and_grad(E, C, x, reduction="none")
