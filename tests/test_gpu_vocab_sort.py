"""GPU parity of vocabulary sorting ("Cut Your Losses in Large-Vocabulary
Language Models", section "Vocabulary Sorting"), through the C ABI.

* the radix sort is index work: its order must equal the oracle's stable
  ascending order of the same fp32 keys exactly;
* the logit sums are fp32 sums of fp32 products: each must lie within the
  standard error bound gamma_k sum_d |C_vd| sum_i |E_id| (k = N + D terms
  deep at most) of the oracle's fp64 sum;
* the order the device takes from its own sums must be ascending in the
  oracle's sums, up to those bounds (where two sums are closer than their
  bounds, either order is correct);
* the sorted backward: without the filter it is the plain gradient (same
  tolerances as the unsorted path); with the filter it matches the oracle's
  sorted, filtered backward, and on inputs whose frequent tokens are
  scattered through the vocabulary it skips far more tiles than the
  unsorted path.
"""
import numpy as np
import pytest
import torch

import cce_workloads as W
import oracle as O
from tests.gpu_util import (TOL_GRAD, TOL_GRAD_FILTERED, assert_grads_close, bf16_to_f64, rel_fro, to_device)

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24  # unit roundoff of fp32


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests.conftest import build_library
    build_library()


def _gamma(k):
    return k * U32 / (1.0 - k * U32)


# ------------------------------------------------------------------ the order
def _keys(rng, V):
    k = rng.integers(-40, 41, size=V).astype(np.float32) * np.float32(0.25)  # many exact ties
    m = rng.random(V)
    k[m < 0.3] = rng.standard_normal(int((m < 0.3).sum())).astype(np.float32) * np.float32(1e3)
    k[m > 0.97] = np.float32(-0.0)
    k[(m > 0.95) & (m <= 0.97)] = np.float32(0.0)
    if V > 10:
        k[3], k[7] = np.float32(np.inf), np.float32(-np.inf)
        k[9] = np.float32(1e-42)   # subnormal
        k[10] = np.float32(-1e-42)
    return k


@pytest.mark.parametrize("V", [1, 7, 1023, 1024, 1025, 5000, 151936, 256000, 300001])
def test_order_is_the_stable_ascending_order(V):
    import linear_cross_entropy_gb300 as cce
    rng = np.random.default_rng(V)
    k = _keys(rng, V)
    perm = cce.vocab_order(torch.from_numpy(k).cuda()).cpu().numpy().astype(np.int64)
    expect = O.vocab_order(k.astype(np.float64))
    assert np.array_equal(perm, expect)


# --------------------------------------------------------------- the sort key
def _sum_bound(E, C, x, ignore_index=-100):
    V = C.shape[0]
    take = (x != ignore_index) & (x >= 0) & (x < V)
    a = np.abs(E[take]).sum(axis=0)
    return _gamma(E.shape[0] + E.shape[1]) * (np.abs(C) @ a)


CASES = [
    ("tiny", dict(kind="config")),
    ("ragged", dict(kind="small", N=300, D=136, V=5000)),
    ("freq", dict(kind="freq", N=700, D=64, V=9000)),
]


def _inputs(kind, N=None, D=None, V=None):
    if kind == "config":
        return W.make_inputs(W.CONFIGS["tiny"])
    if kind == "small":
        return W.make_inputs(W.small("ragged", N, D, V))
    return W.frequent_token_inputs(N, D, V, n_freq=192, scatter=True, unigram=8.0)


@pytest.mark.parametrize("name,case", CASES)
def test_logit_sums_and_their_order(name, case):
    import linear_cross_entropy_gb300 as cce
    E_bits, C_bits, x = _inputs(**case)
    x = x.copy()
    x[5] = C_bits.shape[0] + 3  # out of range: takes no part (and is not an error here)
    E, C, xt = to_device(E_bits, C_bits, x)
    sums = cce.vocab_logit_sums(E, C, xt).double().cpu().numpy()
    Ef, Cf = O.from_bits(E_bits, C_bits)
    ref, count = O.vocab_logit_sums(Ef, Cf, x)
    bound = _sum_bound(Ef, Cf, x)
    err = np.abs(sums - ref)
    assert np.all(err <= bound), f"logit sum off by {err.max():.3e} (bound {bound[np.argmax(err)]:.3e})"
    # the device's order of its own sums, checked against the oracle's sums
    perm = cce.vocab_order(torch.from_numpy(sums.astype(np.float32)).cuda()).cpu().numpy().astype(np.int64)
    assert np.array_equal(np.sort(perm), np.arange(len(perm)))
    a, b = perm[:-1], perm[1:]
    assert np.all(ref[a] <= ref[b] + bound[a] + bound[b])


# ----------------------------------------------------------- sorted backward
def _run(E_bits, C_bits, x, *, eps, sort, reduction="mean", ignore_index=-100, grad_out=None, softcap=0.0):
    import linear_cross_entropy_gb300 as cce
    E, C, xt = to_device(E_bits, C_bits, x)
    loss, lse = cce.cce_forward(E, C, xt, ignore_index, reduction, softcap=softcap)
    if grad_out is None:
        g = torch.ones(x.shape[0] if reduction == "none" else 1, dtype=torch.float32, device="cuda")
    else:
        g = torch.as_tensor(grad_out, dtype=torch.float32, device="cuda")
    dE, dC, st = cce.cce_backward(E, C, xt, lse, g, ignore_index, reduction, eps, softcap=softcap,
                                  vocab_sort=sort, stats=True)
    torch.cuda.synchronize()
    return {"dE": bf16_to_f64(dE), "dC": bf16_to_f64(dC), "dE_raw": dE, "stats": st,
            "lse": lse.double().cpu().numpy()}


def _oracle(E_bits, C_bits, x, reduction="mean", ignore_index=-100, grad_out=1.0, softcap=0.0):
    Ef, Cf = O.from_bits(E_bits, C_bits)
    f = O.forward(Ef, Cf, x, ignore_index, reduction, softcap=softcap)
    w = O.row_weights(x, ignore_index, reduction, grad_out, f["count"])
    return Ef, Cf, f, w


UNFILTERED = [
    ("tiny", dict(kind="config"), "mean"),
    ("ragged-sum", dict(kind="small", N=300, D=136, V=5000), "sum"),
    ("ragged-none", dict(kind="small", N=300, D=136, V=5000), "none"),
    ("multi-chunk", dict(kind="small", N=200, D=64, V=9000), "mean"),
]


@pytest.mark.parametrize("name,case,reduction", UNFILTERED)
def test_sorted_backward_without_filter_is_the_plain_gradient(name, case, reduction):
    E_bits, C_bits, x = _inputs(**case)
    go = None
    if reduction == "none":
        go = np.random.default_rng(3).standard_normal(x.shape[0])
    got = _run(E_bits, C_bits, x, eps=0.0, sort=True, reduction=reduction, grad_out=go)
    Ef, Cf, f, w = _oracle(E_bits, C_bits, x, reduction, grad_out=1.0 if go is None else go)
    dE, dC = O.backward(Ef, Cf, x, f["lse"], w)
    assert_grads_close(got, dE, dC, TOL_GRAD, x)
    assert got["stats"]["skipped"] == 0


def test_sorted_backward_with_ignore_index_inside_the_vocabulary():
    E_bits, C_bits, x = _inputs("small", 300, 136, 5000)
    x = np.where(x == -100, 5, x)
    x[::11] = 5
    got = _run(E_bits, C_bits, x, eps=0.0, sort=True, reduction="sum", ignore_index=5)
    Ef, Cf, f, w = _oracle(E_bits, C_bits, x, "sum", ignore_index=5)
    dE, dC = O.backward(Ef, Cf, x, f["lse"], w, ignore_index=5)
    assert_grads_close(got, dE, dC, TOL_GRAD, x, ignore_index=5)


def test_sorted_backward_with_softcap():
    E_bits, C_bits, x = _inputs("small", 300, 136, 5000)
    got = _run(E_bits, C_bits, x, eps=0.0, sort=True, softcap=20.0)
    Ef, Cf, f, w = _oracle(E_bits, C_bits, x, softcap=20.0)
    dE, dC = O.backward(Ef, Cf, x, f["lse"], w, softcap=20.0)
    assert_grads_close(got, dE, dC, TOL_GRAD, x)


def test_sorted_filtered_backward_matches_the_oracle_and_skips_more():
    N, D, V = 1024, 128, 20000
    E_bits, C_bits, x = W.frequent_token_inputs(N, D, V, n_freq=256, scatter=True, unigram=8.0)
    got = _run(E_bits, C_bits, x, eps=O.FILTER_EPS, sort=True)
    plain = _run(E_bits, C_bits, x, eps=O.FILTER_EPS, sort=False)
    Ef, Cf, f, w = _oracle(E_bits, C_bits, x)
    perm = O.vocab_order(O.vocab_logit_sums(Ef, Cf, x)[0])
    dEf, dCf, keep = O.backward_filtered(Ef, Cf, x, f["lse"], w, 128, 128, O.FILTER_EPS, compact_ignored=True,
                                         vocab_perm=perm)
    eE, eC = assert_grads_close(got, dEf, dCf, TOL_GRAD_FILTERED, x)
    tiles, skipped = got["stats"]["tiles"], got["stats"]["skipped"]
    assert tiles == keep.size
    assert abs(skipped - int((~keep).sum())) <= max(1, keep.size // 200), (skipped, int((~keep).sum()))
    assert skipped >= plain["stats"]["skipped"] + 0.3 * tiles, (skipped, plain["stats"]["skipped"], tiles)
    # the same gradient as the unsorted path, within the filter's error
    assert rel_fro(got["dE"], plain["dE"]) <= TOL_GRAD_FILTERED
    assert rel_fro(got["dC"], plain["dC"]) <= TOL_GRAD_FILTERED
    print(f"sorted: skipped {skipped}/{tiles} (oracle {int((~keep).sum())}), unsorted skipped "
          f"{plain['stats']['skipped']}; dE err {eE:.2e} dC err {eC:.2e}")


def test_sorted_backward_is_deterministic():
    E_bits, C_bits, x = W.frequent_token_inputs(600, 64, 9000, n_freq=200, scatter=True, unigram=8.0)
    a = _run(E_bits, C_bits, x, eps=O.FILTER_EPS, sort=True)
    b = _run(E_bits, C_bits, x, eps=O.FILTER_EPS, sort=True)
    assert torch.equal(a["dE_raw"].view(torch.int16), b["dE_raw"].view(torch.int16))
    assert np.array_equal(a["dC"], b["dC"]) and a["stats"] == b["stats"]
