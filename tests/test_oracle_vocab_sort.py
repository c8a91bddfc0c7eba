"""Pins of the oracle's vocabulary sorting ("Cut Your Losses in
Large-Vocabulary Language Models", section "Vocabulary Sorting").

The sort key (each token's logit sum over the rows that take part) is pinned
by brute-force loops and by linearity; the order by counting ranks one key
at a time and by a hand-sorted example; the sorted, filtered backward by
three facts that hold whatever the order: the identity order changes
nothing, without the filter any order gives the plain gradient, and the
result does not depend on how the input vocabulary was numbered.  Two
planted mistakes (targets not moved to their sorted positions, dC rows put
back with the inverse order) are shown to fail those pins.
"""
import numpy as np
import pytest

import cce_workloads as W
import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _problem(rng, N, D, V, scale=3.0, ignore=()):
    E = rng.standard_normal((N, D))
    C = rng.standard_normal((V, D)) * scale / np.sqrt(D)
    x = rng.integers(0, V, size=N).astype(np.int64)
    for i in ignore:
        x[i] = O.IGNORE_INDEX
    return E, C, x


# ------------------------------------------------------------------ sort key
def test_logit_sums_by_brute_force(rng):
    E, C, x = _problem(rng, 6, 3, 7)
    x[1] = O.IGNORE_INDEX
    x[4] = 7  # out of range: takes no part
    S, count = O.vocab_logit_sums(E, C, x)
    assert count == 4
    for v in range(7):
        acc = 0.0
        for i in range(6):
            if x[i] == O.IGNORE_INDEX or not (0 <= x[i] < 7):
                continue
            for d in range(3):
                acc += E[i, d] * C[v, d]
        assert abs(S[v] - acc) <= 1e-13 * max(1.0, abs(acc))


def test_logit_sums_are_linear_in_the_rows(rng):
    """sum_i C_v . E_i = C_v . (sum_i E_i); rows that take no part change
    nothing, and moving one row that takes part by delta moves S by C delta."""
    E, C, x = _problem(rng, 300, 24, 500, ignore=(0, 7, 299))
    S, count = O.vocab_logit_sums(E, C, x)
    part = (x != O.IGNORE_INDEX)
    assert count == int(part.sum())
    lin = C @ E[part].sum(axis=0)
    assert np.allclose(S, lin, rtol=1e-11, atol=1e-11)
    E2 = E.copy()
    E2[7] += 100.0
    assert np.array_equal(O.vocab_logit_sums(E2, C, x)[0], S)
    delta = rng.standard_normal(24)
    E2 = E.copy()
    E2[3] += delta
    assert np.allclose(O.vocab_logit_sums(E2, C, x)[0] - S, C @ delta, rtol=1e-9, atol=1e-10)


# ----------------------------------------------------------------- the order
def test_order_hand_sorted_example():
    keys = np.array([3.0, -1.0, 3.0, 0.0, -0.0, 2.0, -1.0])
    # ascending; the two -1 keep token order (1, 6), 0.0 and -0.0 are equal
    # (3, 4), the two 3.0 too (0, 2)
    assert O.vocab_order(keys).tolist() == [1, 6, 3, 4, 5, 0, 2]


def test_order_by_counting_ranks(rng):
    V = 300
    keys = rng.integers(-3, 4, size=V).astype(np.float64)
    keys[::7] = rng.standard_normal(len(keys[::7]))
    keys[5] = -0.0
    keys[9] = 0.0
    perm = O.vocab_order(keys)
    assert sorted(perm.tolist()) == list(range(V))
    for v in range(V):
        rank = 0
        for u in range(V):
            if keys[u] < keys[v] or (keys[u] == keys[v] and u < v):
                rank += 1
        assert perm[rank] == v


# ------------------------------------------------- sorted, filtered backward
def _setup(rng, N=260, D=16, V=700, ignore=(2, 100, 259)):
    E, C, x = _problem(rng, N, D, V, ignore=ignore)
    f = O.forward(E, C, x, reduction="mean")
    w = O.row_weights(x, -100, "mean", 1.0, f["count"])
    return E, C, x, f, w


def test_identity_order_changes_nothing(rng):
    E, C, x, f, w = _setup(rng)
    a = O.backward_filtered(E, C, x, f["lse"], w, 16, 16, 1e-3, compact_ignored=True)
    b = O.backward_filtered(E, C, x, f["lse"], w, 16, 16, 1e-3, compact_ignored=True,
                            vocab_perm=np.arange(C.shape[0]))
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def _check_unfiltered(bwd, E, C, x, f, w, perm):
    dE, dC = O.backward(E, C, x, f["lse"], w)
    sE, sC, keep = bwd(E, C, x, f["lse"], w, 16, 16, 0.0, compact_ignored=True, vocab_perm=perm)
    return keep.all() and np.allclose(sE, dE, rtol=1e-12, atol=1e-15) and \
        np.allclose(sC, dC, rtol=1e-12, atol=1e-15)


def test_any_order_gives_the_plain_gradient_without_filter(rng):
    E, C, x, f, w = _setup(rng)
    perm = rng.permutation(C.shape[0])
    assert _check_unfiltered(O.backward_filtered, E, C, x, f, w, perm)
    keys, _ = O.vocab_logit_sums(E, C, x)
    assert _check_unfiltered(O.backward_filtered, E, C, x, f, w, O.vocab_order(keys))


def test_sorted_result_does_not_depend_on_input_numbering(rng):
    """Relabel the vocabulary by q (C' = C[q], targets moved with it): the
    sorted order finds the same tiles, so dE and the survival map are the
    same and dC' = dC[q]."""
    E, C, x, f, w = _setup(rng)
    V = C.shape[0]
    q = rng.permutation(V)
    qinv = np.empty(V, np.int64)
    qinv[q] = np.arange(V)
    C2 = C[q]
    x2 = np.where(x == O.IGNORE_INDEX, x, qinv[np.where(x == O.IGNORE_INDEX, 0, x)])
    p1 = O.vocab_order(O.vocab_logit_sums(E, C, x)[0])
    p2 = O.vocab_order(O.vocab_logit_sums(E, C2, x2)[0])
    assert np.array_equal(q[p2], p1)  # the same tokens in the same order
    dE1, dC1, k1 = O.backward_filtered(E, C, x, f["lse"], w, 8, 8, 2e-2, compact_ignored=True, vocab_perm=p1)
    dE2, dC2, k2 = O.backward_filtered(E, C2, x2, f["lse"], w, 8, 8, 2e-2, compact_ignored=True,
                                       vocab_perm=p2)
    assert 0.05 < k1.mean() < 0.95
    assert np.array_equal(k1, k2)
    assert np.allclose(dE2, dE1, rtol=1e-13, atol=1e-16)
    assert np.allclose(dC2, dC1[q], rtol=1e-13, atol=1e-16)


def test_custom_ignore_index_inside_the_vocabulary(rng):
    """An ignore index that is itself a token id: a row whose target lands on
    that id's sorted position must still take part."""
    E, C, x = _problem(rng, 120, 8, 300)
    ign = 5
    x[::9] = ign
    f = O.forward(E, C, x, ignore_index=ign, reduction="sum")
    w = O.row_weights(x, ign, "sum", 1.0, f["count"])
    dE, dC = O.backward(E, C, x, f["lse"], w, ignore_index=ign)
    perm = np.roll(np.arange(300), 3)  # position 5 holds token 2
    sE, sC, _ = O.backward_filtered(E, C, x, f["lse"], w, 16, 16, 0.0, ignore_index=ign, compact_ignored=True,
                                    vocab_perm=perm)
    assert np.allclose(sE, dE, rtol=1e-12, atol=1e-15) and np.allclose(sC, dC, rtol=1e-12, atol=1e-15)


def test_sorting_gathers_the_frequent_tokens():
    """On the scattered frequent-token inputs the frequent ids end up in the
    last positions and far fewer tiles survive than in the input order."""
    n_freq = 128
    E_bits, C_bits, x = W.frequent_token_inputs(512, 128, 4096, n_freq=n_freq, scatter=True, unigram=8.0)
    E, C = O.from_bits(E_bits, C_bits)
    f = O.forward(E, C, x, reduction="mean")
    w = O.row_weights(x, -100, "mean", 1.0, f["count"])
    perm = O.vocab_order(O.vocab_logit_sums(E, C, x)[0])
    freq_ids = np.nonzero(np.linalg.norm(C, axis=1) > 2.0)[0]
    assert len(freq_ids) == n_freq
    assert set(perm[-n_freq:].tolist()) == set(freq_ids.tolist())
    _, _, k_in = O.backward_filtered(E, C, x, f["lse"], w, 128, 128, O.FILTER_EPS, compact_ignored=True)
    _, _, k_s = O.backward_filtered(E, C, x, f["lse"], w, 128, 128, O.FILTER_EPS, compact_ignored=True,
                                    vocab_perm=perm)
    assert k_in.mean() > 0.5 and k_s.mean() <= 2.0 / k_s.shape[1] + 1e-12


# ------------------------------------------------------------ planted mistakes
def _targets_not_moved(E, C, x, lse, w, BN, BV, eps, ignore_index=-100, compact_ignored=False, vocab_perm=None):
    p = np.asarray(vocab_perm)
    dE, dCs, keep = O.backward_filtered(E, np.asarray(C)[p], x, lse, w, BN, BV, eps, ignore_index,
                                        compact_ignored=compact_ignored)
    dC = np.empty_like(dCs)
    dC[p] = dCs
    return dE, dC, keep


def _rows_put_back_inverted(E, C, x, lse, w, BN, BV, eps, ignore_index=-100, compact_ignored=False,
                            vocab_perm=None):
    dE, dC, keep = O.backward_filtered(E, C, x, lse, w, BN, BV, eps, ignore_index,
                                       compact_ignored=compact_ignored, vocab_perm=vocab_perm)
    p = np.asarray(vocab_perm)
    dCs = dC[p]  # the rows in sorted order, then put back the wrong way round
    return dE, dCs[p], keep


@pytest.mark.parametrize("mutant", [_targets_not_moved, _rows_put_back_inverted])
def test_planted_sorting_mistakes_are_caught(rng, mutant):
    E, C, x, f, w = _setup(rng)
    perm = rng.permutation(C.shape[0])
    assert not _check_unfiltered(mutant, E, C, x, f, w, perm)
