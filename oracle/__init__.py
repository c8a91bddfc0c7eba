"""fp64 CPU oracle for Cut Cross-Entropy (linear cross-entropy).

TEST INFRASTRUCTURE ONLY.  This package is imported by the tests, by
``__graft_entry__.smoke()`` and by ``bench.py``'s CPU-baseline / reference
legs, and by nothing else.  The product path (``linear_cross_entropy_gb300``)
never imports it, and this package imports nothing from the product: the two
share only the seeded input generator ``cce_workloads``.

What it computes is the plain definition of the loss and its gradient, in
float64, from the bf16-rounded inputs widened exactly to float64:

* logits            a_iv = sum_d E_id C_vd            (one library matmul)
* log-sum-exp       LSE_i = m_i + log sum_v exp(a_iv - m_i),  m_i = max_v a_iv
* loss              loss_i = LSE_i - a_{i, x_i}
* logit gradient    G_iv = exp(a_iv - LSE_i) - [v = x_i]
* input gradients   dE_i = w_i sum_v G_iv C_v ,   dC_v = sum_i w_i G_iv E_i

Passages followed (page title, section):

* "Cut Cross-Entropy: Training Loss Without the Logit Matrix, and Why 0.1%
  Element Sparsity Becomes 50% Block Sparsity" -- section "The decomposition"
  (loss = LSE - target logit; backward G = S - onehot, dE = G C, dC = G^T E);
  section "Gradient filtering: the part that makes it fast" (a tile is
  skipped when every |G| < eps, eps = 2^-12, tested on |S - onehot|).
* "Cut Your Losses in Large-Vocabulary Language Models" -- "The Mathematical
  Decomposition" (the loss splits into an indexed logit and a log-sum-exp),
  "Memory-Efficient Linear-Log-Sum-Exp, Backward Pass (Algorithm 3)",
  "The Combined Backward Pass (Algorithm 4)".  That page writes the
  log-likelihood (target - LSE) and G = onehot - S; the loss here is its
  negative, LSE - target, whose gradient is S - onehot (the first page's
  sign).
* "cut-cross-entropy" kernel card -- "Correctness": ignore_index rows add no
  loss and get exactly zero gradient; a fully masked batch has zero loss and
  zero gradients; reductions none / sum / mean.
* Logit softcapping (Gemma 2's final logits; the paper's backward-pass
  breakdown, "Cut Your Losses ...", Table A2, times it as its own stage):
  with cap > 0 the logits are a'_iv = cap tanh(a_iv / cap); LSE, loss and
  G = softmax(a') - onehot use a', and the gradient reaching E and C is
  G (1 - tanh^2(a / cap)).  The filter tests |G| before that factor.
* Vocabulary sorting ("Cut Your Losses ...", section "Vocabulary Sorting"):
  the vocabulary is reordered by each token's average logit over the batch
  so that tokens with large softmax values share tiles; the filter then
  works on tiles of consecutive sorted positions.  The order (ascending,
  equal keys by token id) follows the argsort the first page names.  Sorting
  changes which tiles exist, never the unfiltered result.
* The single call ("fused-linear-cross-entropy" page, section "2. Fused
  Linear Cross-Entropy (FLCE)"): loss and both gradients computed together
  for a unit upstream gradient, which the backward then multiplies in.
* Reading where the pages are silent: mean divides by the number of
  non-ignored rows, clamped to at least 1 (the chunked-CE code on the
  "fused-linear-cross-entropy" page clamps the count the same way); the LSE of
  an ignored row is still the true LSE of its logits.

The gradient weights w_i follow from the reduction: w_i = g (sum),
g / max(count, 1) (mean), g_i (none), and 0 on ignored rows, where g is the
incoming gradient of the reduced loss.

Pins (tests/test_oracle_pins.py): closed forms (C = 0 gives loss = log V;
N = 1, V = 2 gives a softplus), central finite differences of the loss for dE
and dC, torch.nn.functional.cross_entropy on materialised fp64 logits,
row sums of G equal to zero, vocabulary-permutation invariance, the
pigeonhole bound on entries >= 2^-12 and the eps tie case; for sorting, the
logit sums by brute-force loops and by the linearity C (sum_i E_i), the order
by brute-force rank counting and a hand-sorted example, and the sorted
filtered backward by its independence of the input vocabulary order.  Every function
below is pinned by at least one of them.
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100
FILTER_EPS = 2.0 ** -12  # finfo(bf16).eps / 32

_ROW_BLOCK_BYTES = 1 << 28  # memory bound for one block of dense logit rows


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _row_blocks(n_rows: int, V: int):
    step = max(1, _ROW_BLOCK_BYTES // (8 * max(V, 1)))
    for r0 in range(0, n_rows, step):
        yield r0, min(n_rows, r0 + step)


def logits(E: np.ndarray, C: np.ndarray) -> np.ndarray:
    """a = E C^T for the given rows of E (float64 matmul)."""
    return E @ C.T


def softcap_logits(A: np.ndarray, softcap: float) -> np.ndarray:
    """a' = cap tanh(a / cap) (identity when cap == 0)."""
    return A if not softcap else softcap * np.tanh(A / softcap)


def softcap_slope(A: np.ndarray, softcap: float):
    """d a' / d a = 1 - tanh^2(a / cap) (1 when cap == 0)."""
    return 1.0 if not softcap else 1.0 - np.tanh(A / softcap) ** 2


def log_sum_exp(A: np.ndarray) -> np.ndarray:
    """Row-wise LSE_i = m_i + log sum_v exp(a_iv - m_i)."""
    m = A.max(axis=1)
    return m + np.log(np.exp(A - m[:, None]).sum(axis=1))


def forward(E, C, x, ignore_index=IGNORE_INDEX, reduction="mean", rows=None, softcap=0.0):
    """Forward pass for the listed rows (all rows when rows is None).

    Returns a dict with per-row ``lse``, ``target_logit`` (NaN on ignored
    rows), ``loss_rows`` (0 on ignored rows) and, when all rows were
    computed, ``count`` (non-ignored rows) and the reduced ``loss``.
    """
    E = np.asarray(E, np.float64)
    C = np.asarray(C, np.float64)
    x = np.asarray(x, np.int64)
    V = C.shape[0]
    idx = np.arange(E.shape[0]) if rows is None else np.asarray(rows, np.int64)
    lse = np.empty(len(idx))
    tgt = np.full(len(idx), np.nan)
    for r0, r1 in _row_blocks(len(idx), V):
        rr = idx[r0:r1]
        A = softcap_logits(logits(E[rr], C), softcap)
        lse[r0:r1] = log_sum_exp(A)
        xr = x[rr]
        ok = xr != ignore_index
        if np.any(ok & ((xr < 0) | (xr >= V))):
            raise ValueError("target out of range")
        sel = np.nonzero(ok)[0]
        tgt[r0 + sel] = A[sel, xr[sel]]
    valid = x[idx] != ignore_index
    loss_rows = np.where(valid, lse - np.where(valid, tgt, 0.0), 0.0)
    out = {"lse": lse, "target_logit": tgt, "loss_rows": loss_rows}
    if rows is None:
        count = int(valid.sum())
        out["count"] = count
        out["loss"] = reduce_loss(loss_rows, count, reduction)
    return out


def indexed_logits(E, C, x, ignore_index=IGNORE_INDEX, softcap=0.0):
    """o_i = C[x_i] . E_i, the indexed matrix product (NaN on ignored rows)."""
    E = np.asarray(E, np.float64)
    C = np.asarray(C, np.float64)
    x = np.asarray(x, np.int64)
    ok = x != ignore_index
    out = np.full(E.shape[0], np.nan)
    out[ok] = softcap_logits(np.einsum("nd,nd->n", E[ok], C[x[ok]]), softcap)
    return out


def reduce_loss(loss_rows, count, reduction):
    """none -> the rows; sum -> their sum; mean -> sum / max(count, 1)."""
    if reduction == "none":
        return np.asarray(loss_rows, np.float64)
    s = float(np.sum(loss_rows))
    if reduction == "sum":
        return s
    if reduction == "mean":
        return s / max(count, 1)
    raise ValueError(reduction)


def row_weights(x, ignore_index, reduction, grad_out, count=None):
    """w_i: the factor multiplying row i's logit gradient."""
    x = np.asarray(x, np.int64)
    valid = x != ignore_index
    if reduction == "none":
        g = np.broadcast_to(np.asarray(grad_out, np.float64), x.shape)
        return np.where(valid, g, 0.0)
    g = float(np.asarray(grad_out, np.float64).reshape(()))
    if reduction == "sum":
        return np.where(valid, g, 0.0)
    if reduction == "mean":
        n = int(valid.sum()) if count is None else int(count)
        return np.where(valid, g / max(n, 1), 0.0)
    raise ValueError(reduction)


def grad_logits(A, lse, x_rows, v0=0, ignore_index=IGNORE_INDEX, softcap=0.0):
    """G = exp(A' - LSE) - onehot(x) for a block of raw logits A (A' = the
    softcapped logits; A' = A without a cap).

    A holds rows (tokens) x columns v0 .. v0 + A.shape[1] - 1 of the logit
    matrix; ignored rows are all zero.  This is the gradient with respect to
    A'; the filter tests it.
    """
    G = np.exp(softcap_logits(A, softcap) - np.asarray(lse)[:, None])
    x_rows = np.asarray(x_rows, np.int64)
    r = np.nonzero((x_rows >= v0) & (x_rows < v0 + A.shape[1]))[0]
    G[r, x_rows[r] - v0] -= 1.0
    G[x_rows == ignore_index] = 0.0
    return G


def backward_dE(E, C, x, lse_rows, w_rows, rows, ignore_index=IGNORE_INDEX, softcap=0.0):
    """dE_i = w_i sum_v G_iv s_iv C_v for the listed rows (lse/w given per
    listed row; s = softcap slope, 1 without a cap)."""
    E = np.asarray(E, np.float64)
    C = np.asarray(C, np.float64)
    rows = np.asarray(rows, np.int64)
    out = np.empty((len(rows), E.shape[1]))
    for r0, r1 in _row_blocks(len(rows), C.shape[0]):
        rr = rows[r0:r1]
        A = logits(E[rr], C)
        G = grad_logits(A, lse_rows[r0:r1], x[rr], 0, ignore_index, softcap) * softcap_slope(A, softcap)
        out[r0:r1] = np.asarray(w_rows[r0:r1])[:, None] * (G @ C)
    return out


def backward_dC(E, C, x, lse, w, vrows, ignore_index=IGNORE_INDEX, softcap=0.0):
    """dC_v = sum_i w_i G_iv s_iv E_i for the listed vocabulary rows.

    Needs LSE and w for every token row i.
    """
    E = np.asarray(E, np.float64)
    C = np.asarray(C, np.float64)
    x = np.asarray(x, np.int64)
    vrows = np.asarray(vrows, np.int64)
    A = logits(E, C[vrows])                      # [N, len(vrows)]
    G = np.exp(softcap_logits(A, softcap) - np.asarray(lse)[:, None])
    G -= (x[:, None] == vrows[None, :]).astype(np.float64)
    G[x == ignore_index] = 0.0
    G *= softcap_slope(A, softcap)
    return (np.asarray(w)[:, None] * G).T @ E


def backward(E, C, x, lse, w, ignore_index=IGNORE_INDEX, softcap=0.0):
    """Full dE [N, D] and dC [V, D] (small problems: materialises G)."""
    E = np.asarray(E, np.float64)
    C = np.asarray(C, np.float64)
    A = logits(E, C)
    G = grad_logits(A, lse, x, 0, ignore_index, softcap) * softcap_slope(A, softcap)
    Gw = np.asarray(w)[:, None] * G
    return Gw @ C, Gw.T @ E


def tile_survival(E, C, x, lse, BN, BV, eps=FILTER_EPS, ignore_index=IGNORE_INDEX, softcap=0.0):
    """Filter decision per (BN x BV) tile: True when some in-range entry has
    |G_iv| >= eps (unscaled G = softmax - onehot, before any softcap slope;
    ignored rows contribute nothing)."""
    E = np.asarray(E, np.float64)
    C = np.asarray(C, np.float64)
    return tile_keep(grad_logits(logits(E, C), lse, x, 0, ignore_index, softcap), BN, BV, eps)


def tile_keep(G, BN, BV, eps=FILTER_EPS):
    """Survival of each (BN x BV) tile of a logit-gradient matrix G: the tile
    is skipped iff every |G| < eps, so an entry equal to eps keeps it."""
    G = np.abs(np.asarray(G))
    nbn, nbv = -(-G.shape[0] // BN), -(-G.shape[1] // BV)
    keep = np.zeros((nbn, nbv), dtype=bool)
    for a in range(nbn):
        for b in range(nbv):
            keep[a, b] = bool(np.any(G[a * BN:(a + 1) * BN, b * BV:(b + 1) * BV] >= eps))
    return keep


def backward_filtered(E, C, x, lse, w, BN, BV, eps=FILTER_EPS, ignore_index=IGNORE_INDEX,
                      filter_dE=True, filter_dC=True, softcap=0.0, compact_ignored=False, vocab_perm=None):
    """dE, dC with the contributions of skipped tiles removed from the
    outputs whose filter is on; also returns the survival map.  With eps = 0
    no tile is skipped.  filter_dE only ("Cut Your Losses ...", "Numerical
    Stability Variants": CCE-Kahan-FullC computes dC from every tile) and
    filter_dC only (CCE-Kahan-FullE).

    compact_ignored: remove the ignored rows first ("Cut Your Losses ...",
    Table A1: removing ignored tokens), so the BN-row tiles are made of
    consecutive non-ignored rows; dE rows are returned in the original order
    (ignored rows 0) and the survival map is over the compact rows.

    vocab_perm: the vocabulary in sorted order (vocab_perm[j] = the token at
    position j; "Cut Your Losses ...", section "Vocabulary Sorting").  The
    BV-column tiles are then made of consecutive sorted positions: the
    problem is solved on C[vocab_perm] with each target replaced by its
    sorted position, and the rows of dC are put back in token order.  The
    survival map is over sorted positions."""
    if vocab_perm is not None:
        p = np.asarray(vocab_perm, np.int64)
        V = p.shape[0]
        inv = np.empty(V, np.int64)
        inv[p] = np.arange(V)
        x = np.asarray(x, np.int64)
        take = (x != ignore_index) & (x >= 0) & (x < V)
        # rows that take part get their target's sorted position; the rest get
        # -1, outside [0, V), and -1 becomes the ignore index of the sub-call
        xs = np.where(take, inv[np.where(take, x, 0)], -1)
        dE, dCs, keep = backward_filtered(E, np.asarray(C)[p], xs, lse, w, BN, BV, eps, -1, filter_dE,
                                          filter_dC, softcap, compact_ignored, None)
        dC = np.empty_like(dCs)
        dC[p] = dCs
        return dE, dC, keep
    if compact_ignored:
        x = np.asarray(x, np.int64)
        keep_rows = np.nonzero(x != ignore_index)[0]
        dEc, dC, keep = backward_filtered(np.asarray(E)[keep_rows], C, x[keep_rows], np.asarray(lse)[keep_rows],
                                          np.asarray(w)[keep_rows], BN, BV, eps, ignore_index, filter_dE,
                                          filter_dC, softcap, False)
        dE = np.zeros((x.shape[0], dEc.shape[1]))
        dE[keep_rows] = dEc
        return dE, dC, keep
    E = np.asarray(E, np.float64)
    C = np.asarray(C, np.float64)
    A = logits(E, C)
    G = grad_logits(A, lse, x, 0, ignore_index, softcap)
    keep = tile_keep(G, BN, BV, eps)
    mask = np.repeat(np.repeat(keep, BN, axis=0), BV, axis=1)[:G.shape[0], :G.shape[1]]
    Gw = np.asarray(w)[:, None] * G * softcap_slope(A, softcap)
    Gf = np.where(mask, Gw, 0.0)
    return (Gf if filter_dE else Gw) @ C, (Gf if filter_dC else Gw).T @ E, keep


def loss_and_grad(E, C, x, ignore_index=IGNORE_INDEX, reduction="mean", softcap=0.0, filter_eps=0.0, BN=128,
                  BV=128, filter_dE=True, filter_dC=True):
    """The single-call form of the loss ("fused-linear-cross-entropy" page,
    section "2. Fused Linear Cross-Entropy (FLCE)"): the loss and both
    gradients in one pass, for the reduced loss with a unit upstream gradient;
    the autograd backward only multiplies them by the upstream gradient
    (which is exact: both gradients are linear in it).  Only the sum and mean
    reductions have a scalar upstream gradient, so only they are defined.

    It is forward() followed by backward() with grad_out = 1.  With
    filter_eps > 0 the skipped tiles' contributions are removed as in
    backward_filtered with the ignored rows removed first ("Cut Your Losses
    ...", Table A1: removing ignored tokens), so a filter tile is 128
    consecutive rows that take part x 128 vocabulary entries, as in the
    two-call backward.  Returns {loss, lse, count, dE, dC, keep}."""
    if reduction not in ("sum", "mean"):
        raise ValueError("the single call is defined for the sum and mean reductions")
    E = np.asarray(E, np.float64)
    C = np.asarray(C, np.float64)
    f = forward(E, C, x, ignore_index, reduction, softcap=softcap)
    w = row_weights(x, ignore_index, reduction, 1.0, f["count"])
    if filter_eps:
        dE, dC, keep = backward_filtered(E, C, x, f["lse"], w, BN, BV, filter_eps, ignore_index, filter_dE,
                                         filter_dC, softcap, compact_ignored=True)
    else:
        dE, dC = backward(E, C, x, f["lse"], w, ignore_index, softcap)
        keep = None
    return {"loss": f["loss"], "lse": f["lse"], "count": f["count"], "dE": dE, "dC": dC, "keep": keep}


def vocab_logit_sums(E, C, x, ignore_index=IGNORE_INDEX):
    """The statistic vocabulary sorting orders by ("Cut Your Losses ...",
    section "Vocabulary Sorting"): for every token v, the sum over the rows
    that take part of the logit a_iv = C_v . E_i, and the number of those rows
    (the average logit is sum / count, so both order the vocabulary alike).
    A row takes part when its target is in [0, V) and is not ignore_index.
    Returns (sums [V] float64, count)."""
    E = np.asarray(E, np.float64)
    C = np.asarray(C, np.float64)
    x = np.asarray(x, np.int64)
    V = C.shape[0]
    rows = np.nonzero((x != ignore_index) & (x >= 0) & (x < V))[0]
    S = np.zeros(V)
    for r0, r1 in _row_blocks(len(rows), V):
        S += logits(E[rows[r0:r1]], C).sum(axis=0)
    return S, int(len(rows))


def vocab_order(keys):
    """The sorted vocabulary: perm[j] is the token at position j, with the keys
    in ascending order ("Cut Cross-Entropy: Training Loss Without the Logit
    Matrix ...", section "Gradient filtering: the part that makes it fast",
    sorts with an ascending argsort of the average logit) and equal keys in
    increasing token id (a stable sort; -0.0 equals +0.0)."""
    return np.argsort(np.asarray(keys, np.float64), kind="stable")


def from_bits(E_bits, C_bits):
    """Widen the bf16 inputs of a workload to float64 (E, C)."""
    return widen_bf16(E_bits), widen_bf16(C_bits)


def fwd_bwd_rows(E, C, x, rows, ignore_index=IGNORE_INDEX, reduction="mean", grad_out=1.0, softcap=0.0):
    """Forward + backward of the sub-problem made of the listed token rows
    (a standalone batch): returns (loss, dE_rows, dC).  Used to time the
    oracle on a bounded sample of a workload."""
    rows = np.asarray(rows, np.int64)
    Es, xs = np.asarray(E)[rows], np.asarray(x)[rows]
    f = forward(Es, C, xs, ignore_index, reduction, softcap=softcap)
    w = row_weights(xs, ignore_index, reduction, grad_out, f["count"])
    dE, dC = backward(Es, C, xs, f["lse"], w, ignore_index, softcap)
    return f["loss"], dE, dC
