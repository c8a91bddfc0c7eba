"""GPU-vs-oracle parity on seeded inputs, through the C ABI.

Sizes are small enough for the fp64 oracle to finish in seconds, yet span
several 128 x 256 tiles and ragged tails in N, D and V, several backward
vocabulary chunks, every reduction, ignored rows and the filter on and off.
"""
import numpy as np
import pytest
import torch

import cce_workloads as W
import oracle as O
from tests.gpu_util import (TOL_GRAD, TOL_GRAD_FILTERED, TOL_LSE, TOL_ROW, assert_forward_close,
                            assert_grads_close, bf16_to_f64, make, mixed_survival_inputs, oracle_full, rel_fro,
                            row_max_rel, run_cuda, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests.conftest import build_library
    build_library()


@pytest.mark.parametrize("filter_on", [True, False])
def test_tiny_config(filter_on):
    """The tiny workload (N=256, D=128, V=4096, mean), full comparison."""
    w, (E, C, x) = make("tiny")
    eps = O.FILTER_EPS if filter_on else 0.0
    got = run_cuda(E, C, x, reduction=w.reduction, filter_eps=eps)
    ref = oracle_full(E, C, x, reduction=w.reduction)
    assert_forward_close(got, ref, w.reduction, x)
    assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD_FILTERED if filter_on else TOL_GRAD, x)


@pytest.mark.parametrize("N,D,V", [
    (300, 96, 1000),    # ragged in every dimension; D not a multiple of 64
    (129, 64, 257),     # one row / one column past a tile
    (1, 64, 300),       # a single token
    (1000, 256, 5000),  # several row blocks and vocabulary tiles
    (640, 128, 9000),   # several backward chunks
    (300, 448, 3000),   # two gradient D tiles, the second one ragged (192 of 256 columns)
    (260, 600, 2000),   # three gradient D tiles, the last one ragged (88 of 256 columns)
    (700, 384, 3000),   # D tiles of 256 and 128: CTA pairs run the second with N = 128
])
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_ragged_shapes_unfiltered(N, D, V, reduction):
    w, (E, C, x) = make(W.small("r", N, D, V, reduction=reduction))
    g = np.random.default_rng(N + V).standard_normal(N) if reduction == "none" else 1.0
    got = run_cuda(E, C, x, reduction=reduction, filter_eps=0.0, grad_out=g)
    ref = oracle_full(E, C, x, reduction=reduction, grad_out=g)
    assert_forward_close(got, ref, reduction, x)
    assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD, x)


@pytest.mark.parametrize("ignore_frac", [0.0, 0.1])
def test_many_token_blocks_cta_pairs(ignore_frac):
    """Enough token blocks (65) that the forward and the recompute run as CTA
    pairs, with an odd block count (the last pair half empty) in the forward
    and, after compaction of the ignored rows, in the recompute."""
    N, D, V = 65 * 128, 64, 3000
    w, (E, C, x) = make(W.small("pairs", N, D, V, ignore_frac=ignore_frac))
    got = run_cuda(E, C, x, reduction="mean", filter_eps=0.0)
    ref = oracle_full(E, C, x, reduction="mean")
    assert_forward_close(got, ref, "mean", x)
    assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD, x)


def test_target_in_short_final_panel():
    """'Correctness': a ragged vocabulary with targets inside the short final panel."""
    N, D, V = 200, 64, 1000 + 37
    w, (E, C, x) = make(W.small("p", N, D, V, ignore_frac=0.0))
    x = x.copy()
    x[::3] = V - 1 - (np.arange(len(x[::3])) % 37)
    got = run_cuda(E, C, x, reduction="mean", filter_eps=0.0)
    ref = oracle_full(E, C, x, reduction="mean")
    assert_forward_close(got, ref, "mean", x)
    assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD, x)


def test_multi_chunk_backward():
    """V wide enough for several backward vocabulary chunks (dE accumulates)."""
    import linear_cross_entropy_gb300 as cce
    N, D, V = 256, 64, 40000
    assert cce.memory_report(N, D, V)["bwd_chunk_cols"] < V
    w, (E, C, x) = make(W.small("c", N, D, V))
    got = run_cuda(E, C, x, reduction="mean", filter_eps=0.0)
    ref = oracle_full(E, C, x, reduction="mean")
    assert_forward_close(got, ref, "mean", x)
    assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD, x)


@pytest.mark.parametrize("D", [128, 256])
def test_filter_matches_filtered_oracle(D):
    """Frequent-token inputs: softmax mass sits in the lowest 256 ids, so most
    128 x 128 tiles are skipped.  The filtered result matches the filtered
    oracle tightly and the unfiltered oracle within 1e-2; the skip count
    equals the oracle's tile survival map (no tile lies near eps here).
    D = 256: one full-width gradient D tile, whose MN-major B operand comes in
    one 3-D box of four 64-column groups."""
    N, V = 512, 6000
    E, C, x = W.frequent_token_inputs(N, D, V, n_freq=256, seed=3)
    got = run_cuda(E, C, x, reduction="mean", filter_eps=O.FILTER_EPS)
    ref = oracle_full(E, C, x, reduction="mean", filter_eps=O.FILTER_EPS)
    assert_forward_close(got, ref, "mean", x)
    assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD_FILTERED, x)
    assert rel_fro(got["dE"], ref["dE_f"]) <= TOL_GRAD
    assert rel_fro(got["dC"], ref["dC_f"]) <= TOL_GRAD
    # the filtered oracle takes the same tile decisions: every row agrees too
    assert row_max_rel(got["dE"], ref["dE_f"]) <= TOL_ROW
    assert row_max_rel(got["dC"], ref["dC_f"]) <= TOL_ROW
    keep = ref["keep"]
    st = got["stats"]
    assert st["tiles"] == keep.size
    assert st["skipped"] == int((~keep).sum())
    assert st["skipped"] > keep.size // 2
    # rows of dC in fully skipped vocabulary slices are exact zeros
    dead = np.nonzero(~keep.any(axis=0))[0]
    assert len(dead) > 0
    for b in dead[:8]:
        assert np.all(got["dC"][b * 128:(b + 1) * 128] == 0.0)


@pytest.mark.parametrize("N,words", [(3000, 0), (20000, 1)])
def test_neighbouring_blocks_keep_different_k_blocks(N, words):
    """The gradient GEMM as CTA pairs (D = 256: M = 256 over two neighbouring
    row blocks) where the two blocks of a pair keep different K-blocks: the
    pair runs the union, and a CTA loads zeros for a K-block only its partner
    keeps.  Most token-block pairs differ here (dE), and vocabulary blocks 0
    and 1 do (dC: block 0 keeps every token block, block 1 a third of them).
    words = 1: a work item carries one survival word (64 filter columns), so
    the dC tiles' K range (149 token blocks) is longer than that and the
    producer walks the maps itself, as it does beyond 327,680 rows.  No tile
    lies within 0.1% of eps (checked on the oracle), so the skip count must
    equal the oracle's exactly.  (The skipped tiles' sum is not small against
    the kept one in this input, so only the filtered oracle is the
    reference.)"""
    from linear_cross_entropy_gb300 import _lib
    lib = _lib.load()
    D, V = 256, 1500
    E, C, x = mixed_survival_inputs(N, D, V)
    prev = lib.cce_selftest_pair_map_words(words)
    prev_layout = lib.cce_selftest_grad_layout(1)  # pairs (the automatic choice takes one CTA per tile here)
    try:
        got = run_cuda(E, C, x, reduction="mean", filter_eps=O.FILTER_EPS)
    finally:
        lib.cce_selftest_pair_map_words(prev)
        lib.cce_selftest_grad_layout(prev_layout)
    ref = oracle_full(E, C, x, reduction="mean", filter_eps=O.FILTER_EPS)
    Ef, Cf = O.from_bits(E, C)
    w = O.row_weights(x, O.IGNORE_INDEX, "mean", 1.0, int((x != O.IGNORE_INDEX).sum()))
    keep = ref["keep"]
    for eps in (O.FILTER_EPS * (1 - 1e-3), O.FILTER_EPS * (1 + 1e-3)):
        _, _, k2 = O.backward_filtered(Ef, Cf, x, ref["lse"], w, 128, 128, eps, compact_ignored=True)
        assert np.array_equal(k2, keep), "an input tile lies near eps"
    nb, nv = keep.shape
    assert sum(not np.array_equal(keep[p], keep[p + 1]) for p in range(0, nb - 1, 2)) > nb // 8
    assert not np.array_equal(keep[:, 0], keep[:, 1])
    if words:
        assert (nb + 63) // 64 > words
    assert_forward_close(got, ref, "mean", x)
    st = got["stats"]
    assert st["tiles"] == keep.size
    assert st["skipped"] == int((~keep).sum()) > 0
    assert rel_fro(got["dE"], ref["dE_f"]) <= TOL_GRAD
    assert rel_fro(got["dC"], ref["dC_f"]) <= TOL_GRAD
    assert row_max_rel(got["dE"], ref["dE_f"]) <= TOL_ROW
    assert row_max_rel(got["dC"], ref["dC_f"]) <= TOL_ROW


@pytest.mark.parametrize("D", [256, 384])
@pytest.mark.parametrize("filter_eps", [O.FILTER_EPS, 0.0])
def test_gradient_layouts_agree_bitwise(filter_eps, D):
    """The gradient GEMM as CTA pairs and one CTA per tile accumulate each
    tile's kept K-blocks in the same order (the K-blocks a pair runs only for
    the other tile multiply zeros), so dE and dC are the same bits, on inputs
    whose neighbouring blocks keep different K-blocks; and the automatic
    choice between the two (by the chunk's kept tiles) agrees as well.
    D = 384: the pairs run the 128-column second D tile with N = 128."""
    from linear_cross_entropy_gb300 import _lib
    lib = _lib.load()
    E, C, x = mixed_survival_inputs(3000, D, 1500)
    runs = []
    for layout in (1, 2, 0):
        prev = lib.cce_selftest_grad_layout(layout)
        try:
            runs.append(run_cuda(E, C, x, reduction="mean", filter_eps=filter_eps))
        finally:
            lib.cce_selftest_grad_layout(prev)
    for other in runs[1:]:
        assert np.array_equal(runs[0]["dE"], other["dE"]) and np.array_equal(runs[0]["dC"], other["dC"])
        assert runs[0]["stats"] == other["stats"]


@pytest.mark.parametrize("D,filter_eps", [(64, O.FILTER_EPS), (64, 0.0), (256, 0.0)])
def test_fully_ignored_batch(D, filter_eps):
    """'Correctness': a fully masked batch gives zero loss and finite zero
    gradients, with the filter on or off (off, the dC tiles have no K-block
    at all and nothing marks them as skipped).  D = 256: the gradient GEMM
    runs as CTA pairs."""
    w, (E, C, x) = make(W.small("i", 300, D, 1000))
    x = np.full_like(x, -100)
    got = run_cuda(E, C, x, reduction="mean", filter_eps=filter_eps)
    assert float(got["loss"].reshape(())) == 0.0
    assert np.all(got["dE"] == 0.0) and np.all(got["dC"] == 0.0)
    assert np.all(np.isfinite(got["lse"]))
    if filter_eps == 0.0:
        return
    # the autograd path (its forward skips the rows that take part in nothing: all of them here)
    import linear_cross_entropy_gb300 as cce
    Et, Ct, xt = to_device(E, C, x)
    Et.requires_grad_(True)
    Ct.requires_grad_(True)
    loss = cce.linear_cross_entropy(Et, Ct, xt)
    loss.backward()
    cce.raise_pending_errors()
    assert loss.item() == 0.0
    assert not Et.grad.any() and not Ct.grad.any()


def test_custom_ignore_index():
    w, (E, C, x) = make(W.small("j", 200, 64, 700, ignore_frac=0.0))
    x = x.copy()
    x[5:40] = 7  # rows whose target equals the custom ignore_index are ignored
    got = run_cuda(E, C, x, ignore_index=7, reduction="sum", filter_eps=0.0)
    ref = oracle_full(E, C, x, ignore_index=7, reduction="sum")
    assert_forward_close(got, ref, "sum", x, ignore_index=7)
    assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD, x, ignore_index=7)


def test_repeated_calls_are_bitwise_identical():
    import linear_cross_entropy_gb300 as cce
    from tests.gpu_util import to_device
    w, (E, C, x) = make(W.small("d", 700, 128, 3000))
    Et, Ct, xt = to_device(E, C, x)
    l1, s1 = cce.cce_forward(Et, Ct, xt)
    l2, s2 = cce.cce_forward(Et, Ct, xt)
    assert torch.equal(l1, l2) and torch.equal(s1, s2)
    g = torch.ones(1, device="cuda")
    a = cce.cce_backward(Et, Ct, xt, s1, g)
    b = cce.cce_backward(Et, Ct, xt, s1, g)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_out_of_range_target_is_reported():
    import linear_cross_entropy_gb300 as cce
    from tests.gpu_util import to_device
    w, (E, C, x) = make(W.small("o", 64, 64, 500, ignore_frac=0.0))
    x = x.copy()
    x[3] = 500
    x[9] = -5
    Et, Ct, xt = to_device(E, C, x)
    with pytest.raises(cce.CCEError) as ei:
        cce.cce_forward(Et, Ct, xt)
    assert ei.value.status == 8
    # the row was treated as ignored: the call completed and the context is usable
    loss, lse = cce.cce_forward(Et, Ct, xt, check_errors=False)
    assert torch.isfinite(lse).all()
    with pytest.raises(cce.CCEError):
        cce.cce_backward(Et, Ct, xt, lse, torch.ones(1, device="cuda"))


def test_autograd_path_reports_errors_without_stalling():
    """The autograd wrappers do not wait for the GPU to check the error word:
    the error of a bad target surfaces at raise_pending_errors()."""
    import linear_cross_entropy_gb300 as cce
    from tests.gpu_util import to_device
    w, (E, C, x) = make(W.small("o", 64, 64, 500, ignore_frac=0.0))
    x = x.copy()
    x[5] = 777
    Et, Ct, xt = to_device(E, C, x)
    for fn, calls in ((cce.linear_cross_entropy, 2), (cce.fused_linear_cross_entropy, 1)):
        Eg, Cg = Et.clone().requires_grad_(True), Ct.clone().requires_grad_(True)
        reported = []
        try:  # the backward may already report the forward's word
            fn(Eg, Cg, xt).backward()
        except cce.CCEError as e:
            reported.append(e.status)
        while True:
            try:
                cce.raise_pending_errors()
                break
            except cce.CCEError as e:
                reported.append(e.status)
        # every library call of the step flagged the bad target, each once
        assert reported == [8] * calls
        cce.raise_pending_errors()
    # a clean batch after the bad one raises nothing
    x[5] = 3
    Et, Ct, xt = to_device(E, C, x)
    Eg = Et.clone().requires_grad_(True)
    cce.linear_cross_entropy(Eg, Ct, xt).backward()
    cce.raise_pending_errors()


def test_deferred_error_words_wrap_around_their_ring():
    """More autograd calls than the ring of pinned error words holds: clean
    calls report nothing, and a bad target after them is reported once per
    library call that saw it."""
    import linear_cross_entropy_gb300 as cce
    from tests.gpu_util import to_device
    w, (E, C, x) = make(W.small("o", 64, 64, 500, ignore_frac=0.0))
    Et, Ct, xt = to_device(E, C, x)
    for _ in range(cce._DeferredErrors.SLOTS + 5):  # two calls (forward, backward) each
        Eg = Et.clone().requires_grad_(True)
        cce.linear_cross_entropy(Eg, Ct, xt).backward()
    cce.raise_pending_errors()
    x = x.copy()
    x[7] = 500
    Et, Ct, xt = to_device(E, C, x)
    Eg = Et.clone().requires_grad_(True)
    reported = []
    try:
        cce.linear_cross_entropy(Eg, Ct, xt).backward()
    except cce.CCEError as e:
        reported.append(e.status)
    while True:
        try:
            cce.raise_pending_errors()
            break
        except cce.CCEError as e:
            reported.append(e.status)
    assert reported == [8, 8]


def test_autograd_function_matches_oracle():
    import linear_cross_entropy_gb300 as cce
    from tests.gpu_util import to_device
    w, (E, C, x) = make(W.small("a", 300, 128, 2000))
    Et, Ct, xt = to_device(E, C, x)
    Et.requires_grad_(True)
    Ct.requires_grad_(True)
    loss = cce.linear_cross_entropy(Et, Ct, xt, filter_eps=0.0)
    (2.5 * loss).backward()
    ref = oracle_full(E, C, x, reduction="mean", grad_out=2.5)
    assert abs(loss.item() - ref["loss"]) <= 1e-5 * abs(ref["loss"])
    assert rel_fro(Et.grad.double().cpu().numpy(), ref["dE"]) <= TOL_GRAD
    assert rel_fro(Ct.grad.double().cpu().numpy(), ref["dC"]) <= TOL_GRAD


def test_no_n_by_v_allocation():
    """The caching allocator never sees an N x V-sized block during fwd + bwd."""
    import linear_cross_entropy_gb300 as cce
    from tests.gpu_util import to_device
    N, D, V = 2048, 256, 60000
    w, (E, C, x) = make(W.small("m", N, D, V))
    Et, Ct, xt = to_device(E, C, x)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    loss, lse = cce.cce_forward(Et, Ct, xt)
    dE, dC = cce.cce_backward(Et, Ct, xt, lse, torch.ones(1, device="cuda"))
    torch.cuda.synchronize()
    extra = torch.cuda.max_memory_allocated() - base
    outputs = dE.numel() * 2 + dC.numel() * 2 + lse.numel() * 4 + 4
    assert extra - outputs < N * V * 2, (extra, outputs)


@pytest.mark.parametrize("outputs,fde,fdc", [("dE", True, False), ("dC", False, True), ("none", False, False)])
def test_per_output_filter_flags(outputs, fde, fdc):
    """Per-output filtering (the pages' CCE-Kahan-FullC / FullE variants) on
    the frequent-token workload, against the oracle with the same flags."""
    import linear_cross_entropy_gb300 as cce
    from tests.gpu_util import to_device, bf16_to_f64
    N, D, V = 512, 128, 6000
    E, C, x = W.frequent_token_inputs(N, D, V, n_freq=256, seed=3)
    Et, Ct, xt = to_device(E, C, x)
    loss, lse = cce.cce_forward(Et, Ct, xt)
    dE, dC, st = cce.cce_backward(Et, Ct, xt, lse, torch.ones(1, device="cuda"), filter_outputs=outputs,
                                  stats=True)
    Ef, Cf = O.from_bits(E, C)
    f = O.forward(Ef, Cf, x, reduction="mean")
    w = O.row_weights(x, -100, "mean", 1.0, f["count"])
    rE, rC, keep = O.backward_filtered(Ef, Cf, x, f["lse"], w, 128, 128, O.FILTER_EPS, filter_dE=fde,
                                       filter_dC=fdc, compact_ignored=True)
    assert rel_fro(bf16_to_f64(dE), rE) <= TOL_GRAD
    assert rel_fro(bf16_to_f64(dC), rC) <= TOL_GRAD
    assert row_max_rel(bf16_to_f64(dE), rE) <= TOL_ROW
    assert row_max_rel(bf16_to_f64(dC), rC) <= TOL_ROW
    assert st["skipped"] == int((~keep).sum()) > 0


@pytest.mark.parametrize("filter_on", [False, True])
def test_softcap_against_oracle(filter_on):
    """Gemma-2-style logit softcapping (cap 30 on peaked logits, so the cap bites)."""
    import linear_cross_entropy_gb300 as cce
    from tests.gpu_util import to_device, bf16_to_f64
    cap = 30.0
    N, D, V = 384, 128, 3000
    w, (E, C, x) = make(W.small("s", N, D, V, c_scale=40.0, boost=20.0, ignore_frac=0.05))
    Et, Ct, xt = to_device(E, C, x)
    eps = O.FILTER_EPS if filter_on else 0.0
    loss, lse = cce.cce_forward(Et, Ct, xt, softcap=cap)
    dE, dC = cce.cce_backward(Et, Ct, xt, lse, torch.ones(1, device="cuda"), filter_eps=eps, softcap=cap)
    Ef, Cf = O.from_bits(E, C)
    f = O.forward(Ef, Cf, x, reduction="mean", softcap=cap)
    assert np.max(np.abs(Ef @ Cf.T)) > cap  # the cap changes the logits
    wts = O.row_weights(x, -100, "mean", 1.0, f["count"])
    rE, rC = O.backward(Ef, Cf, x, f["lse"], wts, softcap=cap)
    lse_err = np.max(np.abs(lse.double().cpu().numpy() - f["lse"]) / np.abs(f["lse"]))
    assert lse_err <= 1e-5, lse_err
    assert abs(loss.item() - f["loss"]) <= 1e-5 * abs(f["loss"])
    tol = TOL_GRAD_FILTERED if filter_on else TOL_GRAD
    assert rel_fro(bf16_to_f64(dE), rE) <= tol
    assert rel_fro(bf16_to_f64(dC), rC) <= tol


def test_mostly_ignored_batch_is_compacted():
    """70% of the rows ignored: the backward runs on the compacted rows and
    matches the oracle (unfiltered and filtered); ignored rows stay exact zeros."""
    import linear_cross_entropy_gb300 as cce
    from tests.gpu_util import to_device, bf16_to_f64
    w, (E, C, x) = make(W.small("k", 900, 128, 5000, ignore_frac=0.7, reduction="sum"))
    assert (x == -100).mean() > 0.6
    for eps in (0.0, O.FILTER_EPS):
        got = run_cuda(E, C, x, reduction="sum", filter_eps=eps)
        ref = oracle_full(E, C, x, reduction="sum", filter_eps=eps or None)
        assert_forward_close(got, ref, "sum", x)
        assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD if eps == 0 else TOL_GRAD_FILTERED, x)
        if eps:
            assert rel_fro(got["dE"], ref["dE_f"]) <= TOL_GRAD
            assert row_max_rel(got["dE"], ref["dE_f"]) <= TOL_ROW
            assert got["stats"]["tiles"] == ref["keep"].size


@pytest.mark.parametrize("reduction,ignore_frac", [("mean", 0.3), ("sum", 0.3), ("none", 0.3), ("mean", 0.1)])
def test_forward_skipping_ignored_rows(reduction, ignore_frac):
    """CCE_FWD_SKIP_IGNORED: the GEMM runs over the compacted rows only; the
    loss is the oracle's, the LSE of rows that take part too, and the other
    rows read 0; the backward fed with that LSE gives the oracle's gradients.
    480 rows take part at ignore_frac 0.3 (4 token blocks), 626 at 0.1 (5: the
    forward's last CTA pair is half empty)."""
    import linear_cross_entropy_gb300 as cce
    w = W.small("skip", 700, 136, 5000, ignore_frac=ignore_frac, reduction=reduction)
    E_bits, C_bits, x = W.make_inputs(w)
    x = x.copy()
    x[[3, 4, 5]] = O.IGNORE_INDEX
    E, C, xt = to_device(E_bits, C_bits, x)
    loss, lse = cce.cce_forward(E, C, xt, reduction=reduction, skip_ignored=True)
    g = torch.ones(x.shape[0] if reduction == "none" else 1, dtype=torch.float32, device="cuda")
    dE, dC = cce.cce_backward(E, C, xt, lse, g, reduction=reduction, filter_eps=0.0)
    torch.cuda.synchronize()
    ref = oracle_full(E_bits, C_bits, x, reduction=reduction)
    valid = x != O.IGNORE_INDEX
    lse_got = lse.double().cpu().numpy()
    err = np.abs(lse_got[valid] - ref["lse"][valid]) / np.abs(ref["lse"][valid])
    assert err.max() <= TOL_LSE and np.all(lse_got[~valid] == 0.0)
    if reduction == "none":
        rows = loss.double().cpu().numpy()
        assert np.all(np.abs(rows - ref["loss_rows"]) <= TOL_LSE * np.abs(ref["lse"]) + 1e-30)
        assert np.all(rows[~valid] == 0.0)
    else:
        assert abs(loss.item() - float(ref["loss"])) <= TOL_LSE * abs(float(ref["loss"]))
    got = {"dE": bf16_to_f64(dE), "dC": bf16_to_f64(dC), "dE_raw": dE}
    assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD, x)


@pytest.mark.parametrize("targets", ["uniform", "concentrated"])
def test_filter_threshold_tie(targets):
    """The filter at its tie: C = 0 and V = 4096 make every logit 0, so every
    non-target probability is exactly 1/4096 = 2^-12 = eps ("Cut Cross-Entropy:
    Training Loss Without the Logit Matrix ...", "Gradient filtering: the part
    that makes it fast": eps = finfo(bf16).eps / 32 and at most 4096 entries
    per row reach it).  The pages skip a tile when every |G| < eps, so ties
    survive; a tile whose max |G| lies within 1e-6 relative of eps may flip
    between the GPU's fp32 and the oracle's fp64, so the GPU's skip count must
    lie between the oracle's counts at eps (1 - 1e-6) and eps (1 + 1e-6).
    Every row has the same logits, so the GPU decides every tie the same way:
    its gradients must match the filtered oracle of that decision, and, when
    it keeps the ties (the pages' reading), the unfiltered oracle.
    "uniform": targets spread over the vocabulary (few tiles are decided by
    the tie alone); "concentrated": targets in the first 256 ids, so 30 of
    the 32 vocabulary tiles of every token block are decided by the tie."""
    N, D, V = 512, 64, 4096
    rng = np.random.default_rng(11)
    E_bits = W.f32_to_bf16_bits(rng.standard_normal((N, D)).astype(np.float32))
    C_bits = np.zeros((V, D), dtype=np.uint16)
    hi = V if targets == "uniform" else 256
    x = rng.integers(0, hi, size=N).astype(np.int64)
    got = run_cuda(E_bits, C_bits, x, reduction="mean", filter_eps=O.FILTER_EPS)
    Ef, Cf = O.from_bits(E_bits, C_bits)
    f = O.forward(Ef, Cf, x, reduction="mean")
    assert np.all(f["lse"] == 12.0 * np.log(2.0))  # log V exactly
    lse_err = np.abs(got["lse"] - f["lse"]) / f["lse"]
    assert lse_err.max() <= TOL_LSE
    assert abs(float(got["loss"].reshape(())) - float(f["loss"])) <= TOL_LSE * float(f["loss"])
    wts = O.row_weights(x, O.IGNORE_INDEX, "mean", 1.0, f["count"])
    dE_u, dC_u = O.backward(Ef, Cf, x, f["lse"], wts)
    assert np.all(dE_u == 0.0)  # C = 0
    refs = {}
    for side, eps in (("keep_ties", O.FILTER_EPS * (1 - 1e-6)), ("skip_ties", O.FILTER_EPS * (1 + 1e-6))):
        dEf, dCf, keep = O.backward_filtered(Ef, Cf, x, f["lse"], wts, 128, 128, eps, compact_ignored=True)
        refs[side] = (dCf, int((~keep).sum()), keep.size)
    lo, hi_ = refs["keep_ties"][1], refs["skip_ties"][1]
    assert lo == 0 and hi_ > 0
    st = got["stats"]
    assert st["tiles"] == refs["keep_ties"][2]
    assert lo <= st["skipped"] <= hi_, (st, lo, hi_)
    assert st["skipped"] in (lo, hi_), "every tie is decided the same way"
    # dE = G C is exactly zero whatever the filter keeps
    assert np.all(got["dE"] == 0.0)
    side = "keep_ties" if st["skipped"] == lo else "skip_ties"
    dC_ref = refs[side][0]
    assert rel_fro(got["dC"], dC_ref) <= TOL_GRAD
    assert row_max_rel(got["dC"], dC_ref) <= TOL_ROW
    if side == "keep_ties":
        assert rel_fro(got["dC"], dC_u) <= TOL_GRAD_FILTERED
    elif targets == "uniform":
        # few tiles are decided by the tie alone: within the filtered bar either way
        assert rel_fro(got["dC"], dC_u) <= TOL_GRAD_FILTERED


@pytest.mark.parametrize("cols,sort", [(256, False), (512, False), (256, True), (None, False)])
def test_staging_budget(cols, sort):
    """cce_backward_ex2: the G-hat chunk buffer bounded by max_staging_bytes.
    Budgets of one and two 256-column tiles per chunk (36 and 18 chunks at
    V = 9000, the last one ragged) give the oracle's gradients like the
    default budget does, with and without vocabulary sorting; the chunk width
    follows the budget."""
    import linear_cross_entropy_gb300 as cce
    N, D, V = 640, 128, 9000
    budget = 0 if cols is None else N * cols * 2 + 100
    assert cce.backward_chunk_cols(N, V, budget) == (cols or 4608)
    w, (E, C, x) = make(W.small("b", N, D, V))
    Et, Ct, xt = to_device(E, C, x)
    loss, lse = cce.cce_forward(Et, Ct, xt)
    need = cce.backward_workspace_bytes(N, D, V, vocab_sort=sort, max_staging_bytes=budget)
    assert need <= cce.backward_workspace_bytes(N, D, V, vocab_sort=sort)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for eps in (0.0, O.FILTER_EPS):
        dE, dC, st = cce.cce_backward(Et, Ct, xt, lse, torch.ones(1, device="cuda"), filter_eps=eps,
                                      vocab_sort=sort, max_staging_bytes=budget, workspace=ws, stats=True)
        torch.cuda.synchronize()
        ref = oracle_full(E, C, x, reduction="mean")
        got = {"dE": bf16_to_f64(dE), "dC": bf16_to_f64(dC), "dE_raw": dE}
        assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD if eps == 0 else TOL_GRAD_FILTERED, x)
        assert st["tiles"] == ((x != -100).sum() + 127) // 128 * ((V + 127) // 128)


@pytest.mark.parametrize("D", [8, 16, 24, 40, 72])
def test_small_hidden_sizes(D):
    """Hidden sizes below one 64-column K-block: the logit GEMMs' K box and
    the gradient GEMM's D tile (32 columns wide here, 64 at D = 72) reach past
    D and read zeros there; stores of D tiles stop at D.  Ragged N and V,
    ignored rows, filter off and on, and the single call."""
    import linear_cross_entropy_gb300 as cce
    N, V = 300, 700
    w, (E, C, x) = make(W.small("sd", N, D, V))
    for eps in (0.0, O.FILTER_EPS):
        got = run_cuda(E, C, x, reduction="mean", filter_eps=eps)
        ref = oracle_full(E, C, x, reduction="mean", filter_eps=eps or None)
        assert_forward_close(got, ref, "mean", x)
        assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD if eps == 0 else TOL_GRAD_FILTERED, x)
        if eps:
            assert rel_fro(got["dE"], ref["dE_f"]) <= TOL_GRAD and rel_fro(got["dC"], ref["dC_f"]) <= TOL_GRAD
    Et, Ct, xt = to_device(E, C, x)
    loss, _, dE, dC = cce.cce_loss_and_grad(Et, Ct, xt, filter_eps=0.0)
    ref = oracle_full(E, C, x, reduction="mean")
    assert abs(loss.item() - float(ref["loss"])) <= TOL_LSE * abs(float(ref["loss"]))
    got = {"dE": bf16_to_f64(dE), "dC": bf16_to_f64(dC), "dE_raw": dE}
    assert_grads_close(got, ref["dE"], ref["dC"], TOL_GRAD, x)


@pytest.mark.parametrize("filter_on", [False, True])
def test_single_entry_vocabulary(filter_on):
    """V = 1: every row's only logit is its target logit, so LSE_i = a_i,
    every loss is 0 and G = softmax - onehot = 0 in exact arithmetic.  The
    GPU's fp32 LSE (a max and a log-sum in base 2) may differ from a_i in the
    last bits, so the loss and the gradients must be 0 up to 1e-5 of the LSE
    scale; with the filter on every |G| < eps and the gradients are exact
    zeros."""
    N, D, V = 200, 64, 1
    rng = np.random.default_rng(5)
    E_bits = W.f32_to_bf16_bits(rng.standard_normal((N, D)).astype(np.float32))
    C_bits = W.f32_to_bf16_bits(rng.standard_normal((V, D)).astype(np.float32))
    x = np.zeros(N, dtype=np.int64)
    x[::7] = O.IGNORE_INDEX
    eps = O.FILTER_EPS if filter_on else 0.0
    for reduction in ("mean", "none"):
        got = run_cuda(E_bits, C_bits, x, reduction=reduction, filter_eps=eps)
        Ef, Cf = O.from_bits(E_bits, C_bits)
        f = O.forward(Ef, Cf, x, reduction=reduction)
        scale = float(np.abs(f["lse"]).max())
        assert np.max(np.abs(got["lse"] - f["lse"])) <= TOL_LSE * scale
        assert np.max(np.abs(got["loss"])) <= TOL_LSE * scale
        if filter_on:
            assert np.all(got["dE"] == 0.0) and np.all(got["dC"] == 0.0)
            assert got["stats"]["skipped"] == got["stats"]["tiles"]
        else:
            gscale = np.abs(Ef).max() * np.abs(Cf).max()
            assert np.max(np.abs(got["dE"])) <= TOL_LSE * gscale
            assert np.max(np.abs(got["dC"])) <= TOL_LSE * gscale * N
        ign = x == O.IGNORE_INDEX
        raw = got["dE_raw"][torch.from_numpy(np.nonzero(ign)[0]).cuda()]
        assert not raw.view(torch.int16).any()
