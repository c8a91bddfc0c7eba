"""GPU parity of the single call (loss and both gradients in one pass,
"fused-linear-cross-entropy" page, section "2. Fused Linear Cross-Entropy
(FLCE)") against the fp64 oracle's loss_and_grad, through the C ABI.

Covered: both reductions, ignored rows (compacted away before the GEMMs: the
LSE is checked on the rows that take part and must be 0 on the others), a
ragged vocabulary (V not a multiple of 256), several token chunks (dC
accumulated in fp32 over chunks, dE rows of every chunk), the vocabulary
split of the dE tiles, the filter on inputs where it bites (gradients within
the filtered tolerance of the oracle's filtered gradients, skipped-tile count
against the oracle's map), softcapping, the autograd wrapper with an upstream
gradient other than 1, a fully ignored batch, and determinism.
"""
import numpy as np
import pytest
import torch

import cce_workloads as W
import oracle as O
from tests.gpu_util import TOL_GRAD, TOL_GRAD_FILTERED, TOL_LSE, bf16_to_f64, mixed_survival_inputs, rel_fro, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests.conftest import build_library
    build_library()


def _run(E_bits, C_bits, x, **kw):
    import linear_cross_entropy_gb300 as cce
    E, C, xt = to_device(E_bits, C_bits, x)
    loss, lse, dE, dC, st = cce.cce_loss_and_grad(E, C, xt, stats=True, **kw)
    torch.cuda.synchronize()
    return {"loss": float(loss.item()), "lse": lse.double().cpu().numpy(), "dE": bf16_to_f64(dE),
            "dC": bf16_to_f64(dC), "dE_raw": dE, "stats": st}


def _check(got, ref, x, tol, ignore_index=-100):
    part = (x != ignore_index) & (x >= 0) & (x < ref["dC"].shape[0])
    lse_err = np.abs(got["lse"][part] - ref["lse"][part]) / np.abs(ref["lse"][part])
    assert lse_err.max() <= TOL_LSE, f"LSE rel err {lse_err.max():.3e}"
    assert np.all(got["lse"][~part] == 0.0)
    assert abs(got["loss"] - ref["loss"]) <= TOL_LSE * abs(ref["loss"]), (got["loss"], ref["loss"])
    eE, eC = rel_fro(got["dE"], ref["dE"]), rel_fro(got["dC"], ref["dC"])
    assert eE <= tol and eC <= tol, f"dE {eE:.3e} dC {eC:.3e}"
    ign = np.nonzero(x == ignore_index)[0]
    if len(ign):
        z = got["dE_raw"][torch.from_numpy(ign).cuda()].view(torch.int16)
        assert int(torch.count_nonzero(z)) == 0, "ignored rows of dE are not +0"
    return eE, eC


CASES = [
    # name, workload, reduction, max staging bytes (0 = default: one chunk)
    ("tiny", W.CONFIGS["tiny"], "mean", 0),
    ("ragged-sum", W.small("r", 300, 136, 5000), "sum", 0),
    ("three-chunks", W.small("c", 700, 64, 5000), "mean", 256 * 5120 * 2),
    ("split-dE", W.small("s", 512, 128, 20000), "sum", 256 * 20224 * 2),
    ("wide-D", W.small("w", 300, 600, 3000), "mean", 0),
    ("pairs-split-dE", W.small("p", 700, 256, 20000), "sum", 256 * 20224 * 2),
]


@pytest.mark.parametrize("name,w,reduction,staging", CASES, ids=[c[0] for c in CASES])
def test_single_call_unfiltered(name, w, reduction, staging):
    E_bits, C_bits, x = W.make_inputs(w)
    got = _run(E_bits, C_bits, x, reduction=reduction, filter_eps=0.0, max_staging_bytes=staging)
    Ef, Cf = O.from_bits(E_bits, C_bits)
    ref = O.loss_and_grad(Ef, Cf, x, reduction=reduction)
    _check(got, ref, x, TOL_GRAD)
    assert got["stats"]["skipped"] == 0


@pytest.mark.parametrize("staging", [0, 256 * 9216 * 2], ids=["one-chunk", "several-chunks"])
def test_single_call_filtered(staging):
    N, D, V = 1024, 128, 9000
    E_bits, C_bits, x = W.frequent_token_inputs(N, D, V, n_freq=256)
    got = _run(E_bits, C_bits, x, reduction="mean", filter_eps=O.FILTER_EPS, max_staging_bytes=staging)
    Ef, Cf = O.from_bits(E_bits, C_bits)
    ref = O.loss_and_grad(Ef, Cf, x, reduction="mean", filter_eps=O.FILTER_EPS)
    _check(got, ref, x, TOL_GRAD_FILTERED)
    keep = ref["keep"]
    assert got["stats"]["tiles"] == keep.size
    assert abs(got["stats"]["skipped"] - int((~keep).sum())) <= max(1, keep.size // 200)
    assert got["stats"]["skipped"] > keep.size // 2


def test_single_call_filtered_full_width_d_tile():
    """D = 256 (one full-width gradient D tile, 3-D B boxes) with the filter
    skipping most tiles."""
    E_bits, C_bits, x = W.frequent_token_inputs(1024, 256, 9000, n_freq=256)
    got = _run(E_bits, C_bits, x, reduction="sum", filter_eps=O.FILTER_EPS)
    Ef, Cf = O.from_bits(E_bits, C_bits)
    ref = O.loss_and_grad(Ef, Cf, x, reduction="sum", filter_eps=O.FILTER_EPS)
    _check(got, ref, x, TOL_GRAD_FILTERED)
    keep = ref["keep"]
    assert abs(got["stats"]["skipped"] - int((~keep).sum())) <= max(1, keep.size // 200)
    assert got["stats"]["skipped"] > keep.size // 2


@pytest.mark.parametrize("staging", [0, 256 * 1536 * 2], ids=["one-chunk", "several-chunks"])
def test_single_call_pairs_with_different_survival(staging):
    """D = 256: the single call's gradient GEMM as CTA pairs, on inputs whose
    neighbouring blocks keep different K-blocks (most token-block pairs, and
    vocabulary blocks 0 and 1), so the pairs run the union and load zeros
    where their own tile skips; one token chunk or several.  No tile lies
    within 0.1% of eps (checked on the oracle): the skip count is exact."""
    from linear_cross_entropy_gb300 import _lib
    lib = _lib.load()
    N, D, V = 3000, 256, 1500
    E_bits, C_bits, x = mixed_survival_inputs(N, D, V)
    prev = lib.cce_selftest_grad_layout(1)  # pairs (the automatic choice takes one CTA per tile here)
    try:
        got = _run(E_bits, C_bits, x, reduction="mean", filter_eps=O.FILTER_EPS, max_staging_bytes=staging)
        again = _run(E_bits, C_bits, x, reduction="mean", filter_eps=O.FILTER_EPS, max_staging_bytes=staging)
        lib.cce_selftest_grad_layout(2)
        single = _run(E_bits, C_bits, x, reduction="mean", filter_eps=O.FILTER_EPS, max_staging_bytes=staging)
    finally:
        lib.cce_selftest_grad_layout(prev)
    # the same bits as one CTA per tile (and as a second run)
    assert np.array_equal(got["dE"], single["dE"]) and np.array_equal(got["dC"], single["dC"])
    assert np.array_equal(got["dE"], again["dE"]) and np.array_equal(got["dC"], again["dC"])
    Ef, Cf = O.from_bits(E_bits, C_bits)
    ref = O.loss_and_grad(Ef, Cf, x, reduction="mean", filter_eps=O.FILTER_EPS)
    for eps in (O.FILTER_EPS * (1 - 1e-3), O.FILTER_EPS * (1 + 1e-3)):
        assert np.array_equal(O.loss_and_grad(Ef, Cf, x, reduction="mean", filter_eps=eps)["keep"], ref["keep"])
    keep = ref["keep"]
    assert got["stats"]["tiles"] == keep.size
    assert got["stats"]["skipped"] == int((~keep).sum()) > 0
    _check(got, ref, x, TOL_GRAD_FILTERED)


def test_single_call_softcap():
    w = W.small("cap", 300, 136, 5000)
    E_bits, C_bits, x = W.make_inputs(w)
    got = _run(E_bits, C_bits, x, reduction="mean", filter_eps=0.0, softcap=20.0)
    Ef, Cf = O.from_bits(E_bits, C_bits)
    _check(got, O.loss_and_grad(Ef, Cf, x, reduction="mean", softcap=20.0), x, TOL_GRAD)


def test_single_call_autograd_scales_by_the_upstream_gradient():
    import linear_cross_entropy_gb300 as cce
    w = W.small("ag", 260, 64, 3000)
    E_bits, C_bits, x = W.make_inputs(w)
    E, C, xt = to_device(E_bits, C_bits, x)
    E.requires_grad_(True)
    C.requires_grad_(True)
    loss = cce.fused_linear_cross_entropy(E, C, xt, reduction="sum", filter_eps=0.0)
    (2.5 * loss).backward()
    Ef, Cf = O.from_bits(E_bits, C_bits)
    ref = O.loss_and_grad(Ef, Cf, x, reduction="sum")
    assert abs(loss.item() - ref["loss"]) <= TOL_LSE * abs(ref["loss"])
    assert rel_fro(bf16_to_f64(E.grad), 2.5 * ref["dE"]) <= TOL_GRAD
    assert rel_fro(bf16_to_f64(C.grad), 2.5 * ref["dC"]) <= TOL_GRAD


def test_single_call_is_deterministic():
    E_bits, C_bits, x = W.frequent_token_inputs(600, 64, 9000, n_freq=200)
    a = _run(E_bits, C_bits, x, reduction="mean", max_staging_bytes=256 * 9216 * 2)
    b = _run(E_bits, C_bits, x, reduction="mean", max_staging_bytes=256 * 9216 * 2)
    assert a["loss"] == b["loss"] and np.array_equal(a["lse"], b["lse"])
    assert torch.equal(a["dE_raw"].view(torch.int16), b["dE_raw"].view(torch.int16))
    assert np.array_equal(a["dC"], b["dC"]) and a["stats"] == b["stats"]


@pytest.mark.parametrize("D,filter_eps", [(64, None), (64, 0.0), (256, 0.0)])
def test_single_call_fully_ignored_batch(D, filter_eps):
    """Zero loss and gradients with the filter on or off (off, nothing marks
    the dC tiles, which have no K-block, as skipped); D = 256: CTA pairs."""
    E_bits, C_bits, x = W.make_inputs(W.small("z", 300, D, 3000))
    x = np.full_like(x, -100)
    kw = {} if filter_eps is None else {"filter_eps": filter_eps}
    got = _run(E_bits, C_bits, x, reduction="mean", max_staging_bytes=256 * 3072 * 2, **kw)
    assert got["loss"] == 0.0 and np.all(got["lse"] == 0.0)
    assert np.all(got["dE"] == 0.0) and np.all(got["dC"] == 0.0)
    assert got["stats"]["tiles"] == 0


def test_single_call_rejects_reduction_none():
    import linear_cross_entropy_gb300 as cce
    E_bits, C_bits, x = W.make_inputs(W.CONFIGS["tiny"])
    E, C, xt = to_device(E_bits, C_bits, x)
    with pytest.raises(ValueError):
        cce.cce_loss_and_grad(E, C, xt, reduction="none")
