"""Full-size GPU parity on the four large workloads, in the launch
configuration the benchmark uses.

The fp64 oracle's LSE for every row is stored in tests/golden (written by
tests/golden/make_oracle_lse.py, which calls only oracle/); the input digest
stored beside it proves the box drew the same bytes.  Checked here:

* LSE of every row within 1e-5 relative; the reduced loss within 1e-5
  relative of the oracle's (stored LSE minus the oracle's indexed target
  logits, reduced in fp64);
* dE rows and dC rows on a seeded sample, each computed one by one by the
  oracle, within 5e-3 relative Frobenius error (1e-2 with the filter on);
* every ignored row of dE is bit-exact +0;
* the identity <E, dE> = <C, dC> (both equal sum_i w_i sum_v G_iv a_iv),
  which ties all of dC to dE at any size.

The same checks run with vocabulary sorting on, on the Qwen2.5-0.5B-shaped
head and on the supplementary workload of that shape whose frequent tokens
are scattered through the vocabulary (where sorting must let the filter
skip nearly every tile).
"""
import functools
import os

import numpy as np
import pytest
import torch

import cce_workloads as W
import oracle as O
from tests.gpu_util import TOL_GRAD, TOL_GRAD_FILTERED, TOL_LSE, rel_fro, to_device

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests.conftest import build_library
    build_library()


@functools.lru_cache(maxsize=1)
def _inputs(name):
    w = W.ALL_CONFIGS[name]
    E, C, x = W.make_inputs(w)
    ref = np.load(os.path.join(GOLDEN, f"oracle_lse_{name}.npz"))
    assert str(ref["digest"]) == W.inputs_digest(E, C, x), "inputs differ from the ones the oracle saw"
    assert tuple(ref["sizes"]) == (w.N, w.D, w.V)
    return w, E, C, x, ref["lse"]


CASES = [(n, f, False) for n in ("qwen", "gemma", "llama", "long") for f in W.CONFIGS[n].filter_modes]
CASES += [("qwen", "on", True), ("freq", "on", False), ("freq", "on", True)]


@pytest.mark.parametrize("name,filter_mode,sort", CASES)
def test_full_size(name, filter_mode, sort):
    import linear_cross_entropy_gb300 as cce
    w, E_bits, C_bits, x, lse_ref = _inputs(name)
    eps = O.FILTER_EPS if filter_mode == "on" else 0.0
    tol = TOL_GRAD_FILTERED if filter_mode == "on" else TOL_GRAD
    E, C, xt = to_device(E_bits, C_bits, x)
    loss, lse = cce.cce_forward(E, C, xt, reduction=w.reduction)
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    dE, dC, stats = cce.cce_backward(E, C, xt, lse, g, reduction=w.reduction, filter_eps=eps, stats=True,
                                     vocab_sort=sort)
    torch.cuda.synchronize()

    # forward: every row
    lse_gpu = lse.double().cpu().numpy()
    err = np.abs(lse_gpu - lse_ref) / np.abs(lse_ref)
    assert err.max() <= TOL_LSE, f"LSE rel err {err.max():.3e}"
    Ef, Cf = O.from_bits(E_bits, C_bits)
    valid = x != O.IGNORE_INDEX
    count = int(valid.sum())
    tgt = O.indexed_logits(Ef, Cf, x)
    loss_rows = np.where(valid, lse_ref - np.where(valid, tgt, 0.0), 0.0)
    loss_ref = O.reduce_loss(loss_rows, count, w.reduction)
    assert abs(loss.item() - loss_ref) <= TOL_LSE * abs(loss_ref), (loss.item(), loss_ref)

    # backward: sampled rows, each computed one by one by the oracle
    rng = np.random.default_rng(11)
    wts = O.row_weights(x, O.IGNORE_INDEX, w.reduction, 1.0, count)
    rows = np.unique(np.concatenate([[0, w.N - 1], rng.choice(w.N, 30, replace=False)]))
    dE_ref = O.backward_dE(Ef, Cf, x, lse_ref[rows], wts[rows], rows)
    dE_got = dE[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    e_dE = rel_fro(dE_got, dE_ref)
    assert e_dE <= tol, f"dE sample rel err {e_dE:.3e}"
    freq = np.bincount(x[valid], minlength=w.V).argsort()[::-1][:12]
    vrows = np.unique(np.concatenate([freq, [0, w.V - 1], rng.choice(w.V, 20, replace=False)]))
    dC_ref = O.backward_dC(Ef, Cf, x, lse_ref, wts, vrows)
    dC_got = dC[torch.from_numpy(vrows).cuda()].double().cpu().numpy()
    e_dC = rel_fro(dC_got, dC_ref)
    assert e_dC <= tol, f"dC sample rel err {e_dC:.3e}"

    # ignored rows: bit-exact zero
    ign = np.nonzero(~valid)[0]
    if len(ign):
        z = dE[torch.from_numpy(ign).cuda()].view(torch.int16)
        assert int(torch.count_nonzero(z)) == 0

    # <E, dE> = <C, dC>
    lhs = float((E.double() * dE.double()).sum())
    rhs = float((C.double() * dC.double()).sum())
    assert abs(lhs - rhs) <= 2e-2 * max(abs(lhs), abs(rhs)), (lhs, rhs)
    if name == "freq" and sort:
        # 256 frequent tokens: sorted, they fill the last two or three 128-wide
        # vocabulary tiles, so nearly every other tile is skipped
        assert stats["skipped"] >= 0.97 * stats["tiles"], stats
    print(f"{name} filter={filter_mode} sort={sort}: loss {loss.item():.6f} (oracle {loss_ref:.6f}) lse err {err.max():.2e} "
          f"dE err {e_dE:.2e} dC err {e_dC:.2e} tiles skipped {stats['skipped']}/{stats['tiles']} "
          f"<E,dE>={lhs:.6e} <C,dC>={rhs:.6e}")
    del E, C, dE, dC
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["qwen", "llama"])
def test_full_size_single_call(name):
    """The single call at full size (the Llama-shaped head takes two token
    chunks at the default staging budget, so dC goes through the fp32
    accumulator): LSE of every row, the loss, sampled dE and dC rows against
    the oracle, ignored rows +0, and <E, dE> = <C, dC>."""
    import linear_cross_entropy_gb300 as cce
    w, E_bits, C_bits, x, lse_ref = _inputs(name)
    E, C, xt = to_device(E_bits, C_bits, x)
    loss, lse, dE, dC, stats = cce.cce_loss_and_grad(E, C, xt, reduction=w.reduction, stats=True)
    torch.cuda.synchronize()
    valid = x != O.IGNORE_INDEX
    lse_got = lse.double().cpu().numpy()
    err = np.abs(lse_got[valid] - lse_ref[valid]) / np.abs(lse_ref[valid])
    assert err.max() <= TOL_LSE, f"LSE rel err {err.max():.3e}"
    assert np.all(lse_got[~valid] == 0.0)  # the single call skips the rows that take no part
    Ef, Cf = O.from_bits(E_bits, C_bits)
    count = int(valid.sum())
    tgt = O.indexed_logits(Ef, Cf, x)
    loss_ref = O.reduce_loss(np.where(valid, lse_ref - np.where(valid, tgt, 0.0), 0.0), count, w.reduction)
    assert abs(loss.item() - loss_ref) <= TOL_LSE * abs(loss_ref), (loss.item(), loss_ref)
    rng = np.random.default_rng(12)
    wts = O.row_weights(x, O.IGNORE_INDEX, w.reduction, 1.0, count)
    rows = np.unique(np.concatenate([[0, w.N - 1], rng.choice(w.N, 30, replace=False)]))
    dE_ref = O.backward_dE(Ef, Cf, x, lse_ref[rows], wts[rows], rows)
    e_dE = rel_fro(dE[torch.from_numpy(rows).cuda()].double().cpu().numpy(), dE_ref)
    assert e_dE <= TOL_GRAD_FILTERED, f"dE sample rel err {e_dE:.3e}"
    freq = np.bincount(x[valid], minlength=w.V).argsort()[::-1][:12]
    vrows = np.unique(np.concatenate([freq, [0, w.V - 1], rng.choice(w.V, 20, replace=False)]))
    dC_ref = O.backward_dC(Ef, Cf, x, lse_ref, wts, vrows)
    e_dC = rel_fro(dC[torch.from_numpy(vrows).cuda()].double().cpu().numpy(), dC_ref)
    assert e_dC <= TOL_GRAD_FILTERED, f"dC sample rel err {e_dC:.3e}"
    ign = np.nonzero(~valid)[0]
    if len(ign):
        assert int(torch.count_nonzero(dE[torch.from_numpy(ign).cuda()].view(torch.int16))) == 0
    lhs = float((E.double() * dE.double()).sum())
    rhs = float((C.double() * dC.double()).sum())
    assert abs(lhs - rhs) <= 2e-2 * max(abs(lhs), abs(rhs)), (lhs, rhs)
    print(f"{name} single call: loss {loss.item():.6f} (oracle {loss_ref:.6f}) lse err {err.max():.2e} "
          f"dE err {e_dE:.2e} dC err {e_dC:.2e} tiles skipped {stats['skipped']}/{stats['tiles']}")
    del E, C, dE, dC
    torch.cuda.empty_cache()
