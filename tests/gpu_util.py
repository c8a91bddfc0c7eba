"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding (C ABI) and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import cce_workloads as W
import oracle as O

# Tolerances (fixed for this operator): loss and LSE within 1e-5 relative;
# per-row loss within 1e-5 * LSE_i (cancellation in LSE - target); dE and dC
# within 5e-3 relative Frobenius error unfiltered and 1e-2 with the filter on;
# ignored rows bit-exact zero.
TOL_LSE = 1e-5
TOL_GRAD = 5e-3
TOL_GRAD_FILTERED = 1e-2


def to_device(E_bits, C_bits, x, device="cuda"):
    E = torch.from_numpy(np.ascontiguousarray(E_bits).view(np.int16)).to(device).view(torch.bfloat16)
    C = torch.from_numpy(np.ascontiguousarray(C_bits).view(np.int16)).to(device).view(torch.bfloat16)
    xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.int64)).to(device)
    return E, C, xt


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_cuda(E_bits, C_bits, x, ignore_index=-100, reduction="mean", filter_eps=O.FILTER_EPS, grad_out=None):
    import linear_cross_entropy_gb300 as cce
    E, C, xt = to_device(E_bits, C_bits, x)
    loss, lse = cce.cce_forward(E, C, xt, ignore_index, reduction)
    if grad_out is None:
        g = torch.ones(x.shape[0] if reduction == "none" else 1, dtype=torch.float32, device="cuda")
    else:
        g = torch.as_tensor(grad_out, dtype=torch.float32, device="cuda")
    dE, dC, stats = cce.cce_backward(E, C, xt, lse, g, ignore_index, reduction, filter_eps, stats=True)
    torch.cuda.synchronize()
    return {
        "loss": loss.detach().cpu().numpy().astype(np.float64),
        "lse": lse.cpu().numpy().astype(np.float64),
        "dE": bf16_to_f64(dE),
        "dC": bf16_to_f64(dC),
        "dE_raw": dE,
        "stats": stats,
    }


def rel_fro(a, b) -> float:
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def oracle_full(E_bits, C_bits, x, ignore_index=-100, reduction="mean", grad_out=1.0, filter_eps=None,
                tile=(128, 128)):
    E, C = O.from_bits(E_bits, C_bits)
    f = O.forward(E, C, x, ignore_index, reduction)
    w = O.row_weights(x, ignore_index, reduction, grad_out, f["count"])
    dE, dC = O.backward(E, C, x, f["lse"], w, ignore_index)
    out = {"loss": f["loss"], "lse": f["lse"], "loss_rows": f["loss_rows"], "dE": dE, "dC": dC}
    if filter_eps:
        dEf, dCf, keep = O.backward_filtered(E, C, x, f["lse"], w, tile[0], tile[1], filter_eps, ignore_index,
                                             compact_ignored=True)
        out.update(dE_f=dEf, dC_f=dCf, keep=keep)
    return out


def assert_forward_close(got, ref, reduction, x, ignore_index=-100):
    lse_err = np.abs(got["lse"] - ref["lse"]) / np.abs(ref["lse"])
    assert lse_err.max() <= TOL_LSE, f"LSE rel err {lse_err.max():.3e}"
    if reduction == "none":
        err = np.abs(got["loss"] - ref["loss_rows"])
        assert np.all(err <= TOL_LSE * np.abs(ref["lse"]) + 1e-30), f"row loss err {err.max():.3e}"
        ign = x == ignore_index
        assert np.all(got["loss"][ign] == 0.0)
    else:
        r = float(np.asarray(ref["loss"]))
        g = float(np.asarray(got["loss"]).reshape(()))
        if r == 0.0:
            assert g == 0.0
        else:
            assert abs(g - r) <= TOL_LSE * abs(r), f"loss {g!r} vs {r!r}"


# Per-row bound beside the Frobenius one: the relative error of every row of
# dE and dC, with the row's reference norm floored at ROW_FLOOR x the RMS row
# norm (rows whose reference is nearly zero are measured on that scale).  A
# single wrong row or ragged tile that the Frobenius figure would dilute
# fails it; bf16 rounding alone gives about 2e-3 per row.
TOL_ROW = 5e-2
ROW_FLOOR = 0.05


def row_max_rel(a, b) -> float:
    """Largest per-row relative error of a against the reference b (2-D)."""
    a = np.asarray(a, dtype=np.float64).reshape(a.shape[0], -1)
    b = np.asarray(b, dtype=np.float64).reshape(b.shape[0], -1)
    den = np.linalg.norm(b, axis=1)
    rms = float(np.sqrt(np.mean(den * den)))
    if rms == 0.0:
        return float(np.abs(a).max()) if a.size else 0.0
    num = np.linalg.norm(a - b, axis=1)
    return float(np.max(num / np.maximum(den, ROW_FLOOR * rms)))


def assert_grads_close(got, ref_dE, ref_dC, tol, x, ignore_index=-100, row_tol="auto"):
    """Relative Frobenius error of dE and dC within tol, ignored rows of dE
    bit-exact +0, and (when the reference takes the same filter decisions
    as the GPU: row_tol "auto" applies it to unfiltered comparisons, tol <=
    TOL_GRAD) every row within row_tol."""
    eE, eC = rel_fro(got["dE"], ref_dE), rel_fro(got["dC"], ref_dC)
    rE, rC = row_max_rel(got["dE"], ref_dE), row_max_rel(got["dC"], ref_dC)
    assert eE <= tol, f"dE rel Frobenius err {eE:.3e} > {tol} (worst row {rE:.3e})"
    assert eC <= tol, f"dC rel Frobenius err {eC:.3e} > {tol} (worst row {rC:.3e})"
    if row_tol == "auto":
        row_tol = TOL_ROW if tol <= TOL_GRAD else None
    if row_tol is not None:
        assert rE <= row_tol, f"dE worst row rel err {rE:.3e} > {row_tol} (Frobenius {eE:.3e})"
        assert rC <= row_tol, f"dC worst row rel err {rC:.3e} > {row_tol} (Frobenius {eC:.3e})"
    ign = x == ignore_index
    if np.any(ign):
        raw = got["dE_raw"][torch.from_numpy(np.nonzero(ign)[0]).cuda()]
        assert torch.equal(raw.view(torch.int16), torch.zeros_like(raw.view(torch.int16))), \
            "ignored rows of dE are not bit-exact +0"
    return eE, eC


def make(name_or_w, **kw):
    w = W.CONFIGS[name_or_w] if isinstance(name_or_w, str) else name_or_w
    if kw:
        w = w.with_(**kw)
    return w, W.make_inputs(w)


def mixed_survival_inputs(N, D=256, V=1500, seed=5):
    """Frequent-token inputs (128 frequent ids: vocabulary block 0) whose
    token blocks differ in what the filter keeps: every third 128-row block
    has its hidden states scaled by 0.01 (a near-uniform softmax: every tile
    kept), the others point at their target's classifier row (0.35 C_x: the
    target takes over 99% of the mass, so only vocabulary block 0 is kept)."""
    E, C, x = W.frequent_token_inputs(N, D, V, n_freq=128, seed=seed)
    Ef = W.bf16_bits_to_f32(E).astype(np.float32)
    Cf = W.bf16_bits_to_f32(C).astype(np.float32)
    for b in range((N + 127) // 128):
        r = slice(b * 128, min(N, (b + 1) * 128))
        if b % 3 == 0:
            Ef[r] *= np.float32(0.01)
        else:
            t = x[r]
            live = t != O.IGNORE_INDEX
            Ef[r][live] = np.float32(0.35) * Cf[t[live]]
    return W.f32_to_bf16_bits(Ef), C, x
