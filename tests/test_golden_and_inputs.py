"""Page-printed values (tests/golden) and the seeded input generator."""
import math
import os

import numpy as np
import pytest

import cce_workloads as W
import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = float(v)
    return out


def test_memory_arithmetic_identities():
    g = read_golden("memory_arithmetic.txt")
    MiB = 1 << 20
    N, V, D = int(g["N"]), int(g["V"]), int(g["D"])
    assert N * V * 4 / MiB == g["logits_fp32_MiB"]
    assert 3 * g["logits_fp32_MiB"] == g["baseline_MB"]
    assert V * D * 2 / MiB == g["dC_bf16_MiB"]
    assert N * D * 2 / MiB == g["dE_bf16_MiB"]
    assert g["dC_bf16_MiB"] + g["dE_bf16_MiB"] == g["lower_bound_MiB"]
    assert g["cce_total_MiB"] - g["lower_bound_MiB"] == 3


def test_filter_threshold_values():
    g = read_golden("filter_threshold.txt")
    import torch
    assert torch.finfo(torch.bfloat16).eps == g["bf16_eps"]
    assert g["bf16_eps"] / 32 == g["filter_eps"] == 2.0 ** g["filter_eps_log2"]
    assert O.FILTER_EPS == g["filter_eps"]
    assert 1 / g["filter_eps"] == g["max_entries_row"]


def test_generator_is_deterministic_and_block_independent(monkeypatch):
    w = W.small("t", 300, 64, 5000)
    a = W.make_inputs(w)
    monkeypatch.setenv("CCE_GEN_WORKERS", "1")
    b = W.make_inputs(w)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    assert W.inputs_digest(*a) == W.inputs_digest(*b)


def test_generator_distributions():
    w = W.small("t", 4000, 256, 20000, ignore_frac=0.1)
    E, C, x = W.make_inputs(w)
    Cf = W.bf16_bits_to_f32(C).astype(np.float64)
    assert abs(Cf.std() * math.sqrt(256) - 4.0) < 0.02
    assert abs(Cf.mean()) < 1e-3
    ign = x == W.IGNORE_INDEX
    assert 0.08 < ign.mean() < 0.12
    xv = x[~ign]
    assert xv.min() >= 0 and xv.max() < 20000
    # Zipf: the most frequent id holds about 1 / H_{V,1.1} of the mass
    top = np.bincount(xv).max() / len(xv)
    H = sum(r ** -1.1 for r in range(1, 20001))
    assert abs(top - 1 / H) < 0.02
    # boost: E_i . C[x_i] / ||C[x_i]|| has mean close to the boost (3)
    Ef = W.bf16_bits_to_f32(E).astype(np.float64)
    cx = Cf[np.where(ign, 0, x)]
    proj = (Ef * cx).sum(1) / np.linalg.norm(cx, axis=1)
    assert abs(proj[~ign].mean() - 3.0) < 0.1


def test_tiny_config_recipe():
    w = W.CONFIGS["tiny"]
    E, C, x = W.make_inputs(w)
    assert E.shape == (256, 128) and C.shape == (4096, 128) and x.dtype == np.int64
    assert np.all((x >= 0) & (x < 4096))
    Ef = W.bf16_bits_to_f32(E)
    assert abs(Ef.std() - 1.0) < 0.02


def test_norm_ppf_against_scipy():
    st = pytest.importorskip("scipy.stats")
    u = np.linspace(1e-10, 1 - 1e-10, 100001)
    assert np.max(np.abs(W._norm_ppf(u) - st.norm.ppf(u))) < 1e-7
