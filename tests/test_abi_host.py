"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol include/cce.h declares, sizes its workspaces, reproduces the
page's memory arithmetic, and rejects bad arguments before launching."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from tests.conftest import build_library
    build_library()
    from linear_cross_entropy_gb300 import _lib
    return _lib.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "cce.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cce_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "cce_forward" in names and "cce_backward" in names
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings(lib):
    assert lib.cce_abi_version() == 101
    for s in range(10):
        assert lib.cce_status_string(s)


def test_memory_arithmetic_of_the_page(lib):
    """'The memory numbers hold up': 8192 x 256000 x 4 B = 8000 MiB of fp32
    logits; dC = 1125 MiB and dE = 36 MiB, lower bound 1161 MiB."""
    import linear_cross_entropy_gb300 as cce
    from tests.test_golden_and_inputs import read_golden
    g = read_golden("memory_arithmetic.txt")
    r = cce.memory_report(int(g["N"]), int(g["D"]), int(g["V"]))
    MiB = 1 << 20
    assert r["logits_fp32_bytes"] / MiB == g["logits_fp32_MiB"]
    assert r["dC_bytes"] / MiB == g["dC_bf16_MiB"]
    assert r["dE_bytes"] / MiB == g["dE_bf16_MiB"]
    assert (r["dC_bytes"] + r["dE_bytes"]) / MiB == g["lower_bound_MiB"]
    # no workspace ever approaches an N x V buffer
    assert r["fwd_workspace_bytes"] < r["logits_fp32_bytes"] / 50
    assert r["bwd_workspace_bytes"] < r["logits_fp32_bytes"] / 8
    assert r["bwd_chunk_cols"] < 256000


@pytest.mark.parametrize("N,D,V", [(256, 128, 4096), (4096, 896, 151936), (8192, 2304, 256000),
                                   (16384, 4096, 128256), (65536, 2048, 128256), (1, 8, 1), (1000, 96, 5000)])
def test_workspace_queries(lib, N, D, V):
    f = lib.cce_forward_workspace_bytes(N, D, V)
    b = lib.cce_backward_workspace_bytes(N, D, V)
    assert f > 0 and b > 0
    assert b >= N * D * 4  # holds the fp32 dE accumulator
    import linear_cross_entropy_gb300 as cce
    r = cce.memory_report(N, D, V)
    # The backward's G buffer holds one vocabulary chunk: fewer columns than V
    # (never an N x V buffer) and at most 512 MiB plus one 256-column tile row.
    if V > 256:
        assert r["bwd_chunk_cols"] < V
    assert N * r["bwd_chunk_cols"] * 2 <= max(512 << 20, N * 256 * 2)
    compaction = N * (4 + 4 + 8 + 4 + 4) + N * D * 2  # row map + compact x, LSE, grad_out and E
    zero_box = 128 * 128 * 2  # the A operand a CTA pair's gradient GEMM loads where its own tile skips
    assert b <= (N * D * 4 + N * r["bwd_chunk_cols"] * 2 + 2 * (N // 128 + 1) * (V // 128 + 1) + compaction
                 + zero_box + 8192)
    assert f < N * V * 4 or V < 1024


@pytest.mark.parametrize("N,D,V", [(256, 128, 4096), (4096, 896, 151936), (65536, 2048, 128256), (1, 8, 1)])
def test_sorted_workspace_adds_keys_order_and_two_chunks(lib, N, D, V):
    """With vocabulary sorting the backward adds the keys, the order and its
    inverse (4 bytes each per token), the sort scratch, and one chunk of C in
    sorted order -- never a V x D copy when V spans several chunks."""
    import linear_cross_entropy_gb300 as cce
    b = lib.cce_backward_workspace_bytes(N, D, V)
    for flags in (0, 1, 2, 3):
        assert lib.cce_backward_workspace_bytes_ex(N, D, V, flags) == b
    bs = lib.cce_backward_workspace_bytes_ex(N, D, V, 4 | 3)
    vc = cce.memory_report(N, D, V)["bwd_chunk_cols"]
    extra = bs - b
    assert extra >= 12 * V + vc * D * 2
    scratch = lib.cce_vocab_sort_workspace_bytes(N, D, V)
    # ping-pong keys and values (12 bytes a token), four passes of per-block digit counts
    assert 12 * V <= scratch <= 12 * V + 4 * (4 * 256 * (V // 1024 + 1) + D * (N // 32 + 2)) + 4096
    assert extra <= 12 * V + scratch + vc * D * 2 + 8 * 256
    assert lib.cce_backward_workspace_bytes_ex(N, D, V, 8) == 0


@pytest.mark.parametrize("N,D,V", [(4096, 896, 151936), (16384, 4096, 128256), (300, 136, 5000)])
def test_single_call_workspace(lib, N, D, V):
    """The single call's workspace holds the compacted rows (E and x), one
    chunk of fp16 staged logits within the staging budget (whole 256-row
    chunks, at least one) with its 32-column maxima, dE slabs and, with
    several chunks, an fp32 dC accumulator."""
    vp_ = -(-V // 256) * 256
    for budget in (0, 64 << 20, 1):
        b = lib.cce_loss_and_grad_workspace_bytes(N, D, V, budget)
        cap = (2 << 30) if budget == 0 else budget
        nc = min(max(256, cap // (vp_ * 2) // 256 * 256), -(-N // 256) * 256)
        chunks = -(-N // nc)
        assert b >= nc * vp_ * 2 + N * D * 4 + N * D * 2 + (V * D * 4 if chunks > 1 else 0)
        assert b <= nc * vp_ * 2 + 8 * (-(-N // 128) * 128) * D * 4 + (V * D * 4 if chunks > 1 else 0) \
            + N * D * 2 + 4 * (vp_ // 32) * nc + 8 * (vp_ // 1024 + 1) * nc + 32 * N \
            + 3 * (nc // 128 + 1) * (V // 128 + 1) \
            + 64 * 1024  # compact rows, chunk maxima, split partials, LSE, maps and loss blocks, survival maps


def test_workspace_rejects_bad_sizes(lib):
    for N, D, V in [(0, 64, 10), (10, 0, 10), (10, 64, 0), (10, 12, 10), (1 << 31, 64, 10)]:
        assert lib.cce_forward_workspace_bytes(N, D, V) == 0
        assert lib.cce_backward_workspace_bytes(N, D, V) == 0


FAKE = 1 << 20  # an aligned non-null host integer: never dereferenced, checks fail first


def _fwd(lib, **kw):
    a = dict(E=FAKE, C=FAKE, x=FAKE, N=256, D=128, V=4096, ign=-100, red=2, loss=FAKE, lse=FAKE, ws=FAKE,
             wsb=1 << 40, err=0, stream=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.cce_forward(vp(a["E"]), vp(a["C"]), vp(a["x"]), a["N"], a["D"], a["V"], a["ign"], a["red"],
                           vp(a["loss"]), vp(a["lse"]), vp(a["ws"]), a["wsb"], vp(a["err"]), vp(a["stream"]))


def _bwd(lib, **kw):
    a = dict(E=FAKE, C=FAKE, x=FAKE, lse=FAKE, g=FAKE, N=256, D=128, V=4096, ign=-100, red=2, eps=2.0 ** -12,
             dE=FAKE, dC=FAKE, ws=FAKE, wsb=1 << 40, err=0, stats=0, stream=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.cce_backward(vp(a["E"]), vp(a["C"]), vp(a["x"]), vp(a["lse"]), vp(a["g"]), a["N"], a["D"], a["V"],
                            a["ign"], a["red"], a["eps"], vp(a["dE"]), vp(a["dC"]), vp(a["ws"]), a["wsb"],
                            vp(a["err"]), vp(a["stats"]), vp(a["stream"]))


@pytest.mark.parametrize("kw,status", [
    (dict(E=0), 1), (dict(C=0), 1), (dict(x=0), 1), (dict(loss=0), 1), (dict(lse=0), 1), (dict(ws=0), 1),
    (dict(N=0), 2), (dict(V=0), 2), (dict(D=12), 2), (dict(D=0), 2), (dict(N=1 << 31), 2),
    (dict(E=FAKE + 2), 3), (dict(C=FAKE + 8), 3), (dict(lse=FAKE + 4), 3), (dict(x=FAKE + 4), 3),
    (dict(red=3), 4), (dict(red=-1), 4), (dict(wsb=16), 5),
])
def test_forward_rejects_without_launch(lib, kw, status):
    assert _fwd(lib, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(g=0), 1), (dict(dE=0), 1), (dict(dC=0), 1), (dict(lse=0), 1),
    (dict(D=100), 2), (dict(dE=FAKE + 2), 3), (dict(stats=FAKE + 4), 3),
    (dict(eps=-1.0), 4), (dict(eps=float("nan")), 4), (dict(eps=float("inf")), 4), (dict(red=7), 4),
    (dict(wsb=1024), 5),
])
def test_backward_rejects_without_launch(lib, kw, status):
    assert _bwd(lib, **kw) == status


@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on fake pointers when a GPU is present")
def test_valid_arguments_without_gpu_report_cuda_error(lib):
    """Without a GPU the device check fails with a status, nothing is launched."""
    assert _fwd(lib) in (6, 7)
    assert _bwd(lib) in (6, 7)


def test_binding_refuses_cpu_tensors(lib):
    import linear_cross_entropy_gb300 as cce
    E = torch.zeros(4, 8, dtype=torch.bfloat16)
    C = torch.zeros(5, 8, dtype=torch.bfloat16)
    x = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA"):
        cce.cce_forward(E, C, x)


def test_extended_entry_points_reject_bad_options(lib):
    vp = ctypes.c_void_p
    args = [vp(FAKE), vp(FAKE), vp(FAKE), 256, 128, 4096, -100, 2]
    for cap in (-1.0, float("nan"), float("inf")):
        assert lib.cce_forward_ex(*args, cap, vp(FAKE), vp(FAKE), vp(FAKE), 1 << 40, vp(0), vp(0)) == 4
    bargs = [vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 256, 128, 4096, -100, 2]
    tail = [vp(FAKE), vp(FAKE), vp(FAKE), 1 << 40, vp(0), vp(0), vp(0)]
    fargs = [vp(FAKE), vp(FAKE), vp(FAKE), 256, 128, 4096, -100]
    ftail = [vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1 << 40, vp(0), vp(0), vp(0)]
    assert lib.cce_loss_and_grad(*fargs, 0, 0.0, 2.0 ** -12, 3, 0, *ftail) == 4   # reduction none
    assert lib.cce_loss_and_grad(*fargs, 2, 0.0, 2.0 ** -12, 4 | 3, 0, *ftail) == 4  # sorting not offered
    assert lib.cce_loss_and_grad(*fargs, 2, -1.0, 2.0 ** -12, 3, 0, *ftail) == 4  # negative softcap
    assert lib.cce_forward_ex2(*args, 0.0, 2, vp(FAKE), vp(FAKE), vp(FAKE), 1 << 40, vp(0), vp(0)) == 4  # bad flag
    assert lib.cce_forward_workspace_bytes_ex(256, 128, 4096, 2) == 0
    assert lib.cce_forward_workspace_bytes_ex(256, 128, 4096, 0) == lib.cce_forward_workspace_bytes(256, 128, 4096)
    assert lib.cce_forward_workspace_bytes_ex(256, 128, 4096, 1) >= \
        lib.cce_forward_workspace_bytes(256, 128, 4096) + 256 * 128 * 2 + 256 * 24
    assert lib.cce_backward_ex(*bargs, 0.0, 2.0 ** -12, 8, *tail) == 4      # unknown flag bit
    assert lib.cce_backward_ex(*bargs, 0.0, 2.0 ** -12, 4 | 16, *tail) == 4  # sort plus an unknown bit
    assert lib.cce_backward_ex(*bargs, -3.0, 2.0 ** -12, 3, *tail) == 4     # negative softcap


def test_pair_map_words_hook(lib):
    """The test hook that caps the survival words of a gradient-GEMM pair's
    work item: returns the previous cap, and out-of-range values restore the
    default of 40 (host only, no device work)."""
    prev = lib.cce_selftest_pair_map_words(3)
    try:
        assert prev == 40
        assert lib.cce_selftest_pair_map_words(0) == 3
        assert lib.cce_selftest_pair_map_words(41) == 40
        assert lib.cce_selftest_pair_map_words(-5) == 40
    finally:
        lib.cce_selftest_pair_map_words(prev)
    assert lib.cce_selftest_pair_map_words(0) == 40


def test_grad_layout_hook(lib):
    """The test hook that forces the gradient GEMM's layout: returns the
    previous setting; out-of-range values restore the automatic choice (0)."""
    prev = lib.cce_selftest_grad_layout(1)
    try:
        assert prev == 0
        assert lib.cce_selftest_grad_layout(2) == 1
        assert lib.cce_selftest_grad_layout(7) == 2
        assert lib.cce_selftest_grad_layout(-1) == 0
    finally:
        lib.cce_selftest_grad_layout(prev)
    assert lib.cce_selftest_grad_layout(0) == 0
