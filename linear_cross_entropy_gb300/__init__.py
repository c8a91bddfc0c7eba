"""Cut Cross-Entropy for GB300 (sm_103a): the classifier-head matmul fused with
cross-entropy, forward and backward, without writing the N x V logit matrix.

Python binding of libcce.so.  Every step of the computation runs in the
library's CUDA kernels; this module only marshals arguments (PyTorch provides
device memory and streams).  There is no CPU fallback: importing fails when
the library is not built, and calls fail on tensors that are not CUDA tensors.

    loss = linear_cross_entropy(E, C, x)     # E [N,D] bf16, C [V,D] bf16, x [N] int64
    loss.backward()                          # E.grad, C.grad (bf16)

Semantics ("Cut Your Losses in Large-Vocabulary Language Models", section
"The Mathematical Decomposition"; "cut-cross-entropy" kernel card,
"Correctness"): loss_i = LSE_i - C[x_i] . E_i; rows with x_i == ignore_index
add no loss and get exactly zero gradient; reduction none / sum / mean (mean
over non-ignored rows, 0 for a fully ignored batch).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import CCEError, DEVERR_TARGET_RANGE, DEVERR_TIMEOUT, RED

FILTER_EPS = 2.0 ** -12  # finfo(bf16).eps / 32

__all__ = [
    "linear_cross_entropy", "cce_forward", "cce_backward", "CCEError", "FILTER_EPS",
    "forward_workspace_bytes", "backward_workspace_bytes", "backward_chunk_cols", "memory_report", "kernel_launch_count",
    "Profiler", "vocab_logit_sums", "vocab_order", "cce_loss_and_grad", "fused_linear_cross_entropy",
    "loss_and_grad_workspace_bytes", "raise_pending_errors",
]

_lib.load()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_handle(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_inputs(E, C, x):
    for name, t, dt in (("E", E, torch.bfloat16), ("C", C, torch.bfloat16), ("x", x, torch.int64)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
        if t.dtype != dt:
            raise ValueError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if E.dim() != 2 or C.dim() != 2 or x.dim() != 1:
        raise ValueError("expected E [N, D], C [V, D], x [N]")
    if E.shape[1] != C.shape[1] or E.shape[0] != x.shape[0]:
        raise ValueError(f"shape mismatch: E {tuple(E.shape)}, C {tuple(C.shape)}, x {tuple(x.shape)}")


def forward_workspace_bytes(N, D, V, *, skip_ignored=False) -> int:
    return int(_lib.load().cce_forward_workspace_bytes_ex(N, D, V, _lib.FWD_SKIP_IGNORED if skip_ignored else 0))


def backward_workspace_bytes(N, D, V, *, filter_outputs="both", vocab_sort=False, max_staging_bytes=0) -> int:
    flags = FILTER_OUTPUTS[filter_outputs] | (_lib.SORT_VOCAB if vocab_sort else 0)
    return int(_lib.load().cce_backward_workspace_bytes_ex2(N, D, V, flags, int(max_staging_bytes)))


def backward_chunk_cols(N, V, max_staging_bytes=0) -> int:
    """Vocabulary columns per backward chunk for this G-hat staging budget."""
    return int(_lib.load().cce_backward_chunk_cols(N, V, int(max_staging_bytes)))


def memory_report(N, D, V) -> dict:
    rep = _lib.MemoryReport()
    _lib.check(_lib.load().cce_memory_accounting(N, D, V, ctypes.byref(rep)), "cce_memory_accounting")
    return {k: int(getattr(rep, k)) for k, _ in _lib.MemoryReport._fields_}


def kernel_launch_count() -> int:
    return int(_lib.load().cce_kernel_launch_count())


def _raise_word(v, what=""):
    where = f" ({what})" if what else ""
    if v & DEVERR_TIMEOUT:
        raise CCEError(9, "a kernel pipeline wait timed out" + where)
    if v & DEVERR_TARGET_RANGE:
        raise CCEError(8, "target index outside [0, V) and not ignore_index" + where)


def _raise_dev_err(dev_err):
    _raise_word(int(dev_err.item()))


class _DeferredErrors:
    """Device error words of the autograd calls, checked without stalling the
    host.  Each call's word is copied to pinned host memory behind its kernels
    and read once that copy has landed: at a later call, or in
    raise_pending_errors().  A training step therefore never waits for the
    GPU mid-step; an error surfaces one call or more after the call that set
    it (the kernels treat the offending rows as ignored and complete), and
    each call's word is reported at most once.  The pinned words and events
    are a ring per device, allocated once: no pinned allocation per call."""

    SLOTS = 64

    def __init__(self):
        self._pending = []  # (pinned word, event, call name), in issue order
        self._rings = {}  # device index -> [pinned int32 words, events, next slot]
        self._found = []  # errors read while freeing a slot, raised at the next poll, in order

    def _make_ring(self, device):
        return [torch.zeros(self.SLOTS, dtype=torch.int32, pin_memory=True), [None] * self.SLOTS, 0]

    def _record(self, word, events, slot, dev_err):
        """Copies *dev_err into the pinned word behind the call's kernels and
        returns the event that marks the copy's completion."""
        with torch.cuda.device(dev_err.device):
            word.copy_(dev_err, non_blocking=True)
            if events[slot] is None:
                events[slot] = torch.cuda.Event()
            events[slot].record()
        return events[slot]

    def watch(self, dev_err, what):
        key = dev_err.device.index
        ring = self._rings.get(key)
        if ring is None:
            ring = self._make_ring(dev_err.device)
            self._rings[key] = ring
        words, events, slot = ring
        ring[2] = (slot + 1) % self.SLOTS
        word = words[slot:slot + 1]
        # The slot's previous word is read before the slot is reused.  An
        # error found there is kept, not raised yet, so that this call's own
        # word is recorded (and reported later) whatever the older one holds.
        while any(w.data_ptr() == word.data_ptr() for w, _, _ in self._pending):
            try:
                self._take_oldest(wait=True)
            except CCEError as e:
                self._found.append(e)
        self._pending.append((word, self._record(word, events, slot, dev_err), what))
        self.poll(keep_last=True)

    def _take_oldest(self, wait):
        word, ev, what = self._pending[0]
        if wait:
            ev.synchronize()
        elif not ev.query():
            return False
        self._pending.pop(0)
        _raise_word(int(word[0]), what)
        return True

    def poll(self, wait=False, keep_last=False):
        """Raises for the oldest landed word that is not clean; keep_last
        leaves the newest call's word for later."""
        if self._found:
            raise self._found.pop(0)
        while len(self._pending) > (1 if keep_last else 0):
            if not self._take_oldest(wait):
                return


_deferred = _DeferredErrors()


def raise_pending_errors():
    """Waits for the autograd calls issued so far (linear_cross_entropy,
    fused_linear_cross_entropy) and raises CCEError if one of them set a
    device error word."""
    _deferred.poll(wait=True)


def cce_forward(E, C, x, ignore_index=-100, reduction="mean", *, softcap=0.0, skip_ignored=False, stream=None,
                check_errors=True, workspace=None, dev_err=None):
    """Returns (loss, lse).  loss is [N] for reduction='none', else a 0-d tensor.
    softcap > 0 caps the logits as softcap * tanh(logit / softcap).
    skip_ignored: compact away the rows that take part in no loss before the
    GEMM (their lse, and loss for 'none', are then 0; the loss is unchanged)."""
    _check_inputs(E, C, x)
    N, D = E.shape
    V = C.shape[0]
    lib = _lib.load()
    red = RED[reduction]
    dev = E.device
    loss = torch.empty(N if red == 0 else 1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    flags = _lib.FWD_SKIP_IGNORED if skip_ignored else 0
    need = int(lib.cce_forward_workspace_bytes_ex(N, D, V, flags))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if dev_err is None:
        dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        st = lib.cce_forward_ex2(_ptr(E), _ptr(C), _ptr(x), N, D, V, int(ignore_index), red, float(softcap), flags,
                                 _ptr(loss), _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(dev_err),
                                 _stream_handle(stream))
    _lib.check(st, "cce_forward")
    if check_errors:
        _raise_dev_err(dev_err)
    return (loss if red == 0 else loss.reshape(())), lse


FILTER_OUTPUTS = {"both": 3, "dE": 1, "dC": 2, "none": 0}


def cce_backward(E, C, x, lse, grad_out, ignore_index=-100, reduction="mean", filter_eps=FILTER_EPS, *,
                 filter_outputs="both", softcap=0.0, vocab_sort=False, max_staging_bytes=0, stream=None,
                 check_errors=True, workspace=None, dev_err=None, stats=False, dE=None, dC=None):
    """Returns (dE, dC) or (dE, dC, {tiles, skipped}) with stats=True.

    filter_outputs: which gradients skip the filtered tiles -- "both" (plain
    CCE), "dE" (dC from every tile: CCE-Kahan-FullC), "dC" (FullE) or "none".
    vocab_sort: filter over the vocabulary sorted by average logit (the
    gradients are the same; the tiles, and so what the filter skips, differ).
    max_staging_bytes: bound of the bf16 G-hat chunk buffer in the workspace
    (0: the default 512 MiB); a smaller budget means more vocabulary chunks."""
    _check_inputs(E, C, x)
    N, D = E.shape
    V = C.shape[0]
    lib = _lib.load()
    red = RED[reduction]
    dev = E.device
    g = grad_out.to(device=dev, dtype=torch.float32).contiguous().reshape(-1)
    if g.numel() != (N if red == 0 else 1):
        raise ValueError("grad_out must have N elements for reduction='none', else 1")
    lse = lse.contiguous()
    if dE is None:
        dE = torch.empty_like(E)
    if dC is None:
        dC = torch.empty_like(C)
    flags = FILTER_OUTPUTS[filter_outputs] | (_lib.SORT_VOCAB if vocab_sort else 0)
    need = int(lib.cce_backward_workspace_bytes_ex2(N, D, V, flags, int(max_staging_bytes)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if dev_err is None:
        dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    st_t = torch.zeros(2, dtype=torch.int64, device=dev) if stats else None
    with torch.cuda.device(dev):
        st = lib.cce_backward_ex2(_ptr(E), _ptr(C), _ptr(x), _ptr(lse), _ptr(g), N, D, V, int(ignore_index), red,
                                  float(softcap), float(filter_eps), flags, int(max_staging_bytes), _ptr(dE),
                                  _ptr(dC), _ptr(workspace), workspace.numel(), _ptr(dev_err), _ptr(st_t),
                                  _stream_handle(stream))
    _lib.check(st, "cce_backward")
    if check_errors:
        _raise_dev_err(dev_err)
    if stats:
        s = st_t.tolist()
        return dE, dC, {"tiles": s[0], "skipped": s[1]}
    return dE, dC


class LinearCrossEntropyFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, E, C, x, ignore_index, reduction, filter_eps, filter_outputs, softcap, vocab_sort,
                max_staging_bytes):
        err = torch.zeros(1, dtype=torch.int32, device=E.device)
        # The LSE is kept only for the backward, which reads it on the rows
        # that take part; so the forward GEMM skips the other rows
        # (CCE_FWD_SKIP_IGNORED: same loss, per-row loss 0 where ignored).
        loss, lse = cce_forward(E, C, x, ignore_index, reduction, softcap=softcap, skip_ignored=True,
                                check_errors=False, dev_err=err)
        _deferred.watch(err, "cce_forward")
        ctx.save_for_backward(E, C, x, lse)
        ctx.cfg = (ignore_index, reduction, filter_eps, filter_outputs, softcap, vocab_sort, max_staging_bytes)
        return loss

    @staticmethod
    def backward(ctx, grad_loss):
        E, C, x, lse = ctx.saved_tensors
        ignore_index, reduction, filter_eps, filter_outputs, softcap, vocab_sort, max_staging_bytes = ctx.cfg
        err = torch.zeros(1, dtype=torch.int32, device=E.device)
        dE, dC = cce_backward(E, C, x, lse, grad_loss, ignore_index, reduction, filter_eps,
                              filter_outputs=filter_outputs, softcap=softcap, vocab_sort=vocab_sort,
                              max_staging_bytes=max_staging_bytes, check_errors=False, dev_err=err)
        _deferred.watch(err, "cce_backward")
        return dE, dC, None, None, None, None, None, None, None, None


def linear_cross_entropy(E, C, x, ignore_index=-100, reduction="mean", filter_eps=FILTER_EPS,
                         filter_outputs="both", softcap=0.0, vocab_sort=False, max_staging_bytes=0):
    """Cross-entropy of the logits E @ C^T against targets x, never materialised.

    E [N, D] bf16 (hidden states), C [V, D] bf16 (classifier weight), x [N]
    int64.  filter_eps is the backward's tile-skip threshold (0 disables);
    filter_outputs picks which gradients it applies to ("both", "dE", "dC",
    "none"); softcap > 0 caps the logits as softcap * tanh(logit / softcap);
    vocab_sort filters over the vocabulary sorted by average logit;
    max_staging_bytes bounds the backward's G-hat chunk buffer (0: default).
    Device errors (a target outside [0, V)) are raised without stalling the
    step: at a later call or at raise_pending_errors()."""
    return LinearCrossEntropyFunction.apply(E, C, x, ignore_index, reduction, filter_eps, filter_outputs,
                                            softcap, vocab_sort, max_staging_bytes)


def loss_and_grad_workspace_bytes(N, D, V, max_staging_bytes=0) -> int:
    return int(_lib.load().cce_loss_and_grad_workspace_bytes(N, D, V, int(max_staging_bytes)))


def cce_loss_and_grad(E, C, x, ignore_index=-100, reduction="mean", filter_eps=FILTER_EPS, *,
                      filter_outputs="both", softcap=0.0, max_staging_bytes=0, stream=None, check_errors=True,
                      workspace=None, dev_err=None, stats=False, lse=True, dE=None, dC=None):
    """The single call: (loss, lse, dE, dC) or, with stats=True, also
    {tiles, skipped}.  dE and dC are the gradients of the reduced loss for a
    unit upstream gradient.  reduction: "sum" or "mean".  lse=False skips
    writing the per-row LSE (returns None for it)."""
    _check_inputs(E, C, x)
    if reduction not in ("sum", "mean"):
        raise ValueError("the single call supports reduction 'sum' and 'mean'")
    N, D = E.shape
    V = C.shape[0]
    lib = _lib.load()
    dev = E.device
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse_t = torch.empty(N, dtype=torch.float32, device=dev) if lse else None
    if dE is None:
        dE = torch.empty_like(E)
    if dC is None:
        dC = torch.empty_like(C)
    need = int(lib.cce_loss_and_grad_workspace_bytes(N, D, V, int(max_staging_bytes)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if dev_err is None:
        dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    st_t = torch.zeros(2, dtype=torch.int64, device=dev) if stats else None
    with torch.cuda.device(dev):
        st = lib.cce_loss_and_grad(_ptr(E), _ptr(C), _ptr(x), N, D, V, int(ignore_index), RED[reduction],
                                   float(softcap), float(filter_eps), FILTER_OUTPUTS[filter_outputs],
                                   int(max_staging_bytes), _ptr(loss), _ptr(lse_t), _ptr(dE), _ptr(dC),
                                   _ptr(workspace), workspace.numel(), _ptr(dev_err), _ptr(st_t),
                                   _stream_handle(stream))
    _lib.check(st, "cce_loss_and_grad")
    if check_errors:
        _raise_dev_err(dev_err)
    out = (loss.reshape(()), lse_t, dE, dC)
    if stats:
        s = st_t.tolist()
        return out + ({"tiles": s[0], "skipped": s[1]},)
    return out


class FusedLinearCrossEntropyFunction(torch.autograd.Function):
    """The loss and both gradients come from one library call in the forward;
    the backward only multiplies them by the upstream gradient."""

    @staticmethod
    def forward(ctx, E, C, x, ignore_index, reduction, filter_eps, filter_outputs, softcap, max_staging_bytes):
        err = torch.zeros(1, dtype=torch.int32, device=E.device)
        loss, _, dE, dC = cce_loss_and_grad(E, C, x, ignore_index, reduction, filter_eps,
                                            filter_outputs=filter_outputs, softcap=softcap,
                                            max_staging_bytes=max_staging_bytes, lse=False,
                                            check_errors=False, dev_err=err)
        _deferred.watch(err, "cce_loss_and_grad")
        ctx.save_for_backward(dE, dC)
        return loss

    @staticmethod
    def backward(ctx, grad_loss):
        dE, dC = ctx.saved_tensors
        g = grad_loss.to(device=dE.device, dtype=torch.float32).contiguous().reshape(1)
        with torch.cuda.device(dE.device):
            st = _lib.load().cce_scale_grads(_ptr(dE), dE.numel(), _ptr(dC), dC.numel(), _ptr(g),
                                             _stream_handle(None))
        _lib.check(st, "cce_scale_grads")
        return dE, dC, None, None, None, None, None, None, None


def fused_linear_cross_entropy(E, C, x, ignore_index=-100, reduction="mean", filter_eps=FILTER_EPS,
                               filter_outputs="both", softcap=0.0, max_staging_bytes=0):
    """linear_cross_entropy computed by the single call: loss and gradients in
    the forward (token chunks of staged logits, no recompute), the backward
    only scales.  reduction "sum" or "mean".  Device errors are raised as
    for linear_cross_entropy."""
    return FusedLinearCrossEntropyFunction.apply(E, C, x, ignore_index, reduction, filter_eps, filter_outputs,
                                                 softcap, max_staging_bytes)


def vocab_logit_sums(E, C, x, ignore_index=-100, *, stream=None):
    """sums[v] = sum of the logits C_v . E_i over the rows that take part
    (fp32 [V]); the statistic vocabulary sorting orders by."""
    _check_inputs(E, C, x)
    N, D = E.shape
    V = C.shape[0]
    lib = _lib.load()
    ws = torch.empty(max(int(lib.cce_vocab_sort_workspace_bytes(N, D, V)), 16), dtype=torch.uint8,
                     device=E.device)
    sums = torch.empty(V, dtype=torch.float32, device=E.device)
    with torch.cuda.device(E.device):
        st = lib.cce_vocab_logit_sums(_ptr(E), _ptr(C), _ptr(x), N, D, V, int(ignore_index), _ptr(sums), _ptr(ws),
                                      ws.numel(), _stream_handle(stream))
    _lib.check(st, "cce_vocab_logit_sums")
    return sums


def vocab_order(keys, *, stream=None):
    """perm (int32 [V]): the stable ascending order of the fp32 keys."""
    if not keys.is_cuda or keys.dtype != torch.float32 or keys.dim() != 1:
        raise ValueError("keys must be a 1-D float32 CUDA tensor")
    keys = keys.contiguous()
    V = keys.numel()
    lib = _lib.load()
    ws = torch.empty(max(int(lib.cce_vocab_sort_workspace_bytes(1, 8, V)), 16), dtype=torch.uint8,
                     device=keys.device)
    perm = torch.empty(V, dtype=torch.int32, device=keys.device)
    with torch.cuda.device(keys.device):
        st = lib.cce_vocab_order(_ptr(keys), V, _ptr(perm), _ptr(ws), ws.numel(), _stream_handle(stream))
    _lib.check(st, "cce_vocab_order")
    return perm


@dataclass
class PhaseTimes:
    ms: dict
    launches: dict


class Profiler:
    """Per-phase CUDA-event timing recorded by the library on its stream."""

    def __enter__(self):
        lib = _lib.load()
        lib.cce_profile_reset()
        lib.cce_profile_enable(1)
        return self

    def __exit__(self, *exc):
        _lib.load().cce_profile_enable(0)
        return False

    @staticmethod
    def read() -> PhaseTimes:
        lib = _lib.load()
        ms = (ctypes.c_double * _lib.NUM_PHASES)()
        cnt = (ctypes.c_int64 * _lib.NUM_PHASES)()
        _lib.check(lib.cce_profile_read(ms, cnt), "cce_profile_read")
        names = [lib.cce_profile_phase_name(i).decode() for i in range(_lib.NUM_PHASES)]
        return PhaseTimes({n: ms[i] for i, n in enumerate(names)}, {n: cnt[i] for i, n in enumerate(names)})
