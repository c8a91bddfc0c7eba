"""ctypes binding of libcce.so (declarations in include/cce.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch  # noqa: F401  (loads the CUDA runtime libcce.so links against)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcce.so")

CCE_OK = 0
STATUS_NAMES = {
    0: "CCE_OK", 1: "CCE_ERR_NULL", 2: "CCE_ERR_SHAPE", 3: "CCE_ERR_ALIGN", 4: "CCE_ERR_ARG",
    5: "CCE_ERR_WORKSPACE", 6: "CCE_ERR_DEVICE", 7: "CCE_ERR_CUDA", 8: "CCE_ERR_TARGET_RANGE",
    9: "CCE_ERR_TIMEOUT",
}
RED = {"none": 0, "sum": 1, "mean": 2}
DEVERR_TARGET_RANGE = 1
DEVERR_TIMEOUT = 2
NUM_PHASES = 8
SORT_VOCAB = 4
FWD_SKIP_IGNORED = 1


class CCEError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{what}: {name}" if what else name)


class MemoryReport(ctypes.Structure):
    _fields_ = [
        ("logits_fp32_bytes", ctypes.c_uint64),
        ("dE_bytes", ctypes.c_uint64),
        ("dC_bytes", ctypes.c_uint64),
        ("lse_bytes", ctypes.c_uint64),
        ("fwd_workspace_bytes", ctypes.c_uint64),
        ("bwd_workspace_bytes", ctypes.c_uint64),
        ("bwd_chunk_cols", ctypes.c_uint64),
        ("fwd_vocab_splits", ctypes.c_uint64),
    ]


_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -m linear_cross_entropy_gb300.build` "
            "(there is no non-CUDA fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.cce_forward_workspace_bytes.argtypes = [i64, i64, i64]
    lib.cce_forward_workspace_bytes.restype = sz
    lib.cce_backward_workspace_bytes.argtypes = [i64, i64, i64]
    lib.cce_backward_workspace_bytes.restype = sz
    lib.cce_forward.argtypes = [vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, vp, vp, vp, sz, vp, vp]
    lib.cce_forward.restype = ctypes.c_int
    lib.cce_backward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float,
                                 vp, vp, vp, sz, vp, vp, vp]
    lib.cce_backward.restype = ctypes.c_int
    lib.cce_forward_ex.argtypes = [vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float, vp, vp, vp, sz,
                                   vp, vp]
    lib.cce_forward_ex.restype = ctypes.c_int
    lib.cce_backward_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float,
                                    ctypes.c_float, ctypes.c_int, vp, vp, vp, sz, vp, vp, vp]
    lib.cce_backward_ex.restype = ctypes.c_int
    lib.cce_backward_workspace_bytes_ex.argtypes = [i64, i64, i64, ctypes.c_int]
    lib.cce_backward_workspace_bytes_ex.restype = sz
    lib.cce_backward_ex2.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float,
                                     ctypes.c_float, ctypes.c_int, sz, vp, vp, vp, sz, vp, vp, vp]
    lib.cce_backward_ex2.restype = ctypes.c_int
    lib.cce_backward_workspace_bytes_ex2.argtypes = [i64, i64, i64, ctypes.c_int, sz]
    lib.cce_backward_workspace_bytes_ex2.restype = sz
    lib.cce_backward_chunk_cols.argtypes = [i64, i64, sz]
    lib.cce_backward_chunk_cols.restype = ctypes.c_uint64
    lib.cce_vocab_sort_workspace_bytes.argtypes = [i64, i64, i64]
    lib.cce_vocab_sort_workspace_bytes.restype = sz
    lib.cce_vocab_logit_sums.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, vp, sz, vp]
    lib.cce_vocab_logit_sums.restype = ctypes.c_int
    lib.cce_vocab_order.argtypes = [vp, i64, vp, vp, sz, vp]
    lib.cce_vocab_order.restype = ctypes.c_int
    lib.cce_forward_workspace_bytes_ex.argtypes = [i64, i64, i64, ctypes.c_int]
    lib.cce_forward_workspace_bytes_ex.restype = sz
    lib.cce_forward_ex2.argtypes = [vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float, ctypes.c_int, vp,
                                    vp, vp, sz, vp, vp]
    lib.cce_forward_ex2.restype = ctypes.c_int
    lib.cce_loss_and_grad_workspace_bytes.argtypes = [i64, i64, i64, sz]
    lib.cce_loss_and_grad_workspace_bytes.restype = sz
    lib.cce_loss_and_grad.argtypes = [vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_int, sz, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    lib.cce_loss_and_grad.restype = ctypes.c_int
    lib.cce_scale_grads.argtypes = [vp, i64, vp, i64, vp, vp]
    lib.cce_scale_grads.restype = ctypes.c_int
    lib.cce_forward_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, vp, vp, vp, vp]
    lib.cce_forward_noalloc.restype = ctypes.c_int
    lib.cce_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint32, vp]
    lib.cce_selftest_wait_timeout.restype = ctypes.c_int
    lib.cce_selftest_pair_timeout.argtypes = [vp, ctypes.c_uint32, ctypes.c_int, vp]
    lib.cce_selftest_pair_timeout.restype = ctypes.c_int
    lib.cce_selftest_pair_map_words.argtypes = [ctypes.c_int]
    lib.cce_selftest_pair_map_words.restype = ctypes.c_int
    lib.cce_selftest_grad_layout.argtypes = [ctypes.c_int]
    lib.cce_selftest_grad_layout.restype = ctypes.c_int
    lib.cce_memory_accounting.argtypes = [i64, i64, i64, ctypes.POINTER(MemoryReport)]
    lib.cce_memory_accounting.restype = ctypes.c_int
    lib.cce_status_string.argtypes = [ctypes.c_int]
    lib.cce_status_string.restype = ctypes.c_char_p
    lib.cce_abi_version.argtypes = []
    lib.cce_abi_version.restype = ctypes.c_int
    lib.cce_kernel_launch_count.argtypes = []
    lib.cce_kernel_launch_count.restype = ctypes.c_uint64
    lib.cce_profile_enable.argtypes = [ctypes.c_int]
    lib.cce_profile_enable.restype = ctypes.c_int
    lib.cce_profile_reset.argtypes = []
    lib.cce_profile_reset.restype = ctypes.c_int
    lib.cce_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]
    lib.cce_profile_read.restype = ctypes.c_int
    lib.cce_profile_phase_name.argtypes = [ctypes.c_int]
    lib.cce_profile_phase_name.restype = ctypes.c_char_p
    _lib = lib
    return lib


def check(status: int, what: str = "") -> None:
    if status != CCE_OK:
        raise CCEError(status, what)
