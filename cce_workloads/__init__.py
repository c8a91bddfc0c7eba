"""Seeded synthetic inputs for the Cut Cross-Entropy workloads.

This module is shared by the fp64 oracle (``oracle/``), the tests and the
benchmark.  It holds none of the method's arithmetic: it only draws the
inputs E [N, D] (bf16 bits), C [V, D] (bf16 bits) and x [N] (int64).

The inputs stand in for the pages' real workloads, which need model weights
and datasets that are not available here:

* Gemma 2 2B-Instruct hidden states on Alpaca, N=8192, |V|=256000, D=2304
  ("Cut Your Losses in Large-Vocabulary Language Models", Table 1);
* Qwen2.5-0.5B hidden states on blog prose, |V|=151936, D=896, 4096 tokens
  ("Cut Cross-Entropy: Training Loss Without the Logit Matrix ...",
  section "Gradient filtering: the part that makes it fast");
* 65,536 tokens against a 128,256-entry vocabulary at D=2048
  ("cut-cross-entropy" kernel card, section "Measured").

Every draw is bit-reproducible on any platform: random bits come from numpy's
PCG64 (integer arithmetic only), and the only floating-point operations used
on them are +, -, *, /, sqrt, floor, frexp and ldexp, which IEEE 754 fixes
exactly.  numpy's transcendental functions (whose last bit may differ between
x86 and Arm builds) are never used; ``_log`` and ``_exp`` below are written
out from their series.  Large tensors are drawn in independent blocks of
2**22 elements, each seeded by (seed, stream, block), so the result does not
depend on how many worker threads draw them.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

IGNORE_INDEX = -100
BLOCK = 1 << 22

# Stream ids of the independent random streams.
_S_C, _S_E, _S_XRANK, _S_XPERM, _S_IGNORE, _S_XUNIF = 1, 2, 3, 4, 5, 6

_LN2 = 0.6931471805599453  # nearest double to ln 2


# ----------------------------------------------------------------------------
# Platform-exact elementary functions (float64, basic IEEE operations only).
# ----------------------------------------------------------------------------
def _log(p: np.ndarray) -> np.ndarray:
    """Natural log of positive float64 values.

    p = m * 2**e with m in [0.5, 1) (exact frexp); m is moved into
    [sqrt(1/2), sqrt(2)) and ln m = 2 * atanh(z), z = (m-1)/(m+1), summed as
    the odd power series of atanh (|z| < 0.172, 14 terms reach 1e-17).
    """
    p = np.asarray(p, dtype=np.float64)
    m, e = np.frexp(p)
    small = m < 0.7071067811865476
    m = np.where(small, m * 2.0, m)
    e = np.where(small, e - 1, e).astype(np.float64)
    z = (m - 1.0) / (m + 1.0)
    z2 = z * z
    acc = np.zeros_like(z)
    for k in range(27, 0, -2):  # Horner over 1/k for k = 27, 25, ..., 1
        acc = acc * z2 + 1.0 / k
    return e * _LN2 + 2.0 * z * acc


def _exp(y: np.ndarray) -> np.ndarray:
    """exp of float64 values in a moderate range (|y| < 700).

    y = k ln2 + r with r in [0, ln2); exp(r) by its Taylor series (22 terms),
    then scaled by 2**k with ldexp (exact).
    """
    y = np.asarray(y, dtype=np.float64)
    k = np.floor(y / _LN2)
    r = y - k * _LN2
    acc = np.ones_like(r)
    for n in range(22, 0, -1):  # Horner: 1 + r/1 (1 + r/2 (1 + ...))
        acc = 1.0 + acc * r / n
    return np.ldexp(acc, k.astype(np.int64))


# Inverse normal CDF: P. J. Acklam, "An algorithm for computing the inverse
# normal cumulative distribution function" (2003); relative error < 1.15e-9,
# far below the bf16 resolution the draws are rounded to.
_A = (-3.969683028665376e+01, 2.209460984245205e+02, -2.759285104469687e+02,
      1.383577518672690e+02, -3.066479806614716e+01, 2.506628277459239e+00)
_B = (-5.447609879822406e+01, 1.615858368580409e+02, -1.556989798598866e+02,
      6.680131188771972e+01, -1.328068155288572e+01)
_Cc = (-7.784894002430293e-03, -3.223964580411365e-01, -2.400758277161838e+00,
       -2.549732539343734e+00, 4.374664141464968e+00, 2.938163982698783e+00)
_Dd = (7.784695709041462e-03, 3.224671290700398e-01, 2.445134137142996e+00,
       3.754408661907416e+00)
_P_LOW = 0.02425


def _norm_ppf(p: np.ndarray) -> np.ndarray:
    out = np.empty_like(p)
    lo = p < _P_LOW
    hi = p > 1.0 - _P_LOW
    mid = ~(lo | hi)
    q = p[mid] - 0.5
    r = q * q
    num = ((((_A[0] * r + _A[1]) * r + _A[2]) * r + _A[3]) * r + _A[4]) * r + _A[5]
    den = ((((_B[0] * r + _B[1]) * r + _B[2]) * r + _B[3]) * r + _B[4]) * r + 1.0
    out[mid] = num * q / den
    for mask, sign, base in ((lo, 1.0, p[lo]), (hi, -1.0, 1.0 - p[hi])):
        if base.size == 0:
            continue
        q = np.sqrt(-2.0 * _log(base))
        num = ((((_Cc[0] * q + _Cc[1]) * q + _Cc[2]) * q + _Cc[3]) * q + _Cc[4]) * q + _Cc[5]
        den = (((_Dd[0] * q + _Dd[1]) * q + _Dd[2]) * q + _Dd[3]) * q + 1.0
        out[mask] = sign * num / den
    return out


def _uniform_open(gen: np.random.Generator, n: int) -> np.ndarray:
    """n doubles uniform on (0, 1): (k + 0.5) / 2**53 with k a 53-bit integer."""
    k = gen.bit_generator.random_raw(n) >> np.uint64(11)
    return (k.astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def _gen(seed: int, stream: int, block: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, block])))


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even); returns uint16 bits."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_block(args):
    seed, stream, block, n, sigma = args
    g = _gen(seed, stream, block)
    z = _norm_ppf(_uniform_open(g, n))
    return f32_to_bf16_bits((z * sigma).astype(np.float32))


def _pool_workers(nblocks: int) -> int:
    env = os.environ.get("CCE_GEN_WORKERS")
    if env is not None:
        return max(1, int(env))
    return max(1, min(nblocks, os.cpu_count() or 1, 16))


def normal_bf16(seed: int, stream: int, n: int, sigma: float) -> np.ndarray:
    """n draws of N(0, sigma^2) rounded to bf16, as uint16 bits."""
    nblocks = (n + BLOCK - 1) // BLOCK
    jobs = [(seed, stream, b, min(BLOCK, n - b * BLOCK), sigma) for b in range(nblocks)]
    workers = _pool_workers(nblocks)
    if workers <= 1 or nblocks <= 2:
        parts = [_normal_block(j) for j in jobs]
    else:
        # Threads, not processes: numpy releases the GIL in its array loops,
        # and no process is forked from one that may hold a CUDA context.
        with ThreadPoolExecutor(max_workers=workers) as ex:
            parts = list(ex.map(_normal_block, jobs))
    return np.concatenate(parts) if parts else np.zeros(0, np.uint16)


def normal_f64(seed: int, stream: int, n: int) -> np.ndarray:
    """n draws of N(0, 1) in float64 (used before the E rows are boosted)."""
    out = []
    for b in range((n + BLOCK - 1) // BLOCK):
        g = _gen(seed, stream, b)
        out.append(_norm_ppf(_uniform_open(g, min(BLOCK, n - b * BLOCK))))
    return np.concatenate(out) if out else np.zeros(0)


def zipf_targets(seed: int, n: int, V: int, s: float) -> np.ndarray:
    """Zipf(s) ranks truncated to 1..V (p(r) ~ r**-s), mapped to token ids
    through a seeded random permutation of [0, V)."""
    r = np.arange(1, V + 1, dtype=np.float64)
    w = _exp(-s * _log(r))
    cdf = np.cumsum(w)  # sequential, so exact order is fixed
    u = _uniform_open(_gen(seed, _S_XRANK), n) * cdf[-1]
    rank = np.searchsorted(cdf, u, side="right")
    rank = np.minimum(rank, V - 1)  # rank index 0 = most frequent
    perm = _gen(seed, _S_XPERM).permutation(V)
    return perm[rank].astype(np.int64)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: sizes, value distributions and loss settings."""
    name: str
    N: int
    D: int
    V: int
    c_scale: float          # C ~ N(0, (c_scale / sqrt(D))^2)
    targets: str            # "uniform", "zipf" or "frequent_scattered"
    zipf_s: float = 1.1
    boost: float = 0.0      # E_i += boost * C[x_i] / ||C[x_i]||
    ignore_frac: float = 0.0
    reduction: str = "mean"
    filter_modes: tuple = ("on",)
    seed: int = 0

    @property
    def c_sigma(self) -> float:
        return self.c_scale / math.sqrt(self.D)

    def flops_fwd_bwd(self) -> int:
        """Unfiltered algorithmic flops of forward + backward: 8 N D V."""
        return 8 * self.N * self.D * self.V

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads (sizes and recipes as specified for this operator).
CONFIGS = {
    "tiny": Workload("tiny", 256, 128, 4096, 2.0, "uniform", reduction="mean"),
    "qwen": Workload("qwen", 4096, 896, 151936, 4.0, "zipf", boost=3.0,
                     ignore_frac=0.05, reduction="mean"),
    "gemma": Workload("gemma", 8192, 2304, 256000, 4.0, "zipf", boost=3.0,
                      ignore_frac=0.0, reduction="mean", filter_modes=("on", "off")),
    "llama": Workload("llama", 16384, 4096, 128256, 4.0, "zipf", boost=3.0,
                      ignore_frac=0.05, reduction="sum"),
    "long": Workload("long", 65536, 2048, 128256, 6.0, "zipf", boost=5.0,
                     ignore_frac=0.10, reduction="mean", filter_modes=("on", "off")),
}
CONFIG_ORDER = ("tiny", "qwen", "gemma", "llama", "long")

# Supplementary workloads (not among the five above): the Qwen2.5-0.5B head
# shape with the softmax mass on 256 frequent tokens that a random vocabulary
# order scatters (frequent_token_inputs with scatter=True, unigram=8) -- the
# case vocabulary sorting is for -- at 4,096 tokens and at 16,384 and 65,536
# (the sort's cost is per vocabulary, its saving per token).
SUPPLEMENTARY = {
    "freq": Workload("freq", 4096, 896, 151936, 0.0, "frequent_scattered", ignore_frac=0.05,
                     reduction="mean", filter_modes=("on",)),
    "freq16k": Workload("freq16k", 16384, 896, 151936, 0.0, "frequent_scattered", ignore_frac=0.05,
                        reduction="mean", filter_modes=("on",)),
    "freq64k": Workload("freq64k", 65536, 896, 151936, 0.0, "frequent_scattered", ignore_frac=0.05,
                        reduction="mean", filter_modes=("on",)),
}
ALL_CONFIGS = {**CONFIGS, **SUPPLEMENTARY}


def make_inputs(w: Workload):
    """Draw (E_bits [N,D] uint16, C_bits [V,D] uint16, x [N] int64) for w.

    Order of operations (fixed): C is drawn and rounded to bf16; the targets
    are drawn; E's base normals are drawn in float64; the boost uses the bf16
    C rows of the drawn targets (norms accumulated column by column in
    float64); E is rounded to float32 then bf16; finally the ignore mask
    replaces a Bernoulli(ignore_frac) subset of targets with -100 (the boost
    was applied to those rows too).
    """
    N, D, V = w.N, w.D, w.V
    if w.targets == "frequent_scattered":
        return frequent_token_inputs(N, D, V, n_freq=256, seed=w.seed, ignore_frac=w.ignore_frac, scatter=True,
                                     unigram=8.0)
    C_bits = normal_bf16(w.seed, _S_C, V * D, w.c_sigma).reshape(V, D)
    if w.targets == "uniform":
        x = _gen(w.seed, _S_XUNIF).integers(0, V, size=N, dtype=np.int64)
    elif w.targets == "zipf":
        x = zipf_targets(w.seed, N, V, w.zipf_s)
    else:
        raise ValueError(w.targets)
    E = normal_f64(w.seed, _S_E, N * D).reshape(N, D)
    if w.boost != 0.0:
        cx = bf16_bits_to_f32(C_bits[x]).astype(np.float64)
        sq = np.zeros(N)
        for d in range(D):
            col = cx[:, d]
            sq = sq + col * col
        norm = np.sqrt(sq)
        norm = np.where(norm > 0.0, norm, 1.0)
        E = E + (w.boost / norm)[:, None] * cx
    E_bits = f32_to_bf16_bits(E.astype(np.float32))
    if w.ignore_frac > 0.0:
        u = _uniform_open(_gen(w.seed, _S_IGNORE), N)
        x = np.where(u < w.ignore_frac, np.int64(IGNORE_INDEX), x)
    return E_bits, C_bits, x


def inputs_digest(E_bits, C_bits, x) -> str:
    """sha256 over the exact input bytes (detects any cross-platform drift)."""
    h = hashlib.sha256()
    for a in (E_bits, C_bits, x):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def small(name: str, N: int, D: int, V: int, **kw) -> Workload:
    """A small custom workload (parity and edge cases)."""
    base = dict(c_scale=4.0, targets="zipf", boost=3.0, ignore_frac=0.05, reduction="mean")
    base.update(kw)
    return Workload(name, N, D, V, **base)


def frequent_token_inputs(N: int, D: int, V: int, n_freq: int = 256, seed: int = 0,
                          ignore_frac: float = 0.05, scatter: bool = False, unigram: float = 0.0):
    """A supplementary workload where the gradient filter bites: the n_freq
    lowest ids are "frequent tokens" with large classifier rows (as byte-pair
    merge order puts frequent tokens at low ids), every other row is small,
    and targets are drawn uniformly among the frequent ids.  Softmax mass then
    sits in the first n_freq columns, so most 128 x 128 tiles are skippable.

    unigram > 0: every hidden state gets a common component 4 u along a fixed
    random unit direction u and every frequent row gets (unigram / 4) u, so
    the frequent tokens' logits are raised by about `unigram` on every row --
    the shared "frequent token" bias of a trained head, which makes the
    average logit a useful sort key.
    scatter: token ids are relabelled by a seeded random permutation of
    [0, V), so the frequent tokens are spread over the whole vocabulary (an
    arbitrary vocabulary order; "Cut Cross-Entropy: Training Loss Without the
    Logit Matrix ...", section "Gradient filtering: the part that makes it
    fast", measures the filter under a random vocabulary permutation).
    Defaults reproduce the original draw bit for bit.
    Returns (E_bits, C_bits, x)."""
    g = _gen(seed, 7)
    big = normal_bf16(seed, 8, n_freq * D, 6.0 / math.sqrt(D))
    small = normal_bf16(seed, 9, (V - n_freq) * D, 0.5 / math.sqrt(D))
    C_bits = np.concatenate([big, small]).reshape(V, D)
    E_bits = normal_bf16(seed, 10, N * D, 1.0).reshape(N, D)
    x = g.integers(0, n_freq, size=N, dtype=np.int64)
    if unigram > 0.0:
        u = normal_f64(seed, 12, D)
        sq = 0.0
        for d in range(D):
            sq += u[d] * u[d]
        u = u / math.sqrt(sq)
        E = bf16_bits_to_f32(E_bits).astype(np.float64) + 4.0 * u[None, :]
        E_bits = f32_to_bf16_bits(E.astype(np.float32))
        Cf = bf16_bits_to_f32(C_bits[:n_freq]).astype(np.float64) + (unigram / 4.0) * u[None, :]
        C_bits[:n_freq] = f32_to_bf16_bits(Cf.astype(np.float32))
    if scatter:
        perm = _gen(seed, 13).permutation(V)  # natural id j -> token id perm[j]
        C_s = np.empty_like(C_bits)
        C_s[perm] = C_bits
        C_bits = C_s
        x = perm[x].astype(np.int64)
    u = _uniform_open(_gen(seed, 11), N)
    x = np.where(u < ignore_frac, np.int64(IGNORE_INDEX), x)
    return E_bits, C_bits, x


# A supplementary benchmark workload (not one of the five above): the
# Qwen2.5-0.5B head shape with softmax mass on 256 frequent tokens that a
# random vocabulary order scatters; the case vocabulary sorting is for.
FREQ_SCATTERED = dict(N=4096, D=896, V=151936, n_freq=256, seed=0, ignore_frac=0.05, scatter=True,
                      unigram=8.0)
