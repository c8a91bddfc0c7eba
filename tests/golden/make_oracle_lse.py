"""Write the fp64 oracle's LSE for every row of the full-size workloads.

Usage: python tests/golden/make_oracle_lse.py qwen gemma llama long freq

For each workload this draws the seeded inputs (cce_workloads), runs
oracle.forward over all rows and stores tests/golden/oracle_lse_<name>.npz
with the per-row LSE (float64), the input digest and the workload sizes.  It
calls only oracle/ and cce_workloads; nothing here touches the GPU path.  The
full-size GPU parity tests use the stored LSE to evaluate dC rows (which need
every row's LSE) without recomputing the whole forward on the GPU machine.
"""
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import cce_workloads as W  # noqa: E402
import oracle  # noqa: E402


def main(names):
    for name in names:
        w = W.ALL_CONFIGS[name]
        t0 = time.time()
        E_bits, C_bits, x = W.make_inputs(w)
        digest = W.inputs_digest(E_bits, C_bits, x)
        E, C = oracle.from_bits(E_bits, C_bits)
        del E_bits, C_bits
        f = oracle.forward(E, C, x, reduction=w.reduction)
        out = os.path.join(os.path.dirname(os.path.abspath(__file__)), f"oracle_lse_{name}.npz")
        np.savez_compressed(out, lse=f["lse"], digest=np.array(digest),
                            sizes=np.array([w.N, w.D, w.V], np.int64), seed=np.array(w.seed))
        print(f"{name}: N={w.N} D={w.D} V={w.V} loss={f['loss']!r} count={f['count']} "
              f"digest={digest[:16]} {time.time() - t0:.0f}s", flush=True)


if __name__ == "__main__":
    main(sys.argv[1:] or ["qwen", "gemma", "llama", "long", "freq"])
