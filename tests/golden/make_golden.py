"""Write tests/golden/oracle_small.json from the CPU oracle alone.

The fixture freezes the oracle's output for a few small seeded problems so
that the same numbers are demanded on every machine the tests run on (the
x86 build host and the Arm GPU host compile oracle.c with different fmaf
implementations and OpenMP runtimes).  Inputs are regenerated from
gemm_inputs at test time; a SHA-256 of their bytes is stored to catch any
drift in the generator.  Run: python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import gemm_inputs as gi  # noqa: E402
import oracle  # noqa: E402

CASES = [
    # name, transA, transB, M, N, K, alpha, beta, seed
    ("nn_7x5x9", "N", "N", 7, 5, 9, 1.0, 0.0, 1001),
    ("tn_6x11x4", "T", "N", 6, 11, 4, -1.5, 0.25, 1002),
    ("nt_9x8x33", "N", "T", 9, 8, 33, 0.5, -1.0, 1003),
    ("tt_13x3x17", "T", "T", 13, 3, 17, 2.0, 1.0, 1004),
]


def case_inputs(ta, tb, M, N, K, seed):
    ra, ca = (M, K) if ta == "N" else (K, M)
    rb, cb = (K, N) if tb == "N" else (N, K)
    A = gi.random_matrix(seed, ra, ca)
    B = gi.random_matrix(seed + 1, rb, cb)
    C = gi.random_matrix(seed + 2, M, N)
    return A, B, C


def fingerprint(*arrays):
    h = hashlib.sha256()
    for a in arrays:
        h.update(np.ascontiguousarray(a, np.float32).tobytes())
    return h.hexdigest()


def main():
    out = {"source": "oracle/oracle.c via oracle.gemm_f64 and oracle.gemm_f32_seq",
           "cases": []}
    for name, ta, tb, M, N, K, alpha, beta, seed in CASES:
        A, B, C = case_inputs(ta, tb, M, N, K, seed)
        args = (ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta, C, N)
        ref, bound = oracle.gemm_f64(*args)
        f32 = oracle.gemm_f32_seq(*args)
        out["cases"].append({
            "name": name, "transA": ta, "transB": tb, "M": M, "N": N, "K": K,
            "alpha": alpha, "beta": beta, "seed": seed,
            "inputs_sha256": fingerprint(A, B, C),
            "ref_f64_hex": [float(v).hex() for v in ref.reshape(-1)],
            "bound_f64_hex": [float(v).hex() for v in bound.reshape(-1)],
            "f32_seq_bits": [int(v) for v in f32.reshape(-1).view(np.uint32)],
        })
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
