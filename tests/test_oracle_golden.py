"""The oracle reproduces its frozen small-case outputs bit for bit.

The fixture (tests/golden/oracle_small.json) is written by
tests/golden/make_golden.py, which calls only the oracle.  This test runs on
every machine the suite runs on, so the oracle's results cannot silently
differ between the build host and the GPU host.
"""
import json
import os

import numpy as np

from tests.golden.make_golden import case_inputs, fingerprint

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_frozen_fixture(oracle_mod):
    with open(os.path.join(HERE, "golden", "oracle_small.json")) as f:
        fx = json.load(f)
    assert len(fx["cases"]) >= 4
    for c in fx["cases"]:
        ta, tb, M, N, K = c["transA"], c["transB"], c["M"], c["N"], c["K"]
        A, B, C = case_inputs(ta, tb, M, N, K, c["seed"])
        assert fingerprint(A, B, C) == c["inputs_sha256"], c["name"]
        args = (ta, tb, M, N, K, c["alpha"], A, A.shape[1], B, B.shape[1],
                c["beta"], C, N)
        ref, bound = oracle_mod.gemm_f64(*args)
        f32 = oracle_mod.gemm_f32_seq(*args)
        assert [float(v).hex() for v in ref.reshape(-1)] == c["ref_f64_hex"], c["name"]
        assert [float(v).hex() for v in bound.reshape(-1)] == c["bound_f64_hex"], c["name"]
        assert f32.reshape(-1).view(np.uint32).tolist() == c["f32_seq_bits"], c["name"]
