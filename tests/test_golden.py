"""The oracle still reproduces its committed regression fixtures
(tests/golden/oracle_small.json and gdn2_small.json, written by
tests/golden/make_golden.py)."""
import json
import os

import numpy as np

import oracle


def test_oracle_reproduces_golden_fixture():
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_small.json")
    rec = json.load(open(path))
    p = {k: np.asarray(v, dtype=np.float64) for k, v in rec["inputs"].items()}
    out = oracle.kda_reference(p["q"], p["k"], p["v"], p["g"], p["beta"], p["A_log"],
                               p["dt_bias"], p["cu_seqlens"].astype(np.int64), p["dO"],
                               scale=rec["scale"], lower_bound=rec["lower_bound"], eps=rec["eps"])
    for k, v in rec["outputs"].items():
        np.testing.assert_allclose(out[k], np.asarray(v), rtol=1e-12, atol=1e-14, err_msg=k)


def test_gdn2_oracle_reproduces_golden_fixture():
    path = os.path.join(os.path.dirname(__file__), "golden", "gdn2_small.json")
    rec = json.load(open(path))
    p = {k: np.asarray(v, dtype=np.float64) for k, v in rec["inputs"].items()}
    out = oracle.gdn2_reference(p["q"], p["k"], p["v"], p["g"], p["erase"], p["write"], p["A_log"],
                                p["dt_bias"], p["cu_seqlens"].astype(np.int64), p["dO"],
                                scale=rec["scale"], lower_bound=rec["lower_bound"], eps=rec["eps"])
    for k, v in rec["outputs"].items():
        np.testing.assert_allclose(out[k], np.asarray(v), rtol=1e-12, atol=1e-14, err_msg=k)
