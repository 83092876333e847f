"""Writes tests/golden/oracle_small.json and tests/golden/gdn2_small.json by
calling only the oracle.

The pages print no worked numerical example for KDA or GDN-2, so these
fixtures are regression records of the pinned oracle on small seeded
problems (two packed sequences of 5 and 11 tokens, H=2, D=8, nonzero A_log /
dt_bias, scale 0.5; the GDN-2 one with channel-wise erase / write gates in
place of beta).
Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def problem():
    rng = np.random.default_rng(20260)
    lengths = [5, 11]
    S, H, D = sum(lengths), 2, 8
    p = dict(q=rng.standard_normal((S, H, D)), k=rng.standard_normal((S, H, D)),
             v=rng.standard_normal((S, H, D)), g=rng.standard_normal((S, H, D)),
             beta=rng.standard_normal((S, H)), A_log=rng.standard_normal(H) * 0.5,
             dt_bias=rng.standard_normal((H, D)) * 0.5, dO=rng.standard_normal((S, H, D)))
    # store inputs rounded to float32 so the JSON round-trip is exact
    p = {k: v.astype(np.float32).astype(np.float64) for k, v in p.items()}
    p["cu_seqlens"] = [0, 5, 16]
    return p


def problem_gdn2():
    rng = np.random.default_rng(20261)
    lengths = [5, 11]
    S, H, D = sum(lengths), 2, 8
    p = {n: rng.standard_normal((S, H, D)) for n in ["q", "k", "v", "g", "erase", "write", "dO"]}
    p["A_log"] = rng.standard_normal(H) * 0.5
    p["dt_bias"] = rng.standard_normal((H, D)) * 0.5
    p = {k: v.astype(np.float32).astype(np.float64) for k, v in p.items()}
    p["cu_seqlens"] = [0, 5, 16]
    return p


def write(name, p, out):
    rec = {"inputs": {k: (v.tolist() if hasattr(v, "tolist") else v) for k, v in p.items()},
           "scale": 0.5, "lower_bound": -5.0, "eps": 1e-6,
           "outputs": {k: v.tolist() for k, v in out.items()}}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), name)
    with open(path, "w") as f:
        json.dump(rec, f)
    print("wrote", path)


def main():
    p = problem()
    out = oracle.kda_reference(p["q"], p["k"], p["v"], p["g"], p["beta"], p["A_log"],
                               p["dt_bias"], p["cu_seqlens"], p["dO"], scale=0.5)
    write("oracle_small.json", p, out)
    p = problem_gdn2()
    out = oracle.gdn2_reference(p["q"], p["k"], p["v"], p["g"], p["erase"], p["write"], p["A_log"],
                                p["dt_bias"], p["cu_seqlens"], p["dO"], scale=0.5)
    write("gdn2_small.json", p, out)


if __name__ == "__main__":
    main()
