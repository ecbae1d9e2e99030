"""Writes tests/golden/oracle_regression.json from the CPU oracle alone.

The pages print no worked example, so the stored values here are not the
pages': they record what the fp64 oracle gives on a small deterministic input
(closed-form sin/cos values, no random generator) so that a later change to
the oracle's arithmetic shows up as a diff.  Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def golden_inputs():
    T, Hqk, Hv, K, V = 11, 1, 2, 4, 3
    t = np.arange(T)[:, None, None]
    q = np.sin(0.7 * t + np.arange(K)[None, None, :] * 1.3 + 0.1)
    k = np.cos(0.5 * t - np.arange(K)[None, None, :] * 0.9)
    v = np.sin(0.3 * t * (np.arange(V)[None, None, :] + 1) + np.arange(Hv)[None, :, None])
    a = np.cos(0.4 * np.arange(T)[:, None] + np.arange(Hv)[None, :])
    b = np.sin(0.9 * np.arange(T)[:, None] - np.arange(Hv)[None, :])
    A_log = np.array([0.5, math.log(16.0)])
    dt_bias = np.array([-0.25, 0.75])
    h0 = np.cos(np.arange(Hv * V * K)).reshape(1, Hv, V, K) * 0.1
    return dict(T=T, Hqk=Hqk, Hv=Hv, K=K, V=V, q=q, k=k, v=v, a=a, b=b, A_log=A_log,
                dt_bias=dt_bias, h0=h0, scale=0.5)


def golden_outputs(inp):
    g, beta = oracle.gate_prep(inp["a"], inp["b"], inp["A_log"], inp["dt_bias"])
    o, hT = oracle.gdn_fwd(inp["q"], inp["k"], inp["v"], g, beta, inp["h0"], scale=inp["scale"],
                           l2norm_qk=True)
    M, S = oracle.segment_summary(inp["k"], inp["v"], g, beta, [0, 5, 11], l2norm_qk=True)
    return dict(g=g, beta=beta, o=o, hT=hT, M=M, S_local=S)


if __name__ == "__main__":
    out = {k: v.tolist() for k, v in golden_outputs(golden_inputs()).items()}
    out["_about"] = ("fp64 oracle outputs on the closed-form input of make_golden.py; "
                     "written by tests/golden/make_golden.py")
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=None)
    print("wrote", path)
