"""Writes step_small.json: small MuonH steps computed by the float64 oracle.

Regression fixture only: it pins the oracle to its own earlier output, and the
GPU tests compare the CUDA library against it.  It calls nothing but the
oracle; inputs are drawn here with numpy's seeded generator.

    python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import muonh as om  # noqa: E402

PARAMS = {"lr": 0.02, "beta": 0.95, "ns_steps": 5, "coeffs": [3.4445, -4.775, 2.0315], "eps": 1e-7}
SHAPES = [(4, 6), (6, 4), (5, 5), (1, 8), (3, 1)]


def main():
    rng = np.random.default_rng(20261202)
    cases = []
    ws, gs, ms = [], [], []
    for r, c in SHAPES:
        ws.append((rng.standard_normal((r, c)) * 0.02).astype(np.float32))
        gs.append((rng.standard_normal((r, c)) * 1e-3).astype(np.float32))
        ms.append((rng.standard_normal((r, c)) * 1e-3).astype(np.float32))
    r0 = om.capture_norms(ws)
    p = PARAMS
    out = om.muonh_step(ws, gs, ms, r0, p["lr"], p["beta"], p["ns_steps"], p["coeffs"], p["eps"])
    for i in range(len(SHAPES)):
        cases.append({
            "shape": list(SHAPES[i]),
            "w": ws[i].tolist(), "g": gs[i].tolist(), "m": ms[i].tolist(),
            "r0": float(r0[i]),
            "o": out["o"][i].tolist(),
            "w_new": out["w"][i].astype(np.float32).tolist(),
            "m_new": out["m"][i].astype(np.float32).tolist(),
        })
    doc = {
        "what": "MuonH step (momentum, Newton-Schulz, hyperball) by the float64 oracle",
        "source": "oracle/muonh.py; method from the Puro-2B digest (jacksunwei.me), section "
                  "\"The load-bearing tricks aren't in the abstract\"",
        "params": p,
        "cases": cases,
    }
    with open(os.path.join(HERE, "step_small.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
