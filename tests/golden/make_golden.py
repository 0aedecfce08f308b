"""Writes tiny_favor.json: a small seeded FAVOR+ case and the oracle's outputs for it.

The pages print no worked numeric example, so this fixture is a regression record of the oracle
(it calls only ``oracle`` and ``seeded_inputs``). ``tests/test_golden.py`` checks the stored
outputs two ways: against the oracle as it stands, and against a 50-digit brute-force evaluation
of the explicit sums of the "Performer" paper note's *Normalization* equation (all j for the
non-causal form, j <= i for the causal form of "Performer for vision", *How It Works*, Step 2).

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import seeded_inputs as si  # noqa: E402


def main():
    n, d, m = 6, 4, 8
    seed, omega_seed = 4242, 4343
    Q = si.normal(seed, si.TID_Q, n * d).reshape(1, n, d)
    K = si.normal(seed, si.TID_K, n * d).reshape(1, n, d)
    V = si.normal(seed, si.TID_V, n * d).reshape(1, n, d)
    om = si.build_omega(omega_seed, m, d)
    out = {
        "about": "tiny FAVOR+ case; inputs from seeded_inputs, outputs from the fp64 oracle",
        "n": n, "d": d, "m": m, "seed": seed, "omega_seed": omega_seed,
        "Q": Q[0].tolist(), "K": K[0].tolist(), "V": V[0].tolist(), "Omega": om.tolist(),
    }
    for kind in ("exp", "relu"):
        out[f"Y_noncausal_{kind}"] = oracle.attn_noncausal(Q, K, V, om, kind=kind)[0].tolist()
        out[f"Y_causal_{kind}"] = oracle.attn_causal(Q, K, V, om, kind=kind)[0].tolist()
    out["Phi_Q_row_exp"] = oracle.features(Q, om, stab="row")[0].tolist()
    with open(os.path.join(HERE, "tiny_favor.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
