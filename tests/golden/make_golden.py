"""Write tiny_bwd.json: a small worked example of the intra-chunk backward.

The pages print no worked example, so the stored values are the oracle's, written by this
script, which calls nothing but ``oracle`` and the seeded input recipe of ``kda_inputs``
(bwd_intra page, module docstring: the definitions the oracle writes out).  The inputs are
stored too, so that a change of the recipe or of the oracle shows up in
``tests/test_golden.py``.

    python tests/golden/make_golden.py
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import kda_inputs  # noqa: E402
import oracle  # noqa: E402

# two 8-token chunks, two heads, four channels; steep enough gates that the exponents matter
RECIPE = dict(B=1, T=16, H=2, k_dim=4, bt=8, gate_lo=-2.0, seed=20261202)
ARGS = ("q", "k", "g", "beta", "dAqk", "dAkk")


def make():
    r = RECIPE
    inp = kda_inputs.make_inputs(r["B"], r["T"], r["H"], gate_lo=r["gate_lo"], seed=r["seed"],
                                 k_dim=r["k_dim"], bt=r["bt"])
    out = oracle.intra_bwd(*(inp[n] for n in ARGS), bt=r["bt"])
    return {
        "source": "oracle.intra_bwd (fp64 C) on kda_inputs.make_inputs(**recipe)",
        "recipe": r,
        "inputs": {n: inp[n].double().tolist() for n in ARGS},
        "outputs": {n: v.tolist() for n, v in zip(("dq", "dk", "db", "dg"), out)},
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_bwd.json"), "w") as f:
        json.dump(make(), f, indent=None, separators=(",", ":"))
        f.write("\n")
    print("wrote", os.path.join(HERE, "tiny_bwd.json"))
