"""The stored worked example, tests/golden/tiny_bwd.json (written from the oracle by
tests/golden/make_golden.py; the pages print none of their own): the seeded recipe still
regenerates the stored inputs bit for bit, the oracle still gives the stored outputs, and
an independent method -- torch fp64 autograd of the separable forward -- agrees with them."""

import json
import os

import numpy as np
import pytest

import kda_inputs
import oracle
from tests import _pins

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_bwd.json")
ARGS = ("q", "k", "g", "beta", "dAqk", "dAkk")
NAMES = ("dq", "dk", "db", "dg")


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.abs(a - b).max() / np.abs(b).max())


def test_recipe_regenerates_the_stored_inputs(golden):
    r = golden["recipe"]
    inp = kda_inputs.make_inputs(r["B"], r["T"], r["H"], gate_lo=r["gate_lo"], seed=r["seed"],
                                 k_dim=r["k_dim"], bt=r["bt"])
    for n in ARGS:
        assert np.array_equal(inp[n].double().numpy(), np.asarray(golden["inputs"][n])), n


def test_oracle_reproduces_the_stored_outputs(golden):
    inp = {n: np.asarray(v, dtype=np.float64) for n, v in golden["inputs"].items()}
    out = oracle.intra_bwd(*(inp[n] for n in ARGS), bt=golden["recipe"]["bt"])
    for n, a in zip(NAMES, out):
        assert _rel(a, golden["outputs"][n]) <= 1e-13, n


def test_independent_autograd_agrees_with_the_stored_outputs(golden):
    inp = {n: np.asarray(v, dtype=np.float64) for n, v in golden["inputs"].items()}
    out = _pins.autograd_backward(inp, golden["recipe"]["bt"])
    for n, a in zip(NAMES, out):
        # autograd's dg is with respect to g in log2 units too (the separable forward uses 2^g)
        assert _rel(a, golden["outputs"][n]) <= 1e-10, n
