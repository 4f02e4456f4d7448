"""Planted mistakes in the oracle must be caught by the pins.

Each mutant is the oracle source with one plausible error edited in (a dropped
term, a wrong sign, a swapped index, a wrong mask, a missing factor).  The
mutant is compiled on the CPU into a temporary library and run through the pin
checks; every mutant has to fail at least one of them.  This shows the pins
constrain every part of the oracle, not just that the oracle agrees with itself.
"""

import os

import pytest

import oracle
from tests import _pins

MUTANTS = {
    "drop_dk_column_term": ("dk[S * K + d] += aqk * qr * E;", ""),
    "dk_column_term_on_wrong_row": ("dk[S * K + d] += aqk * qr * E;",
                                    "dk[R * K + d] += aqk * qr * E;"),
    "dg_source_sign": ("dg[S * K + d] -= LN2 * wq;", "dg[S * K + d] += LN2 * wq;"),
    "dg_missing_ln2": ("dg[R * K + d] += LN2 * wk;", "dg[R * K + d] += wk;"),
    "dkk_includes_diagonal": ("const double akk = (s < r) ? dAkk[R * BT + s] : 0.0;",
                              "const double akk = dAkk[R * BT + s];",
                              "                    if (s < r) {",
                              "                    if (s <= r) {"),
    "db_times_beta": ("db[R] += akk * kr * ks * E;", "db[R] += akk * beta[R] * kr * ks * E;"),
    "gate_sign_swapped_bwd": (
        "const double E = exp2(g[R * K + d] - g[S * K + d]);\n\n",
        "const double E = exp2(g[S * K + d] - g[R * K + d]);\n\n"),
    "natural_exp_bwd": (
        "const double E = exp2(g[R * K + d] - g[S * K + d]);\n\n",
        "const double E = exp(g[R * K + d] - g[S * K + d]);\n\n"),
    "dk_row_term_uses_source_beta": ("dk[R * K + d] += akk * beta[R] * ks * E;",
                                     "dk[R * K + d] += akk * beta[S] * ks * E;"),
    "fwd_akk_missing_beta": ("Akk[R * BT + s] = (s < r) ? beta[R] * skk : 0.0;",
                             "Akk[R * BT + s] = (s < r) ? skk : 0.0;"),
    "fwd_aqk_strict_mask": ("Aqk[R * BT + s] = (s <= r) ? sqk : 0.0;",
                            "Aqk[R * BT + s] = (s < r) ? sqk : 0.0;"),
    "dq_uses_query_row": ("dq[R * K + d] += aqk * ks * E;", "dq[R * K + d] += aqk * kr * E;"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, source, name):
    edits = MUTANTS[name]
    mutated = source
    for old, new in zip(edits[0::2], edits[1::2]):
        assert mutated.count(old) == 1, f"mutation anchor for {name} not unique/found"
        mutated = mutated.replace(old, new)
    src = tmp_path / "mutant.c"
    src.write_text(mutated)
    lib = oracle.load(oracle.build(str(src), str(tmp_path / "libmutant.so")))
    inp = _pins.tiny_inputs(1, 16, 2, 4, 8, gate_lo=-1.0, seed=3)
    fails = _pins.run_all(lib, inp, 8, with_fd=False)
    assert fails, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(tmp_path, source):
    src = tmp_path / "copy.c"
    src.write_text(source)
    lib = oracle.load(oracle.build(str(src), str(tmp_path / "libcopy.so")))
    inp = _pins.tiny_inputs(1, 16, 2, 4, 8, gate_lo=-1.0, seed=3)
    assert not _pins.run_all(lib, inp, 8, with_fd=False)
    assert os.path.exists(tmp_path / "libcopy.so")
