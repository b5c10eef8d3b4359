"""The oracle against its stored record (tests/golden/oracle_small_cases.json).

The pages print no numeric worked example, so the stored outputs are the
oracle's own, written by tests/golden/make_oracle_golden.py from oracle/
only; the oracle is pinned to the mathematics by test_oracle_pins.py.  This
file holds it to that record: a change to the oracle's arithmetic, or to the
seeded input recipe, fails here until the fixture is regenerated with the
passage that justifies the change.
"""

import json
import os

import numpy as np
import pytest

import oracle
from mamba_selective_scan_gb300.inputs import make_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_small_cases.json")


def _cases():
    with open(GOLDEN, encoding="utf-8") as fh:
        return json.load(fh)["cases"]


def _arr(rec):
    return np.asarray(rec["data"], dtype=np.float64).reshape(rec["shape"])


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_seeded_recipe_reproduces_stored_inputs(case):
    sh = case["shape"]
    inp = make_inputs(sh["batch"], sh["seq_len"], sh["d_inner"], act=case["act"], seed=case["seed"],
                      random_params=case["random_params"])
    for k, rec in case["inputs"].items():
        assert np.array_equal(np.asarray(inp[k], dtype=np.float64), _arr(rec)), k


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_oracle_reproduces_stored_outputs(case):
    inp = {k: _arr(rec) for k, rec in case["inputs"].items()}
    f = oracle.forward(inp)
    g = oracle.backward(inp, chunk=case["chunk"])
    # float64 throughout; the bound leaves room for a compiler that fuses
    # multiply-adds differently on another host
    for part, got in (("forward", f), ("backward", g)):
        for k, rec in case[part].items():
            want = _arr(rec)
            scale = max(1.0, float(np.abs(want).max()))
            np.testing.assert_allclose(got[k], want, rtol=1e-10, atol=1e-12 * scale, err_msg=f"{part} {k}")
