"""Pins for the oracle's stable ascending sort (the step before
ApplyTopKTopPWithSorted, section 6.1 of the CANN ops-nn
ApplyTopKTopPWithSorted guide), checked against things other than the
library routine it calls: rows sorted by hand (tests/golden/sort_rows.json)
and the definition itself -- a permutation under which (value, index) rises
strictly, with -0 equal to +0 -- checked pair by pair in plain Python."""
import json
import os

import numpy as np
import pytest

import oracle as O
from rawutil import to_raw

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _sorted_indices(orc, raw, dtype):
    return orc.stable_ascending_sort(orc.decode(raw, dtype))[1]


def pin_sort_hand_rows(orc):
    with open(os.path.join(GOLDEN, "sort_rows.json")) as f:
        rows = json.load(f)["rows"]
    for row in rows:
        raw = to_raw(row["x"], row["dtype"])
        assert _sorted_indices(orc, raw, row["dtype"]).tolist() == row["indices"], row["name"]


def pin_sort_definition(orc):
    rng = np.random.default_rng(17)
    for trial in range(60):
        dt = ("f32", "f16", "bf16")[trial % 3]
        V = int(rng.integers(1, 300))
        v = np.round(rng.standard_normal(V), 1)
        v[rng.random(V) < 0.1] = -0.0
        v[rng.random(V) < 0.05] = -np.inf
        raw = to_raw(v, dt)
        vals = [float(t) for t in orc.decode(raw, dt)]
        idx = [int(i) for i in _sorted_indices(orc, raw, dt)]
        assert sorted(idx) == list(range(V))
        for j in range(V - 1):
            a, b = vals[idx[j]], vals[idx[j + 1]]
            assert a < b or (a == b and idx[j] < idx[j + 1]), (dt, j)


PINS = [pin_sort_hand_rows, pin_sort_definition]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_sort_oracle_pin(pin):
    pin(O)


def test_sort_pins_catch_an_unstable_order():
    import importlib.util
    import oracle.oracle as om
    spec = importlib.util.spec_from_file_location("oracle_sort_mutant", om.__file__)
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)

    def reversed_ties(x):
        idx = np.lexsort((-np.arange(len(x)), x))
        return x[idx], idx
    m.stable_ascending_sort = reversed_ties
    caught = 0
    for pin in PINS:
        try:
            pin(m)
        except AssertionError:
            caught += 1
    assert caught == len(PINS)
