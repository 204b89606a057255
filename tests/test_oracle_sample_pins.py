"""Pins for the oracle's post-filter stage (min-p and the sample), checked
against things other than the oracle itself.

* golden rows worked by hand (tests/golden/sample_rows.json) from the min-p
  step and the None / QSample modes of the aclnnTopKTopPSampleV2 page;
* a closed form: for 0 < minP < 1, min-p keeps exactly the survivors with
  x >= max + ln(minP) (the normaliser cancels in probs < max_prob * minP);
* probability theory: with q drawn i.i.d. from Exp(1), the index of the
  largest probs / q is distributed as probs (the exponential race), so the
  token frequencies over many draws must match the softmax;
* invariants: outputs are the input bits or -inf, the kept set is a top set
  of the survivors that always holds the largest element, it shrinks as minP
  grows, and the token is a kept element.

The last test plants plausible mistakes into a private copy of the oracle and
checks that at least one pin catches each of them.
"""
import importlib.util
import json
import math
import os

import numpy as np
import pytest

import oracle as O
from rawutil import NEG_INF, bits, to_raw

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def pin_sample_hand_rows(orc):
    for row in _load("sample_rows.json")["rows"]:
        dt = row["dtype"]
        x = to_raw(row["x"], dt)
        q = None if row["q"] is None else np.asarray(row["q"], dtype=np.float32)
        out, token, _ = orc.sample_row(x, dt, row["min_p"], q)
        assert np.array_equal(bits(out, dt), bits(to_raw(row["expected"], dt), dt)), row["name"]
        assert token == row["token"], (row["name"], token)


def pin_sample_minp_closed_form(orc):
    rng = np.random.default_rng(11)
    checked = 0
    for _ in range(60):
        V = 300
        x = (2.0 * rng.standard_normal(V)).astype(np.float32)
        x[rng.random(V) < 0.3] = -np.inf          # earlier filter stages
        mp = float(np.float32(rng.uniform(0.001, 0.9)))
        finite = x[np.isfinite(x)].astype(np.float64)
        bound = finite.max() + math.log(mp)
        if np.min(np.abs(finite - bound)) < 1e-9:
            continue                               # a value on the boundary decides nothing here
        out, _, _ = orc.sample_row(x, "f32", mp, None)
        want = np.where(np.isfinite(x) & (x.astype(np.float64) >= bound), x, -np.inf).astype(np.float32)
        assert np.array_equal(out.view(np.uint32), want.view(np.uint32))
        checked += 1
    assert checked > 40


def pin_sample_exponential_race(orc):
    # P(argmax_i probs_i / q_i = j) = probs_j when q_i ~ Exp(1) i.i.d.
    x = np.array([0.0, 0.5, 1.0, -1.0, 0.2, -np.inf], dtype=np.float32)
    fin = x[:5].astype(np.float64)
    probs = np.exp(fin - fin.max())
    probs /= probs.sum()
    rng = np.random.default_rng(5)
    n = 12000
    counts = np.zeros(6)
    qs = rng.exponential(1.0, size=(n, 6)).astype(np.float32)
    for i in range(n):
        _, t, _ = orc.sample_row(x, "f32", None, qs[i], 1e-10)
        counts[t] += 1
    assert counts[5] == 0
    freq = counts[:5] / n
    sigma = np.sqrt(probs * (1 - probs) / n)
    assert np.all(np.abs(freq - probs) <= 5 * sigma), (freq, probs)


def pin_sample_invariants(orc):
    rng = np.random.default_rng(23)
    for trial in range(80):
        dt = ("f32", "f16", "bf16")[trial % 3]
        V = int(rng.integers(1, 60))
        vals = np.round(2.0 * rng.standard_normal(V), 1)   # ties on purpose
        vals[rng.random(V) < 0.3] = -np.inf
        if not np.isfinite(vals).any():
            vals[int(rng.integers(V))] = 0.5
        x = to_raw(vals, dt)
        xv = O.decode(x, dt)
        q = rng.exponential(1.0, V).astype(np.float32) if trial % 2 else None
        prev = None
        for mp in (0.0, 0.05, 0.3, 0.7, 1.0):
            out, token, _ = orc.sample_row(x, dt, mp, q)
            ob = bits(out, dt)
            keep = ob != NEG_INF[dt]
            assert np.all(ob[keep] == bits(x, dt)[keep])
            assert not np.any(keep & ~np.isfinite(xv))
            top = xv[np.isfinite(xv)].max()
            last = int(np.flatnonzero(xv == top)[-1])
            assert keep[last]
            if keep.any():
                lo = xv[keep].min()
                assert np.all(keep[np.isfinite(xv) & (xv > lo)])      # a top set of the survivors
            assert keep[token]
            if prev is not None:
                assert not np.any(keep & ~prev)                      # shrinks as minP grows
            prev = keep
        assert int(np.sum(prev)) == 1                                # minP = 1 keeps one element


PINS = [pin_sample_hand_rows, pin_sample_minp_closed_form, pin_sample_exponential_race, pin_sample_invariants]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_sample_oracle_pin(pin):
    pin(O)


# ------------------------------------------------------------- planted mistakes
def _fresh_oracle_copy():
    import oracle.oracle as om
    spec = importlib.util.spec_from_file_location("oracle_sample_mutant", om.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _mut_multiply_by_q(m):
    def f(probs, keep, last, q, eps):
        if q is None:
            return last, None
        r = np.where(keep, probs * (np.asarray(q, np.float64) + eps), -np.inf)
        return int(np.flatnonzero(r == r.max())[-1]), r
    m.sample_token = f


def _mut_first_of_ties(m):
    orig = m.survivor_probs

    def f(vals):
        alive, last, e, probs = orig(vals)
        first = int(np.flatnonzero(alive & (vals == vals[alive].max()))[0])
        return alive, first, e, probs
    m.survivor_probs = f


def _mut_minp_from_smallest(m):
    def f(alive, probs, last, mp):
        if mp is None or not (mp > 0.0):
            return alive.copy()
        if mp >= 1.0:
            keep = np.zeros(alive.shape[0], bool)
            keep[last] = True
            return keep
        return alive & ~(probs < probs[alive].min() * mp)
    m.min_p_keep = f


def _mut_minp_one_keeps_all_max(m):
    def f(alive, probs, last, mp):
        if mp is None or not (mp > 0.0):
            return alive.copy()
        return alive & ~(probs < probs[last] * mp)
    m.min_p_keep = f


def _mut_sample_ignores_minp(m):
    orig = m.sample_token

    def f(probs, keep, last, q, eps):
        return orig(probs, probs > 0, last, q, eps)
    m.sample_token = f


def _mut_softmax_over_all(m):
    def f(vals):
        alive = vals != -np.inf
        mx = vals[alive].max()
        last = int(np.flatnonzero(alive & (vals == mx))[-1])
        e = np.where(alive, np.exp(np.where(alive, vals - mx, 0.0)), 1.0)   # masked elements keep weight
        return alive | True, last, e, e / e.sum()
    m.survivor_probs = f


MUTANTS = [_mut_multiply_by_q, _mut_first_of_ties, _mut_minp_from_smallest, _mut_minp_one_keeps_all_max,
           _mut_sample_ignores_minp, _mut_softmax_over_all]


@pytest.mark.parametrize("mutate", MUTANTS, ids=[m.__name__ for m in MUTANTS])
def test_sample_pins_catch_planted_mistake(mutate):
    m = _fresh_oracle_copy()
    mutate(m)
    caught = []
    for pin in PINS:
        try:
            pin(m)
        except (AssertionError, IndexError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {mutate.__name__}"
