"""Pins for the TopKTopPSampleV2 oracle (oracle/v2.py), checked against
things other than the oracle itself:

* golden rows worked by hand from the page aclnnTopKTopPSampleV2
  (tests/golden/v2_rows.json), one rule per row, including the two top-p
  forms at exact equality and the ks_max rounding;
* closed forms built without the oracle's sort: top-k alone keeps the first
  k of a lexicographic (-value, index) order; the kept positions are a
  prefix of that order, found by brute force over prefixes in exact
  rational arithmetic for probability inputs;
* probability theory: with q drawn i.i.d. from Exp(1), the QSample index is
  distributed as the probabilities of the kept positions;
* invariants: outputs are the input bits or defLogit, at least one
  position is kept, the kept set shrinks as min-p grows.

The last test plants plausible mistakes into a private copy of the oracle
and checks that at least one pin catches each of them."""
import importlib.util
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle.v2 as OV
from rawutil import NEG_INF, bits, to_raw

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "v2_rows.json")) as f:
        return json.load(f)


def _f32(vals):
    return np.array([{"-inf": -np.inf}.get(v, v) if isinstance(v, str) else v for v in vals], dtype=np.float32)


def pin_golden_rows(ov):
    for r in _golden()["rows"]:
        dt = r["dtype"]
        x = to_raw(r["x"], dt)
        q = None if r["q"] is None else np.array(r["q"], dtype=np.float32)
        sel, tok, idx, sm, _ = ov.v2_row(x, dt, r["k"], r["p"], r["min_p"], q, r.get("eps", 1e-10), r["ks_max"],
                                         r["logits"])
        assert np.array_equal(bits(sel, dt), bits(to_raw(r["select"], dt), dt)), (r["name"], sel)
        assert tok == r["token"], (r["name"], tok)
        assert np.array_equal(idx, np.array(r["logits_idx"])), (r["name"], idx)
        assert np.array_equal(sm.view(np.uint32), _f32(r["sort_masked"]).view(np.uint32)), (r["name"], sm)


def pin_ks_max(ov):
    for c in _golden()["ks_max"]["cases"]:
        assert ov.topk_runs(c["k"], c["V"], c["ks_max"]) == c["runs"], c


def _lex_order(vals):
    """Descending by value, equal values by increasing index, with -0 == +0:
    a plain sort of (-value, index) pairs."""
    return [i for _, i in sorted(((-float(v) + 0.0, i) for i, v in enumerate(vals)))]


def pin_topk_closed_form(ov, seed=3):
    rng = np.random.default_rng(seed)
    for dt in ("f32", "f16", "bf16"):
        for _ in range(25):
            V = int(rng.integers(2, 200))
            x = to_raw(np.round(rng.standard_normal(V) * 2, 0), dt)      # many ties
            xv = ov.decode(x, dt)
            k = int(rng.integers(1, min(V, 64) + 1))
            sel, tok, idx, _, _ = ov.v2_row(x, dt, k, None, None, None, 1e-10, 64, True)
            first = _lex_order(xv)[:k]
            want = np.full(V, NEG_INF[dt], dtype=bits(x, dt).dtype)
            want[first] = bits(x, dt)[first]
            assert np.array_equal(bits(sel, dt), want)
            assert tok == first[0]
            assert list(idx[:k]) == first and (idx[k:] == -1).all()


def _dyadic_row(rng, V):
    """Probabilities that are multiples of 1/64 summing to 1 (exact in fp32)."""
    cuts = np.sort(rng.choice(np.arange(1, 64), size=V - 1, replace=True))
    w = np.diff(np.concatenate([[0], cuts, [64]]))
    return w.astype(np.float32) / np.float32(64)


def pin_topp_prefix_brute_force(ov, seed=5, trials=200):
    """Probability inputs (no softmax), exact rationals: after a top-k stage
    the kept prefix is the longest one whose every position has mass before
    it <= p; without top-k, the longest whose every position has its own and
    all later mass > 1 - p.  Brute force over every prefix length."""
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        V = int(rng.integers(1, 9))
        x = _dyadic_row(rng, V)
        p = float(np.float32(rng.choice([0.0, 0.25, 0.5, 0.75, 0.999, rng.random()])))
        k = int(rng.choice([0, V])) if V > 1 else 0
        sel, _, _, _, info = ov.v2_row(x, "f32", k, p, None, None, 1e-10, 8, False)
        order = _lex_order(x)
        fr = [Fraction(float(x[i])) for i in order]
        p_exact = Fraction(p)
        thr = Fraction(float(np.float32(np.float32(1.0) - np.float32(p))))
        best = 1
        for L in range(1, V + 1):
            if 1 <= k <= V:
                ok = all(sum(fr[:j]) <= p_exact for j in range(L))
            else:
                ok = all(sum(fr[j:]) > thr for j in range(L))
            if ok:
                best = L
        assert info.n_kept == best, (x, k, p, info.n_kept, best)
        want = np.zeros(V, dtype=np.float32)           # defLogit is 0 for probability input
        want[order[:best]] = x[order[:best]]
        assert np.array_equal(sel.view(np.uint32), want.view(np.uint32)), (x, k, p)


def pin_qsample_distribution(ov, seed=7, draws=12000):
    """q i.i.d. Exp(1): the sampled index follows the kept probabilities."""
    rng = np.random.default_rng(seed)
    x = to_raw([2.0, 1.0, 0.5, 0.0, -1.0, 3.0], "f32")
    counts = np.zeros(6)
    sel0, _, _, _, info = ov.v2_row(x, "f32", 4, None, None, None, 0.0, 8, True)
    for _ in range(draws):
        q = rng.exponential(1.0, size=6).astype(np.float32)
        _, tok, _, _, _ = ov.v2_row(x, "f32", 4, None, None, q, 0.0, 8, True)
        counts[tok] += 1
    xv = ov.decode(x, "f32")
    top4 = _lex_order(xv)[:4]
    e = np.exp(xv[top4] - xv[top4].max())
    want = np.zeros(6)
    want[top4] = e / e.sum()
    sd = np.sqrt(draws * want * (1 - want)) + 1e-9
    assert np.all(np.abs(counts - draws * want) <= 5 * sd + 1), (counts, draws * want)


def pin_invariants(ov, seed=11):
    rng = np.random.default_rng(seed)
    for dt in ("f32", "bf16"):
        for _ in range(30):
            V = int(rng.integers(1, 300))
            x = to_raw(np.round(rng.standard_normal(V) * 3, 1), dt)
            b = bits(x, dt)
            k = int(rng.integers(-1, V + 2))
            p = float(rng.random())
            prev = None
            for mp in (0.0, 0.01, 0.1, 0.5, 1.0):
                sel, tok, idx, sm, info = ov.v2_row(x, dt, k, p, mp, None, 1e-10, 1024, True)
                sb = bits(sel, dt)
                kept = sb != NEG_INF[dt]
                assert kept.sum() >= 1
                assert np.all((sb == b) | (sb == NEG_INF[dt]))
                assert kept[tok]
                if prev is not None:
                    assert np.all(prev | ~kept), "the kept set shrinks as min-p grows"
                prev = kept


PINS = [pin_golden_rows, pin_ks_max, pin_topk_closed_form, pin_topp_prefix_brute_force, pin_qsample_distribution,
        pin_invariants]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_v2_oracle_pin(pin):
    pin(OV)


# ------------------------------------------------------------- planted mistakes
def _fresh():
    spec = importlib.util.spec_from_file_location("oracle.v2_mutant", OV.__file__,
                                                  submodule_search_locations=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    spec.loader.exec_module(mod)
    return mod


def _mut_ties_high_index_first(m):
    m.stable_descending_order = lambda vals: np.lexsort((-np.arange(len(vals)), -vals))


def _mut_no_ks_alignment(m):
    m.ks_max_aligned = lambda ks: int(ks)


def _mut_topk_keeps_all_ties(m):
    orig = m.v2_row

    def f(x_raw, dtype, k=None, *a, **kw):
        if k is not None and 1 <= int(k) < x_raw.shape[0]:
            v = m.decode(x_raw, dtype)
            kth = np.sort(v)[::-1][int(k) - 1]
            k = int((v >= kth).sum())
        return orig(x_raw, dtype, k, *a, **kw)
    m.v2_row = f


def _mut_topp_strict(m):
    src = open(OV.__file__).read().replace("keep = before <= p32", "keep = before < p32")
    exec(compile(src, OV.__file__, "exec"), m.__dict__)


def _mut_softmax_over_all(m):
    src = open(OV.__file__).read().replace(
        "e = np.exp(s[:n] - s[0])\n        prob32 = (e / e.sum()).astype(np.float32)",
        "e = np.exp(s - s[0])\n        prob32 = (e / e.sum()).astype(np.float32)[:n]")
    exec(compile(src, OV.__file__, "exec"), m.__dict__)


def _mut_minp_from_smallest(m):
    src = open(OV.__file__).read().replace("thd = pr[0] * mp", "thd = pr[n_topp - 1] * mp")
    exec(compile(src, OV.__file__, "exec"), m.__dict__)


def _mut_q_by_original_index(m):
    src = open(OV.__file__).read().replace(
        "qv = np.asarray(q, dtype=np.float32).astype(np.float64)[:n_kept]",
        "qv = np.asarray(q, dtype=np.float32).astype(np.float64)[order][:n_kept]")
    exec(compile(src, OV.__file__, "exec"), m.__dict__)


MUTANTS = [_mut_ties_high_index_first, _mut_no_ks_alignment, _mut_topk_keeps_all_ties, _mut_topp_strict,
           _mut_softmax_over_all, _mut_minp_from_smallest, _mut_q_by_original_index]


@pytest.mark.parametrize("mutate", MUTANTS, ids=[m.__name__ for m in MUTANTS])
def test_v2_pins_catch_planted_mistake(mutate):
    m = _fresh()
    mutate(m)
    caught = []
    for pin in PINS:
        try:
            if pin is pin_qsample_distribution:
                pin(m, draws=3000)
            elif pin is pin_topp_prefix_brute_force:
                pin(m, trials=80)
            else:
                pin(m)
        except (AssertionError, IndexError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {mutate.__name__}"
