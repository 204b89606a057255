"""Pins for the CPU oracle, checked against things other than the oracle itself.

* golden rows: the example inputs the page prints (section 7 of the CANN
  ops-nn ApplyTopKTopPWithSorted guide) and rows worked by hand from its
  eight-step formula (section 2), stored under tests/golden/ with derivations;
* brute force on tiny rows: the kept set must be the smallest top set, in
  (value, index) order, whose probability mass reaches 1 - thr -- checked by
  enumerating every subset with high-precision exp (no sort, no cumsum);
* closed forms: top-k alone equals a library selection (np.partition);
* invariants: outputs are the input bits or -inf, at least one token is kept,
  the kept set is upward closed, and it grows with p and with k.

The last test plants plausible mistakes into a private copy of the oracle and
checks that at least one pin catches each of them.
"""
import importlib.util
import itertools
import json
import os

import numpy as np
import pytest

import oracle as O
from rawutil import NEG_INF, bits, to_raw

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ pin bodies
# Each pin takes an oracle module so the mutation test can rerun it on a
# mutated copy; each returns None or raises AssertionError.

def _expected_bits(expected, dtype):
    return bits(to_raw(expected, dtype), dtype)


def pin_page_example(orc):
    g = _load("page_example.json")
    dt = g["dtype"]
    for row in g["rows"]:
        x = to_raw(row["x"], dt)
        p = to_raw([row["p"]], dt)[0]
        out, _ = orc.apply_row(x, dt, p, row["k"])
        assert np.array_equal(bits(out, dt), _expected_bits(row["expected"], dt)), row


def pin_hand_rows(orc):
    g = _load("hand_rows.json")
    for row in g["rows"]:
        dt = row["dtype"]
        if "x_fill" in row:
            val, n = row["x_fill"]
            x = to_raw([val] * int(n), dt)
            exp = np.full(int(n), NEG_INF[dt], dtype=bits(x, dt).dtype)
            kf = row["expected_kept_from"]
            exp[kf:] = bits(x, dt)[kf:]
        else:
            x = to_raw(row["x"], dt)
            exp = _expected_bits(row["expected"], dt)
        p = None if row["p"] is None else to_raw([row["p"]], dt)[0]
        out, _ = orc.apply_row(x, dt, p, row["k"])
        assert np.array_equal(bits(out, dt), exp), row["name"]


def pin_thresholds(orc):
    g = _load("hand_rows.json")["thresholds"]
    for c in g["cases"]:
        p = to_raw([c["p"]], c["dtype"])[0]
        assert float(orc.top_p_threshold(p, c["dtype"])) == c["thr"], c


def _brute_kept(x, k, p_eff):
    """Kept set by subset enumeration (mpmath exp, 50 digits): returns
    (lo, hi, topk_set, order) where lo..hi bounds |kept| allowing exact ties."""
    import mpmath
    mpmath.mp.dps = 50
    V = len(x)
    if k is not None and 1 <= k <= V - 1:
        surv = [v for v in range(V) if sum(1 for u in range(V) if x[u] > x[v]) < k]
    else:
        surv = list(range(V))
    w = {v: mpmath.e ** mpmath.mpf(float(x[v])) for v in surv}
    tot = sum(w.values())
    tol = mpmath.mpf("1e-6")

    def nstar(target):
        best = len(surv)
        for r in range(0, len(surv) + 1):
            if any(sum((w[a] for a in A), mpmath.mpf(0)) / tot >= target
                   for A in itertools.combinations(surv, r)):
                best = r
                break
        return max(best, 1)

    if p_eff is None:
        return len(surv), len(surv), set(surv)
    return nstar(mpmath.mpf(float(p_eff)) + tol), nstar(mpmath.mpf(float(p_eff)) - tol), set(surv)


def pin_brute_force(orc, trials=150, seed=7):
    rng = np.random.default_rng(seed)
    for t in range(trials):
        V = int(rng.integers(1, 9))
        # small integer grid -> many exact ties
        x = (rng.integers(-3, 4, size=V) * 0.75).astype(np.float32)
        k = int(rng.integers(-1, V + 2)) if rng.random() < 0.8 else None
        use_p = rng.random() < 0.8 or k is None
        p = np.float32(rng.choice([0.0, 1.0, rng.random()])) if use_p else None
        out, info = orc.apply_row(x, "f32", p, k)
        kept = bits(out, "f32") != NEG_INF["f32"]
        p_eff = None if p is None else 1.0 - float(info.thr)
        lo, hi, topk_set = _brute_kept(x, k, p_eff)
        kept_set = set(np.nonzero(kept)[0].tolist())
        assert kept_set <= topk_set, (x, k, p)
        # upward closed in (value, index) order
        for v in kept_set:
            for u in range(V):
                if (x[u], u) > (x[v], v):
                    assert u in kept_set, (x, k, p)
        assert hi <= len(kept_set) <= lo, (x, k, p, lo, hi, kept_set)
        # kept elements keep their bits
        assert np.array_equal(bits(out, "f32")[kept], bits(x, "f32")[kept])


def pin_topk_partition(orc, seed=3):
    rng = np.random.default_rng(seed)
    for dt in ("f32", "f16", "bf16"):
        for _ in range(20):
            V = int(rng.integers(2, 300))
            xf = np.round(rng.standard_normal(V) * 4, 1).astype(np.float32)
            x = to_raw(xf, dt)
            xv = orc.decode(x, dt)
            k = int(rng.integers(1, V))
            kth = np.partition(xv, V - k)[V - k]
            exp = np.where(xv >= kth, bits(x, dt), NEG_INF[dt]).astype(bits(x, dt).dtype)
            out, _ = orc.apply_row(x, dt, None, k)
            assert np.array_equal(bits(out, dt), exp)


def pin_invariants(orc, seed=11):
    rng = np.random.default_rng(seed)
    for dt in ("f32", "f16", "bf16"):
        for _ in range(15):
            V = int(rng.integers(1, 400))
            x = to_raw(np.round(rng.standard_normal(V) * 3, 2), dt)
            b = bits(x, dt)
            ps = sorted(rng.random(3).tolist() + [0.0, 1.0])
            k = int(rng.integers(0, V + 1))
            prev = None
            for pv in ps:
                p = to_raw([pv], dt)[0]
                out, _ = orc.apply_row(x, dt, p, k)
                ob = bits(out, dt)
                kept = ob != NEG_INF[dt]
                assert kept.sum() >= 1
                assert np.all((ob == b) | (ob == NEG_INF[dt]))
                if prev is not None:
                    assert np.all(kept | ~prev), "kept set must grow with p"
                prev = kept
            # p = 1 with top-k off is the identity (no exp underflow at this range)
            out, _ = orc.apply_row(x, dt, to_raw([1.0], dt)[0], 0)
            assert np.array_equal(bits(out, dt), b)
            # k = 1 alone keeps exactly the maximum value(s)
            if V >= 2:
                xv = orc.decode(x, dt)
                out, _ = orc.apply_row(x, dt, None, 1)
                kept = bits(out, dt) != NEG_INF[dt]
                assert np.array_equal(kept, xv == xv.max())
            # kept set grows with k
            prev = None
            for kk in range(1, min(V, 12)):
                out, _ = orc.apply_row(x, dt, None, kk)
                kept = bits(out, dt) != NEG_INF[dt]
                if prev is not None:
                    assert np.all(kept | ~prev)
                prev = kept


def pin_sorted_matches_unsorted(orc, seed=5):
    rng = np.random.default_rng(seed)
    for dt in ("f32", "bf16"):
        V = 257
        x = to_raw(np.round(rng.standard_normal(V) * 2, 1), dt)
        xv = orc.decode(x, dt)
        idx = np.argsort(xv, kind="stable")
        sv = x[idx]
        for k, pv in [(5, 0.3), (0, 0.9), (100, None), (1, 1.0)]:
            p = None if pv is None else to_raw([pv], dt)[0]
            a, _ = orc.apply_row(x, dt, p, k)
            s, _ = orc.apply_sorted_row(sv, idx.astype(np.int32), dt, p, k)
            assert np.array_equal(bits(a, dt), bits(s, dt))


def pin_bf16_codec(orc):
    # round-to-nearest-even at the bf16 boundary, and exact decode
    cases = [(1.0 + 2 ** -8, 1.0), (1.0 + 3 * 2 ** -8, 1.015625), (-2.0 - 2 ** -7, -2.0), (0.1, 0.10009765625)]
    for v, want in cases:
        assert float(orc.round_to_dtype_f32(np.array([v], np.float32), "bf16")[0]) == want
    assert orc.decode(np.array([0x3F80, 0xC000, 0x8000], np.uint16), "bf16").tolist() == [1.0, -2.0, -0.0]


def pin_topk_survivors(orc, seed=13):
    """topk_survivors, the helper that tells the parity check a top-k
    decision (never allowed to differ) from a top-p one, pinned three ways:
    hand-worked sorted rows; its definition on every k for tiny rows sorted
    by numpy, not by the oracle (kept iff fewer than k elements are strictly
    larger); and the RowInfo that apply_row / apply_sorted_row hand to the
    tests, against the same definition in the stable order."""
    g = _load("hand_rows.json")["topk_survivors"]
    for c in g["cases"]:
        s = np.asarray(to_raw(c["s"], "f32"), dtype=np.float32).astype(np.float64)
        got = orc.topk_survivors(s, len(s), c["k"])
        assert np.array_equal(got, np.asarray(c["kept"], dtype=bool)), c
    rng = np.random.default_rng(seed)
    for _ in range(200):
        V = int(rng.integers(1, 9))
        x = (rng.integers(-3, 4, size=V) * 0.5).astype(np.float64)
        s = np.sort(x)
        for k in range(-1, V + 2):
            want = np.array([(not (1 <= k <= V - 1)) or int((s > s[j]).sum()) < k for j in range(V)])
            assert np.array_equal(orc.topk_survivors(s, V, k), want), (s, k)
    for dt in ("f32", "bf16"):
        V = 61
        x = to_raw(np.round(rng.standard_normal(V), 0), dt)   # heavy ties
        xv = orc.decode(x, dt)
        idx = np.argsort(xv, kind="stable")
        for k in (1, 2, 5, 30, V - 1, 0, V):
            for info in (orc.apply_row(x, dt, None, k)[1],
                         orc.apply_sorted_row(x[idx], idx.astype(np.int32), dt, to_raw([0.5], dt)[0], k)[1]):
                vals = xv[info.idx]
                want = np.array([(not (1 <= k <= V - 1)) or int((xv > v).sum()) < k for v in vals])
                assert np.array_equal(info.topk_kept, want), (dt, k)


PINS = [pin_page_example, pin_hand_rows, pin_thresholds, pin_brute_force,
        pin_topk_partition, pin_invariants, pin_sorted_matches_unsorted, pin_bf16_codec,
        pin_topk_survivors]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pytest.importorskip("mpmath") if pin is pin_brute_force else None
    pin(O)


# ------------------------------------------------------------- planted mistakes
def _fresh_oracle_copy():
    import oracle.oracle as om
    spec = importlib.util.spec_from_file_location("oracle_mutant", om.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _mut_topk_le(m):
    def f(s, V, k, thr):
        kept = np.ones(V, bool)
        vals = s.copy()
        if m.topk_enabled(k, V):
            msk = s <= s[V - int(k)]
            kept &= ~msk
            vals[msk] = -np.inf
        C = None
        if thr is not None:
            e = np.exp(vals - vals[V - 1]) if np.isfinite(vals[V - 1]) else np.ones(V)
            q = (e / e.sum()).astype(np.float32)
            C = np.cumsum(q.astype(np.float64)).astype(np.float32)
            tm = C <= thr
            tm[V - 1] = False
            kept &= ~tm
        return kept, C
    m.filter_sorted_row = f


def _mut_topp_lt(m):
    def f(s, V, k, thr):
        kept = np.ones(V, bool)
        vals = s.copy()
        if m.topk_enabled(k, V):
            msk = s < s[V - int(k)]
            kept &= ~msk
            vals[msk] = -np.inf
        C = None
        if thr is not None:
            e = np.exp(vals - vals[V - 1])
            q = (e / e.sum()).astype(np.float32)
            C = np.cumsum(q.astype(np.float64)).astype(np.float32)
            tm = C < thr
            tm[V - 1] = False
            kept &= ~tm
        return kept, C
    m.filter_sorted_row = f


def _mut_no_last_guard(m):
    def f(s, V, k, thr):
        kept = np.ones(V, bool)
        vals = s.copy()
        if m.topk_enabled(k, V):
            msk = s < s[V - int(k)]
            kept &= ~msk
            vals[msk] = -np.inf
        C = None
        if thr is not None:
            e = np.exp(vals - vals[V - 1])
            q = (e / e.sum()).astype(np.float32)
            C = np.cumsum(q.astype(np.float64)).astype(np.float32)
            kept &= ~(C <= thr)
        return kept, C
    m.filter_sorted_row = f


def _mut_softmax_ignores_topk(m):
    def f(s, V, k, thr):
        kept = np.ones(V, bool)
        if m.topk_enabled(k, V):
            kept &= ~(s < s[V - int(k)])
        C = None
        if thr is not None:
            e = np.exp(s - s[V - 1])
            q = (e / e.sum()).astype(np.float32)
            C = np.cumsum(q.astype(np.float64)).astype(np.float32)
            tm = C <= thr
            tm[V - 1] = False
            kept &= ~tm
        return kept, C
    m.filter_sorted_row = f


def _mut_kth_off_by_one(m):
    orig = m.filter_sorted_row

    def f(s, V, k, thr):
        if m.topk_enabled(k, V) and int(k) < V - 1:
            return orig(s, V, int(k) + 1, thr)
        return orig(s, V, k, thr)
    m.filter_sorted_row = f


def _mut_ties_reversed(m):
    def srt(x):
        idx = np.lexsort((-np.arange(len(x)), x))
        return x[idx], idx
    m.stable_ascending_sort = srt


def _mut_gather(m):
    def sc(raw_sorted_bits, idx, kept, dtype):
        return np.where(kept, raw_sorted_bits, m.neg_inf_bits(dtype))[idx]
    m.scatter_back = sc


def _mut_thr_unrounded(m):
    def thr(p_raw, dtype):
        p32 = np.float32(m.decode(np.asarray([p_raw]), dtype)[0])
        return np.float32(np.float32(1.0) - p32)
    m.top_p_threshold = thr


def _mut_cumsum_descending(m):
    def f(s, V, k, thr):
        kept = np.ones(V, bool)
        vals = s.copy()
        if m.topk_enabled(k, V):
            msk = s < s[V - int(k)]
            kept &= ~msk
            vals[msk] = -np.inf
        C = None
        if thr is not None:
            e = np.exp(vals - vals[V - 1])
            q = (e / e.sum()).astype(np.float32)
            C = np.cumsum(q[::-1].astype(np.float64))[::-1].astype(np.float32)
            tm = C <= thr
            tm[V - 1] = False
            kept &= ~tm
        return kept, C
    m.filter_sorted_row = f


def _mut_survivors_off_by_one(m):
    def f(s, V, k):
        if not m.topk_enabled(k, V):
            return np.ones(V, dtype=bool)
        return ~(s < s[V - int(k) - 1])
    m.topk_survivors = f


def _mut_survivors_le(m):
    def f(s, V, k):
        if not m.topk_enabled(k, V):
            return np.ones(V, dtype=bool)
        return ~(s <= s[V - int(k)])
    m.topk_survivors = f


MUTANTS = [_mut_topk_le, _mut_topp_lt, _mut_no_last_guard, _mut_softmax_ignores_topk,
           _mut_kth_off_by_one, _mut_ties_reversed, _mut_gather, _mut_thr_unrounded,
           _mut_cumsum_descending, _mut_survivors_off_by_one, _mut_survivors_le]


@pytest.mark.parametrize("mutate", MUTANTS, ids=[m.__name__ for m in MUTANTS])
def test_pins_catch_planted_mistake(mutate):
    pytest.importorskip("mpmath")
    m = _fresh_oracle_copy()
    mutate(m)
    caught = []
    for pin in PINS:
        try:
            if pin is pin_brute_force:
                pin(m, trials=60)
            else:
                pin(m)
        except (AssertionError, IndexError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {mutate.__name__}"
