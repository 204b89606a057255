"""The seeded input recipes (top_logit_filter_gb300.workloads): shapes,
dtypes, value distributions and the k / p / min_p / q recipes each workload
promises, on reduced sizes.  Host logic only."""
import numpy as np
import pytest

import oracle as O
from top_logit_filter_gb300 import workloads as W


def _vals(w):
    return O.decode(w["x"], w["dtype"])


@pytest.mark.parametrize("wl", [1, 2, 3, 4, 5])
def test_shapes_dtypes_and_seeding(wl):
    spec = W.WORKLOADS[wl]
    B = min(spec["B"], 64)
    V = min(spec["V"], 4096)
    a = W.make(wl, B=B, V=V)
    b = W.make(wl, B=B, V=V)
    assert a["x"].shape == (B, V) and a["dtype"] == spec["dtype"]
    assert a["x"].dtype == {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[spec["dtype"]]
    assert np.array_equal(a["x"], b["x"])                       # same seed, same inputs
    assert not np.array_equal(a["x"], W.make(wl, B=B, V=V, seed=1)["x"])
    assert (a["k"] is not None) == spec["topk"] and (a["p"] is not None) == spec["topp"]
    assert np.isfinite(_vals(a)).all()


def test_value_distributions():
    x3 = _vals(W.make(3, B=16, V=20000))
    assert abs(x3.mean()) < 0.05 and abs(x3.std() - 2.0) < 0.05
    x1 = _vals(W.make(1))
    assert abs(x1.std() - 3.0) < 0.1
    x2 = _vals(W.make(2, B=16, V=32000))
    assert abs(x2.std() - 2.5) < 0.05
    # 20 tokens per row boosted by +8: the row maxima sit near 8 + 2.5 * 1.9,
    # above the about 2.5 * 4.1 that 32000 unboosted draws reach
    assert np.median(x2.max(axis=1)) > 11.5
    x4 = W.make(4, B=32, V=20000)
    sd = _vals(x4).std(axis=1)                   # N(0,1)/T with T ~ U[0.3, 1.5]
    assert sd.min() > 1 / 1.5 - 0.05 and sd.max() < 1 / 0.3 + 0.1


def test_k_and_p_recipes():
    w1 = W.make(1)
    assert w1["k"].tolist() == [1, 10, 0, 2000]
    assert np.allclose(O.decode(w1["p"], "f32"), [0.9, 0.5, 1.0, 0.0])
    w3 = W.make(3)
    k, p = w3["k"], O.decode(w3["p"], "bf16")
    assert k.dtype == np.int32 and (k == 0).sum() == round(0.10 * 256)
    assert k[k > 0].min() >= 1 and k.max() <= 1024
    assert (p == 1.0).sum() >= round(0.05 * 256) and p.min() >= 0.5 and p.max() <= 1.0
    w4 = W.make(4, B=64, V=256)
    assert w4["p"] is None and w4["k"].min() >= 1 and w4["k"].max() <= 64
    w5 = W.make(5, B=64, V=256)
    p5 = O.decode(w5["p"], "bf16")
    assert p5.min() >= 0.099 and p5.max() <= 0.951


def test_presorted_input_is_the_stable_ascending_order():
    w = W.make(5, B=6, V=3001)
    sv, si, x = w["sorted_value"], w["sorted_indices"], w["x"]
    assert si.dtype == np.int32
    for b in range(6):
        assert sorted(si[b].tolist()) == list(range(3001))            # a permutation
        assert np.array_equal(sv[b], x[b][si[b]])
        v = O.decode(sv[b], "bf16")
        assert np.all(np.diff(v) >= 0)                                  # ascending
        ties = np.diff(v) == 0
        assert np.all(np.diff(si[b])[ties] > 0)                         # equal values keep index order


def test_filtered_rows_recipe():
    d = W.make_filtered(40, 5000, "bf16", seed=3, empty_rows=2)
    v = O.decode(d["x"], "bf16")
    alive = np.isfinite(v)
    assert not alive[-2:].any() and alive[:-2].any(axis=1).all()
    # every row is a top set: all values at or above its smallest survivor are kept
    for b in range(38):
        lo = v[b][alive[b]].min()
        assert alive[b][v[b] >= lo].all()
    assert d["min_p"].dtype == np.float32 and (d["min_p"] == 0).sum() == 4 and (d["min_p"] == 1).sum() == 2
    assert d["q"].dtype == np.float32 and d["q"].shape == (40, 5000) and (d["q"] > 0).all()
    assert abs(d["q"].mean() - 1.0) < 0.02                              # Exp(1)
