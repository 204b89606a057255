"""GPU parity of the pre-sorted entry point (ApplyTopKTopPWithSorted,
sections 2-4 of the CANN ops-nn ApplyTopKTopPWithSorted guide) through the C
ABI, against the CPU oracle.

Small ragged rows sweep dtypes, modes, tie-heavy rows and signed zeros, with
and without the optional logits, under every cluster size the planner may
pick.  The pre-sorted workload (B=512, V=152064 bf16, peaked logits) then
runs at full size: sampled rows against the oracle element by element, every
row against properties that hold at any size."""
import numpy as np
import pytest

import flipstats
import oracle as O
from parity import compare_row
from rawutil import NEG_INF, bits, raw_to_torch, torch_to_raw
from test_gpu_parity import _kp, _rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DTS = ("f32", "f16", "bf16")
# TOPKP_FORCE_SORTED_PLAN: CTAs per row (cluster size); "" = the planner's choice
CLUSTERS = ["", "1", "2", "4", "8"]


@pytest.fixture(scope="module")
def tk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_logit_filter_gb300 import build
    build.build()
    import top_logit_filter_gb300 as m
    return m


def _presort(x, dtype):
    from top_logit_filter_gb300 import workloads
    return workloads.presort(x, dtype)


def _run_sorted(tk, sv, si, dtype, p, k, logits=None):
    svt = raw_to_torch(sv, dtype, "cuda")
    sit = torch.from_numpy(si).cuda()
    pt = None if p is None else raw_to_torch(p, dtype, "cuda")
    kt = None if k is None else torch.from_numpy(k).cuda()
    lt = None if logits is None else raw_to_torch(logits, dtype, "cuda")
    o = tk.apply_sorted(svt, sit, p=pt, k=kt, logits=lt)
    torch.cuda.synchronize()
    return torch_to_raw(o, dtype)


def _check_rows(out, x, sv, si, dtype, p, k, rows, where):
    flips = 0
    for b in rows:
        _, info = O.apply_sorted_row(sv[b], si[b], dtype, None if p is None else p[b],
                                     None if k is None else int(k[b]))
        flips += compare_row(out[b], x[b], info, dtype, where=f"{where} row {b}")
    return flips


@pytest.mark.parametrize("dtype", DTS)
@pytest.mark.parametrize("V", [1, 2, 7, 64, 1000, 5003])
@pytest.mark.parametrize("mode", ["k", "p", "kp"])
def test_small_sorted_rows(tk, monkeypatch, dtype, V, mode):
    rng = np.random.default_rng(V * 11 + len(mode))
    B = 9
    for kind in ("normal", "ties", "zeros"):
        x = _rows(rng, B, V, dtype, kind)
        sv, si = _presort(x, dtype)
        k, p = _kp(rng, B, V, dtype, mode)
        for clusters in CLUSTERS:
            monkeypatch.setenv("TOPKP_FORCE_SORTED_PLAN", clusters)
            for with_logits in (False, True):
                out = _run_sorted(tk, sv, si, dtype, p, k, x if with_logits else None)
                _check_rows(out, x, sv, si, dtype, p, k, range(B),
                            f"{dtype} V={V} {mode} {kind} clusters={clusters!r} logits={with_logits}")


def test_sorted_without_logits_uses_indices(tk):
    """Without logits the output is a scatter through sorted_indices: a
    non-identity permutation of a row must land where the indices say."""
    rng = np.random.default_rng(5)
    B, V, dtype = 3, 4099, "bf16"
    x = _rows(rng, B, V, dtype, "normal")
    sv, si = _presort(x, dtype)
    k = np.array([5, 0, 4098], dtype=np.int32)
    p = None
    out = _run_sorted(tk, sv, si, dtype, p, k)
    _check_rows(out, x, sv, si, dtype, p, k, range(B), "scatter")
    # every kept element sits at its source column
    ob, xb = bits(out, dtype), bits(x, dtype)
    kept = ob != NEG_INF[dtype]
    assert (ob[kept] == xb[kept]).all()


def _suffix_in_stable_order(out_row, x_row, dtype):
    """The kept set is a non-empty suffix of the stable ascending order."""
    ob, xb = bits(out_row, dtype), bits(x_row, dtype)
    assert ((ob == xb) | (ob == NEG_INF[dtype])).all()
    kept = ob == xb
    order = np.argsort(O.decode(x_row, dtype), kind="stable")
    ks = kept[order]
    assert ks[-1], "the last sorted position is always kept"
    first = int(np.argmax(ks))
    assert ks[first:].all(), "kept set is not a top suffix of the stable order"
    return int(ks.sum())


def test_workload5_full_size(tk):
    """All 512 rows of the pre-sorted workload, with and without logits,
    element by element against the oracle, plus the properties that hold at
    any size (a top suffix of the stable order; nothing below the k-th
    largest)."""
    from top_logit_filter_gb300 import workloads
    w = workloads.make(5)
    dtype = w["dtype"]
    x, sv, si, p, k = w["x"], w["sorted_value"], w["sorted_indices"], w["p"], w["k"]
    infos = [O.apply_sorted_row(sv[b], si[b], dtype, p[b], int(k[b]))[1] for b in range(w["B"])]
    for with_logits in (True, False):
        out = _run_sorted(tk, sv, si, dtype, p, k, x if with_logits else None)
        flips = 0
        for b in range(w["B"]):
            flips += compare_row(out[b], x[b], infos[b], dtype, where=f"wl5 logits={with_logits} row {b}")
            _suffix_in_stable_order(out[b], x[b], dtype)
            # top-k bound: nothing below the k-th largest survives
            kth = O.decode(sv[b][w["V"] - int(k[b])], dtype) if 1 <= int(k[b]) < w["V"] else -np.inf
            kept_vals = O.decode(x[b], dtype)[bits(out[b], dtype) != NEG_INF[dtype]]
            assert (kept_vals >= kth).all(), b
        flipstats.record(f"workload 5 ({w['name']}, logits={'given' if with_logits else 'absent'})", w["B"], flips)


def test_workload5_top_p_only_full_size(tk):
    """The pre-sorted batch with top-k off: the top-p sum and cut run over the
    whole sorted row (152064 elements), split over the rows' CTAs.  32 rows
    element by element against the oracle, with and without logits."""
    from top_logit_filter_gb300 import workloads
    w = workloads.make(5)
    dtype = w["dtype"]
    rows = list(range(0, w["B"], w["B"] // 32))
    x, sv, si, p = w["x"][rows], w["sorted_value"][rows], w["sorted_indices"][rows], w["p"][rows]
    infos = [O.apply_sorted_row(sv[b], si[b], dtype, p[b], None)[1] for b in range(len(rows))]
    for with_logits in (True, False):
        out = _run_sorted(tk, sv, si, dtype, p, None, x if with_logits else None)
        flips = 0
        for b in range(len(rows)):
            flips += compare_row(out[b], x[b], infos[b], dtype, where=f"wl5 top-p only logits={with_logits} row {b}")
            _suffix_in_stable_order(out[b], x[b], dtype)
        flipstats.record(f"workload 5 as top-p only (logits={'given' if with_logits else 'absent'})", len(rows), flips)
