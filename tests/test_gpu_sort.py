"""GPU parity of the stable sort (topkp_sort, the l0op::Sort step before
ApplyTopKTopPWithSorted, section 6.1 of the CANN ops-nn
ApplyTopKTopPWithSorted guide) through the C ABI, against the oracle's
stable ascending sort: values bit for bit and indices exactly."""
import numpy as np
import pytest

import oracle as O
from rawutil import bits, raw_to_torch, to_raw, torch_to_raw

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DTS = ("f32", "f16", "bf16")


@pytest.fixture(scope="module")
def tk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_logit_filter_gb300 import build
    build.build()
    import top_logit_filter_gb300 as m
    return m


def _gpu_sort(tk, x, dtype, ld_pad=0):
    B, V = x.shape
    t = raw_to_torch(x, dtype, "cuda")
    if ld_pad:
        base = torch.zeros((B, V + ld_pad), dtype=t.dtype, device="cuda")
        base[:, ld_pad:] = t
        t = base[:, ld_pad:]
    sv, si = tk.sort(t)
    torch.cuda.synchronize()
    return torch_to_raw(sv, dtype), si.cpu().numpy()


def _check(x, dtype, sv, si, where):
    for b in range(x.shape[0]):
        _, idx = O.stable_ascending_sort(O.decode(x[b], dtype))
        assert np.array_equal(si[b], idx), f"{where} row {b}: indices differ at {np.nonzero(si[b] != idx)[0][:8]}"
        assert np.array_equal(bits(sv[b], dtype), bits(x[b], dtype)[idx]), f"{where} row {b}: values differ"


def _rows(B, V, dtype, seed):
    rng = np.random.default_rng(seed)
    v = np.round(2.0 * rng.standard_normal((B, V)), 1)      # many ties
    v[rng.random((B, V)) < 0.02] = -0.0                       # signed zeros tie with +0
    v[rng.random((B, V)) < 0.01] = -np.inf
    return np.stack([to_raw(r, dtype) for r in v])


@pytest.mark.parametrize("dtype", DTS)
@pytest.mark.parametrize("V", [1, 2, 7, 513, 1000, 5003])
def test_sort_small_rows(tk, dtype, V):
    x = _rows(4, V, dtype, seed=V)
    sv, si = _gpu_sort(tk, x, dtype)
    _check(x, dtype, sv, si, f"{dtype} V={V}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B", [1, 20, 50, 100, 160])
def test_sort_row_split_over_clusters(tk, dtype, B):
    """Batches of 1 to 160 rows: the planner runs a row on a cluster of 8,
    4, 2 or 1 CTAs (each counting its slice of every pass's source); the
    result is the same stable sort."""
    x = _rows(B, 5003, dtype, seed=B)
    sv, si = _gpu_sort(tk, x, dtype)
    _check(x, dtype, sv, si, f"{dtype} B={B}")


@pytest.mark.parametrize("dtype", DTS)
def test_sort_strided_rows(tk, dtype):
    x = _rows(3, 2053, dtype, seed=5)
    sv, si = _gpu_sort(tk, x, dtype, ld_pad=3)
    _check(x, dtype, sv, si, f"{dtype} strided")


def test_sort_decode_rows_and_feed_the_sorted_filter(tk):
    """16 rows of the pre-sorted workload (V=152064 bf16): the sort matches
    the oracle, and topkp_apply_sorted on it matches the oracle's filter."""
    from top_logit_filter_gb300 import workloads
    from parity import compare_row
    w = workloads.make(5, B=16)
    x, p, k = w["x"], w["p"], w["k"]
    sv, si = _gpu_sort(tk, x, "bf16")
    _check(x, "bf16", sv, si, "wl5")
    out = tk.apply_sorted(raw_to_torch(sv, "bf16", "cuda"), torch.from_numpy(si).cuda(),
                          p=raw_to_torch(p, "bf16", "cuda"), k=torch.from_numpy(k).cuda())
    out = torch_to_raw(out, "bf16")
    for b in range(4):
        _, info = O.apply_row(x[b], "bf16", p[b], int(k[b]))
        compare_row(out[b], x[b], info, "bf16", where=f"sort + apply_sorted row {b}")


def test_sort_fp32_long_rows(tk):
    from top_logit_filter_gb300 import workloads
    w = workloads.make(4, B=4)
    sv, si = _gpu_sort(tk, w["x"], "f32")
    _check(w["x"], "f32", sv, si, "wl4")
