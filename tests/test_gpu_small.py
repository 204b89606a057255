"""GPU parity of the short-row kernels (small.cu): rows of at most 4096
elements sorted in shared memory, 16-bit rows of at most 32768 elements
counted per key in registers.

Two bars.  Against the main filter kernel (apply.cu, forced with the plan
"c1"): the same output bits, since both compute the filter of the CANN
ops-nn ApplyTopKTopPWithSorted guide (section 2) with the same per-element
fixed-point masses and exact integer sums.  Against the CPU oracle: the
parity rule of tests/parity.py (top-k exact, top-p flips only inside the
1e-5 band)."""
import numpy as np
import pytest

import flipstats
from rawutil import bits, raw_to_torch, torch_to_raw
from test_gpu_parity import DTS, _check_all, _infos, _kp, _rows, _run_apply

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

KINDS = ("normal", "ties", "zeros", "wide", "logprob", "shifted", "late_max")


@pytest.fixture(scope="module")
def tk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_logit_filter_gb300 import build
    build.build()
    import top_logit_filter_gb300 as m
    return m


def _both(tk, monkeypatch, x, dt, p, k, plan="small"):
    monkeypatch.setenv("TOPKP_FORCE_PLAN", plan)
    a = _run_apply(tk, x, dt, p, k)
    monkeypatch.setenv("TOPKP_FORCE_PLAN", "c1")
    b = _run_apply(tk, x, dt, p, k)
    return a, b


def _same(a, b, dt, where):
    ba, bb = bits(a, dt), bits(b, dt)
    if not np.array_equal(ba, bb):
        r, c = np.argwhere(ba != bb)[0]
        raise AssertionError(f"{where}: short-row kernel and main kernel differ first at row {r} col {c} "
                             f"({ba[r, c]:#x} vs {bb[r, c]:#x})")


@pytest.mark.parametrize("dtype", DTS)
@pytest.mark.parametrize("V", [1, 3, 31, 1024, 2049, 4096])
@pytest.mark.parametrize("mode", ["k", "p", "kp"])
def test_sort_path(tk, monkeypatch, dtype, V, mode):
    rng = np.random.default_rng(V * 13 + len(mode))
    B = 9
    for kind in KINDS:
        x = _rows(rng, B, V, dtype, kind)
        k, p = _kp(rng, B, V, dtype, mode)
        a, b = _both(tk, monkeypatch, x, dtype, p, k)
        _same(a, b, dtype, f"{dtype} V={V} {mode} {kind}")
        _check_all(a, x, dtype, p, k, f"sort path {dtype} V={V} {mode} {kind}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("V", [4097, 8191, 20000, 32000, 32768])
@pytest.mark.parametrize("mode", ["k", "p", "kp"])
@pytest.mark.parametrize("plan", ["small1", "small2"])
def test_table_path(tk, monkeypatch, dtype, V, mode, plan):
    """One CTA per row, and a cluster of two CTAs per row (each counts half
    the row; the bucket sums, scans and tie ranks go through the cluster)."""
    rng = np.random.default_rng(V * 17 + len(mode))
    B = 9
    for kind in KINDS:
        x = _rows(rng, B, V, dtype, kind)
        k, p = _kp(rng, B, V, dtype, mode)
        a, b = _both(tk, monkeypatch, x, dtype, p, k, plan)
        _same(a, b, dtype, f"{plan} {dtype} V={V} {mode} {kind}")
        if kind in ("normal", "ties", "zeros"):
            _check_all(a, x, dtype, p, k, f"table path {plan} {dtype} V={V} {mode} {kind}")


@pytest.mark.parametrize("dtype", DTS)
@pytest.mark.parametrize("V", [3001, 20011])
@pytest.mark.parametrize("plan", ["small1", "small2"])
def test_strided_unaligned_and_in_place(tk, monkeypatch, dtype, V, plan):
    """Misaligned row starts, row strides above V, a separate misaligned
    output with untouched padding, and in place."""
    monkeypatch.setenv("TOPKP_FORCE_PLAN", plan)
    rng = np.random.default_rng(V)
    B = 5
    x = _rows(rng, B, V, dtype, "normal")
    k, p = _kp(rng, B, V, dtype, "kp")
    infos = _infos(x, dtype, p, k)
    pt = raw_to_torch(p, dtype, "cuda")
    kt = torch.from_numpy(k).cuda()
    big = torch.zeros((B, V + 9), dtype=raw_to_torch(x, dtype).dtype, device="cuda")
    big[:, 1:V + 1] = raw_to_torch(x, dtype, "cuda")
    obig = torch.zeros_like(big)
    out = tk.apply(big[:, 1:V + 1], p=pt, k=kt, out=obig[:, 3:V + 3])
    torch.cuda.synchronize()
    _check_all(torch_to_raw(out, dtype), x, dtype, p, k, f"{dtype} V={V} strided", infos)
    assert torch.count_nonzero(obig[:, :3]) == 0 and torch.count_nonzero(obig[:, V + 3:]) == 0
    xt = raw_to_torch(x, dtype, "cuda")
    r = tk.apply(xt, p=pt, k=kt, out=xt)
    torch.cuda.synchronize()
    assert r.data_ptr() == xt.data_ptr()
    _check_all(torch_to_raw(xt, dtype), x, dtype, p, k, f"{dtype} V={V} in place", infos)


@pytest.mark.parametrize("wl", [1, 2])
def test_small_workloads_full_size(tk, monkeypatch, wl):
    """The 4 x 1024 fp32 joint and 64 x 32000 fp16 top-p-only batches: the
    planner's choice (the short-row kernels) against the main kernel and the
    oracle on every row."""
    from top_logit_filter_gb300 import workloads
    w = workloads.make(wl)
    dt = w["dtype"]
    monkeypatch.setenv("TOPKP_FORCE_PLAN", "")
    a = _run_apply(tk, w["x"], dt, w["p"], w["k"])
    monkeypatch.setenv("TOPKP_FORCE_PLAN", "c1")
    b = _run_apply(tk, w["x"], dt, w["p"], w["k"])
    _same(a, b, dt, w["name"])
    flips = _check_all(a, w["x"], dt, w["p"], w["k"], w["name"])
    flipstats.record(f"workload {wl} ({w['name']}) on the short-row kernel", w["B"], flips,
                     "top-p flips inside the band")
