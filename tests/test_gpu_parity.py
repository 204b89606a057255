"""GPU parity: libtopkp.so (through the C ABI) against the CPU oracle.

Small cases sweep dtypes, ragged row lengths, every launch plan, the k / p
edge values of sections 4 and 2 of the CANN ops-nn ApplyTopKTopPWithSorted
guide, tie-heavy rows, signed zeros, strided, unaligned and in-place buffers.
The five workloads then run at full size, in the launch configuration the
benchmark uses, checked row by row on a sample (and by closed forms on every
row where one exists)."""
import numpy as np
import pytest

import flipstats
import oracle as O
from parity import compare_row
from rawutil import NEG_INF, bits, raw_to_torch, to_raw, torch_to_raw

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


def _rows(rng, B, V, dtype, kind):
    if kind == "normal":
        x = rng.standard_normal((B, V)).astype(np.float32) * 3
    elif kind == "ties":
        x = (rng.integers(-6, 7, size=(B, V)) * 0.5).astype(np.float32)
    elif kind == "wide":
        # magnitudes over dozens of binades, both signs: a 16-bit row then
        # touches more key buckets than the key-count path has blocks
        lo, hi = (-20.0, 14.0) if dtype == "f16" else (-60.0, 60.0)
        sign = np.where(rng.random((B, V)) < 0.5, -1.0, 1.0)
        x = (sign * np.exp2(rng.uniform(lo, hi, size=(B, V)))).astype(np.float32)
    elif kind == "logprob":
        # every value negative (log-probabilities)
        x = (-np.abs(rng.standard_normal((B, V))) * 3 - 0.01).astype(np.float32)
    elif kind == "shifted":
        # every value far above zero: no negative value carries mass
        x = (rng.standard_normal((B, V)) * 2 + 40).astype(np.float32)
    elif kind == "late_max":
        # negative rows whose maximum sits in the last percent of the row,
        # after the first load group of every warp
        x = (-np.abs(rng.standard_normal((B, V))) * 3 - 1).astype(np.float32)
        for b in range(B):
            x[b, V - 1 - int(rng.integers(0, max(1, V // 100)))] = 2.5 + b
    else:  # "zeros": signed zeros and a few values
        x = rng.choice(np.array([-0.0, 0.0, 1.0, -1.0, 2.0], dtype=np.float32), size=(B, V))
    return np.stack([to_raw(r, dtype) for r in x])


def _kp(rng, B, V, dtype, mode):
    kcand = [-1, 0, 1, 2, max(1, V // 3), V - 1, V, V + 5, int(rng.integers(1, max(2, V)))]
    pcand = [0.0, 0.3, 0.9, 1.0, float(rng.random()), 0.5]
    k = np.array([kcand[i % len(kcand)] for i in range(B)], dtype=np.int32) if mode != "p" else None
    p = to_raw([pcand[i % len(pcand)] for i in range(B)], dtype) if mode != "k" else None
    return k, p


def _run_apply(tk, x, dtype, p, k, out=None):
    xt = raw_to_torch(x, dtype, "cuda")
    pt = None if p is None else raw_to_torch(p, dtype, "cuda")
    kt = None if k is None else torch.from_numpy(k).cuda()
    o = tk.apply(xt, p=pt, k=kt, out=out)
    torch.cuda.synchronize()
    return torch_to_raw(o, dtype)


def _infos(x, dtype, p, k):
    return [O.apply_row(x[b], dtype, None if p is None else p[b], None if k is None else int(k[b]))[1]
            for b in range(x.shape[0])]


def _check_all(out, x, dtype, p, k, where, infos=None):
    flips = 0
    infos = _infos(x, dtype, p, k) if infos is None else infos
    for b in range(x.shape[0]):
        flips += compare_row(out[b], x[b], infos[b], dtype, where=f"{where} row {b}")
    return flips


# TOPKP_FORCE_PLAN: "" = the planner's choice; "generic" = every row that
# needs a cut takes the generic radix path; "cN" = every row is split over a
# cluster of N CTAs (slices may be short or empty), "mN" = mixed clusters of
# N (a row without top-k split over the cluster, or N rows with top-k, one
# per CTA), alone or after "generic,".
PLANS = ["", "generic", "c2", "c8", "generic,c4", "m4"]


@pytest.mark.parametrize("dtype", DTS)
@pytest.mark.parametrize("V", [1, 2, 7, 64, 1000, 5003])
@pytest.mark.parametrize("mode", ["k", "p", "kp"])
def test_small_rows_all_plans(tk, monkeypatch, dtype, V, mode):
    rng = np.random.default_rng(V * 7 + len(mode))
    B = 9
    for kind in ("normal", "ties", "zeros", "wide", "logprob", "shifted"):
        x = _rows(rng, B, V, dtype, kind)
        k, p = _kp(rng, B, V, dtype, mode)
        infos = _infos(x, dtype, p, k)
        for plan in PLANS:
            monkeypatch.setenv("TOPKP_FORCE_PLAN", plan)
            out = _run_apply(tk, x, dtype, p, k)
            _check_all(out, x, dtype, p, k, f"{dtype} V={V} {mode} {kind} plan={plan!r}", infos)


@pytest.mark.parametrize("dtype", DTS)
def test_multi_slice_rows(tk, monkeypatch, dtype):
    """Rows long enough that every warp sweeps several load groups, with a
    partial last warp step and a tail shorter than 16 bytes."""
    rng = np.random.default_rng(3)
    B, V = 6, 40011
    for kind in ("normal", "ties", "wide", "logprob", "shifted", "late_max"):
        x = _rows(rng, B, V, dtype, kind)
        k, p = _kp(rng, B, V, dtype, "kp")
        k[:3] = [0, 37, 900]
        infos_kp, infos_p = _infos(x, dtype, p, k), _infos(x, dtype, p, None)
        for plan in PLANS + ["c4"]:
            monkeypatch.setenv("TOPKP_FORCE_PLAN", plan)
            out = _run_apply(tk, x, dtype, p, k)
            _check_all(out, x, dtype, p, k, f"{dtype} {kind} plan={plan!r}", infos_kp)
            # top-p only (k absent): the mass-table and window paths
            out = _run_apply(tk, x, dtype, p, None)
            _check_all(out, x, dtype, p, None, f"{dtype} {kind} top-p only plan={plan!r}", infos_p)


@pytest.mark.parametrize("plan", ["", "c2", "c4"])
@pytest.mark.parametrize("dtype", DTS)
def test_strided_unaligned_and_in_place(tk, monkeypatch, dtype, plan):
    monkeypatch.setenv("TOPKP_FORCE_PLAN", plan)
    rng = np.random.default_rng(11)
    B, V = 5, 3001
    x = _rows(rng, B, V, dtype, "normal")
    k, p = _kp(rng, B, V, dtype, "kp")
    pt = raw_to_torch(p, dtype, "cuda")
    kt = torch.from_numpy(k).cuda()
    big = torch.zeros((B, V + 9), dtype=raw_to_torch(x, dtype).dtype, device="cuda")
    big[:, 1:V + 1] = raw_to_torch(x, dtype, "cuda")       # misaligned base, stride V+9
    view = big[:, 1:V + 1]
    obig = torch.zeros_like(big)
    out = tk.apply(view, p=pt, k=kt, out=obig[:, 3:V + 3])
    torch.cuda.synchronize()
    _check_all(torch_to_raw(out, dtype), x, dtype, p, k, f"{dtype} strided")
    # untouched padding
    assert torch.count_nonzero(obig[:, :3]) == 0 and torch.count_nonzero(obig[:, V + 3:]) == 0
    # in place
    xt = raw_to_torch(x, dtype, "cuda")
    r = tk.apply(xt, p=pt, k=kt, out=xt)
    torch.cuda.synchronize()
    assert r.data_ptr() == xt.data_ptr()
    _check_all(torch_to_raw(xt, dtype), x, dtype, p, k, f"{dtype} in place")


def test_empty_and_single_column(tk):
    x = torch.zeros((0, 5), device="cuda")
    assert tk.apply(x, k=torch.zeros(0, dtype=torch.int32, device="cuda")).shape == (0, 5)
    x = torch.zeros((3, 0), device="cuda")
    assert tk.apply(x, k=torch.ones(3, dtype=torch.int32, device="cuda")).shape == (3, 0)
    x = torch.tensor([[-1.5], [2.0], [0.0]], device="cuda")
    o = tk.apply(x, p=torch.tensor([0.0, 0.5, 1.0], device="cuda"), k=torch.ones(3, dtype=torch.int32, device="cuda"))
    assert torch.equal(o, x)


def test_deterministic(tk):
    from top_logit_filter_gb300 import workloads
    w = workloads.make(3, B=32)
    xt = raw_to_torch(w["x"], "bf16", "cuda")
    pt = raw_to_torch(w["p"], "bf16", "cuda")
    kt = torch.from_numpy(w["k"]).cuda()
    a = tk.apply(xt, p=pt, k=kt)
    for _ in range(3):
        b = tk.apply(xt, p=pt, k=kt)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    tk.device_status()


# ------------------------------------------------------------ full workloads
def _workload_inputs(w):
    dt = w["dtype"]
    xt = raw_to_torch(w["x"], dt, "cuda")
    pt = None if w["p"] is None else raw_to_torch(w["p"], dt, "cuda")
    kt = None if w["k"] is None else torch.from_numpy(w["k"]).cuda()
    return xt, pt, kt


@pytest.mark.parametrize("wl,sample", [(1, None), (2, None), (3, None), (4, 48)])
def test_workload_full_size(tk, wl, sample):
    from top_logit_filter_gb300 import workloads
    w = workloads.make(wl)
    dt = w["dtype"]
    xt, pt, kt = _workload_inputs(w)
    out = torch_to_raw(tk.apply(xt, p=pt, k=kt), dt)
    tk.device_status()
    B = w["B"]
    rows = range(B) if sample is None else np.random.default_rng(wl).choice(B, sample, replace=False)
    flips = 0
    for b in rows:
        _, info = O.apply_row(w["x"][b], dt, None if w["p"] is None else w["p"][b],
                              None if w["k"] is None else int(w["k"][b]))
        flips += compare_row(out[b], w["x"][b], info, dt, where=f"workload {wl} row {b}")
    flipstats.record(f"workload {wl} ({w['name']})", len(rows), flips)
    if wl == 4:
        # top-k alone on every row: out == where(x >= k-th largest, x, -inf)
        xv = O.decode(w["x"], dt)
        ob = bits(out, dt)
        for b in range(B):
            kk = int(w["k"][b])
            kth = np.partition(xv[b], w["V"] - kk)[w["V"] - kk]
            exp = np.where(xv[b] >= kth, bits(w["x"][b], dt), NEG_INF[dt])
            assert np.array_equal(ob[b], exp), f"row {b}"


def test_workload3_every_split_full_size(tk, monkeypatch):
    """All 256 rows of the B=256 x V=128256 bf16 batch against the oracle
    under every split of a row over a cluster, and the planner's own."""
    from top_logit_filter_gb300 import workloads
    w = workloads.make(3)
    dt = w["dtype"]
    xt, pt, kt = _workload_inputs(w)
    infos = _infos(w["x"], dt, w["p"], w["k"])
    for plan in ("c1", "c2", "c4", "c8", "m2", "m8", ""):
        monkeypatch.setenv("TOPKP_FORCE_PLAN", plan)
        out = torch_to_raw(tk.apply(xt, p=pt, k=kt), dt)
        tk.device_status()
        flips = _check_all(out, w["x"], dt, w["p"], w["k"], f"workload 3 plan={plan!r}", infos)
        flipstats.record(f"workload 3 split plan {plan or 'planner'!r}", w["B"], flips)


@pytest.mark.parametrize("mode", ["topp_only", "topk_only", "all_rows_joint"])
def test_workload3_mode_variants_full_size(tk, mode):
    """The B=256 x V=128256 bf16 rows with one filter dropped (or every row
    joint), so each launch runs one kernel path on every row."""
    from top_logit_filter_gb300 import workloads
    w = workloads.make(3)
    dt = "bf16"
    k = None if mode == "topp_only" else np.where(w["k"] > 0, w["k"], 512).astype(np.int32)
    p = None if mode == "topk_only" else w["p"]
    xt = raw_to_torch(w["x"], dt, "cuda")
    out = torch_to_raw(tk.apply(xt, p=None if p is None else raw_to_torch(p, dt, "cuda"),
                                k=None if k is None else torch.from_numpy(k).cuda()), dt)
    tk.device_status()
    flips = 0
    rows = np.random.default_rng(7).choice(w["B"], 40, replace=False)
    for b in rows:
        _, info = O.apply_row(w["x"][b], dt, None if p is None else p[b], None if k is None else int(k[b]))
        flips += compare_row(out[b], w["x"][b], info, dt, where=f"{mode} row {b}")
    flipstats.record(f"workload 3 as {mode}", len(rows), flips)


@pytest.mark.parametrize("dtype", ("f16", "bf16"))
def test_top_p_cut_among_signed_zeros(tk, monkeypatch, dtype):
    """Top-p-only rows whose cut falls inside a run of zeros, -0 and +0
    mixed: the two compare equal, so they rank as ties in index order and
    the first kept zero may be either."""
    rng = np.random.default_rng(17)
    V = 4000
    vals = np.array([-1.0, -0.0, 0.0, 1.0, 2.0], dtype=np.float32)
    ps = np.linspace(0.80, 0.98, 16)
    x = np.stack([to_raw(rng.permutation(np.repeat(vals, V // len(vals))), dtype) for _ in ps])
    p = to_raw(ps, dtype)
    # the oracle's first kept element is -0 in some rows and +0 in others
    cut_bits = set()
    for b in range(len(ps)):
        _, info = O.apply_row(x[b], dtype, p[b], None)
        first = info.idx[np.argmax(info.kept)]
        cut_bits.add(int(bits(x[b][first:first + 1], dtype)[0]))
    assert {int(bits(to_raw(np.array([-0.0], np.float32), dtype), dtype)[0]),
            int(bits(to_raw(np.array([0.0], np.float32), dtype), dtype)[0])} <= cut_bits
    for plan in PLANS:
        monkeypatch.setenv("TOPKP_FORCE_PLAN", plan)
        out = _run_apply(tk, x, dtype, p, None)
        _check_all(out, x, dtype, p, None, f"{dtype} signed zeros plan={plan!r}")


@pytest.mark.parametrize("plan", ["", "c2", "c4"])
@pytest.mark.parametrize("dtype", DTS)
def test_sampled_bound_too_high_restarts(tk, monkeypatch, dtype, plan):
    """Rows whose first load groups (the sample that bounds top-k candidates
    in a single pass) hold one large value per vector and the rest of the
    row nothing comparable: the sampled bound then has fewer than k elements
    above it, and the row must restart with the exact two-pass bound."""
    rng = np.random.default_rng(29)
    B, V = 2, 131072
    x = rng.standard_normal((B, V)).astype(np.float32)
    per_warp = V // 8 // 16                     # 16-byte vectors per warp (16-bit rows)
    if dtype == "f32":
        per_warp = V // 4 // 16
    vec = 8 if dtype != "f32" else 4
    big = 10.0 + 0.25 * np.arange(16 * 128, dtype=np.float32)
    rng.shuffle(big)
    i = 0
    for w in range(16):
        for t in range(128):                    # the first 128 vectors of warp w
            x[:, (w * per_warp + t) * vec] = big[i]
            i += 1
    xr = np.stack([to_raw(r, dtype) for r in x])
    k = np.array([1000, 1300], dtype=np.int32)
    monkeypatch.setenv("TOPKP_FORCE_PLAN", plan)
    for p in (None, to_raw([0.9, 0.5], dtype)):
        out = _run_apply(tk, xr, dtype, p, k)
        _check_all(out, xr, dtype, p, k, f"{dtype} sampled bound restart p={p is not None}")


def _two_cluster_rows(dtype):
    """fp16/bf16 rows with a cluster of values near -2 and one near +3 (and
    nothing between), sized so that the mass below the gap is close to
    1 - p: the rigorous window of the top-p cut then reaches from one
    cluster across zero to the other, over a thousand empty buckets."""
    rng = np.random.default_rng(41)
    V = 8192
    rows = []
    for ratio in np.linspace(2.10, 2.55, 16):
        n2 = int(round((V - 1) / (1 + ratio)))
        n1 = V - 1 - n2
        v = np.concatenate([rng.uniform(-2.0, -1.9, n1), rng.uniform(2.9, 3.0, n2), [3.0]]).astype(np.float32)
        rows.append(rng.permutation(v))
    x = np.stack([to_raw(r, dtype) for r in rows])
    p = to_raw(np.full(len(rows), 1.0 - 1.0 / 64.0, dtype=np.float32), dtype)
    return x, p


@pytest.mark.parametrize("plan", ["", "c2", "c8"])
@pytest.mark.parametrize("dtype", ("f16", "bf16"))
def test_top_p_window_across_empty_buckets(tk, monkeypatch, dtype, plan):
    monkeypatch.setenv("TOPKP_FORCE_PLAN", plan)
    x, p = _two_cluster_rows(dtype)
    out = _run_apply(tk, x, dtype, p, None)
    _check_all(out, x, dtype, p, None, f"{dtype} two clusters plan={plan!r}")
