"""GPU parity of topkp_apply_sample: the filter of the CANN ops-nn
ApplyTopKTopPWithSorted guide (section 2) and, on its survivors, the min-p
step and the sample of the page aclnnTopKTopPSampleV2, in one pass.

Two bars.  Against the GPU's own two-call path (topkp_apply, then
topkp_sample on its output): the same token and the same output bits, since
both compute the same arithmetic.  Against the CPU oracle (oracle.apply_row,
then oracle.sample_row on its output): the tolerances of the two stages, a
top-p flip inside the filter's band (tests/parity.py) and a min-p or race
decision inside the sample's band (tests/test_gpu_sample.py)."""
import numpy as np
import pytest

import flipstats
import oracle as O
from rawutil import NEG_INF, bits, raw_to_torch, to_raw, torch_to_raw
from test_gpu_parity import _kp, _rows
from test_gpu_sample import _check as check_sample, EPS

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DTS = ("f32", "f16", "bf16")
PLANS = ["", "generic", "c2", "m4"]


@pytest.fixture(scope="module")
def tk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_logit_filter_gb300 import build
    build.build()
    import top_logit_filter_gb300 as m
    return m


def _t(a, dt=None):
    if a is None:
        return None
    if dt is not None:
        return raw_to_torch(a, dt, "cuda")
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _two_call(tk, x, dt, p, k, mp, q):
    f = tk.apply(_t(x, dt), p=_t(p, dt), k=_t(k))
    tok, o = tk.sample(f, min_p=_t(mp), q=_t(q), eps=EPS)
    torch.cuda.synchronize()
    return torch_to_raw(f, dt), torch_to_raw(o, dt), tok.cpu().numpy()


def _fused(tk, x, dt, p, k, mp, q, mode="out"):
    xt = _t(x, dt)
    if mode == "inplace":
        tok, o = tk.apply_sample(xt, p=_t(p, dt), k=_t(k), min_p=_t(mp), q=_t(q), eps=EPS, out=xt)
    elif mode == "token":
        tok, o = tk.apply_sample(xt, p=_t(p, dt), k=_t(k), min_p=_t(mp), q=_t(q), eps=EPS, want_out=False)
        assert o is None
    else:
        tok, o = tk.apply_sample(xt, p=_t(p, dt), k=_t(k), min_p=_t(mp), q=_t(q), eps=EPS)
    torch.cuda.synchronize()
    return (None if o is None else torch_to_raw(o, dt)), tok.cpu().numpy()


def _min_p(rng, B):
    mp = rng.uniform(0.001, 0.3, size=B).astype(np.float32)
    mp[::7] = 0.0
    mp[3::11] = 1.0
    return mp


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("V", [1, 7, 1000, 5003])
@pytest.mark.parametrize("mode", ["k", "p", "kp"])
def test_fused_equals_two_calls(tk, monkeypatch, dt, V, mode):
    rng = np.random.default_rng(V * 5 + len(mode))
    B = 9
    for kind in ("normal", "ties", "zeros", "wide"):
        x = _rows(rng, B, V, dt, kind)
        k, p = _kp(rng, B, V, dt, mode)
        mp = _min_p(rng, B)
        q = rng.exponential(1.0, size=(B, V)).astype(np.float32)
        for plan in PLANS:
            monkeypatch.setenv("TOPKP_FORCE_PLAN", plan)
            for mpa, qa in ((mp, q), (None, q), (mp, None), (None, None)):
                f, o2, t2 = _two_call(tk, x, dt, p, k, mpa, qa)
                for m in ("out", "inplace", "token"):
                    o1, t1 = _fused(tk, x, dt, p, k, mpa, qa, m)
                    where = f"{dt} V={V} {mode} {kind} plan={plan!r} mp={mpa is not None} q={qa is not None} {m}"
                    assert np.array_equal(t1, t2), f"{where}: tokens {t1} vs {t2}"
                    if o1 is not None:
                        assert np.array_equal(bits(o1, dt), bits(o2, dt)), f"{where}: outputs differ"


@pytest.mark.parametrize("dt", DTS)
def test_fused_against_the_oracle(tk, dt):
    """Output and token against oracle.sample_row on oracle.apply_row's
    output, row by row."""
    rng = np.random.default_rng(17)
    B, V = 12, 20011
    x = _rows(rng, B, V, dt, "normal")
    k, p = _kp(rng, B, V, dt, "kp")
    mp = _min_p(rng, B)
    q = rng.exponential(1.0, size=(B, V)).astype(np.float32)
    o, tok = _fused(tk, x, dt, p, k, mp, q)
    f = np.stack([O.apply_row(x[b], dt, p[b], int(k[b]))[0] for b in range(B)])
    check_sample(f, dt, mp, q, o, tok, where=f"fused {dt}")
    o, tok = _fused(tk, x, dt, p, k, None, None)
    check_sample(f, dt, None, None, o, tok, where=f"fused {dt} argmax")


def test_fused_full_size_bench_batch(tk):
    """The B=256 x V=128256 bf16 joint batch with min_p and q: fused against
    the two calls on every row, and against the oracle on 32 rows."""
    from top_logit_filter_gb300 import workloads
    w = workloads.make(3)
    dt = "bf16"
    rng = np.random.default_rng(33)
    mp = _min_p(rng, w["B"])
    q = rng.exponential(1.0, size=(w["B"], w["V"])).astype(np.float32)
    f, o2, t2 = _two_call(tk, w["x"], dt, w["p"], w["k"], mp, q)
    o1, t1 = _fused(tk, w["x"], dt, w["p"], w["k"], mp, q)
    assert np.array_equal(t1, t2)
    assert np.array_equal(bits(o1, dt), bits(o2, dt))
    _, t3 = _fused(tk, w["x"], dt, w["p"], w["k"], mp, q, "token")
    assert np.array_equal(t3, t2)
    rows = list(range(32))
    fo = np.stack([O.apply_row(w["x"][b], dt, w["p"][b], int(w["k"][b]))[0] for b in rows])
    flips, tdiff = check_sample(fo, dt, mp[:32], q[:32], None, t1[:32], where="fused full")
    flipstats.record("fused filter + sample, B=256 x V=128256 bf16 (first 32 rows)", 32, tdiff,
                     "QSample tokens differing within the band")
