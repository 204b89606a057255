"""GPU parity of the post-filter stage (topkp_sample: the min-p step and the
None / QSample modes of the aclnnTopKTopPSampleV2 page) through the C ABI,
against the CPU oracle.

The bar: every output element is bit-identical to the oracle's, except a
min-p decision at an element whose exp(x - max) lies within BAND (relative)
of min_p; the None-mode token is exact; a QSample token is a kept element
whose probs / (q + eps) is within BAND (relative) of the largest one."""
import numpy as np
import pytest

import flipstats
import oracle as O
from rawutil import NEG_INF, bits, raw_to_torch, torch_to_raw

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BAND = 1e-5
EPS = 1e-10
DTS = ("f32", "f16", "bf16")


@pytest.fixture(scope="module")
def tk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_logit_filter_gb300 import build
    build.build()
    import top_logit_filter_gb300 as m
    return m


def _inputs(B, V, dt, seed, empty_rows=0):
    from top_logit_filter_gb300 import workloads
    return workloads.make_filtered(B, V, dt, seed, empty_rows=empty_rows)


def _run(tk, f, dt, min_p, q, mode="out", ld_pad=0):
    """mode: "out" (separate output), "inplace", or "token" (no output)."""
    B, V = f.shape
    if ld_pad:
        base = torch.full((B, V + ld_pad), float("nan"), dtype=torch.float32).to(
            {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dt]).cuda()
        ft = base[:, ld_pad:]
        ft.copy_(raw_to_torch(f, dt, "cuda"))
    else:
        ft = raw_to_torch(f, dt, "cuda")
    mpt = None if min_p is None else torch.from_numpy(min_p).cuda()
    qt = None if q is None else torch.from_numpy(q).cuda()
    if mode == "inplace":
        tok, o = tk.sample(ft, min_p=mpt, q=qt, eps=EPS, out=ft)
    elif mode == "token":
        tok, o = tk.sample(ft, min_p=mpt, q=qt, eps=EPS, want_out=False)
        assert o is None
    else:
        tok, o = tk.sample(ft, min_p=mpt, q=qt, eps=EPS)
    torch.cuda.synchronize()
    return (None if o is None else torch_to_raw(o, dt)), tok.cpu().numpy()


def _check(f, dt, min_p, q, out, tok, rows=None, where=""):
    """Returns (min-p flips, token differences) over the checked rows."""
    flips = tdiff = 0
    neg = NEG_INF[dt]
    for b in (range(f.shape[0]) if rows is None else rows):
        mp = None if min_p is None else min_p[b]
        qb = None if q is None else q[b]
        ref, t_ref, info = O.sample_row(f[b], dt, mp, qb, EPS)
        w = f"{where} row {b}"
        if t_ref < 0:
            assert tok[b] == -1, w
            if out is not None:
                assert np.array_equal(bits(out[b], dt), bits(f[b], dt)), w
            continue
        fb = bits(f[b], dt)
        if out is not None:
            ob = bits(out[b], dt)
            assert np.all((ob == fb) | (ob == neg)), f"{w}: output neither the input nor -inf"
            gk = ob != neg
            diff = np.nonzero(gk != info.keep)[0]
            if diff.size:
                assert mp is not None and 0.0 < float(mp) < 1.0, f"{w}: differs without min-p at {diff[:8]}"
                rel = np.abs(info.e[diff] - float(np.float32(mp))) / float(np.float32(mp))
                assert np.all(rel <= BAND) and np.all(info.alive[diff]), (
                    f"{w}: min-p flip outside the band at {diff[rel > BAND][:8]}")
                flips += int(diff.size)
        else:
            gk = info.keep
        t = int(tok[b])
        if q is None:
            assert t == t_ref, f"{w}: argmax token {t} != {t_ref}"
            continue
        assert 0 <= t < f.shape[1] and info.alive[t], f"{w}: token {t} is not a survivor"
        if out is not None:
            assert gk[t], f"{w}: token {t} was removed by the GPU's own min-p"
        qv = q[b].astype(np.float64) + float(np.float32(EPS))
        r = np.where(gk, info.e / qv, -np.inf)
        assert info.e[t] / qv[t] >= r.max() * (1.0 - BAND), f"{w}: token {t} is not a largest ratio"
        tdiff += int(t != t_ref)
    return flips, tdiff


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("V", [1, 7, 1000, 4099])
@pytest.mark.parametrize("use_mp,use_q", [(False, False), (True, False), (False, True), (True, True)])
def test_sample_small(tk, dt, V, use_mp, use_q):
    d = _inputs(6, V, dt, seed=100 + V, empty_rows=1)
    mp = d["min_p"] if use_mp else None
    q = d["q"] if use_q else None
    out, tok = _run(tk, d["x"], dt, mp, q)
    _check(d["x"], dt, mp, q, out, tok, where=f"{dt} V={V}")


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("mode", ["inplace", "token"])
def test_sample_in_place_and_token_only(tk, dt, mode):
    d = _inputs(8, 3001, dt, seed=7)
    out, tok = _run(tk, d["x"], dt, d["min_p"], d["q"], mode=mode)
    _check(d["x"], dt, d["min_p"], d["q"], out, tok, where=mode)


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
def test_sample_strided_unaligned_rows(tk, dt):
    d = _inputs(5, 2053, dt, seed=9)
    out, tok = _run(tk, d["x"], dt, d["min_p"], d["q"], ld_pad=3)
    _check(d["x"], dt, d["min_p"], d["q"], out, tok, where="strided")


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("mode", ["out", "inplace", "token"])
def test_sample_dense_rows(tk, dt, mode):
    """Rows with more survivors than the kernel lists in shared memory (every
    element finite, V = 12289): the second pass reads the row again."""
    rng = np.random.default_rng(31)
    from rawutil import to_raw
    B, V = 6, 12289
    f = np.stack([to_raw(2.0 * rng.standard_normal(V), dt) for _ in range(B)])
    mp = np.array([0.0, 0.01, 0.2, 1.0, 0.5, 0.05], np.float32)
    q = rng.exponential(1.0, size=(B, V)).astype(np.float32)
    out, tok = _run(tk, f, dt, mp, q, mode=mode)
    _check(f, dt, mp, q, out, tok, where=f"dense {mode}")
    out, tok = _run(tk, f, dt, mp, None, mode=mode)
    _check(f, dt, mp, None, out, tok, where=f"dense argmax {mode}")


def test_sample_edge_rows(tk):
    dt = "f32"
    rows = [
        [1.0, 3.0, 2.0, 3.0],                 # tied maximum
        ["-inf", "-inf", 5.0, "-inf"],        # one survivor
        ["-inf", "-inf", "-inf", "-inf"],     # none (token -1, copied)
        [0.0, "-0", "-inf", -1.0],            # signed zeros tie as the maximum
    ]
    from rawutil import to_raw
    f = np.stack([to_raw(r, dt) for r in rows])
    for mp in (np.array([1.0, 1.0, 1.0, 1.0], np.float32), np.array([0.5, 0.0, 0.2, 0.4], np.float32), None):
        for q in (None, np.array([[1, 5, 1, 1], [1, 1, 1, 1], [1, 1, 1, 1], [2, 1, 1, 1]], np.float32)):
            out, tok = _run(tk, f, dt, mp, q)
            _check(f, dt, mp, q, out, tok, where="edge")
    out, tok = _run(tk, f, dt, np.ones(4, np.float32), None)
    assert tok.tolist() == [3, 2, -1, 1]
    assert np.array_equal(bits(out[0], dt), bits(to_raw(["-inf", "-inf", "-inf", 3.0], dt), dt))


def test_sample_full_size_bf16(tk):
    """B=256 x V=128256 bf16 (the filter's decode batch), every row against
    the oracle, QSample with min-p; the GPU and the oracle should agree on
    (nearly) every token."""
    d = _inputs(256, 128256, "bf16", seed=3, empty_rows=2)
    out, tok = _run(tk, d["x"], "bf16", d["min_p"], d["q"])
    flips, tdiff = _check(d["x"], "bf16", d["min_p"], d["q"], out, tok, where="full")
    assert tdiff <= 2, tdiff
    flipstats.record("sample stage, B=256 x V=128256 bf16 filtered rows", 256, flips, "min-p flips inside the band")
    flipstats.record("sample stage, B=256 x V=128256 bf16 filtered rows", 256, tdiff, "QSample tokens differing within the band")


def test_filter_then_sample_pipeline(tk):
    """The oracle's filter output of 32 rows of the B=256 x V=128256 bf16
    decode batch (joint top-k + top-p) feeds the GPU sample stage."""
    from top_logit_filter_gb300 import workloads
    w = workloads.make(3)
    rows = list(range(32))
    f, _ = O.apply(w["x"][:32], "bf16", w["p"][:32], w["k"][:32])
    rng = np.random.default_rng(77)
    q = rng.exponential(1.0, size=f.shape).astype(np.float32)
    mp = rng.uniform(0.001, 0.2, size=32).astype(np.float32)
    out, tok = _run(tk, f, "bf16", mp, q)
    _check(f, "bf16", mp, q, out, tok, rows=rows, where="pipeline")
    out, tok = _run(tk, f, "bf16", None, None)
    _check(f, "bf16", None, None, out, tok, rows=rows, where="pipeline argmax")
