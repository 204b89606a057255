"""GPU parity of topkp_sample_v2 (the TopKTopPSampleV2 semantics of the page
aclnnTopKTopPSampleV2) through the C ABI, against the CPU oracle
(oracle/v2.py).

The bar.  The sorted order and its indices are exact.  The kept positions
form a prefix of that order; its length may differ from the oracle's only
through decisions inside the band: a top-p decision whose cumulative
probability lies within BAND of its threshold, or a min-p decision whose
probability lies within BAND (relative) of prob[0] * min_p.  Without q the
token is exact; with q it is a kept position whose prob / (q + eps) is
within BAND (relative) of the largest.  Probabilities agree within PROB_RTOL
(fp32 exponentials and one fp32 division against the exact value rounded
once: a few units in the last place)."""
import numpy as np
import pytest

import flipstats
import oracle.v2 as OV
from rawutil import NEG_INF, bits, raw_to_torch, to_raw, torch_to_raw

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BAND = 1e-5
PROB_RTOL = 1e-5
EPS = 1e-10


@pytest.fixture(scope="module")
def tk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_logit_filter_gb300 import build
    build.build()
    import top_logit_filter_gb300 as m
    return m


def _run(tk, x, dt, k, p, mp, q, ks_max, logits, need):
    xt = raw_to_torch(x, dt, "cuda")
    kt = None if k is None else torch.from_numpy(np.asarray(k, dtype=np.int32)).cuda()
    pt = None if p is None else torch.from_numpy(np.asarray(p, dtype=np.float32)).cuda()
    mt = None if mp is None else torch.from_numpy(np.asarray(mp, dtype=np.float32)).cuda()
    qt = None if q is None else torch.from_numpy(q).cuda()
    a, b = tk.sample_v2(xt, k=kt, p=pt, min_p=mt, q=qt, eps=EPS, ks_max=ks_max, input_is_logits=logits,
                        need_sample_result=need)
    torch.cuda.synchronize()
    if need:
        return a.cpu().numpy(), b.cpu().numpy()
    return a.cpu().numpy(), torch_to_raw(b, dt)


def _band_ok(info, lo, hi, mp):
    """Every sorted position in [lo, hi) decided inside the band."""
    for j in range(lo, hi):
        ok = False
        if info.topp_stat is not None:
            stat, thr = info.topp_stat
            if j < len(stat) and abs(float(stat[j]) - float(thr)) <= BAND:
                ok = True
        if info.thd is not None and j < len(info.prob32):
            if abs(float(info.prob32[j]) - info.thd) <= BAND * info.thd:
                ok = True
        if not ok:
            return False
    return True


def _check_row(x, dt, info, sel, tok, idx, sm, q, logits, where):
    V = x.shape[0]
    order = info.order
    n_kept_o = info.n_kept
    flips = 0
    if sel is not None:
        xb, sb = bits(x, dt), bits(sel, dt)
        d = NEG_INF[dt] if logits else 0
        assert np.all((sb == xb) | (sb == d)), f"{where}: output neither the input nor defLogit"
        kept = (sb == xb)[order]
        n_kept_g = int(np.argmin(kept)) if not kept.all() else V
        assert not kept[n_kept_g:].any(), f"{where}: kept positions are not a prefix of the order"
    else:
        fill = np.float32(0.0) if (info.minp_ran or not logits) else np.float32(-np.inf)
        live = ~((sm == fill) | np.isnan(sm))
        n_kept_g = int(np.argmin(live)) if not live.all() else V
    if n_kept_g != n_kept_o:
        lo, hi = sorted((n_kept_g, n_kept_o))
        assert _band_ok(info, lo, hi, None), f"{where}: kept {n_kept_g} positions, oracle {n_kept_o}, outside the band"
        flips = hi - lo
    if tok is not None:
        if q is None:
            assert tok == order[0], f"{where}: token {tok}, want {order[0]}"
        else:
            pos = int(np.flatnonzero(order == tok)[0])
            n = min(n_kept_g, n_kept_o)
            assert pos < max(n_kept_g, n_kept_o), f"{where}: token outside the kept prefix"
            r = info.prob32[:n].astype(np.float64) / (q[:n].astype(np.float64) + float(np.float32(EPS)))
            mine = float(info.prob32[pos]) / (float(q[pos]) + float(np.float32(EPS)))
            assert mine >= r.max() * (1 - BAND), f"{where}: token {tok} ratio {mine} vs best {r.max()}"
    if idx is not None:
        n = info.n
        assert np.array_equal(idx[:n], order[:n]), f"{where}: logits_idx differs"
        assert (idx[n:] == -1).all(), f"{where}: logits_idx past n"
        m = min(n_kept_g, n_kept_o)
        np.testing.assert_allclose(sm[:m], info.prob32[:m], rtol=PROB_RTOL, atol=1e-12, err_msg=where)
        hi = max(n_kept_g, n_kept_o)
        fill = np.float32(0.0) if (info.minp_ran or not logits) else np.float32(-np.inf)
        assert np.array_equal(sm[hi:].view(np.uint32), np.full(V - hi, fill, np.float32).view(np.uint32)), \
            f"{where}: removed positions hold the wrong value"
    return flips


def _rows(rng, B, V, dt, logits, kind):
    if logits:
        if kind == "ties":
            x = (rng.integers(-6, 7, size=(B, V)) * 0.5).astype(np.float32)
        else:
            x = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    else:
        # probabilities in (0, 1), summing to 1 in exact arithmetic only approximately
        w = rng.random((B, V)) + 0.01
        x = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return np.stack([to_raw(r, dt) for r in x])


@pytest.mark.parametrize("dt", ("f32", "f16", "bf16"))
@pytest.mark.parametrize("V", [1, 7, 1000, 5003])
@pytest.mark.parametrize("logits", [True, False])
def test_small_rows(tk, dt, V, logits):
    rng = np.random.default_rng(V * 3 + (7 if logits else 1))
    B = 12
    for kind in ("normal", "ties"):
        x = _rows(rng, B, V, dt, logits, kind)
        for ks_max in (8, 13, 1024):
            ka = min(1024, (ks_max + 7) // 8 * 8)
            kc = [-1, 0, 1, 2, 5, ka, ka + 1, V, max(1, V - 1), 1024, int(rng.integers(1, max(2, V))), 3]
            k = np.array(kc[:B], dtype=np.int32)
            p = np.array([0.0, 0.5, 0.9, 1.0, 0.999, 0.3, 0.7, 0.95, 0.1, 0.6, 0.8, 0.99], dtype=np.float32)[:B]
            mp = np.array([0.0, 0.05, 0.3, 1.0, 0.0, 0.01, 0.2, 0.0, 0.5, 0.02, 0.0, 0.1], dtype=np.float32)[:B]
            q = rng.exponential(1.0, size=(B, V)).astype(np.float32)
            for args in ((k, p, mp, q), (k, None, None, None), (None, p, mp, q), (k, p, None, None)):
                ka_, pa, ma, qa = args
                tok, sel = _run(tk, x, dt, ka_, pa, ma, qa, ks_max, logits, False)
                idx, sm = _run(tk, x, dt, ka_, pa, ma, qa, ks_max, logits, True)
                for b in range(B):
                    _, _, _, _, info = OV.v2_row(x[b], dt, None if ka_ is None else int(ka_[b]),
                                                 None if pa is None else pa[b], None if ma is None else ma[b],
                                                 None if qa is None else qa[b], EPS, ks_max, logits)
                    where = f"{dt} V={V} logits={logits} {kind} ks_max={ks_max} row {b}"
                    _check_row(x[b], dt, info, sel[b], int(tok[b]), None, None, None if qa is None else qa[b],
                               logits, where)
                    _check_row(x[b], dt, info, None, None, idx[b], sm[b], None, logits, where + " (sorted)")


def test_decode_batch_full_size(tk):
    """B=64 x V=152064 bf16 logits 2*N(0,1): k ~ U{1..1024} with 10% of the
    rows at 0 (top-k skipped), p ~ U[0.5, 1], min_p ~ U[0, 0.2], q ~ Exp(1),
    ks_max = 1024; every row against the oracle, both output modes."""
    rng = np.random.default_rng(2026)
    B, V, dt = 64, 152064, "bf16"
    x = to_raw((rng.standard_normal((B, V)) * 2).astype(np.float32).ravel(), dt).reshape(B, V)
    k = rng.integers(1, 1025, size=B).astype(np.int32)
    k[rng.random(B) < 0.1] = 0
    p = rng.uniform(0.5, 1.0, size=B).astype(np.float32)
    mp = rng.uniform(0.0, 0.2, size=B).astype(np.float32)
    q = rng.exponential(1.0, size=(B, V)).astype(np.float32)
    tok, sel = _run(tk, x, dt, k, p, mp, q, 1024, True, False)
    idx, sm = _run(tk, x, dt, k, p, mp, q, 1024, True, True)
    flips = 0
    for b in range(B):
        _, _, _, _, info = OV.v2_row(x[b], dt, int(k[b]), p[b], mp[b], q[b], EPS, 1024, True)
        flips += _check_row(x[b], dt, info, sel[b], int(tok[b]), None, None, q[b], True, f"full row {b}")
        _check_row(x[b], dt, info, None, None, idx[b], sm[b], None, True, f"full row {b} (sorted)")
    flipstats.record("V2 semantics, B=64 x V=152064 bf16", B, flips, "top-p / min-p decisions inside the band")
