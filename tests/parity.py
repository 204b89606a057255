"""Parity checks of GPU output against the oracle's per-row results.

The bar: every output element is bit-identical to the oracle's, except a
top-p decision at a sorted position whose oracle cumulative probability lies
within BAND of round_D(1 - p); such flips are counted and returned.  Top-k
decisions must match exactly."""
import numpy as np

from rawutil import NEG_INF, bits

BAND = 1e-5


def compare_row(out_raw, x_raw, info, dtype, band=BAND, where=""):
    ob, xb = bits(out_raw, dtype), bits(x_raw, dtype)
    neg = NEG_INF[dtype]
    bad = ~((ob == xb) | (ob == neg))
    assert not bad.any(), f"{where}: output is neither the input nor -inf at {np.nonzero(bad)[0][:8]}"
    gk = ob[info.idx] != neg              # GPU survivors, in stable sorted order
    diff = np.nonzero(gk != info.kept)[0]
    if diff.size == 0:
        return 0
    topk_err = gk[diff] & ~info.topk_kept[diff]
    assert not topk_err.any(), f"{where}: kept a value below the k-th largest at sorted {diff[topk_err][:8]}"
    assert info.C is not None, f"{where}: top-k-only row differs at sorted positions {diff[:8]}"
    dist = np.abs(info.C[diff].astype(np.float64) - float(info.thr))
    assert (dist <= band).all(), (
        f"{where}: top-p flip outside the band at sorted {diff[dist > band][:8]}, "
        f"C={info.C[diff[dist > band]][:4]}, thr={info.thr}")
    return int(diff.size)
