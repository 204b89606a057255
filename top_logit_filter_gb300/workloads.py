"""Seeded synthetic inputs for the top-k / top-p filter.

These generators serve both the CUDA path (tests, benchmark) and the CPU
oracle, so they hold none of the filter's arithmetic: they draw random numbers
and cast them to the storage dtype, nothing else.  The one exception to "no
sort" is the pre-sorted workload, whose *input* is by definition the stable
ascending sort of a logits row (the page's ApplyTopKTopPWithSorted contract:
sorted_value ascending, sorted_indices the matching int32 positions).

Raw arrays: fp32 -> np.float32, fp16 -> np.float16, bf16 -> np.uint16 bit
patterns (numpy has no bfloat16).

The five workloads mirror decode-time logits of common LLM vocabularies:

  1  apply, joint top-k + top-p   B=4    V=1024    fp32  3*N(0,1)
  2  apply, top-p only            B=64   V=32000   fp16  2.5*N(0,1), 20 tokens/row +8
  3  apply, joint top-k + top-p   B=256  V=128256  bf16  2*N(0,1)
  4  apply, top-k only            B=1024 V=151936  fp32  N(0,1)/T, T~U[0.3,1.5]
  5  apply_sorted (+logits)       B=512  V=152064  bf16  2*N(0,1)/0.3, pre-sorted
"""

from __future__ import annotations

import numpy as np

WORKLOADS = {
    1: dict(name="apply_joint_B4_V1024_f32", B=4, V=1024, dtype="f32", call="apply", topk=True, topp=True),
    2: dict(name="apply_topp_B64_V32000_f16", B=64, V=32000, dtype="f16", call="apply", topk=False, topp=True),
    3: dict(name="apply_joint_B256_V128256_bf16", B=256, V=128256, dtype="bf16", call="apply", topk=True, topp=True),
    4: dict(name="apply_topk_B1024_V151936_f32", B=1024, V=151936, dtype="f32", call="apply", topk=True, topp=False),
    5: dict(name="apply_sorted_B512_V152064_bf16", B=512, V=152064, dtype="bf16", call="apply_sorted", topk=True, topp=True),
}

SEED_BASE = 20260


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Cast fp32 to bfloat16 bit patterns, round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF).astype(np.uint16)


def cast(v: np.ndarray, dtype: str) -> np.ndarray:
    v = np.asarray(v, dtype=np.float32)
    if dtype == "f32":
        return v
    if dtype == "f16":
        return v.astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16_bits(v)
    raise ValueError(dtype)


def _pick_rows(rng, B: int, frac: float) -> np.ndarray:
    n = int(np.floor(frac * B + 0.5))
    return rng.choice(B, size=n, replace=False) if n else np.zeros(0, dtype=np.int64)


def make(wl: int, B: int | None = None, V: int | None = None, seed: int | None = None) -> dict:
    """Inputs of workload ``wl`` (1..5).  B and V may be shrunk for quick tests;
    the value distributions and the k / p recipes stay the same."""
    spec = WORKLOADS[wl]
    B = spec["B"] if B is None else int(B)
    V = spec["V"] if V is None else int(V)
    dt = spec["dtype"]
    rng = np.random.default_rng(SEED_BASE + wl if seed is None else seed)
    out = dict(wl=wl, name=spec["name"], B=B, V=V, dtype=dt, call=spec["call"])

    if wl == 1:
        x = 3.0 * rng.standard_normal((B, V), dtype=np.float32)
        k = np.resize(np.array([1, 10, 0, 2000], dtype=np.int32), B)
        p = np.resize(np.array([0.9, 0.5, 1.0, 0.0], dtype=np.float32), B)
    elif wl == 2:
        x = 2.5 * rng.standard_normal((B, V), dtype=np.float32)
        for b in range(B):
            hot = rng.choice(V, size=min(20, V), replace=False)
            x[b, hot] += 8.0
        k = None
        p = rng.uniform(0.8, 0.99, size=B).astype(np.float32)
    elif wl == 3:
        x = 2.0 * rng.standard_normal((B, V), dtype=np.float32)
        k = rng.integers(1, 1025, size=B, dtype=np.int32)
        k[_pick_rows(rng, B, 0.10)] = 0
        p = rng.uniform(0.5, 1.0, size=B).astype(np.float32)
        p[_pick_rows(rng, B, 0.05)] = 1.0
    elif wl == 4:
        x = rng.standard_normal((B, V), dtype=np.float32)
        temp = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
        x /= temp[:, None]
        k = rng.integers(1, 65, size=B, dtype=np.int32)
        p = None
    elif wl == 5:
        x = 2.0 * rng.standard_normal((B, V), dtype=np.float32) / np.float32(0.3)
        k = rng.integers(1, 1025, size=B, dtype=np.int32)
        p = rng.uniform(0.1, 0.95, size=B).astype(np.float32)
    else:
        raise ValueError(wl)

    xr = cast(x, dt)
    out["x"] = xr
    out["k"] = None if k is None else np.ascontiguousarray(k, dtype=np.int32)
    out["p"] = None if p is None else cast(p, dt)
    if spec["call"] == "apply_sorted":
        out["sorted_value"], out["sorted_indices"] = presort(xr, dt)
    return out


def _as_sortable(xr: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return (xr.astype(np.uint32) << 16).view(np.float32)
    return xr


def presort(xr: np.ndarray, dtype: str):
    """Input preparation for the pre-sorted entry point: per row, the stable
    ascending order of the logits and the int32 positions it came from."""
    keyv = _as_sortable(xr, dtype)
    idx = np.argsort(keyv, axis=-1, kind="stable")
    sv = np.take_along_axis(xr, idx, axis=-1)
    return np.ascontiguousarray(sv), np.ascontiguousarray(idx.astype(np.int32))


def make_filtered(B: int, V: int, dtype: str, seed: int, scale: float = 2.0, empty_rows: int = 0) -> dict:
    """Inputs of the post-filter stage (min-p and the sample): rows as a
    filter leaves them.  Logits are scale*N(0,1) cast to dtype; every value
    below a per-row cut drawn from U[0, 2*scale] becomes -inf (the last
    ``empty_rows`` rows are all -inf).  min_p is U[0.001, 0.3] per row with
    10% of rows 0 (min-p off) and 5% at 1.0; q holds Exp(1) variates (fp32).
    Nothing here computes the stage itself."""
    rng = np.random.default_rng(seed)
    x = scale * rng.standard_normal((B, V), dtype=np.float32)
    cut = rng.uniform(0.0, 2.0 * scale, size=B).astype(np.float32)
    x = np.where(x >= cut[:, None], x, np.float32(-np.inf)).astype(np.float32)
    if empty_rows:
        x[B - empty_rows:] = -np.inf
    min_p = rng.uniform(0.001, 0.3, size=B).astype(np.float32)
    min_p[_pick_rows(rng, B, 0.10)] = 0.0
    min_p[_pick_rows(rng, B, 0.05)] = 1.0
    q = rng.exponential(1.0, size=(B, V)).astype(np.float32)
    return dict(B=B, V=V, dtype=dtype, x=cast(x, dtype), min_p=min_p, q=q)
