"""CPU oracle for the fused top-k / top-p logit filter -- TEST INFRASTRUCTURE ONLY.

This module is the plain, slow, obviously-correct statement of what the filter
computes.  Only the test suite, the smoke check and the CPU-baseline leg of the
benchmark may import it; the library itself never does, and it shares no code
with the CUDA path.

Source.  "[guide]" below is the web page "CANN ops-nn 算子实战：
ApplyTopKTopPWithSorted 的 top-k/top-p 采样过滤原理与 aclnn 调用指南"; its
numbered sections are cited as §1..§10 (§2 = 计算流程与公式, the eight-step
formula and the golden PyTorch transcription; §3 = 参数说明; §4 = 约束说明;
§6 = 源码级原理剖析).

Readings where the page is silent or garbled (each one is listed again in the
design notes with its reason):

  R1  Step 8 is printed as a gather but the golden code scatters
      (``scatter_(dim=-1, index=logits_idx, src=logits_sort)``): the oracle
      scatters, out[idx[j]] = s[j].
  R2  The comparison operators were lost in extraction.  Top-k masks values
      strictly below the k-th largest (the text says 严格小于); top-p masks
      positions whose cumulative probability is <= 1-p (the text says 小于等于).
  R3  k <= 0 or k >= V disables top-k for that row (§4, stated for the aclnn
      interface); the same rule is applied to the pre-sorted entry point.
  R4  The page fixes the precision of the softmax and cumsum *outputs* (fp32:
      ``.to(torch.float32).softmax`` then ``cumsum``) but not how they are
      accumulated.  Each output is taken as the exact value rounded once to
      fp32: q_j = fp32(e_j / S) and C_j = fp32(sum_{i<=j} q_i), both formed
      in fp64.  (A sequential fp32 accumulation over 1e5 terms drifts by
      ~2e-5, larger than the 1e-5 tolerance band the parity tests use.)
  R5  ``1 - p`` is evaluated on a p tensor of the logits dtype (§3 says p has
      the logits dtype), so the threshold is round_D(fp32(1 - p)) compared
      against the fp32 cumsum.
  R6  Inputs are finite; p lies in [0, 1]; NaN / inf logits are undefined.

Every floating-point value is decoded exactly to fp64 before it is compared,
so the sort, the top-k threshold and the top-k mask are exact.
"""

from __future__ import annotations

import numpy as np

# dtype names accepted by the oracle: raw arrays are np.float32, np.float16 or
# np.uint16 holding bfloat16 bit patterns.
F32, F16, BF16 = "f32", "f16", "bf16"

_NEG_INF_BITS = {F32: np.uint32(0xFF800000), F16: np.uint16(0xFC00), BF16: np.uint16(0xFF80)}


# ---------------------------------------------------------------- dtype codec
def decode(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 values of a raw dtype array (bf16 = upper half of an fp32)."""
    if dtype == F32:
        return np.asarray(raw, dtype=np.float32).astype(np.float64)
    if dtype == F16:
        return np.asarray(raw, dtype=np.float16).astype(np.float64)
    if dtype == BF16:
        bits = np.asarray(raw, dtype=np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def round_to_dtype_f32(v: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 values to dtype D (round-to-nearest-even), returned as fp32."""
    v = np.asarray(v, dtype=np.float32)
    if dtype == F32:
        return v
    if dtype == F16:
        return v.astype(np.float16).astype(np.float32)
    if dtype == BF16:
        u = v.view(np.uint32).astype(np.uint64)
        lsb = (u >> 16) & 1
        r = ((u + 0x7FFF + lsb) >> 16) & 0xFFFF
        return (r.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


def neg_inf_bits(dtype: str):
    return _NEG_INF_BITS[dtype]


def raw_bits(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Bit patterns of a raw array as unsigned ints (for bit-exact comparison)."""
    if dtype == F32:
        return np.asarray(raw, dtype=np.float32).view(np.uint32)
    if dtype == F16:
        return np.asarray(raw, dtype=np.float16).view(np.uint16)
    return np.asarray(raw, dtype=np.uint16)


# ------------------------------------------------------------------ the steps
def topk_enabled(k: int | None, V: int) -> bool:
    """[guide] §4: k <= 0 or k >= V means no top-k filtering (reading R3)."""
    return k is not None and 1 <= int(k) <= V - 1


def top_p_threshold(p_raw, dtype: str) -> np.float32:
    """round_D(fp32(1 - p)) as fp32 -- the golden code's ``1 - p`` on a p
    tensor of the logits dtype ([guide] §2 golden code, §3; reading R5)."""
    p32 = np.float32(decode(np.asarray([p_raw]), dtype)[0])
    one_minus = np.float32(np.float32(1.0) - p32)
    return np.float32(round_to_dtype_f32(np.asarray([one_minus]), dtype)[0])


def stable_ascending_sort(x: np.ndarray):
    """Step 0 of the aclnn path ([guide] §6.1: l0op::Sort(..., descending=false,
    stable=true)): ascending by value, equal values keep index order.  -0 and
    +0 compare equal, so they too keep index order."""
    idx = np.argsort(x, kind="stable")
    return x[idx], idx


def filter_sorted_row(s: np.ndarray, V: int, k: int | None, thr: np.float32 | None):
    """Steps 1-7 of [guide] §2 on one ascending row s (fp64 values).

    Returns (kept, C): kept[j] says whether sorted position j survives, and C
    is the fp32 cumulative probability (None when top-p is off)."""
    kept = np.ones(V, dtype=bool)
    vals = s.copy()
    # Steps 1-3: k-th largest is s[V-k]; strictly smaller values become -inf.
    if topk_enabled(k, V):
        kth_value = s[V - int(k)]
        topk_mask = s < kth_value
        kept &= ~topk_mask
        vals[topk_mask] = -np.inf
    C = None
    if thr is not None:
        # Step 4: fp32 softmax over the filtered row (reading R4: each output
        # is the fp64 value rounded once to fp32).
        m = vals[V - 1]
        e = np.exp(vals - m)            # exp(-inf) = 0
        q = (e / e.sum()).astype(np.float32)
        # Step 5: ascending cumulative sum, fp32 outputs (reading R4).
        C = np.cumsum(q.astype(np.float64)).astype(np.float32)
        # Step 6: mask C <= 1-p, except that the last position never masks.
        topp_mask = C <= thr
        topp_mask[V - 1] = False
        # Step 7.
        kept &= ~topp_mask
    return kept, C


def topk_survivors(s: np.ndarray, V: int, k: int | None) -> np.ndarray:
    """Sorted positions that survive steps 1-3 alone (reported to the tests,
    which must tell a top-k difference -- never allowed -- from a top-p one)."""
    if not topk_enabled(k, V):
        return np.ones(V, dtype=bool)
    return ~(s < s[V - int(k)])


def scatter_back(raw_sorted_bits: np.ndarray, idx: np.ndarray, kept: np.ndarray, dtype: str):
    """Step 8 ([guide] §2 golden ``scatter_``; reading R1): out[idx[j]] is the
    sorted element's bits if kept, else the dtype's -inf."""
    V = idx.shape[0]
    src = np.where(kept, raw_sorted_bits, neg_inf_bits(dtype))
    out = np.empty(V, dtype=raw_sorted_bits.dtype)
    out[idx] = src
    return out


# --------------------------------------------------------------- entry points
class RowInfo:
    """Per-row intermediate results, kept for the tests' tolerance checks."""

    __slots__ = ("idx", "kept", "C", "thr", "topk_kept")

    def __init__(self, idx, kept, C, thr, topk_kept=None):
        self.idx, self.kept, self.C, self.thr, self.topk_kept = idx, kept, C, thr, topk_kept


def _bits_to_raw(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == F32:
        return bits.view(np.float32)
    if dtype == F16:
        return bits.view(np.float16)
    return bits


def apply_row(x_raw: np.ndarray, dtype: str, p_raw=None, k=None):
    """One row of aclnnApplyTopKTopP ([guide] §2 and §6.1): sort internally,
    filter, scatter back.  Returns (out_raw, RowInfo)."""
    V = int(x_raw.shape[0])
    bits = raw_bits(x_raw, dtype)
    vals = decode(x_raw, dtype)
    s, idx = stable_ascending_sort(vals)
    thr = None if p_raw is None else top_p_threshold(p_raw, dtype)
    kept, C = filter_sorted_row(s, V, k, thr)
    out_bits = scatter_back(bits[idx], idx, kept, dtype)
    return _bits_to_raw(out_bits, dtype), RowInfo(idx, kept, C, thr, topk_survivors(s, V, k))


def apply_sorted_row(sv_raw: np.ndarray, si: np.ndarray, dtype: str, p_raw=None, k=None):
    """One row of ApplyTopKTopPWithSorted ([guide] §2, §3): the input is already
    ascending; step 8 scatters through sorted_indices.  When logits are also
    given, the page's contract is that sorted_value is their stable sort, so
    the result is the same scatter."""
    V = int(sv_raw.shape[0])
    s = decode(sv_raw, dtype)
    idx = np.asarray(si, dtype=np.int64)
    thr = None if p_raw is None else top_p_threshold(p_raw, dtype)
    kept, C = filter_sorted_row(s, V, k, thr)
    out_bits = scatter_back(raw_bits(sv_raw, dtype), idx, kept, dtype)
    return _bits_to_raw(out_bits, dtype), RowInfo(idx, kept, C, thr, topk_survivors(s, V, k))


def apply(x_raw: np.ndarray, dtype: str, p_raw=None, k=None, rows=None):
    """Batched aclnnApplyTopKTopP over a [B, V] raw array.  ``rows`` restricts
    the work to a subset of row numbers (the others are returned as zeros).
    Returns (out_raw, {row: RowInfo})."""
    x_raw = np.asarray(x_raw)
    B = x_raw.shape[0]
    out = np.zeros_like(x_raw)
    infos = {}
    for b in (range(B) if rows is None else rows):
        pb = None if p_raw is None else p_raw[b]
        kb = None if k is None else int(k[b])
        out[b], infos[b] = apply_row(x_raw[b], dtype, pb, kb)
    return out, infos


def apply_sorted(sv_raw, si, dtype, p_raw=None, k=None, rows=None):
    """Batched ApplyTopKTopPWithSorted over [B, V] arrays."""
    sv_raw = np.asarray(sv_raw)
    B = sv_raw.shape[0]
    out = np.zeros_like(sv_raw)
    infos = {}
    for b in (range(B) if rows is None else rows):
        pb = None if p_raw is None else p_raw[b]
        kb = None if k is None else int(k[b])
        out[b], infos[b] = apply_sorted_row(sv_raw[b], si[b], dtype, pb, kb)
    return out, infos


# ------------------------------------------ post-filter stage: min-p and sampling
# "[V2]" is the page "aclnnTopKTopPSampleV2" (CANN community edition API
# reference), cited by its headings: "Formula / minP sampling" and
# "Formula / Subsequent processing" (its None and QSample modes), plus
# "Constraints".  That operator runs top-k, top-p, min-p and the sample in
# one call on a sorted row; this stage takes the filter's output instead
# (original order, masked elements -inf) and applies the last two steps.
#
# Readings (listed again in the design notes):
#   S1  The probabilities are the softmax over the filter's survivors.  [V2]
#       forms them over the top-k survivors before the top-p mask; min-p
#       (probs < max_prob * minP) and the sample (argmax of probs / (q +
#       eps)) compare ratios of probabilities, in which the normaliser
#       cancels, so the choice of normaliser changes no decision.
#   S2  minP <= 0 skips min-p; minP >= 1 keeps the one element of largest
#       value ([V2] Formula / minP sampling, "in other cases"); among equal
#       largest values, the one that comes last in the stable ascending order
#       (the largest index) -- the position the top-p step never masks.
#   S3  q is one fp32 variate per element in original index order ([V2]
#       Constraints: q has the logits' shape); [V2] indexes it by sorted
#       position, which this stage does not have.
#   S4  ArgMax ties go to the element that comes last in the stable
#       ascending order (the largest index among equal values), so that
#       the None mode returns the element the filter always keeps.
#   S5  eps is not given a value by [V2]; it is an argument here.
#   S6  Probabilities, thresholds and ratios are formed in fp64 from the
#       exactly decoded inputs (q and eps as fp32 values).


class SampleInfo:
    """Per-row intermediates of the sample stage, for the tests' tolerances."""

    __slots__ = ("alive", "e", "keep", "ratio", "min_p", "last")

    def __init__(self, alive, e, keep, ratio, min_p, last):
        self.alive, self.e, self.keep, self.ratio, self.min_p, self.last = alive, e, keep, ratio, min_p, last


def survivor_probs(vals: np.ndarray):
    """Softmax over the filter's survivors (S1).  Returns (alive, last, e,
    probs): alive marks the elements that are not -inf, last is the index
    of the largest value that comes last in the stable ascending order (S2,
    S4), e = exp(x - max) and probs = e / sum(e), both fp64."""
    alive = vals != -np.inf
    m = vals[alive].max()
    last = int(np.flatnonzero(alive & (vals == m))[-1])
    e = np.where(alive, np.exp(np.where(alive, vals - m, 0.0)), 0.0)
    return alive, last, e, e / e.sum()


def min_p_keep(alive: np.ndarray, probs: np.ndarray, last: int, mp):
    """[V2] Formula / minP sampling: minPThd = max(probs) * minP, and
    elements with probs < minPThd are removed; minP <= 0 skips the step and
    minP >= 1 keeps the largest element alone (S2)."""
    if mp is None or not (mp > 0.0):
        return alive.copy()
    if mp >= 1.0:
        keep = np.zeros(alive.shape[0], dtype=bool)
        keep[last] = True
        return keep
    thd = probs[last] * mp
    return alive & ~(probs < thd)


def sample_token(probs: np.ndarray, keep: np.ndarray, last: int, q, eps: float):
    """[V2] Formula / Subsequent processing.  None mode (q None): ArgMax of
    the probabilities, i.e. the largest element (S4).  QSample mode: ArgMax of
    probs / (q + eps) over the kept elements, ties to the largest index.
    Returns (token, ratio)."""
    if q is None:
        return last, None
    qv = np.asarray(q, dtype=np.float32).astype(np.float64)
    ratio = np.where(keep, probs / (qv + float(np.float32(eps))), -np.inf)
    return int(np.flatnonzero(ratio == ratio.max())[-1]), ratio


def sample_row(f_raw: np.ndarray, dtype: str, min_p=None, q=None, eps: float = 1e-10):
    """Min-p and the sample on one filtered row (readings S1-S6).

    Returns (out_raw, token, SampleInfo).  out_raw is the row with the
    elements that min-p removes set to -inf; token is the original index
    chosen by ArgMax of the probabilities (q None, [V2] Subsequent
    processing / None) or of probs / (q + eps) (QSample).  A row without a
    finite element (outside the filter's contract) is returned unchanged
    with token -1."""
    V = int(f_raw.shape[0])
    bits = raw_bits(f_raw, dtype)
    vals = decode(f_raw, dtype)
    if not (vals != -np.inf).any():
        return _bits_to_raw(bits.copy(), dtype), -1, SampleInfo(vals != -np.inf, np.zeros(V), vals != -np.inf,
                                                                None, None, -1)
    alive, last, e, probs = survivor_probs(vals)
    mp = None if min_p is None else float(np.float32(min_p))
    keep = min_p_keep(alive, probs, last, mp)
    out_bits = np.where(keep, bits, neg_inf_bits(dtype)).astype(bits.dtype)
    token, ratio = sample_token(probs, keep, last, q, eps)
    return _bits_to_raw(out_bits, dtype), token, SampleInfo(alive, e, keep, ratio, mp, last)


def sample(f_raw, dtype, min_p=None, q=None, eps: float = 1e-10, rows=None):
    """Batched sample stage over [B, V]; min_p is [B] fp32 or None, q is
    [B, V] fp32 or None.  Returns (out_raw, tokens, {row: SampleInfo})."""
    f_raw = np.asarray(f_raw)
    B = f_raw.shape[0]
    out = np.zeros_like(f_raw)
    tokens = np.full(B, -1, dtype=np.int64)
    infos = {}
    for b in (range(B) if rows is None else rows):
        mp = None if min_p is None else min_p[b]
        qb = None if q is None else q[b]
        out[b], tokens[b], infos[b] = sample_row(f_raw[b], dtype, mp, qb, eps)
    return out, tokens, infos
