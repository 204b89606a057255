"""CPU oracle of the TopKTopPSampleV2 semantics -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this module; the library never does, and it shares no code with the
CUDA path.

Source.  "[V2]" is the API reference page "aclnnTopKTopPSampleV2" (CANN
community edition), cited by its headings: "Formula / TopK sampling",
"Formula / TopP sampling", "Formula / minP sampling", "Formula / Optional
output", "Formula / Subsequent processing" and "Constraints".  Per row it
runs, on the row sorted from the largest value down, a top-k stage, a
top-p stage, a min-p stage and a sample, and reports either the sampled
index and the filtered row in original order, or the sorted, masked
probabilities and their original indices.

Parts of the extracted page are lost (its tables, the p-strategy rules, the
GuessK definition, defaults, output dtypes).  The readings below fill them;
each is listed again in the design notes.

  V1  Sort order.  The stages run on the row in descending order of value;
      equal values keep increasing original index (a stable descending
      sort).  [V2] names the order only as "sort(..., descendant)".
  V2  ks_max is an argument in [1, 1024], rounded up to a multiple of 8
      ([V2] TopK sampling: "must be rounded up to a multiple of 8"; its
      default is lost).  Top-k runs iff 1 <= k <= min(V, ks_max aligned)
      ([V2] TopK sampling, valid range; Constraints: k <= 0, or k above the
      aligned ks_max, skips the stage).  When it runs it keeps exactly the
      first k positions of the sorted row (Card(topKValue) = topK).
  V3  Probabilities.  With input_is_logits, the softmax over the top-k
      survivors (all V positions when top-k is skipped); otherwise the
      input values themselves ([V2] TopP sampling).  Each probability is the
      exact value rounded once to fp32.
  V4  Top-p runs iff p < 1 ([V2] Constraints: p >= 1 skips it); p is fp32.
      After a top-k stage, position j stays iff the probabilities of the
      positions before it sum to <= p ([V2] TopP sampling, first form).
      When top-k was skipped, position j stays iff the probabilities of j
      and every position after it sum to > fp32(1 - p) ([V2] TopP sampling,
      second form, "probSum <= 1 - p" masked).  Sums are exact over the fp32
      probabilities.  The GuessK shortcut of that form only saves work when
      the first GuessK positions already hold mass p: it is read as giving
      the same kept set, so it has no separate step here.  Position 0 (the
      largest value) always stays, as the min-p stage's "one token" rule
      keeps it too.
  V5  Min-p ([V2] minP sampling): min_p <= 0 skips it; 0 < min_p < 1 keeps
      the positions whose probability is >= prob[0] * min_p (in fp64 from
      the fp32 values); min_p >= 1 keeps position 0 alone.
  V6  The kept positions form a prefix of the sorted row (each stage keeps
      a prefix); n_kept is its length.
  V7  The sample ([V2] Subsequent processing): without q, the index of
      position 0 (ArgMax of probs, first on ties); with q (fp32, indexed by
      sorted position, q[b, :n_kept]), the original index of the kept
      position with the largest prob / (q + eps), the first one on ties.
  V8  Outputs ([V2] Optional output, Subsequent processing).  The filtered
      row in original order holds the input element where its position was
      kept and defLogit elsewhere: -inf with input_is_logits, else 0.
      The intermediate outputs are V long: logits_idx[j] is the original
      index of sorted position j for j < n (n = k after a top-k stage, V
      otherwise) and -1 past n; sort_masked[j] is the fp32 probability of a
      kept position; a position not kept holds 0 when min-p ran and defLogit
      when it did not (the page zeroes what the min-p mask removed, and
      every removed position is below the min-p threshold).
"""

from __future__ import annotations

import numpy as np

from .oracle import decode, raw_bits, neg_inf_bits


def ks_max_aligned(ks_max: int) -> int:
    """ks_max rounded up to a multiple of 8, at most 1024 (reading V2)."""
    ks = int(ks_max)
    if not 1 <= ks <= 1024:
        raise ValueError("ks_max must lie in [1, 1024]")
    return min(1024, (ks + 7) // 8 * 8)


def topk_runs(k, V: int, ks_max: int) -> bool:
    """[V2] TopK sampling valid range (reading V2)."""
    return k is not None and 1 <= int(k) <= min(V, ks_max_aligned(ks_max))


def stable_descending_order(vals: np.ndarray) -> np.ndarray:
    """Indices of the row from the largest value down; equal values keep
    increasing index (reading V1).  -0 and +0 compare equal."""
    # a stable ascending sort of the negated values keeps index order on ties
    return np.argsort(-vals, kind="stable")


class V2Info:
    __slots__ = ("order", "n", "topk", "prob32", "n_topp", "n_kept", "minp_ran", "token", "ratio",
                 "topp_stat", "minp_stat", "thd")

    def __init__(self, **kw):
        for k, v in kw.items():
            setattr(self, k, v)


def v2_row(x_raw: np.ndarray, dtype: str, k=None, p=None, min_p=None, q=None, eps: float = 1e-10,
           ks_max: int = 1024, input_is_logits: bool = True):
    """One row of the TopKTopPSampleV2 semantics (readings V1-V8).

    Returns (select_raw, token, logits_idx, sort_masked, V2Info):
    select_raw is the filtered row in original order (dtype bits), token the
    sampled original index, logits_idx (int64, V) and sort_masked (float32,
    V) the intermediate outputs."""
    V = int(x_raw.shape[0])
    bits = raw_bits(x_raw, dtype)
    vals = decode(x_raw, dtype)
    order = stable_descending_order(vals)
    s = vals[order]
    topk = topk_runs(k, V, ks_max)
    n = int(k) if topk else V                  # sorted positions that exist after top-k
    # probabilities over the positions that exist (reading V3)
    if input_is_logits:
        e = np.exp(s[:n] - s[0])
        prob32 = (e / e.sum()).astype(np.float32)
    else:
        prob32 = s[:n].astype(np.float32)
    pr = prob32.astype(np.float64)
    # top-p (reading V4): a prefix of length n_topp
    n_topp = n
    topp_stat = None
    if p is not None and float(np.float32(p)) < 1.0:
        p32 = float(np.float32(p))
        if topk:
            before = np.concatenate([[0.0], np.cumsum(pr)[:-1]])      # mass before position j
            keep = before <= p32
            topp_stat = (before, p32)
        else:
            after = np.cumsum(pr[::-1])[::-1]                          # mass of j and every later position
            thr = float(np.float32(np.float32(1.0) - np.float32(p32)))
            keep = after > thr
            topp_stat = (after, thr)
        keep[0] = True
        n_topp = int(np.argmin(keep)) if not keep.all() else n
    # min-p (reading V5)
    n_kept = n_topp
    minp_ran = min_p is not None and float(np.float32(min_p)) > 0.0
    thd = None
    if minp_ran:
        mp = float(np.float32(min_p))
        if mp >= 1.0:
            n_kept = 1
        else:
            thd = pr[0] * mp
            n_kept = int(np.count_nonzero(pr[:n_topp] >= thd))
    n_kept = max(1, n_kept)
    # the sample (reading V7)
    ratio = None
    if q is None:
        tok = 0
    else:
        qv = np.asarray(q, dtype=np.float32).astype(np.float64)[:n_kept]
        ratio = pr[:n_kept] / (qv + float(np.float32(eps)))
        tok = int(np.argmax(ratio))
    token = int(order[tok])
    # outputs (reading V8)
    def_bits = neg_inf_bits(dtype) if input_is_logits else bits.dtype.type(0)
    sel = np.full(V, def_bits, dtype=bits.dtype)
    sel[order[:n_kept]] = bits[order[:n_kept]]
    logits_idx = np.full(V, -1, dtype=np.int64)
    logits_idx[:n] = order[:n]
    fill = np.float32(0.0) if (minp_ran or not input_is_logits) else np.float32(-np.inf)
    sort_masked = np.full(V, fill, dtype=np.float32)
    sort_masked[:n_kept] = prob32[:n_kept]
    info = V2Info(order=order, n=n, topk=topk, prob32=prob32, n_topp=n_topp, n_kept=n_kept, minp_ran=minp_ran,
                  token=token, ratio=ratio, topp_stat=topp_stat, minp_stat=None, thd=thd)
    if dtype == "f32":
        sel_raw = sel.view(np.float32)
    elif dtype == "f16":
        sel_raw = sel.view(np.float16)
    else:
        sel_raw = sel
    return sel_raw, token, logits_idx, sort_masked, info


def v2(x_raw, dtype, k=None, p=None, min_p=None, q=None, eps: float = 1e-10, ks_max: int = 1024,
       input_is_logits: bool = True, rows=None):
    """Batched form over [B, V]; k [B] int, p [B] fp32, min_p [B] fp32, q
    [B, V] fp32, each optional.  Returns (select, tokens, logits_idx,
    sort_masked, {row: V2Info})."""
    x_raw = np.asarray(x_raw)
    B, V = x_raw.shape
    select = np.zeros_like(x_raw)
    tokens = np.full(B, -1, dtype=np.int64)
    idx = np.full((B, V), -1, dtype=np.int64)
    sm = np.zeros((B, V), dtype=np.float32)
    infos = {}
    for b in (range(B) if rows is None else rows):
        select[b], tokens[b], idx[b], sm[b], infos[b] = v2_row(
            x_raw[b], dtype, None if k is None else int(k[b]), None if p is None else p[b],
            None if min_p is None else min_p[b], None if q is None else q[b], eps, ks_max, input_is_logits)
    return select, tokens, idx, sm, infos
