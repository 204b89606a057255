"""GB300-native fused top-k / top-p logit filter.

Python face of libtopkp.so (include/topkp.h).  This module only marshals
arguments: every step of the filter runs in the library's CUDA kernels, and
there is no CPU path -- without the built library, or without a CUDA tensor,
the calls raise.

    out = apply(logits, p=None, k=None, out=None)
    out = apply_sorted(sorted_value, sorted_indices, p=None, k=None, logits=None, out=None)
    token, out = sample(filtered, min_p=None, q=None, eps=1e-10, out=None, want_out=True)
    sorted_value, sorted_indices = sort(logits)

Semantics: section 2 of the web page "CANN ops-nn 算子实战：
ApplyTopKTopPWithSorted 的 top-k/top-p 采样过滤原理与 aclnn 调用指南" --
per row, values strictly below the k-th largest become -inf, then sorted
positions whose fp32 cumulative softmax probability is <= 1-p become -inf
(never the largest), and every other element keeps its bits.  ``sample``
runs the min-p step and the sample of the page "aclnnTopKTopPSampleV2" on
such filtered rows.
"""
from __future__ import annotations

from . import _lib
from ._lib import (TOPKP_ERR_DEVICE_TIMEOUT, TOPKP_ERR_LAUNCH, TOPKP_ERR_PARAM_INVALID,  # noqa: F401
                   TOPKP_ERR_PARAM_NULLPTR, TOPKP_MAX_V, TOPKP_SUCCESS)


class TopKPError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[{status}] {message}")
        self.status = status


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    codes = {torch.float32: _lib.TOPKP_F32, torch.float16: _lib.TOPKP_F16, torch.bfloat16: _lib.TOPKP_BF16}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype} (float32, float16 or bfloat16)")
    return codes[t.dtype]


def _check(status: int):
    if status != _lib.TOPKP_SUCCESS:
        raise TopKPError(status, _lib.last_error())


# Address passed for a tensor that is present but empty (its data pointer can
# be NULL, which the C ABI reads as "absent"); empty problems return before
# any pointer is dereferenced.
_EMPTY = 16


def _ptr(t):
    if t is None:
        return None
    return t.data_ptr() or (_EMPTY if t.numel() == 0 else None)


def _stream(device):
    return _torch().cuda.current_stream(device).cuda_stream


def _vec(t, n, dtype, name, device):
    torch = _torch()
    if t is None:
        return None
    if not torch.is_tensor(t):
        t = torch.as_tensor(t, dtype=dtype, device=device)
    if t.device != device or t.dtype != dtype or t.dim() != 1 or t.shape[0] != n:
        raise ValueError(f"{name} must be a 1-D {dtype} tensor of length {n} on {device}")
    return t.contiguous()


def apply(logits, p=None, k=None, out=None):
    """aclnnApplyTopKTopP: filter a [B, V] CUDA tensor of logits.

    p: [B] tensor of the logits dtype (or None); k: [B] int32 (or None); at
    least one is required.  Rows may be strided along B (stride(1) must be
    1).  Returns ``out`` (allocated when None; may be ``logits`` itself)."""
    torch = _torch()
    lib = _lib.load()
    if not torch.is_tensor(logits) or logits.dim() != 2 or not logits.is_cuda:
        raise ValueError("logits must be a 2-D CUDA tensor")
    dt = _dtype_code(logits)
    if logits.stride(1) != 1:
        logits = logits.contiguous()
    B, V = logits.shape
    dev = logits.device
    p = _vec(p, B, logits.dtype, "p", dev)
    k = _vec(k, B, torch.int32, "k", dev)
    if out is None:
        out = torch.empty((B, V), dtype=logits.dtype, device=dev)
    if out.shape != logits.shape or out.dtype != logits.dtype or out.device != dev or out.stride(1) != 1:
        raise ValueError("out must match logits in shape, dtype and device, with stride(1) == 1")
    with torch.cuda.device(dev):
        _check(lib.topkp_apply(_ptr(logits), B, V, logits.stride(0) if B > 1 else V, dt, _ptr(p), _ptr(k),
                               _ptr(out), out.stride(0) if B > 1 else V, _stream(dev)))
    return out


def apply_sample(logits, p=None, k=None, min_p=None, q=None, eps: float = 1e-10, out=None, want_out: bool = True):
    """The filter and the sample in one pass (topkp_apply_sample): the same
    result as ``sample(apply(logits, p, k), min_p, q, eps)``.  Returns
    (token, out): token is [B] int32; out holds the rows after the filter and
    min-p (``logits`` itself may be passed), or None when ``want_out`` is
    false (then only the token is written)."""
    torch = _torch()
    lib = _lib.load()
    if not torch.is_tensor(logits) or logits.dim() != 2 or not logits.is_cuda:
        raise ValueError("logits must be a 2-D CUDA tensor")
    dt = _dtype_code(logits)
    if logits.stride(1) != 1:
        logits = logits.contiguous()
    B, V = logits.shape
    dev = logits.device
    p = _vec(p, B, logits.dtype, "p", dev)
    k = _vec(k, B, torch.int32, "k", dev)
    min_p = _vec(min_p, B, torch.float32, "min_p", dev)
    if q is not None:
        if not torch.is_tensor(q) or q.shape != (B, V) or q.dtype != torch.float32 or q.device != dev:
            raise ValueError("q must be a float32 tensor shaped like logits on the same device")
        if q.stride(1) != 1:
            q = q.contiguous()
    if want_out and out is None:
        out = torch.empty((B, V), dtype=logits.dtype, device=dev)
    if out is not None and (out.shape != (B, V) or out.dtype != logits.dtype or out.device != dev
                            or out.stride(1) != 1):
        raise ValueError("out must match logits in shape, dtype and device, with stride(1) == 1")
    token = torch.empty(B, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib.topkp_apply_sample(_ptr(logits), B, V, logits.stride(0) if B > 1 else V, dt, _ptr(p), _ptr(k),
                                      _ptr(min_p), _ptr(q), (q.stride(0) if B > 1 else V) if q is not None else V,
                                      float(eps), _ptr(out), (out.stride(0) if B > 1 else V) if out is not None else V,
                                      _ptr(token), _stream(dev)))
    return token, out


def apply_sorted(sorted_value, sorted_indices, p=None, k=None, logits=None, out=None):
    """ApplyTopKTopPWithSorted: filter pre-sorted rows.

    sorted_value: [B, V] ascending per row (stable order); sorted_indices:
    [B, V] int32 source columns; logits (optional): the unsorted rows."""
    torch = _torch()
    lib = _lib.load()
    for name, t in (("sorted_value", sorted_value), ("sorted_indices", sorted_indices)):
        if not torch.is_tensor(t) or t.dim() != 2 or not t.is_cuda:
            raise ValueError(f"{name} must be a 2-D CUDA tensor")
    dt = _dtype_code(sorted_value)
    B, V = sorted_value.shape
    dev = sorted_value.device
    if sorted_indices.shape != (B, V) or sorted_indices.dtype != torch.int32 or sorted_indices.device != dev:
        raise ValueError("sorted_indices must be an int32 tensor shaped like sorted_value")
    sorted_value = sorted_value.contiguous()
    sorted_indices = sorted_indices.contiguous()
    if logits is not None:
        if logits.shape != (B, V) or logits.dtype != sorted_value.dtype or logits.device != dev:
            raise ValueError("logits must match sorted_value in shape, dtype and device")
        logits = logits.contiguous()
    p = _vec(p, B, sorted_value.dtype, "p", dev)
    k = _vec(k, B, torch.int32, "k", dev)
    if out is None:
        out = torch.empty((B, V), dtype=sorted_value.dtype, device=dev)
    if out.shape != (B, V) or out.dtype != sorted_value.dtype or out.device != dev or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like sorted_value")
    with torch.cuda.device(dev):
        _check(lib.topkp_apply_sorted(_ptr(sorted_value), _ptr(sorted_indices), B, V, dt, _ptr(p), _ptr(k),
                                      _ptr(logits), _ptr(out), _stream(dev)))
    return out


def sample(filtered, min_p=None, q=None, eps: float = 1e-10, out=None, want_out: bool = True):
    """Min-p and the exponential-race sample on filtered rows (topkp_sample).

    filtered: [B, V] CUDA tensor (the output of ``apply`` / ``apply_sorted``:
    logits or -inf).  min_p: [B] float32 (or None).  q: [B, V] float32
    variates, e.g. drawn from Exp(1), or None for ArgMax.  Returns
    (token, out): token is a [B] int32 tensor of original indices; out holds
    the rows after min-p (``filtered`` itself may be passed as out), or None
    when ``want_out`` is false."""
    torch = _torch()
    lib = _lib.load()
    if not torch.is_tensor(filtered) or filtered.dim() != 2 or not filtered.is_cuda:
        raise ValueError("filtered must be a 2-D CUDA tensor")
    dt = _dtype_code(filtered)
    if filtered.stride(1) != 1:
        filtered = filtered.contiguous()
    B, V = filtered.shape
    dev = filtered.device
    min_p = _vec(min_p, B, torch.float32, "min_p", dev)
    if q is not None:
        if not torch.is_tensor(q) or q.shape != (B, V) or q.dtype != torch.float32 or q.device != dev:
            raise ValueError("q must be a float32 tensor shaped like filtered on the same device")
        if q.stride(1) != 1:
            q = q.contiguous()
    if want_out and out is None:
        out = torch.empty((B, V), dtype=filtered.dtype, device=dev)
    if out is not None and (out.shape != (B, V) or out.dtype != filtered.dtype or out.device != dev
                            or out.stride(1) != 1):
        raise ValueError("out must match filtered in shape, dtype and device, with stride(1) == 1")
    token = torch.empty(B, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib.topkp_sample(_ptr(filtered), B, V, filtered.stride(0) if B > 1 else V, dt, _ptr(min_p),
                                _ptr(q), (q.stride(0) if B > 1 else V) if q is not None else V, float(eps),
                                _ptr(out), (out.stride(0) if B > 1 else V) if out is not None else V,
                                _ptr(token), _stream(dev)))
    return token, out


def sample_v2(logits, k=None, p=None, min_p=None, q=None, eps: float = 1e-10, ks_max: int = 1024,
              input_is_logits: bool = True, need_sample_result: bool = False, workspace=None):
    """The TopKTopPSampleV2 semantics (topkp_sample_v2) on a [B, V] CUDA tensor.

    k: [B] int32; p, min_p: [B] float32; q: [B, V] float32 read by sorted
    position; each optional.  With ``need_sample_result`` false returns
    (token, select): token is [B] int32 (logitsSelectIdx), select the rows
    in original order with removed elements -inf (0 for probability input,
    logitsTopKPSelect).  Otherwise returns (logits_idx, sort_masked): [B, V]
    int32 original indices of the sorted positions (-1 past the top-k
    survivors) and [B, V] float32 masked probabilities."""
    torch = _torch()
    lib = _lib.load()
    if not torch.is_tensor(logits) or logits.dim() != 2 or not logits.is_cuda:
        raise ValueError("logits must be a 2-D CUDA tensor")
    dt = _dtype_code(logits)
    if logits.stride(1) != 1:
        logits = logits.contiguous()
    B, V = logits.shape
    dev = logits.device
    k = _vec(k, B, torch.int32, "k", dev)
    p = _vec(p, B, torch.float32, "p", dev)
    min_p = _vec(min_p, B, torch.float32, "min_p", dev)
    if q is not None:
        if not torch.is_tensor(q) or q.shape != (B, V) or q.dtype != torch.float32 or q.device != dev:
            raise ValueError("q must be a float32 tensor shaped like logits on the same device")
        if q.stride(1) != 1:
            q = q.contiguous()
    need = int(lib.topkp_sample_v2_workspace_size(B, V, dt))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if workspace.dtype != torch.uint8 or workspace.device != dev or workspace.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of at least {need} bytes on {dev}")
    token = select = idx = sm = None
    if need_sample_result:
        idx = torch.empty((B, V), dtype=torch.int32, device=dev)
        sm = torch.empty((B, V), dtype=torch.float32, device=dev)
    else:
        token = torch.empty(B, dtype=torch.int32, device=dev)
        select = torch.empty((B, V), dtype=logits.dtype, device=dev)
    with torch.cuda.device(dev):
        _check(lib.topkp_sample_v2(_ptr(logits), B, V, logits.stride(0) if B > 1 else V, dt, _ptr(k), _ptr(p),
                                   _ptr(min_p), _ptr(q), (q.stride(0) if B > 1 else V) if q is not None else V,
                                   float(eps), int(ks_max), 1 if input_is_logits else 0, _ptr(select), V,
                                   _ptr(token), _ptr(idx), _ptr(sm), _ptr(workspace), workspace.numel(),
                                   _stream(dev)))
    return (idx, sm) if need_sample_result else (token, select)


def sort(logits, workspace=None):
    """The stable ascending sort of every row (topkp_sort): returns
    (sorted_value, sorted_indices), the inputs of ``apply_sorted``.
    ``workspace`` is a uint8 CUDA tensor of at least
    ``sort_workspace_size(B, V, dtype)`` bytes (allocated when None)."""
    torch = _torch()
    lib = _lib.load()
    if not torch.is_tensor(logits) or logits.dim() != 2 or not logits.is_cuda:
        raise ValueError("logits must be a 2-D CUDA tensor")
    dt = _dtype_code(logits)
    if logits.stride(1) != 1:
        logits = logits.contiguous()
    B, V = logits.shape
    dev = logits.device
    need = int(lib.topkp_sort_workspace_size(B, V, dt))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if workspace.dtype != torch.uint8 or workspace.device != dev or workspace.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of at least {need} bytes on {dev}")
    sv = torch.empty((B, V), dtype=logits.dtype, device=dev)
    si = torch.empty((B, V), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib.topkp_sort(_ptr(logits), B, V, logits.stride(0) if B > 1 else V, dt, _ptr(sv), _ptr(si),
                              _ptr(workspace), workspace.numel(), _stream(dev)))
    return sv, si


def sort_workspace_size(B: int, V: int, dtype) -> int:
    """Bytes of workspace ``sort`` needs for a [B, V] tensor of ``dtype``."""
    torch = _torch()
    codes = {torch.float32: _lib.TOPKP_F32, torch.float16: _lib.TOPKP_F16, torch.bfloat16: _lib.TOPKP_BF16}
    return int(_lib.load().topkp_sort_workspace_size(B, V, codes[dtype]))


def device_status(device=None) -> None:
    """Synchronises the current stream and raises if a kernel gave up a
    bounded wait since the last check."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(_lib.load().topkp_device_status(_stream(dev)))


def last_launch_count() -> int:
    """Kernel launches enqueued by the most recent successful call."""
    return _lib.load().topkp_last_launch_count()
