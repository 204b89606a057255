"""Test helpers: raw dtype arrays <-> Python values and torch tensors.

Nothing here computes any part of the filter."""
import numpy as np

NP_RAW = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}


def to_raw(values, dtype):
    """Python floats (or "-inf"/"-0"/"0" strings) -> raw dtype array."""
    vals = []
    for v in values:
        if isinstance(v, str):
            v = {"-inf": -np.inf, "-0": -0.0, "0": 0.0, "inf": np.inf}[v]
        vals.append(v)
    f = np.array(vals, dtype=np.float32)
    if dtype == "f32":
        return f
    if dtype == "f16":
        return f.astype(np.float16)
    u = f.view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF).astype(np.uint16)


def bits(raw, dtype):
    if dtype == "f32":
        return np.asarray(raw, dtype=np.float32).view(np.uint32)
    if dtype == "f16":
        return np.asarray(raw, dtype=np.float16).view(np.uint16)
    return np.asarray(raw, dtype=np.uint16)


NEG_INF = {"f32": 0xFF800000, "f16": 0xFC00, "bf16": 0xFF80}


def torch_dtype(dtype):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def raw_to_torch(raw, dtype, device="cpu"):
    import torch
    a = np.ascontiguousarray(raw)
    if dtype == "bf16":
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    return t.to(device)


def torch_to_raw(t, dtype):
    import torch
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
