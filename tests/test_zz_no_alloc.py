"""topkp_sort_static, the sort for callers that cannot allocate device memory
when they sort (code running inside a memory pool it does not own, a plugin
handed only its tensors, a process that has already reserved the GPU's
memory): its scratch is a fixed 16 MiB array of the library's own device
memory.  Through the C ABI it must give exactly what topkp_sort gives with a
caller workspace, on two calls in a row that reuse the same array with
different rows; match the CPU oracle's stable sort; leave the device's free
memory unchanged once the first call has loaded it; and refuse a problem too
large for the array.  This file is collected last so that, run with -x,
every other test has run first; it also passes alone in a fresh process."""
import numpy as np
import pytest

import oracle as O
from rawutil import raw_to_torch, to_raw, torch_to_raw

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32, F16, BF16 = 0, 1, 2
CODE = {"f32": F32, "f16": F16, "bf16": BF16}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_logit_filter_gb300 import build, _lib
    build.build()
    return _lib.load()


def _rows(B, V, dtype, seed, ld=None):
    """[B, V] rows with ties and signed zeros, as a view of a [B, ld] buffer."""
    rng = np.random.default_rng(seed)
    ld = V if ld is None else ld
    v = np.round(2.0 * rng.standard_normal((B, ld)), 1)   # ties
    v[rng.random((B, ld)) < 0.02] = -0.0
    return raw_to_torch(np.stack([to_raw(r, dtype) for r in v]), dtype, "cuda")[:, :V]


def _outputs(x):
    B, V = x.shape
    return torch.empty((B, V), dtype=x.dtype, device="cuda"), torch.empty((B, V), dtype=torch.int32, device="cuda")


def _sort_with_workspace(lib, x, dtype):
    B, V = x.shape
    need = lib.topkp_sort_workspace_size(B, V, CODE[dtype])
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    sv, si = _outputs(x)
    st = lib.topkp_sort(x.data_ptr(), B, V, x.stride(0), CODE[dtype], sv.data_ptr(), si.data_ptr(), ws.data_ptr(),
                        need, torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.topkp_last_error_string()
    return sv, si


def _sort_static(lib, x, dtype, out=None):
    B, V = x.shape
    sv, si = _outputs(x) if out is None else out
    st = lib.topkp_sort_static(x.data_ptr(), B, V, x.stride(0), CODE[dtype], sv.data_ptr(), si.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.topkp_last_error_string()
    return sv, si


def _ints(t, dtype):
    return t.view(torch.int16 if dtype != "f32" else torch.int32)


# the largest problem the 16 MiB scratch takes: 20 x 139808 elements need
# round256(4n) + round256(2n) = 16,776,960 bytes, 256 below the limit; one
# element more per row needs 16,777,472
AT_LIMIT = ("bf16", 20, 139808, None)


@pytest.mark.parametrize("dtype,B,V,ld", [("bf16", 8, 152064, None), ("f32", 3, 151936, 151936 + 37),
                                          ("f16", 5, 4099, 4099 + 3), AT_LIMIT])
def test_static_scratch_sort_matches_the_workspace_sort_twice(lib, dtype, B, V, ld):
    for seed in (1, 2):    # two calls in a row on the same scratch, different rows
        x = _rows(B, V, dtype, seed, ld)
        ref_v, ref_i = _sort_with_workspace(lib, x, dtype)
        got_v, got_i = _sort_static(lib, x, dtype)
        torch.cuda.synchronize()
        assert torch.equal(got_i, ref_i)
        assert torch.equal(_ints(got_v, dtype), _ints(ref_v, dtype))


def test_static_scratch_sort_matches_the_oracle(lib):
    """Directly against the CPU oracle's stable ascending sort, on rows whose
    ties and signed zeros make the index order matter."""
    dtype, B, V = "bf16", 4, 30011
    x = _rows(B, V, dtype, 7, V + 5)
    sv, si = _sort_static(lib, x, dtype)
    torch.cuda.synchronize()
    xr, svr, sir = torch_to_raw(x, dtype), torch_to_raw(sv, dtype), si.cpu().numpy()
    for b in range(B):
        _, idx = O.stable_ascending_sort(O.decode(xr[b], dtype))
        assert np.array_equal(sir[b], idx), b
        assert np.array_equal(svr[b], xr[b][idx]), b


def test_static_scratch_sort_allocates_nothing(lib):
    """Once the first call has loaded the sort on this device (and with it
    the static array), further calls leave the device's free memory as it
    was: the outputs are the caller's, the scratch is the library's own."""
    dtype, B, V = AT_LIMIT[:3]
    x = _rows(B, V, dtype, 3)
    out = _outputs(x)
    _sort_static(lib, x, dtype, out)          # warm-up: loads the module
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        _sort_static(lib, x, dtype, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)


@pytest.mark.parametrize("B,V", [(64, 152064), (20, 139809)])
def test_static_scratch_refuses_a_problem_above_its_size(lib, B, V):
    # 64 x 152064 needs about 58 MB of scratch; 20 x 139809 just 512 bytes
    # more than the 16 MiB the array holds
    x = torch.zeros((B, V), dtype=torch.bfloat16, device="cuda")
    sv, si = torch.empty_like(x), torch.empty(x.shape, dtype=torch.int32, device="cuda")
    assert lib.topkp_sort_workspace_size(B, V, BF16) > (16 << 20)
    st = lib.topkp_sort_static(x.data_ptr(), B, V, V, BF16, sv.data_ptr(), si.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert st == 161002
    assert b"scratch" in lib.topkp_last_error_string()
    assert lib.topkp_last_launch_count() == 0
