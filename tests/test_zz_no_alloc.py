"""topkp_sort_static, the sort for callers that cannot allocate device memory
when they sort: its scratch is a fixed array of the library's own device
memory.  Through the C ABI it must give exactly what topkp_sort gives with a
caller workspace, on two calls in a row that reuse the same array with
different rows, and it must refuse a problem too large for the array.  This
file is collected last so that, run with -x, every other test has run first;
it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest

from rawutil import raw_to_torch, to_raw

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


def _rows(B, V, dtype, seed):
    rng = np.random.default_rng(seed)
    v = np.round(2.0 * rng.standard_normal((B, V)), 1)   # ties
    v[rng.random((B, V)) < 0.02] = -0.0
    return raw_to_torch(np.stack([to_raw(r, dtype) for r in v]), dtype, "cuda")


def _sort_with_workspace(lib, x, dtype):
    B, V = x.shape
    need = lib.topkp_sort_workspace_size(B, V, CODE[dtype])
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    sv, si = torch.empty_like(x), torch.empty((B, V), dtype=torch.int32, device="cuda")
    st = lib.topkp_sort(x.data_ptr(), B, V, V, CODE[dtype], sv.data_ptr(), si.data_ptr(), ws.data_ptr(), need,
                        torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.topkp_last_error_string()
    return sv, si


def _sort_static(lib, x, dtype):
    B, V = x.shape
    sv, si = torch.empty_like(x), torch.empty((B, V), dtype=torch.int32, device="cuda")
    st = lib.topkp_sort_static(x.data_ptr(), B, V, V, CODE[dtype], sv.data_ptr(), si.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.topkp_last_error_string()
    return sv, si


@pytest.mark.parametrize("dtype,B,V", [("bf16", 8, 152064), ("f32", 3, 151936), ("f16", 5, 4099)])
def test_static_scratch_sort_matches_the_workspace_sort_twice(lib, dtype, B, V):
    for seed in (1, 2):    # two calls in a row on the same scratch, different rows
        x = _rows(B, V, dtype, seed)
        ref_v, ref_i = _sort_with_workspace(lib, x, dtype)
        got_v, got_i = _sort_static(lib, x, dtype)
        torch.cuda.synchronize()
        assert torch.equal(got_i, ref_i)
        assert torch.equal(got_v.view(torch.int16 if dtype != "f32" else torch.int32),
                           ref_v.view(torch.int16 if dtype != "f32" else torch.int32))


def test_static_scratch_refuses_a_problem_above_its_size(lib):
    x = torch.zeros((64, 152064), dtype=torch.bfloat16, device="cuda")   # about 58 MB of scratch
    sv, si = torch.empty_like(x), torch.empty(x.shape, dtype=torch.int32, device="cuda")
    st = lib.topkp_sort_static(x.data_ptr(), 64, 152064, 152064, BF16, sv.data_ptr(), si.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert st == 161002
    assert b"scratch" in lib.topkp_last_error_string()
    assert lib.topkp_last_launch_count() == 0
