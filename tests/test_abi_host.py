"""The C ABI without a GPU: the library builds, loads, exports every entry
point that include/topkp.h declares, and rejects bad arguments with the
page's status codes before touching the device (section 5.3 of the CANN
ops-nn ApplyTopKTopPWithSorted guide: 161001 null pointer, 161002 invalid)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "topkp.h")


@pytest.fixture(scope="module")
def lib():
    from top_logit_filter_gb300 import build, _lib
    build.build()
    return _lib.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(topkp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_expected_calls():
    assert _declared() == sorted(["topkp_apply", "topkp_apply_sample", "topkp_apply_sorted", "topkp_sample",
                                  "topkp_sample_v2",
                                  "topkp_sample_v2_workspace_size", "topkp_sort", "topkp_sort_workspace_size",
                                  "topkp_sort_static", "topkp_last_error_string", "topkp_device_status",
                                  "topkp_last_launch_count"])


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(os.path.join(ROOT, "top_logit_filter_gb300", "libtopkp.so"))
    for name in _declared():
        assert hasattr(raw, name), name


def test_binding_names_every_export():
    from top_logit_filter_gb300 import _lib
    assert sorted(_lib.EXPORTS) == _declared()


F32, F16, BF16 = 0, 1, 2
NULLPTR, INVALID, LAUNCH = 161001, 161002, 561000
FAKE = 1 << 20  # never dereferenced: every check below fails before a launch


def _apply(lib, x=FAKE, B=2, V=8, ldx=None, dt=F32, p=None, k=FAKE + 4096, out=FAKE + 8192, ldo=None):
    return lib.topkp_apply(x, B, V, V if ldx is None else ldx, dt, p, k, out, V if ldo is None else ldo, None)


def test_apply_argument_errors(lib):
    assert _apply(lib, p=None, k=None) == NULLPTR
    assert b"both NULL" in lib.topkp_last_error_string()
    assert _apply(lib, dt=7) == INVALID
    assert _apply(lib, B=-1) == INVALID
    assert _apply(lib, V=-3) == INVALID
    assert _apply(lib, V=(1 << 23) + 1) == INVALID
    assert _apply(lib, x=None) == NULLPTR
    assert _apply(lib, out=None) == NULLPTR
    assert _apply(lib, ldx=7) == INVALID
    assert _apply(lib, ldo=4) == INVALID
    # out overlapping logits without being the same buffer
    assert _apply(lib, x=FAKE, out=FAKE + 4) == INVALID
    assert _apply(lib, x=FAKE, out=FAKE, ldx=8, ldo=9) == INVALID
    # out overlapping k or p
    assert _apply(lib, k=FAKE + 8192, out=FAKE + 8192 - 4) == INVALID
    assert _apply(lib, p=FAKE + 8200, k=None) == INVALID


def test_apply_empty_problems_succeed_without_launch(lib):
    assert _apply(lib, B=0) == 0
    assert _apply(lib, V=0, x=None, out=None) == 0
    assert lib.topkp_last_launch_count() == 0


def test_sorted_argument_errors(lib):
    def call(sv=FAKE, si=FAKE + 4096, B=2, V=8, dt=BF16, p=FAKE + 12000, k=None, lg=None, out=FAKE + 8192):
        return lib.topkp_apply_sorted(sv, si, B, V, dt, p, k, lg, out, None)
    assert call(p=None, k=None) == NULLPTR
    assert call(dt=3) == INVALID
    assert call(B=-2) == INVALID
    assert call(sv=None) == NULLPTR
    assert call(si=None) == NULLPTR
    assert call(out=None) == NULLPTR
    assert call(out=FAKE + 8) == INVALID          # overlaps sorted_value
    assert call(lg=FAKE + 8190) == INVALID        # overlaps out
    assert call(B=0) == 0


def test_sample_argument_errors(lib):
    def call(x=FAKE, B=2, V=8, ld=8, dt=BF16, mp=None, q=FAKE + 4096, ldq=8, eps=1e-10, out=FAKE + 8192, ldo=8,
             tok=FAKE + 12288):
        return lib.topkp_sample(x, B, V, ld, dt, mp, q, ldq, eps, out, ldo, tok, None)
    assert call(out=None, tok=None) == NULLPTR
    assert call(x=None) == NULLPTR
    assert call(dt=5) == INVALID
    assert call(B=-1) == INVALID
    assert call(ld=7) == INVALID
    assert call(ldq=4) == INVALID
    assert call(ldo=2) == INVALID
    assert call(eps=-1.0) == INVALID
    assert call(tok=FAKE + 12289) == INVALID          # token not 4-byte aligned
    assert call(out=FAKE + 8) == INVALID              # out partially overlaps filtered
    assert call(out=FAKE + 4096 + 16) == INVALID      # out overlaps q
    assert call(tok=FAKE + 4) == INVALID              # token overlaps filtered
    assert call(B=0) == 0
    assert call(V=0, x=None) == 0
    assert lib.topkp_last_launch_count() == 0


def test_sort_workspace_and_argument_errors(lib):
    ws = lib.topkp_sort_workspace_size(2, 8, BF16)
    assert ws == 256 + 256                      # 64 B of indices and 32 B of values, each rounded to 256
    assert lib.topkp_sort_workspace_size(3, 1000, F32) == 12032 + 12032
    assert lib.topkp_sort_workspace_size(0, 8, BF16) == 0 and lib.topkp_sort_workspace_size(2, 8, 9) == 0

    def call(x=FAKE, B=2, V=8, ld=8, dt=BF16, sv=FAKE + 8192, si=FAKE + 12288, w=FAKE + 16384, wn=512):
        return lib.topkp_sort(x, B, V, ld, dt, sv, si, w, wn, None)
    assert call(x=None) == NULLPTR
    assert call(sv=None) == NULLPTR
    assert call(w=None) == NULLPTR
    assert call(dt=4) == INVALID
    assert call(ld=7) == INVALID
    assert call(wn=511) == INVALID               # workspace too small
    assert call(w=FAKE + 16384 + 16) == INVALID  # workspace not 256-byte aligned
    assert call(sv=FAKE + 4) == INVALID          # overlaps the logits
    assert call(si=FAKE + 8192 + 8) == INVALID   # overlaps sorted_value
    assert call(B=0) == 0


def test_sort_static_argument_errors(lib):
    def call(x=FAKE, B=2, V=8, ld=8, dt=BF16, sv=FAKE + 8192, si=FAKE + 12288):
        return lib.topkp_sort_static(x, B, V, ld, dt, sv, si, None)
    assert call(dt=7) == INVALID
    assert call(B=-1) == INVALID
    assert call(B=64, V=152064) == INVALID             # needs more than the fixed 16 MiB scratch
    assert b"scratch" in lib.topkp_last_error_string()
    assert call(x=None) == NULLPTR
    assert call(si=None) == NULLPTR
    assert call(ld=7) == INVALID
    assert call(sv=FAKE + 4) == INVALID                # overlaps the logits
    assert call(B=0) == 0 and call(V=0) == 0
    assert lib.topkp_last_launch_count() == 0


def test_no_device_fails_loudly_instead_of_falling_back(lib):
    """Valid arguments but no usable GPU: the call must report a launch error
    (there is no CPU path)."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _apply(lib) == LAUNCH
    assert b"device" in lib.topkp_last_error_string()
    assert lib.topkp_sample(FAKE, 2, 8, 8, BF16, None, None, 8, 1e-10, None, 8, FAKE + 8192, None) == LAUNCH
    assert lib.topkp_sort(FAKE, 2, 8, 8, BF16, FAKE + 8192, FAKE + 12288, FAKE + 16384, 512, None) == LAUNCH
    assert lib.topkp_sort_static(FAKE, 2, 8, 8, BF16, FAKE + 8192, FAKE + 12288, None) == LAUNCH


def test_python_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    import top_logit_filter_gb300 as tk
    with pytest.raises(ValueError):
        tk.apply(torch.zeros(2, 8), k=torch.ones(2, dtype=torch.int32))
