"""Host checks of the kernels' fixed-point helpers against exact rational
arithmetic: the float -> integer rounding used for probability masses and
the floor(thr * S) target of the top-p cut.  The helpers are plain integer
code shared by host and device, compiled here for the host with nvcc."""
import os
import random
import shutil
import struct
import subprocess
from fractions import Fraction

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("fp") / "fixed_point_probe")
    subprocess.check_call([nvcc, "-O2", "-std=c++17", "-I", os.path.join(ROOT, "include"),
                           "-I", os.path.join(ROOT, "top_logit_filter_gb300", "csrc"),
                           os.path.join(HERE, "fixed_point_probe.cu"), "-o", exe])

    def run(lines):
        out = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True)
        return [int(v) for v in out.stdout.split()]
    return run


def f32(bits):
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def bits_of(x):
    return struct.unpack("<I", struct.pack("<f", x))[0]


def round_half_even(q: Fraction) -> int:
    n = q.numerator // q.denominator
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n


def test_f2ull_rn_matches_exact_rounding(probe):
    rng = random.Random(7)
    cases = [0, 1, bits_of(0.5), bits_of(1.5), bits_of(2.5), bits_of(3.5), bits_of(0.49999997),
             bits_of(0.50000006), bits_of(2.0 ** 40), bits_of(2.0 ** 41 - 2 ** 17), bits_of(2.0 ** 62),
             0x00000001, 0x007fffff, 0x00800000, bits_of(1e-30)]
    # every exponent that matters, random mantissas, plus exact halves
    for e in range(100, 190):
        for _ in range(40):
            cases.append((e << 23) | rng.getrandbits(23))
    for k in range(1, 25):
        cases.append(bits_of(float(Fraction(2 * rng.getrandbits(20) + 1, 2))))
        cases.append(((127 + 23 - k) << 23) | (1 << (k - 1)))  # m * 2^-k with remainder exactly half
    got = probe([f"f {b:x}" for b in cases])
    for b, g in zip(cases, got):
        assert g == round_half_even(Fraction(f32(b))), hex(b)


def test_mass_target_is_exact_floor(probe):
    rng = random.Random(11)
    cases = [(0.0, 123), (1.0, 456), (0.5, 7), (0.5, 2 ** 63 - 1), (0.1, 10 ** 15), (2.0 ** -40, 2 ** 62),
             (1e-45, 2 ** 63), (0.99999994, 2 ** 64 - 1)]
    for _ in range(400):
        thr = struct.unpack("<f", struct.pack("<f", rng.random()))[0]
        cases.append((thr, rng.getrandbits(rng.choice([10, 40, 50, 63, 64]))))
    cases = [(f32(bits_of(t)), S) for t, S in cases]  # thresholds are fp32 values
    got = probe([f"t {bits_of(t):x} {S}" for t, S in cases])
    for (t, S), g in zip(cases, got):
        want = S if t >= 1.0 else (0 if t <= 0 else int(Fraction(t) * S))
        assert g == want, (t, S)
