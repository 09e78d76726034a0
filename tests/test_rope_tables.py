"""The fused K kernel's angle constants (csrc/rope_tables.h), on CPU: the
committed header is exactly what its generator prints, and its values agree
with pi computed another way (the Gauss-Legendre iteration in decimal
arithmetic, where the generator uses Machin's formula) and with the
platform's binary64 sin and cos."""
import decimal
import math
import os
import re
import struct
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_cache_fill_gb300", "csrc")


def header() -> str:
    with open(os.path.join(CSRC, "rope_tables.h")) as f:
        return f.read()


def pi_gauss_legendre(digits: int) -> decimal.Decimal:
    decimal.getcontext().prec = digits + 10
    D = decimal.Decimal
    a, b, t, p = D(1), D(1) / D(2).sqrt(), D(1) / 4, D(1)
    for _ in range(12):  # the digits double per step: 12 steps give thousands
        an = (a + b) / 2
        b = (a * b).sqrt()
        t -= p * (a - an) ** 2
        a, p = an, 2 * p
    return (a + b) ** 2 / (4 * t)


def f32(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def test_header_is_the_generator_output():
    out = subprocess.run([sys.executable, os.path.join(CSRC, "gen_rope_tables.py")], capture_output=True, text=True,
                         timeout=120, check=True).stdout
    assert out == header()


def test_inverse_two_pi_limbs_match_an_independent_pi():
    limbs = [int(x, 16) for x in re.findall(r"0x([0-9a-f]{16})ull", header())]
    assert len(limbs) == 4
    inv = (limbs[0] << 192) | (limbs[1] << 128) | (limbs[2] << 64) | limbs[3]
    pi = pi_gauss_legendre(120)
    want = int((decimal.Decimal(2) ** 256 / (2 * pi)).to_integral_value(rounding=decimal.ROUND_FLOOR))
    assert inv == want


def test_two_pi_over_2p32_pair():
    hi, lo = (float(x) for x in re.findall(r"kTwoPiOver2p32(?:Hi|Lo) = ([-0-9.e]+)f", header()))
    pi = pi_gauss_legendre(60)
    exact = 2 * pi / decimal.Decimal(2) ** 32
    err = abs(decimal.Decimal(hi) + decimal.Decimal(lo) - exact) / exact
    assert err < decimal.Decimal(2) ** -47
    assert abs(lo) <= abs(hi) * 2 ** -24  # a normalised pair


def test_turn_table_values():
    words = [int(x, 16) for x in re.findall(r"0x([0-9a-f]{8})u,", header())]
    assert len(words) == 2048 * 4
    for m in range(2048):
        sh, sl, ch, cl = (f32(w) for w in words[4 * m:4 * m + 4])
        a = 2 * math.pi * m / 2048
        # binary64 sin/cos of the binary64 angle: within a few 2^-53 of the
        # pair (which is within ~2^-48 of the exact value)
        assert abs((sh + sl) - math.sin(a)) < 2 ** -46, m
        assert abs((ch + cl) - math.cos(a)) < 2 ** -46, m
        assert abs(sl) <= abs(sh) * 2 ** -24 and abs(cl) <= abs(ch) * 2 ** -24, m
    # exact values where the kernel relies on them (its fast two-sums need
    # sin A == 0 or |sin A| >= sin(2 pi / 2048), and the same for cos)
    for m, want in ((0, (0.0, 0.0, 1.0, 0.0)), (512, (1.0, 0.0, 0.0, 0.0)), (1024, (0.0, 0.0, -1.0, 0.0)),
                    (1536, (-1.0, 0.0, 0.0, 0.0))):
        assert tuple(abs(v) if v == 0 else v for v in (f32(w) for w in words[4 * m:4 * m + 4])) == want, m
    small = math.sin(2 * math.pi / 2048) * (1 - 2 ** -20)
    for m in range(2048):
        sh, ch = f32(words[4 * m]), f32(words[4 * m + 2])
        assert sh == 0.0 or abs(sh) >= small, m
        assert ch == 0.0 or abs(ch) >= small, m
