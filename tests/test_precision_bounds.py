"""The error bounds that the attention kernels' 16-bit operands rely on,
checked on CPU by emulating each rounding in numpy (float32 -> float16 and
the BF16 conversions round to nearest even, as the kernels' cvt.rn
instructions do) over weights spanning their whole range, in steps, around
the regime edges, and over every BF16 bit pattern.

Chunked prefill (BF16, FP8-K and FP8 K+V calls):
  the weights enter the PV product as one f16 rounding of 2^7 P, P <= 2^8:
      |f16(x) - x| <= 2^-11 x for x >= 2^-14 (P >= 2^-21), 2^-25 below;
  a BF16 V value v enters it as f16(v * 2^-8):
      exact for 2^-6 <= |v| < 2^24, within 2^-17 (in units of v) below,
      and non-finite from 2^24 up (outside the supported range).
Decode (mma.sync), P <= 1 against the exact running max:
  BF16 V: hi = bf16(P), lo = bf16(P - hi):  |P - hi - lo| <= 2^-16 P;
  E4M3 V: x = 2^8 P, hi = f16(x), lo = f16(x - hi):
      |x - hi - lo| <= max(2^-22 x, 2^-25)."""
import numpy as np


def _weights(lo_exp, hi_exp, edges):
    rng = np.random.default_rng(7)
    x = np.exp2(rng.uniform(lo_exp, hi_exp, 1_000_000)).astype(np.float32)
    parts = [x]
    for e in edges:
        c = int(np.float32(2.0 ** e).view(np.uint32))
        parts.append(np.arange(c - (1 << 21), c + (1 << 21), 5, dtype=np.uint32).view(np.float32))
    x = np.concatenate(parts)
    return x[(x > 0) & (x <= 2.0 ** hi_exp)]


def _bf16_rn(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest BF16 (ties to even), as float32; finite inputs."""
    b = x.view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return r.astype(np.uint32).view(np.float32)


def test_bf16_rounding_helper_is_round_to_nearest_even():
    # the emulation above against exact rationals on a few ties and non-ties
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -7)
    x = np.array([one + ulp / 2, one + ulp * 1.5, one + ulp / 4, one + ulp * 0.75], np.float32)
    want = np.array([one, one + 2 * ulp, one, one + ulp], np.float32)
    assert (_bf16_rn(x) == want).all()


def test_prefill_single_f16_weight():
    x = _weights(-40, 15, (-14, -24, 15, -3)).astype(np.float32)   # x = 2^7 P, P <= 2^8
    r = x.astype(np.float16).astype(np.float64)
    x64 = x.astype(np.float64)
    err = np.abs(r - x64)
    normal = x64 >= 2.0 ** -14
    assert (err[normal] <= 2.0 ** -11 * x64[normal]).all()
    assert (err[~normal] <= 2.0 ** -25).all()
    assert np.isfinite(r).all()                                     # 2^15 stays inside f16's range
    # the relative bound is tight: some weight is rounded by more than 2^-12
    assert (err[normal] > 2.0 ** -12 * x64[normal]).any()


def test_prefill_bf16_v_scaled_to_f16_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32)
    v = (bits << 16).view(np.float32)
    fin = np.isfinite(v)
    v, bits = v[fin], bits[fin]
    with np.errstate(over="ignore"):                     # 2^24 and up overflow f16, as checked below
        back = (v * np.float32(2.0 ** -8)).astype(np.float16).astype(np.float64) * 2.0 ** 8
    a = np.abs(v.astype(np.float64))
    exact = (a >= 2.0 ** -6) & (a < 2.0 ** 24)
    assert (back[exact] == v[exact]).all()
    small = a < 2.0 ** -6
    assert (np.abs(back[small] - v[small]) <= 2.0 ** -17).all()
    assert (~np.isfinite(back[a >= 2.0 ** 24])).all()
    # the largest BF16 value below 2^24 converts exactly
    assert a[exact].max() == float(np.float32(2.0 ** 24 - 2.0 ** 16))


def test_decode_bf16_split():
    p = _weights(-60, 0, (-3, -20, 0))                    # P <= 1
    hi = _bf16_rn(p)
    lo = _bf16_rn(p - hi)                                 # p - hi exact in binary32
    err = np.abs(p.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    assert (err <= 2.0 ** -16 * p.astype(np.float64)).all()


def test_decode_f16_split_of_an_e4m3_v_cache():
    x = _weights(-52, 8, (-3, -14, -24, 8))               # x = 2^8 P
    hi = x.astype(np.float16)
    r = x - hi.astype(np.float32)                         # exact in binary32
    lo = r.astype(np.float16)
    err = np.abs(x.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    assert (err <= np.maximum(2.0 ** -22 * x.astype(np.float64), 2.0 ** -25)).all()
    assert np.isfinite(hi).all()
