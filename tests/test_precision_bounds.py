"""The error bounds the chunked prefill's P split relies on, checked on CPU
by emulating the split in numpy over weights spanning their whole range
(2^-40 .. 2^15) and every binary32 value, in steps, around the regime edges.
The PV product multiplies V by the two 16-bit parts hi and lo of each
float32 weight P:
  BF16 V: hi = P truncated to BF16, lo = (P - hi) truncated to BF16:
          |P - hi - lo| < 2^-15 P;
  f16 V (E4M3 V cache): hi = P truncated to 11 significant bits, then f16;
          lo = (P - truncated P) rounded to f16:
          |P - hi - lo| <= max(2^-21 P, 2^-24)."""
import numpy as np


def _weights():
    rng = np.random.default_rng(7)
    x = np.exp2(rng.uniform(-40, 15, 1_000_000)).astype(np.float32)
    edges = []
    for e in (-3, -14, -24, 15):
        c = int(np.float32(2.0 ** e).view(np.uint32))
        edges.append(np.arange(c - (1 << 21), c + (1 << 21), 5, dtype=np.uint32).view(np.float32))
    x = np.concatenate([x] + edges)
    return x[(x > 0) & (x <= 2.0 ** 15)]


def test_bf16_truncation_split():
    x = _weights()
    hi = (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    r = x - hi                                            # exact in binary32
    lo = (r.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    err = np.abs(x.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    assert (err < 2.0 ** -15 * x.astype(np.float64)).all()


def test_f16_split_of_an_e4m3_v_cache():
    x = _weights()
    hi32 = (x.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    hi = hi32.astype(np.float16)
    lo = (x - hi32).astype(np.float16)                    # x - hi32 exact in binary32
    err = np.abs(x.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    assert (err <= np.maximum(2.0 ** -21 * x.astype(np.float64), 2.0 ** -24)).all()
    # both terms are needed: the relative one alone fails for small weights
    assert (err > 2.0 ** -21 * x.astype(np.float64)).any()
    assert np.isfinite(hi).all()                          # 2^15 stays inside f16's range
