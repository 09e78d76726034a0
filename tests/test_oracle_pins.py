"""Pins for the CPU oracle: each test checks the oracle against something that
does not come from the oracle itself — torch's own number-format conversions,
RMSNorm and scaled-dot-product attention, brute-force searches, closed forms
and invariants. A plausible slip anywhere in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong rounding) fails one of
these. CPU only."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import kvgen


# ---------------------------------------------------------------------------
# slot mapping (kv_cache.rs, fill_slots_from_block_table)
# ---------------------------------------------------------------------------
def _slots_by_enumeration(table, block_size):
    """Walk the table block by block and list each block's rows in order: the
    k-th listed slot is the slot of position k."""
    out = []
    for blk in table:
        for row in range(block_size):
            out.append(int(blk) * block_size + row)
    return out


@pytest.mark.parametrize("block_size", [1, 3, 16, 64])
def test_fill_slots_matches_enumeration(oracle_lib, block_size):
    rng = np.random.default_rng(block_size)
    table = rng.permutation(200).astype(np.int32)[:40]
    listed = _slots_by_enumeration(table, block_size)
    for start, count in [(0, 1), (0, 40 * block_size), (5, 17), (block_size - 1, 2 * block_size + 3),
                         (40 * block_size - 1, 1)]:
        count = min(count, 40 * block_size - start)
        got = oracle_lib.fill_slots(table, start, count, block_size)
        assert got.tolist() == listed[start:start + count]
        # invariant: slot / bs is the table's block, slot % bs the row
        pos = np.arange(start, start + count)
        assert np.array_equal(got // block_size, table[pos // block_size])
        assert np.array_equal(got % block_size, pos % block_size)


def test_fill_slots_negative_block_gives_negative_slot(oracle_lib):
    got = oracle_lib.fill_slots(np.array([-1, 3], np.int32), 0, 32, 16)
    assert (got[:16] < 0).all() and (got[16:] >= 48).all()


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_bf16_widening_matches_torch(oracle_lib):
    ref = torch.from_numpy(ALL_BF16.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle_lib.bf16_to_f64(ALL_BF16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_rounding_of_binary32_values_matches_torch(oracle_lib):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32)
    x32 = bits.view(np.float32)
    x32 = x32[np.isfinite(x32)]
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_lib.f64_to_bf16(x32.astype(np.float64))
    assert np.array_equal(got, ref)


def _bf16_finite_sorted():
    vals = torch.from_numpy(ALL_BF16.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    keep = np.isfinite(vals) & ~((vals == 0) & np.signbit(vals))
    order = np.argsort(vals[keep], kind="stable")
    return vals[keep][order], ALL_BF16[keep][order]


def test_bf16_direct_rounding_brute_force(oracle_lib):
    """binary64 -> BF16 in one rounding: nearest BF16 by exact rational
    comparison, ties to the even pattern. Includes exact midpoints and values
    one binary64 ulp either side of them, which a double rounding through
    binary32 would get wrong."""
    vals, pats = _bf16_finite_sorted()
    rng = np.random.default_rng(3)
    i = rng.integers(1, len(vals) - 2, 3000)
    mids = (vals[i] + vals[i + 1]) / 2
    xs = np.concatenate([mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf),
                         rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000)])
    xs = xs[np.abs(xs) < 3.38e38]
    got = oracle_lib.f64_to_bf16(xs)
    for x, g in zip(xs.tolist(), got.tolist()):
        k = np.searchsorted(vals, x)
        lo_i, hi_i = max(k - 1, 0), min(k, len(vals) - 1)
        cands = [(vals[lo_i], pats[lo_i]), (vals[hi_i], pats[hi_i])]
        fx = Fraction(x)
        dists = [abs(Fraction(float(v)) - fx) for v, _ in cands]
        if dists[0] < dists[1]:
            want = cands[0][1]
        elif dists[1] < dists[0]:
            want = cands[1][1]
        else:
            want = cands[0][1] if int(cands[0][1]) % 2 == 0 else cands[1][1]
        if int(want) == 0 and x < 0:
            want = 0x8000                    # a negative value that rounds to zero keeps its sign
        assert int(g) == int(want), (x, hex(g), hex(want))


def test_bf16_rounding_specials(oracle_lib):
    got = oracle_lib.f64_to_bf16(np.array([np.inf, -np.inf, 1e39, -1e39, 0.0, -0.0, np.nan]))
    assert got[:6].tolist() == [0x7F80, 0xFF80, 0x7F80, 0xFF80, 0x0000, 0x8000]
    assert (int(got[6]) & 0x7FFF) > 0x7F80


ALL_E4M3 = np.arange(256, dtype=np.uint16).astype(np.uint8)


def test_e4m3_decode_matches_torch(oracle_lib):
    ref = torch.from_numpy(ALL_E4M3).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle_lib.e4m3_to_f64(ALL_E4M3)
    nan = np.isnan(ref)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def _e4m3_brute_force(x: float) -> int:
    """Nearest non-negative finite E4M3 magnitude by exhaustive search, ties
    to the even code; saturate at 448; sign from the input; NaN -> 0x7F."""
    if np.isnan(x):
        return 0x7F
    sign = 0x80 if np.signbit(x) else 0
    ax = abs(x)
    if ax >= 448:
        return sign | 0x7E
    mags = torch.from_numpy(ALL_E4M3[:0x7F]).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    d = np.abs(mags - ax)  # exact: both sides have few significant bits
    best = np.flatnonzero(d == d.min())
    code = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
    return sign | code


def test_e4m3_encode_exhaustive_over_bf16_inputs(oracle_lib):
    """Every BF16 bit pattern, k_scale = 1: the oracle's code equals the
    brute-force nearest code, and torch's own RNE cast wherever that cast is
    defined (|x| < 448; torch does not saturate)."""
    x = torch.from_numpy(ALL_BF16.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    got = oracle_lib.e4m3_encode(x)
    want = np.array([_e4m3_brute_force(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, want)
    inrange = np.abs(x) < 448
    ref = torch.from_numpy(x[inrange]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[inrange], ref)


def test_e4m3_encode_roundtrip_ties_and_saturation(oracle_lib):
    finite = ALL_E4M3[(ALL_E4M3 & 0x7F) != 0x7F]
    vals = oracle_lib.e4m3_to_f64(finite).astype(np.float32)
    assert np.array_equal(oracle_lib.e4m3_encode(vals), finite)   # every finite code round-trips
    # midpoints between neighbouring magnitudes go to the even code
    mags = oracle_lib.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    codes = oracle_lib.e4m3_encode(mids)
    assert (codes % 2 == 0).all()
    big = np.array([448.0, 448.0 * (1 + 2.0 ** -4), 464.0, 1e30, np.inf], np.float32)
    assert oracle_lib.e4m3_encode(big).tolist() == [0x7E] * 5
    assert oracle_lib.e4m3_encode(-big).tolist() == [0xFE] * 5
    assert oracle_lib.e4m3_encode(np.array([-0.0, 0.0, 2.0 ** -11, -(2.0 ** -11)], np.float32)).tolist() \
        == [0x80, 0x00, 0x00, 0x80]


# ---------------------------------------------------------------------------
# cache writes
# ---------------------------------------------------------------------------
def _pool_u16(nb, bs, H, D):
    return np.full((nb, bs, H, D), kvgen.BF16_NAN, np.uint16)


def _rows(t: torch.Tensor) -> np.ndarray:
    return np.ascontiguousarray(t.view(torch.int16).numpy().view(np.uint16))


def test_write_bf16_then_read_is_identity(oracle_lib):
    w = kvgen.tiny()
    nb, bs, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    slots = np.concatenate([oracle_lib.fill_slots(w.block_tables[s].numpy(), 0, int(L), bs)
                            for s, L in enumerate(w.seq_lens.tolist())])
    key, value = _rows(w.key), _rows(w.value)
    kc, vc = _pool_u16(nb, bs, H, D), _pool_u16(nb, bs, H, D)
    oracle_lib.write_bf16(key, value, kc, vc, slots, len(slots), H, D, bs, H * D, H * D)
    blk, row = slots // bs, slots % bs
    assert np.array_equal(kc[blk, row].reshape(len(slots), H * D), key)
    assert np.array_equal(vc[blk, row].reshape(len(slots), H * D), value)
    untouched = np.ones((nb, bs), bool)
    untouched[blk, row] = False
    assert (kc[untouched] == kvgen.BF16_NAN).all() and (vc[untouched] == kvgen.BF16_NAN).all()


def test_write_strided_rows_and_skipped_slots(oracle_lib):
    H, D, bs, nb = 2, 8, 4, 6
    stride = H * D + 24                      # rows padded, as in a fused QKV buffer
    rng = np.random.default_rng(0)
    src = rng.integers(0, 65535, (5, stride), dtype=np.uint16)
    slots = np.array([3, -1, 17, 0, -5], np.int64)
    vc = _pool_u16(nb, bs, H, D)
    oracle_lib.write_v_only(src, vc, slots, 5, H, D, bs, stride)
    flat = vc.reshape(nb * bs, H * D)
    for t, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(flat[s], src[t, :H * D])
    assert (np.delete(flat, [3, 17, 0], axis=0) == kvgen.BF16_NAN).all()


def test_write_fp8k_codes_are_rounded_quotients(oracle_lib):
    w = kvgen.custom(11, seq_lens=[40, 9], num_q_heads=4, num_kv_heads=2, head_dim=32,
                     block_size=16, fp8=True)
    nb, bs, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    slots = np.concatenate([oracle_lib.fill_slots(w.block_tables[s].numpy(), 0, int(L), bs)
                            for s, L in enumerate(w.seq_lens.tolist())])
    key, value = _rows(w.key), _rows(w.value)
    kc = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    vc = _pool_u16(nb, bs, H, D)
    k_scale = np.float32(w.k_scale)
    oracle_lib.write_fp8k(key, value, kc, vc, slots, len(slots), H, D, bs, H * D, H * D, k_scale)
    # numpy's binary32 division is an independent IEEE division
    quot = w.key.to(torch.float32).numpy() / k_scale
    assert quot.dtype == np.float32
    want = np.array([_e4m3_brute_force(float(v)) for v in quot.ravel()], np.uint8).reshape(quot.shape)
    blk, row = slots // bs, slots % bs
    assert np.array_equal(kc[blk, row].reshape(len(slots), H * D), want)
    assert np.array_equal(vc[blk, row].reshape(len(slots), H * D), value)
    # the outliers (|K| = 20 = max) land exactly on the saturation code
    assert ((want & 0x7F) <= 0x7E).all() and (want[np.abs(quot) >= 447.99] & 0x7F == 0x7E).all()


# ---------------------------------------------------------------------------
# fused K path: RMSNorm, RoPE, one rounding (kv_cache.rs,
# fused_k_norm_rope_cache_write_bf16)
# ---------------------------------------------------------------------------
def test_rmsnorm_matches_torch(oracle_lib):
    rng = np.random.default_rng(1)
    for D in (64, 128, 256):
        x = rng.standard_normal(D) * 7
        w = rng.uniform(0.5, 1.5, D)
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (D,), torch.from_numpy(w), eps=1e-6)
        np.testing.assert_allclose(oracle_lib.rmsnorm_row(x, w, 1e-6), ref.numpy(), rtol=1e-14, atol=0)


def test_rmsnorm_closed_forms(oracle_lib):
    D = 128
    w = np.linspace(0.5, 1.5, D)
    for c in (-3.0, 0.25, 18.0):
        y = oracle_lib.rmsnorm_row(np.full(D, c), w, 1e-6)
        np.testing.assert_allclose(y, np.sign(c) * w / np.sqrt(1 + 1e-6 / c**2), rtol=1e-15)
    x = np.random.default_rng(2).standard_normal(D) * 4
    y = oracle_lib.rmsnorm_row(x, np.ones(D), 0.0)
    assert abs(np.sqrt(np.mean(y**2)) - 1) < 1e-14


def test_rope_position_zero_is_identity(oracle_lib):
    y = np.random.default_rng(3).standard_normal(128)
    assert np.array_equal(oracle_lib.rope_row(y, 128, 0, 1e6), y)


@pytest.mark.parametrize("head_dim,rotary_dim", [(128, 128), (128, 64), (64, 32)])
def test_rope_is_a_rotation_of_half_pairs(oracle_lib, head_dim, rotary_dim):
    """Treat the pair (i, i + rotary_dim/2) as the complex number
    y_i + 1j*y_{i+R/2}: the oracle multiplies it by a unit phasor whose
    angle is pos times a geometric frequency ladder starting at 1, and
    leaves the other dims alone."""
    rng = np.random.default_rng(head_dim + rotary_dim)
    half = rotary_dim // 2
    y = rng.standard_normal(head_dim)
    for pos in (1, 7, 1023, 70000):
        out = oracle_lib.rope_row(y, rotary_dim, pos, 1e6)
        z_in = y[:half] + 1j * y[half:rotary_dim]
        z_out = out[:half] + 1j * out[half:rotary_dim]
        np.testing.assert_allclose(np.abs(z_out), np.abs(z_in), rtol=1e-13)
        assert np.array_equal(out[rotary_dim:], y[rotary_dim:])
        phasor = z_out / z_in
        np.testing.assert_allclose(np.abs(phasor), 1.0, rtol=1e-12)
        if pos == 1:
            ang = np.angle(phasor)                     # small angles, no wrap
            np.testing.assert_allclose(ang[0], 1.0, rtol=1e-12)
            ratios = ang[1:] / ang[:-1]
            np.testing.assert_allclose(ratios, ratios[0], rtol=1e-9)
            np.testing.assert_allclose(ang[-1], 1e6 ** (-(rotary_dim - 2) / rotary_dim), rtol=1e-9)


def test_rope_scores_depend_on_relative_position_only(oracle_lib):
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(128), rng.standard_normal(128)

    def score(m, n):
        return float(oracle_lib.rope_row(q, 128, m, 1e6) @ oracle_lib.rope_row(k, 128, n, 1e6))

    for m, n in [(5, 2), (300, 17), (1023, 1000)]:
        np.testing.assert_allclose(score(m, n), score(m + 111, n + 111), rtol=1e-10, atol=1e-10)
    assert abs(score(10, 3) - score(3, 10)) > 1e-3   # direction matters


def test_fused_row_equals_torch_rmsnorm_then_complex_rotation(oracle_lib):
    w = kvgen.fused_write(seqs=1, tokens_per_seq=64)
    k_in, wt = _rows(w.key), _rows(w.extra["k_norm_weight"].reshape(1, -1)).ravel()
    pos = w.positions.numpy()
    H, D = w.num_kv_heads, w.head_dim
    wt64 = torch.from_numpy(wt.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    inv_freq = 1e6 ** (-np.arange(0, D, 2) / D)
    for t in (0, 1, 33, 63):
        for h in range(H):
            x = w.key[t].view(H, D)[h].to(torch.float64)
            y = torch.nn.functional.rms_norm(x, (D,), wt64, eps=float(np.float32(1e-6))).numpy()
            z = (y[:D // 2] + 1j * y[D // 2:]) * np.exp(1j * pos[t] * inv_freq)
            ref = np.concatenate([z.real, z.imag])
            got = oracle_lib.fused_k_row_f64(k_in, wt, pos, t, h, H, D, D, 1e-6, 1e6)
            np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_fused_write_rounds_once_to_nearest_bf16(oracle_lib):
    w = kvgen.fused_write(seqs=2, tokens_per_seq=48)
    H, D, bs, nb = w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks
    slots = np.concatenate([oracle_lib.fill_slots(w.block_tables[s].numpy(), 0, int(L), bs)
                            for s, L in enumerate(w.seq_lens.tolist())])
    k_in, wt = _rows(w.key), _rows(w.extra["k_norm_weight"].reshape(1, -1)).ravel()
    pos = np.ascontiguousarray(w.positions.numpy())
    kc = _pool_u16(nb, bs, H, D)
    oracle_lib.write_fused_k_norm_rope_bf16(k_in, wt, pos, kc, slots, len(slots), H, D, D, bs,
                                            1e-6, 1e6)
    vals, pats = _bf16_finite_sorted()
    for t in (0, 47, 60):
        for h in (0, H - 1):
            exact = oracle_lib.fused_k_row_f64(k_in, wt, pos, t, h, H, D, D, 1e-6, 1e6)
            stored = kc[slots[t] // bs, slots[t] % bs, h]
            back = oracle_lib.bf16_to_f64(stored)
            # the stored value is a nearest BF16 neighbour of the exact value
            for x, b in zip(exact, back):
                k = np.searchsorted(vals, x)
                assert b in (vals[max(k - 1, 0)], vals[min(k, len(vals) - 1)])
                assert abs(b - x) <= min(abs(vals[max(k - 1, 0)] - x), abs(vals[min(k, len(vals) - 1)] - x))


# ---------------------------------------------------------------------------
# paged decode attention
# ---------------------------------------------------------------------------
def _oracle_cache(oracle_lib, w, fp8=False):
    nb, bs, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    slots = np.concatenate([oracle_lib.fill_slots(w.block_tables[s].numpy(), 0, int(L), bs)
                            for s, L in enumerate(w.seq_lens.tolist())] or [np.zeros(0, np.int64)])
    key, value = _rows(w.key), _rows(w.value)
    vc = _pool_u16(nb, bs, H, D)
    if fp8:
        kc = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
        oracle_lib.write_fp8k(key, value, kc, vc, slots, len(slots), H, D, bs, H * D, H * D,
                              w.k_scale)
    else:
        kc = _pool_u16(nb, bs, H, D)
        oracle_lib.write_bf16(key, value, kc, vc, slots, len(slots), H, D, bs, H * D, H * D)
    return kc, vc


def _dense_reference(w, kc, vc, s, window, fp8=False, fp8_v=False):
    """Gather the sequence's rows by fancy indexing on the pool viewed as
    [num_blocks, block_size, H, D], then torch's own scaled-dot-product
    attention in float64 with the window as a boolean mask."""
    L = int(w.seq_lens[s])
    bs, H, D, Hq = w.block_size, w.num_kv_heads, w.head_dim, w.num_q_heads
    p = np.arange(L)
    blocks = w.block_tables[s].numpy()[p // bs]
    if fp8:
        k = torch.from_numpy(kc[blocks, p % bs]).view(torch.float8_e4m3fn).to(torch.float64) * w.k_scale
    else:
        k = torch.from_numpy(kc[blocks, p % bs].view(np.int16)).view(torch.bfloat16).to(torch.float64)
    if fp8_v:
        v = torch.from_numpy(vc[blocks, p % bs]).view(torch.float8_e4m3fn).to(torch.float64) * w.v_scale
    else:
        v = torch.from_numpy(vc[blocks, p % bs].view(np.int16)).view(torch.bfloat16).to(torch.float64)
    q = w.q[s].view(Hq, D).to(torch.float64)
    g = Hq // H
    k = k.permute(1, 0, 2).repeat_interleave(g, 0)          # [Hq, L, D]
    v = v.permute(1, 0, 2).repeat_interleave(g, 0)
    mask = torch.ones(L, dtype=torch.bool)
    if window:
        mask[: max(0, L - window)] = False
    o = torch.nn.functional.scaled_dot_product_attention(
        q[:, None, :], k, v, attn_mask=mask[None, None, :], scale=float(np.float32(w.inv_sqrt_d)))
    return o[:, 0, :].numpy()


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("window", [0, 1, 16, 50, 1000])
def test_decode_equals_dense_attention(oracle_lib, fp8, window):
    w = kvgen.custom(21, seq_lens=[37, 100, 1, 16, 17], num_q_heads=8, num_kv_heads=2,
                     head_dim=64, block_size=16, fp8=fp8)
    kc, vc = _oracle_cache(oracle_lib, w, fp8)
    q = _rows(w.q)
    args = (w.block_tables.numpy(), w.seq_lens.numpy(), w.max_blocks_per_seq, w.num_seqs,
            w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.inv_sqrt_d)
    if fp8:
        out = oracle_lib.paged_decode_attn_fp8k(q, kc, vc, *args, w.k_scale, w.num_q_heads * w.head_dim, window)
    else:
        out = oracle_lib.paged_decode_attn_bf16(q, kc, vc, *args, w.num_q_heads * w.head_dim, window)
    for s in range(w.num_seqs):
        ref = _dense_reference(w, kc, vc, s, window, fp8)
        np.testing.assert_allclose(out[s], ref, rtol=2.0 ** -24, atol=1e-30)   # one float32 rounding
        for h in (0, w.num_q_heads - 1):
            one = oracle_lib.decode_one(q, None if fp8 else kc, kc if fp8 else None, vc,
                                        w.block_tables.numpy(), w.seq_lens.numpy(),
                                        w.max_blocks_per_seq, w.num_q_heads, w.num_kv_heads,
                                        w.head_dim, w.block_size, w.inv_sqrt_d, w.k_scale,
                                        w.num_q_heads * w.head_dim, window, s, h)
            np.testing.assert_allclose(one, ref[h], rtol=1e-12, atol=1e-12)


def test_decode_special_cases(oracle_lib):
    w = kvgen.custom(22, seq_lens=[1, 40, 0], num_q_heads=4, num_kv_heads=4, head_dim=32,
                     block_size=8)
    kc, vc = _oracle_cache(oracle_lib, w)
    q = _rows(w.q)
    common = (w.block_tables.numpy(), w.seq_lens.numpy(), w.max_blocks_per_seq, w.num_q_heads,
              w.num_kv_heads, w.head_dim, w.block_size, w.inv_sqrt_d, 1.0, w.num_q_heads * w.head_dim)
    bt = w.block_tables.numpy()
    # one position: the output is that position's V row
    o = oracle_lib.decode_one(q, kc, None, vc, *common, 0, 0, 2)
    assert np.array_equal(o, oracle_lib.bf16_to_f64(vc[bt[0, 0], 0, 2]))
    # window 1: the output is the last position's V row
    o = oracle_lib.decode_one(q, kc, None, vc, *common, 1, 1, 3)
    assert np.array_equal(o, oracle_lib.bf16_to_f64(vc[bt[1, 39 // 8], 39 % 8, 3]))
    # empty sequence: zeros
    o = oracle_lib.decode_one(q, kc, None, vc, *common, 0, 2, 1)
    assert not o.any()
    # weights are a distribution over exactly the attended positions
    o, wts = oracle_lib.decode_one(q, kc, None, vc, *common, 10, 1, 0, want_weights=True)
    assert abs(wts.sum() - 1) < 1e-14 and (wts[:30] == 0).all() and (wts[30:] > 0).all()


def test_decode_identical_keys_average_values(oracle_lib):
    w = kvgen.custom(23, seq_lens=[29], num_q_heads=2, num_kv_heads=1, head_dim=16, block_size=4)
    kc, vc = _oracle_cache(oracle_lib, w)
    kc[:] = kc[w.block_tables[0, 0], 0][None, None]         # every key row the same
    o = oracle_lib.decode_one(_rows(w.q), kc, None, vc, w.block_tables.numpy(), w.seq_lens.numpy(),
                              w.max_blocks_per_seq, 2, 1, 16, 4, w.inv_sqrt_d, 1.0, 32, 0, 0, 1)
    p = np.arange(29)
    rows = oracle_lib.bf16_to_f64(vc[w.block_tables[0].numpy()[p // 4], p % 4, 0])
    np.testing.assert_allclose(o, rows.mean(0), rtol=1e-13, atol=1e-15)


def test_decode_block_permutation_invariance(oracle_lib):
    w = kvgen.custom(24, seq_lens=[70, 33], num_q_heads=4, num_kv_heads=2, head_dim=32,
                     block_size=16, fp8=True)
    kc, vc = _oracle_cache(oracle_lib, w, fp8=True)
    q = _rows(w.q)
    args = lambda bt: (bt, w.seq_lens.numpy(), w.max_blocks_per_seq, w.num_seqs, w.num_q_heads,  # noqa: E731
                       w.num_kv_heads, w.head_dim, w.block_size, w.inv_sqrt_d, w.k_scale, 128, 0)
    base = oracle_lib.paged_decode_attn_fp8k(q, kc, vc, *args(w.block_tables.numpy()))
    perm = np.random.default_rng(5).permutation(w.num_blocks)      # new home of each block
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt = w.block_tables.numpy()
    bt2 = np.where(bt >= 0, perm[np.clip(bt, 0, None)], bt).astype(np.int32)
    moved = oracle_lib.paged_decode_attn_fp8k(q, kc2, vc2, *args(bt2))
    assert np.array_equal(base, moved)


# ---------------------------------------------------------------------------
# FP8 K and V (kv_cache.rs, reshape_and_cache_fp8 / paged_decode_attn_fp8)
# ---------------------------------------------------------------------------
def _oracle_cache_fp8(oracle_lib, w):
    nb, bs, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    slots = np.concatenate([oracle_lib.fill_slots(w.block_tables[s].numpy(), 0, int(L), bs)
                            for s, L in enumerate(w.seq_lens.tolist())] or [np.zeros(0, np.int64)])
    kc = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    vc = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    oracle_lib.write_fp8(_rows(w.key), _rows(w.value), kc, vc, slots, len(slots), H, D, bs, w.k_scale,
                         w.v_scale, H * D, H * D)
    return kc, vc


def test_write_fp8_codes_are_rounded_quotients_of_k_and_v(oracle_lib):
    H, D, bs, nb = 2, 32, 16, 7
    n = 40
    ks, vs = H * D + 16, H * D + 48          # rows padded differently, as in fused QKV buffers
    g = torch.Generator().manual_seed(12)
    key = (torch.randn(n, ks, generator=g) * 3).to(torch.bfloat16)
    value = (torch.randn(n, vs, generator=g) * 0.7).to(torch.bfloat16)
    k_scale, v_scale = np.float32(0.021), np.float32(0.0037)
    slots = np.random.default_rng(3).permutation(nb * bs)[:n].astype(np.int64)
    slots[[4, 19]] = -1
    kc = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    vc = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    oracle_lib.write_fp8(_rows(key), _rows(value), kc, vc, slots, n, H, D, bs, k_scale, v_scale, ks, vs)
    flat_k, flat_v = kc.reshape(nb * bs, H * D), vc.reshape(nb * bs, H * D)
    for src, scale, flat in ((key, k_scale, flat_k), (value, v_scale, flat_v)):
        quot = src[:, :H * D].to(torch.float32).numpy() / scale    # numpy's own binary32 division
        assert quot.dtype == np.float32
        for t in range(n):
            if slots[t] >= 0:
                want = [_e4m3_brute_force(float(x)) for x in quot[t]]
                assert np.array_equal(flat[slots[t]], np.array(want, np.uint8)), t
        untouched = np.ones(nb * bs, bool)
        untouched[slots[slots >= 0]] = False
        assert (flat[untouched] == kvgen.E4M3_NAN).all()


@pytest.mark.parametrize("window", [0, 1, 50])
def test_fp8_decode_equals_dense_attention(oracle_lib, window):
    w = kvgen.custom(25, seq_lens=[37, 100, 1, 16, 17], num_q_heads=8, num_kv_heads=2, head_dim=64,
                     block_size=16, fp8=True)
    kc, vc = _oracle_cache_fp8(oracle_lib, w)
    q = _rows(w.q)
    out = oracle_lib.paged_decode_attn_fp8(q, kc, vc, w.block_tables.numpy(), w.seq_lens.numpy(),
                                           w.max_blocks_per_seq, w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                           w.head_dim, w.block_size, w.inv_sqrt_d, w.k_scale, w.v_scale,
                                           w.num_q_heads * w.head_dim, window)
    for s in range(w.num_seqs):
        ref = _dense_reference(w, kc, vc, s, window, fp8=True, fp8_v=True)
        np.testing.assert_allclose(out[s], ref, rtol=2.0 ** -24, atol=1e-30)
        one = oracle_lib.decode_one(q, None, kc, None, w.block_tables.numpy(), w.seq_lens.numpy(),
                                    w.max_blocks_per_seq, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                    w.block_size, w.inv_sqrt_d, w.k_scale, w.num_q_heads * w.head_dim,
                                    window, s, 3, v_cache_fp8=vc, v_scale=w.v_scale)
        np.testing.assert_allclose(one, ref[3], rtol=1e-12, atol=1e-12)


def test_fp8_decode_single_position_and_v_scale_linearity(oracle_lib):
    w = kvgen.custom(26, seq_lens=[1, 90], num_q_heads=4, num_kv_heads=2, head_dim=32, block_size=16,
                     fp8=True)
    kc, vc = _oracle_cache_fp8(oracle_lib, w)
    q = _rows(w.q)
    args = lambda vs: (w.block_tables.numpy(), w.seq_lens.numpy(), w.max_blocks_per_seq, w.num_seqs,  # noqa: E731
                       w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.inv_sqrt_d, w.k_scale, vs,
                       w.num_q_heads * w.head_dim, 0)
    out = oracle_lib.paged_decode_attn_fp8(q, kc, vc, *args(w.v_scale))
    # one position: every query head of a KV head returns that row's codes times v_scale
    b0 = w.block_tables[0, 0].item()
    for h in range(w.num_q_heads):
        row = oracle_lib.e4m3_to_f64(np.ascontiguousarray(vc[b0, 0, h // 2])) * np.float64(np.float32(w.v_scale))
        assert np.array_equal(out[0, h], row.astype(np.float32))
    # the output is linear in v_scale: doubling it doubles every value exactly
    out2 = oracle_lib.paged_decode_attn_fp8(q, kc, vc, *args(2 * w.v_scale))
    assert np.array_equal(out2, 2 * out)


def test_fp8_v_decode_equals_bf16_v_decode_of_the_dequantised_rows(oracle_lib):
    # with v_scale a power of two, code * v_scale is a BF16 value: the FP8-V
    # decode must equal the FP8-K / BF16-V decode of those rows
    w = kvgen.custom(27, seq_lens=[70, 33], num_q_heads=8, num_kv_heads=2, head_dim=32, block_size=16,
                     fp8=True)
    w.v_scale = 2.0 ** -6
    kc, vc = _oracle_cache_fp8(oracle_lib, w)
    deq = oracle_lib.e4m3_to_f64(vc.ravel()) * w.v_scale
    vbf = oracle_lib.f64_to_bf16(np.nan_to_num(deq)).reshape(vc.shape)
    args = (w.block_tables.numpy(), w.seq_lens.numpy(), w.max_blocks_per_seq, w.num_seqs, w.num_q_heads,
            w.num_kv_heads, w.head_dim, w.block_size, w.inv_sqrt_d, w.k_scale)
    a = oracle_lib.paged_decode_attn_fp8(_rows(w.q), kc, vc, *args, w.v_scale, 8 * 32, 0)
    b = oracle_lib.paged_decode_attn_fp8k(_rows(w.q), kc, vbf, *args, 8 * 32, 0)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# multi-token (chunked-prefill) paged attention (kv_cache.rs, "Batched prefill
# variants (N tokens)")
# ---------------------------------------------------------------------------
def _prefill_case(seed, lens, qlens, fp8, Hq=8, H=2, D=32, bs=16):
    w = kvgen.custom(seed, seq_lens=lens, num_q_heads=Hq, num_kv_heads=H, head_dim=D, block_size=bs, fp8=fp8,
                     q_rows=max(sum(qlens), 1))
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    return w, qsl


def _prefill(oracle_lib, w, kc, vc, qsl, window, fp8, seq_lens=None, q=None):
    seq_lens = w.seq_lens.numpy() if seq_lens is None else seq_lens
    q = _rows(w.q) if q is None else q
    return oracle_lib.paged_prefill_attn(q, None if fp8 else kc, kc if fp8 else None, vc, w.block_tables.numpy(),
                                         np.ascontiguousarray(seq_lens, dtype=np.int32), qsl, w.max_blocks_per_seq,
                                         w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                         w.inv_sqrt_d, w.k_scale, w.num_q_heads * w.head_dim, window)


def _dense_causal(w, kc, vc, qsl, s, window, fp8):
    """torch's scaled_dot_product_attention in float64 over the sequence's
    gathered rows, with the causal window as an explicit boolean mask.
    fp8: False (BF16 K and V), True (E4M3 K) or "kv" (E4M3 K and V)."""
    L = int(w.seq_lens[s])
    n = int(qsl[s + 1] - qsl[s])
    bs, H, D, Hq = w.block_size, w.num_kv_heads, w.head_dim, w.num_q_heads
    p = np.arange(L)
    blocks = w.block_tables[s].numpy()[p // bs]
    if fp8:
        k = torch.from_numpy(kc[blocks, p % bs]).view(torch.float8_e4m3fn).to(torch.float64) * w.k_scale
    else:
        k = torch.from_numpy(kc[blocks, p % bs].view(np.int16)).view(torch.bfloat16).to(torch.float64)
    if fp8 == "kv":
        v = torch.from_numpy(vc[blocks, p % bs]).view(torch.float8_e4m3fn).to(torch.float64) * w.v_scale
    else:
        v = torch.from_numpy(vc[blocks, p % bs].view(np.int16)).view(torch.bfloat16).to(torch.float64)
    q = w.q[int(qsl[s]):int(qsl[s + 1])].view(n, Hq, D).permute(1, 0, 2).to(torch.float64)   # [Hq, n, D]
    g = Hq // H
    k = k.permute(1, 0, 2).repeat_interleave(g, 0)
    v = v.permute(1, 0, 2).repeat_interleave(g, 0)
    pos = torch.arange(L - n, L)[:, None]
    keys = torch.arange(L)[None, :]
    mask = keys <= pos
    if window:
        mask &= keys > pos - window
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask[None],
                                                         scale=float(np.float32(w.inv_sqrt_d)))
    return o.permute(1, 0, 2).numpy()                                                      # [n, Hq, D]


@pytest.mark.parametrize("fp8", [False, True, "kv"])
@pytest.mark.parametrize("window", [0, 1, 7, 50])
def test_prefill_equals_dense_causal_attention(oracle_lib, fp8, window):
    lens, qlens = [37, 100, 1, 16, 64], [5, 37, 1, 16, 1]
    w, qsl = _prefill_case(31, lens, qlens, fp8)
    if fp8 == "kv":
        kc, vc = _oracle_cache_fp8(oracle_lib, w)
        out = oracle_lib.paged_prefill_attn(_rows(w.q), None, kc, None, w.block_tables.numpy(), w.seq_lens.numpy(),
                                            qsl, w.max_blocks_per_seq, w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                            w.head_dim, w.block_size, w.inv_sqrt_d, w.k_scale,
                                            w.num_q_heads * w.head_dim, window, v_cache_fp8=vc, v_scale=w.v_scale)
    else:
        kc, vc = _oracle_cache(oracle_lib, w, fp8)
        out = _prefill(oracle_lib, w, kc, vc, qsl, window, fp8)
    for s in range(w.num_seqs):
        ref = _dense_causal(w, kc, vc, qsl, s, window, fp8)
        np.testing.assert_allclose(out[qsl[s]:qsl[s + 1]], ref, rtol=2.0 ** -24, atol=1e-30)


def test_prefill_last_query_is_the_decode_of_its_row(oracle_lib):
    lens, qlens = [37, 100, 16], [4, 9, 16]
    w, qsl = _prefill_case(32, lens, qlens, False)
    kc, vc = _oracle_cache(oracle_lib, w)
    out = _prefill(oracle_lib, w, kc, vc, qsl, 0, False)
    q = _rows(w.q)
    for s in range(w.num_seqs):
        last = q[qsl[s + 1] - 1][None].repeat(w.num_seqs, 0)       # that row as every sequence's query
        dec = oracle_lib.paged_decode_attn_bf16(np.ascontiguousarray(last), kc, vc, w.block_tables.numpy(),
                                                w.seq_lens.numpy(), w.max_blocks_per_seq, w.num_seqs,
                                                w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                                w.inv_sqrt_d, w.num_q_heads * w.head_dim, 0)
        assert np.array_equal(out[qsl[s + 1] - 1], dec[s])


def test_prefill_chunk_split_in_two_calls_gives_the_same_rows(oracle_lib):
    # causal attention: query j's output depends only on positions <= its own,
    # so the first part of a chunk, run with the cache length cut back to its
    # last position, reproduces those rows exactly
    lens, qlens = [90, 40], [30, 17]
    w, qsl = _prefill_case(33, lens, qlens, True)
    kc, vc = _oracle_cache(oracle_lib, w, True)
    full = _prefill(oracle_lib, w, kc, vc, qsl, 20, True)
    first = [12, 5]
    q = _rows(w.q)
    q1 = np.ascontiguousarray(np.concatenate([q[qsl[s]:qsl[s] + first[s]] for s in range(2)]))
    qsl1 = np.array([0, first[0], first[0] + first[1]], np.int32)
    lens1 = np.array([lens[s] - qlens[s] + first[s] for s in range(2)], np.int32)
    part = _prefill(oracle_lib, w, kc, vc, qsl1, 20, True, seq_lens=lens1, q=q1)
    want = np.concatenate([full[qsl[s]:qsl[s] + first[s]] for s in range(2)])
    assert np.array_equal(part, want)


@pytest.mark.parametrize("window", [0, 9])
def test_fp8_v_prefill_equals_bf16_v_prefill_of_the_dequantised_rows(oracle_lib, window):
    # with v_scale a power of two, code * v_scale is a BF16 value: the FP8 K+V
    # prefill must equal the FP8-K / BF16-V prefill of those rows
    lens, qlens = [70, 33, 5], [9, 33, 2]
    w, qsl = _prefill_case(35, lens, qlens, True)
    w.v_scale = 2.0 ** -6
    kc, vc = _oracle_cache_fp8(oracle_lib, w)
    deq = oracle_lib.e4m3_to_f64(vc.ravel()) * w.v_scale
    vbf = oracle_lib.f64_to_bf16(np.nan_to_num(deq)).reshape(vc.shape)
    a = oracle_lib.paged_prefill_attn(_rows(w.q), None, kc, None, w.block_tables.numpy(), w.seq_lens.numpy(), qsl,
                                      w.max_blocks_per_seq, w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                      w.block_size, w.inv_sqrt_d, w.k_scale, w.num_q_heads * w.head_dim, window,
                                      v_cache_fp8=vc, v_scale=w.v_scale)
    b = _prefill(oracle_lib, w, kc, vbf, qsl, window, True)
    assert np.array_equal(a, b)


def test_fp8_kv_prefill_last_query_is_the_fp8_decode_of_its_row(oracle_lib):
    lens, qlens = [37, 100, 16], [4, 9, 16]
    w, qsl = _prefill_case(36, lens, qlens, True)
    kc, vc = _oracle_cache_fp8(oracle_lib, w)
    out = oracle_lib.paged_prefill_attn(_rows(w.q), None, kc, None, w.block_tables.numpy(), w.seq_lens.numpy(),
                                        qsl, w.max_blocks_per_seq, w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                        w.head_dim, w.block_size, w.inv_sqrt_d, w.k_scale,
                                        w.num_q_heads * w.head_dim, 0, v_cache_fp8=vc, v_scale=w.v_scale)
    q = _rows(w.q)
    for s in range(w.num_seqs):
        last = np.ascontiguousarray(q[qsl[s + 1] - 1][None].repeat(w.num_seqs, 0))
        dec = oracle_lib.paged_decode_attn_fp8(last, kc, vc, w.block_tables.numpy(), w.seq_lens.numpy(),
                                               w.max_blocks_per_seq, w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                               w.head_dim, w.block_size, w.inv_sqrt_d, w.k_scale, w.v_scale,
                                               w.num_q_heads * w.head_dim, 0)
        assert np.array_equal(out[qsl[s + 1] - 1], dec[s])


def _prefill_any(oracle_lib, w, kc, vc, qsl, window, fp8, Hq, H, q, q_stride):
    """The oracle prefill for any cache format (fp8: False, True or "kv"),
    with the head counts and query rows given explicitly."""
    kv = fp8 == "kv"
    return oracle_lib.paged_prefill_attn(q, None if fp8 else kc, kc if fp8 else None, None if kv else vc,
                                         w.block_tables.numpy(), w.seq_lens.numpy(), qsl, w.max_blocks_per_seq,
                                         w.num_seqs, Hq, H, w.head_dim, w.block_size, w.inv_sqrt_d, w.k_scale,
                                         q_stride, window, v_cache_fp8=vc if kv else None, v_scale=w.v_scale)


def _cache_any(oracle_lib, w, fp8):
    return _oracle_cache_fp8(oracle_lib, w) if fp8 == "kv" else _oracle_cache(oracle_lib, w, fp8)


@pytest.mark.parametrize("fp8", [False, True, "kv"])
def test_prefill_gqa_equals_mha_over_repeated_kv_heads(oracle_lib, fp8):
    # query head h reads KV head h // g: repeating every KV head g times gives
    # an MHA cache (Hq KV heads) on which the same queries give the same rows
    lens, qlens = [37, 100, 16], [5, 30, 16]
    w, qsl = _prefill_case(37, lens, qlens, fp8, Hq=8, H=2)
    kc, vc = _cache_any(oracle_lib, w, fp8)
    g = w.num_q_heads // w.num_kv_heads
    q = _rows(w.q)
    gqa = _prefill_any(oracle_lib, w, kc, vc, qsl, 9, fp8, 8, 2, q, 8 * w.head_dim)
    kr, vr = (np.ascontiguousarray(np.repeat(c, g, axis=2)) for c in (kc, vc))
    mha = _prefill_any(oracle_lib, w, kr, vr, qsl, 9, fp8, 8, 8, q, 8 * w.head_dim)
    assert np.array_equal(gqa, mha)


@pytest.mark.parametrize("fp8", [False, True, "kv"])
def test_prefill_padded_query_rows_give_the_same_output(oracle_lib, fp8):
    lens, qlens = [37, 100], [5, 30]
    w, qsl = _prefill_case(38, lens, qlens, fp8)
    kc, vc = _cache_any(oracle_lib, w, fp8)
    q = _rows(w.q)
    row = q.shape[1]
    padded = np.full((q.shape[0], row + 40), 0x7FC0, np.uint16)   # NaN padding must never be read
    padded[:, :row] = q
    a = _prefill_any(oracle_lib, w, kc, vc, qsl, 0, fp8, w.num_q_heads, w.num_kv_heads, q, row)
    b = _prefill_any(oracle_lib, w, kc, vc, qsl, 0, fp8, w.num_q_heads, w.num_kv_heads, padded, row + 40)
    assert np.array_equal(a, b) and np.isfinite(a).all()


def test_prefill_queries_before_position_zero_give_zeros(oracle_lib):
    lens, qlens = [3, 10], [5, 2]                # sequence 0 has more queries than positions
    w, qsl = _prefill_case(34, lens, qlens, False)
    kc, vc = _oracle_cache(oracle_lib, w)
    out = _prefill(oracle_lib, w, kc, vc, qsl, 0, False)
    assert not out[:2].any() and np.isfinite(out).all() and out[2:5].any()


# ---------------------------------------------------------------------------
# next rows: MRoPE-interleaved fused write and the FP8-output fused write
# (kv_cache.rs, fused_k_norm_rope_cache_write_bf16_mrope / _fp8)
# ---------------------------------------------------------------------------
def test_mrope_with_equal_positions_is_the_scalar_rope(oracle_lib):
    y = np.random.default_rng(9).standard_normal(128)
    for pos in (0, 5, 1023, 77777):
        assert np.array_equal(oracle_lib.rope_row_mrope(y, 128, [pos, pos, pos], 1e6),
                              oracle_lib.rope_row(y, 128, pos, 1e6))


def test_mrope_pair_uses_position_of_its_index_mod_3(oracle_lib):
    rng = np.random.default_rng(10)
    y = rng.standard_normal(128)
    pos3 = (1, 2, 3)                         # small: no angle wraps
    out = oracle_lib.rope_row_mrope(y, 128, pos3, 1e6)
    z_in = y[:64] + 1j * y[64:]
    z_out = out[:64] + 1j * out[64:]
    np.testing.assert_allclose(np.abs(z_out), np.abs(z_in), rtol=1e-13)
    ang = np.angle(z_out / z_in)
    per_pos = ang / np.array([pos3[i % 3] for i in range(64)])   # the frequency ladder alone
    np.testing.assert_allclose(per_pos[0], 1.0, rtol=1e-12)
    np.testing.assert_allclose(per_pos[1:] / per_pos[:-1], 1e6 ** (-2 / 128), rtol=1e-9)


def test_mrope_fused_row_equals_torch_rmsnorm_then_complex_rotation(oracle_lib):
    w = kvgen.fused_write(seqs=1, tokens_per_seq=16)
    H, D = w.num_kv_heads, w.head_dim
    k_in, wt = _rows(w.key), _rows(w.extra["k_norm_weight"].reshape(1, -1)).ravel()
    rng = np.random.default_rng(11)
    pt, ph, pw = (np.ascontiguousarray(rng.integers(0, 5000, 16).astype(np.int32)) for _ in range(3))
    wt64 = torch.from_numpy(wt.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    inv_freq = 1e6 ** (-np.arange(0, D, 2) / D)
    for t in (0, 7, 15):
        pos = np.array([(pt, ph, pw)[i % 3][t] for i in range(D // 2)], np.float64)
        for h in (0, H - 1):
            x = w.key[t].view(H, D)[h].to(torch.float64)
            y = torch.nn.functional.rms_norm(x, (D,), wt64, eps=float(np.float32(1e-6))).numpy()
            z = (y[:D // 2] + 1j * y[D // 2:]) * np.exp(1j * pos * inv_freq)
            ref = np.concatenate([z.real, z.imag])
            got = oracle_lib.fused_k_row_f64_mrope(k_in, wt, pt, ph, pw, t, h, H, D, D, 1e-6, 1e6)
            np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_e4m3_encode_f64_agrees_with_binary32_encode_and_brute_force(oracle_lib):
    x32 = torch.from_numpy(ALL_BF16.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    with np.errstate(invalid="ignore"):       # the NaN patterns
        assert np.array_equal(oracle_lib.e4m3_encode_f64(x32.astype(np.float64)), oracle_lib.e4m3_encode(x32))
    rng = np.random.default_rng(12)
    xs = rng.standard_normal(4000) * 10.0 ** rng.uniform(-4, 3, 4000)
    got = oracle_lib.e4m3_encode_f64(xs)
    want = np.array([_e4m3_brute_force(float(v)) for v in xs], np.uint8)
    assert np.array_equal(got, want)


def test_fp8_fused_write_codes_are_nearest_to_scaled_exact_rows(oracle_lib):
    w = kvgen.fused_write(seqs=1, tokens_per_seq=32)
    H, D, bs, nb = w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks
    k_in, wt = _rows(w.key), _rows(w.extra["k_norm_weight"].reshape(1, -1)).ravel()
    pos = np.ascontiguousarray(w.positions.numpy())
    slots = oracle_lib.fill_slots(w.block_tables[0].numpy(), 0, 32, bs)
    inv_scale = np.float32(448.0 / 30.0)
    kc = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    oracle_lib.write_fused_k_norm_rope_fp8(k_in, wt, pos, kc, slots, 32, H, D, D, bs, 1e-6, 1e6, inv_scale)
    wt64 = torch.from_numpy(wt.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    inv_freq = 1e6 ** (-np.arange(0, D, 2) / D)
    for t in (0, 31):
        for h in (0, 5):
            x = w.key[t].view(H, D)[h].to(torch.float64)
            y = torch.nn.functional.rms_norm(x, (D,), wt64, eps=float(np.float32(1e-6))).numpy()
            z = (y[:D // 2] + 1j * y[D // 2:]) * np.exp(1j * pos[t] * inv_freq)
            v = np.concatenate([z.real, z.imag]) * float(inv_scale)
            want = np.array([_e4m3_brute_force(float(a)) for a in v], np.uint8)
            assert np.array_equal(kc[slots[t] // bs, slots[t] % bs, h], want)
