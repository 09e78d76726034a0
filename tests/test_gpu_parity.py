"""GPU parity: every C-ABI call against the CPU oracle on the same seeded
inputs. Bit-exact for slot filling, the BF16 copies and the FP8 E4M3 codes;
at most 1 BF16 ulp per element for the fused K norm/RoPE write; decode
outputs within max abs error 2e-3 and max relative error 1e-2 (relative error
taken where |reference| >= 0.2) of the fp64 oracle. Caches start filled with
NaN patterns, so a kernel that touches an unattended row or a padding slot
shows up as NaN or as a changed pool byte."""
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import kvgen
import oracle
import paged_kv_cache_fill_gb300 as pk

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

DEV = torch.device("cuda")
ABS_TOL, REL_TOL, REL_FLOOR = 2e-3, 1e-2, 0.2


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    pk.kv_set_decode_workspace(None)
    _WORKSPACE.clear()


def u16(t: torch.Tensor) -> np.ndarray:
    return np.ascontiguousarray(t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16))


def ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64) & 0xFFFF
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


def assert_decode_close(got: np.ndarray, ref: np.ndarray, what=""):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert err.max() <= ABS_TOL, f"{what}: max abs err {err.max():.3e}"
    big = np.abs(ref) >= REL_FLOOR
    if big.any():
        rel = (err[big] / np.abs(ref[big])).max()
        assert rel <= REL_TOL, f"{what}: max rel err {rel:.3e}"


def oracle_slots(w) -> np.ndarray:
    parts = [oracle.fill_slots(w.block_tables[s].cpu().numpy(), 0, int(L), w.block_size)
             for s, L in enumerate(w.seq_lens.tolist())]
    return np.concatenate(parts) if parts else np.zeros(0, np.int64)


def gpu_slots(w) -> torch.Tensor:
    tables = w.block_tables.to(DEV)
    slots = torch.empty(w.num_tokens, dtype=torch.int64, device=DEV)
    off = 0
    for s, L in enumerate(w.seq_lens.tolist()):
        pk.kv_fill_slots(slots[off:off + L], tables[s], 0, L, w.block_size)
        off += L
    return slots


_WORKSPACE = []  # the registered workspace stays alive until the next registration


def with_workspace(w, on=True):
    _WORKSPACE.clear()
    if not on:
        pk.kv_set_decode_workspace(None)
        return None
    n = pk.kv_decode_workspace_bytes(w.max_blocks_per_seq, w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                     w.head_dim, w.block_size)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    pk.kv_set_decode_workspace(ws)
    _WORKSPACE.append(ws)
    return ws


def test_binding_refuses_host_and_strided_tensors():
    """The C entry points take raw pointers: the binding refuses a host
    tensor and a non-contiguous view before any launch."""
    table = torch.arange(8, dtype=torch.int32, device=DEV)
    slots = torch.empty(16, dtype=torch.int64, device=DEV)
    with pytest.raises(ValueError, match="CUDA device"):
        pk.kv_fill_slots(slots, table.cpu(), 0, 16, 2)
    with pytest.raises(ValueError, match="contiguous"):
        pk.kv_fill_slots(torch.empty(32, dtype=torch.int64, device=DEV)[::2], table, 0, 16, 2)


# ---------------------------------------------------------------------------
# slot filling
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("block_size", [1, 3, 16, 64, 256])
def test_fill_slots_bit_exact(block_size):
    rng = np.random.default_rng(block_size)
    table = rng.permutation(5000).astype(np.int32)[:300]
    table[7] = -1                                     # a padding block
    t_dev = torch.from_numpy(table).to(DEV)
    for start, count in [(0, 1), (0, 300 * block_size), (5, 17), (block_size - 1, 2 * block_size + 3),
                         (300 * block_size - 1, 1), (123, 9999)]:
        count = min(count, 300 * block_size - start)
        got = torch.full((count,), -7, dtype=torch.int64, device=DEV)
        pk.kv_fill_slots(got, t_dev, start, count, block_size)
        assert np.array_equal(got.cpu().numpy(), oracle.fill_slots(table, start, count, block_size))


# ---------------------------------------------------------------------------
# BF16, V-only and FP8-K writes
# ---------------------------------------------------------------------------
def _write_case(key_stride_pad=0, seed=31, H=8, D=128, bs=16, lens=(37, 100, 5, 64)):
    w = kvgen.custom(seed, seq_lens=list(lens), num_q_heads=H, num_kv_heads=H, head_dim=D, block_size=bs)
    row = H * D
    n = w.num_tokens
    stride = row + key_stride_pad
    g = torch.Generator().manual_seed(seed)
    key = torch.randn((n, stride), generator=g).to(torch.bfloat16)
    value = torch.randn((n, stride), generator=g).to(torch.bfloat16)
    slots_ref = oracle_slots(w)
    slots_ref[::11] = -1                              # some padding tokens
    return w, key, value, stride, slots_ref


@pytest.mark.parametrize("pad", [0, 8, 3])           # 3: unaligned rows take the scalar path
def test_write_bf16_and_v_only_bit_exact(pad):
    w, key, value, stride, slots_ref = _write_case(pad)
    H, D, bs, nb, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.num_tokens
    slots = torch.from_numpy(slots_ref).to(DEV)
    kc = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    vc = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    pk.kv_write_bf16(key.to(DEV), value.to(DEV), kc, vc, slots, n, H, D, bs, stride, stride)
    kr = np.full((nb, bs, H, D), kvgen.BF16_NAN, np.uint16)
    vr = kr.copy()
    oracle.write_bf16(u16(key), u16(value), kr, vr, slots_ref, n, H, D, bs, stride, stride)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    v2 = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    pk.kv_write_v_only(value.to(DEV), v2, slots, n, H, D, bs, stride)
    assert np.array_equal(u16(v2), vr)


def _scales_to_sweep():
    """Scales for the exhaustive FP8 tests: workload-like ones, 48 seeded
    log-uniform ones over [2^-60, 2^60] (the division-free quotient's range),
    significands of all ones and of 1 + 2^-23 (the hardest reciprocals), the
    range ends, and scales outside it (the exact-division route)."""
    rng = np.random.default_rng(77)
    sweep = [1.0, 20.0 / 448.0, 3.0e-3, 5.5 / 448.0]
    sweep += list(2.0 ** rng.uniform(-60, 60, 48))
    for e in (-60, -31, -7, 0, 9, 59):
        sweep += [np.nextafter(np.float32(2.0 ** (e + 1)), np.float32(0)), np.float32(2.0 ** e) * np.float32(1 + 2**-23)]
    sweep += [2.0 ** -60, 2.0 ** 60, 2.0 ** -61, 2.0 ** 61, 1e-30, 3e25, 1e-40]
    return [float(np.float32(x)) for x in sweep]


def test_write_fp8k_exhaustive_over_bf16_patterns():
    """All 65536 BF16 bit patterns as K (64 tokens x 1024), over the scale
    sweep: bit-exact codes on both quotient routes."""
    H, D, bs = 8, 128, 16
    n = 64
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(n, H * D)
    key = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16)
    value = torch.randn((n, H * D), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    slots_ref = np.arange(n, dtype=np.int64)[::-1].copy()
    slots = torch.from_numpy(slots_ref).to(DEV)
    for k_scale in _scales_to_sweep():
        kc = kvgen.poisoned_pool(n // bs, bs, H, D, "fp8", DEV)
        vc = kvgen.poisoned_pool(n // bs, bs, H, D, "bf16", DEV)
        pk.kv_write_fp8k(key.to(DEV), value.to(DEV), kc, vc, slots, n, H, D, bs, H * D, H * D, k_scale)
        kr = np.full((n // bs, bs, H, D), kvgen.E4M3_NAN, np.uint8)
        vr = np.full((n // bs, bs, H, D), kvgen.BF16_NAN, np.uint16)
        oracle.write_fp8k(u16(key), u16(value), kr, vr, slots_ref, n, H, D, bs, H * D, H * D, k_scale)
        got = kc.cpu().numpy()
        bad = np.flatnonzero(got.ravel() != kr.ravel())
        assert bad.size == 0, (k_scale, bad[:8], got.ravel()[bad[:8]], kr.ravel()[bad[:8]])
        assert np.array_equal(u16(vc), vr)


@pytest.mark.parametrize("pad", [0, 8, 3])           # 3: unaligned rows take the scalar path
def test_write_fp8_k_and_v_bit_exact(pad):
    w, key, value, stride, slots_ref = _write_case(pad, seed=33)
    H, D, bs, nb, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.num_tokens
    vstride = stride + (8 if pad != 3 else 5)         # K and V rows at different strides
    value = torch.cat([value, torch.randn((n, vstride - stride), generator=torch.Generator().manual_seed(4))
                       .to(torch.bfloat16)], 1).contiguous()
    slots = torch.from_numpy(slots_ref).to(DEV)
    for k_scale, v_scale in ((20.0 / 448.0, 4.5 / 448.0), (1.0, 1.0), (3.0e-3, 0.5)):
        kc = kvgen.poisoned_pool(nb, bs, H, D, "fp8", DEV)
        vc = kvgen.poisoned_pool(nb, bs, H, D, "fp8", DEV)
        pk.kv_write_fp8(key.to(DEV), value.to(DEV), kc, vc, slots, n, H, D, bs, k_scale, v_scale, stride, vstride)
        kr = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
        vr = kr.copy()
        oracle.write_fp8(u16(key), u16(value), kr, vr, slots_ref, n, H, D, bs, k_scale, v_scale, stride, vstride)
        assert np.array_equal(kc.cpu().numpy(), kr) and np.array_equal(vc.cpu().numpy(), vr), (k_scale, v_scale)


def test_write_fp8_v_exhaustive_over_bf16_patterns():
    """All 65536 BF16 bit patterns as V of the FP8 K+V write, with K and V
    scales from the sweep (paired so that some calls mix the two routes)."""
    H, D, bs = 8, 128, 16
    n = 64
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(n, H * D)
    value = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16)
    key = torch.from_numpy(np.ascontiguousarray(pats[::-1]).view(np.int16)).view(torch.bfloat16)
    slots_ref = np.arange(n, dtype=np.int64)
    slots = torch.from_numpy(slots_ref).to(DEV)
    sweep = _scales_to_sweep()
    for k_scale, v_scale in zip(sweep, sweep[7:] + sweep[:7]):
        kc = kvgen.poisoned_pool(n // bs, bs, H, D, "fp8", DEV)
        vc = kvgen.poisoned_pool(n // bs, bs, H, D, "fp8", DEV)
        pk.kv_write_fp8(key.to(DEV), value.to(DEV), kc, vc, slots, n, H, D, bs, k_scale, v_scale, H * D, H * D)
        kr = np.full((n // bs, bs, H, D), kvgen.E4M3_NAN, np.uint8)
        vr = kr.copy()
        oracle.write_fp8(u16(key), u16(value), kr, vr, slots_ref, n, H, D, bs, k_scale, v_scale, H * D, H * D)
        assert np.array_equal(kc.cpu().numpy(), kr), (k_scale, v_scale)
        assert np.array_equal(vc.cpu().numpy(), vr), (k_scale, v_scale)


def test_write_fp8k_workload_bit_exact():
    w = kvgen.custom(41, seq_lens=[300, 17, 1, 64], num_q_heads=8, num_kv_heads=8, head_dim=128,
                     block_size=16, fp8=True)
    H, D, bs, nb, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.num_tokens
    slots_ref = oracle_slots(w)
    slots = gpu_slots(w)
    assert np.array_equal(slots.cpu().numpy(), slots_ref)
    kc = kvgen.poisoned_pool(nb, bs, H, D, "fp8", DEV)
    vc = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    pk.kv_write_fp8k(w.key.to(DEV), w.value.to(DEV), kc, vc, slots, n, H, D, bs, H * D, H * D, w.k_scale)
    kr = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    vr = np.full((nb, bs, H, D), kvgen.BF16_NAN, np.uint16)
    oracle.write_fp8k(u16(w.key), u16(w.value), kr, vr, slots_ref, n, H, D, bs, H * D, H * D, w.k_scale)
    assert np.array_equal(kc.cpu().numpy(), kr) and np.array_equal(u16(vc), vr)


# ---------------------------------------------------------------------------
# fused K norm / RoPE write
# ---------------------------------------------------------------------------
def _fused_check(w, rotary_dim, theta, eps, positions=None, slots_ref=None):
    H, D, bs, nb, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.num_tokens
    wt = w.extra.get("k_norm_weight")
    if wt is None:
        wt = (torch.rand(D, generator=torch.Generator().manual_seed(D)) + 0.5).to(torch.bfloat16)
    pos = positions if positions is not None else w.positions
    if slots_ref is None:
        slots_ref = oracle_slots(w)
    slots = torch.from_numpy(slots_ref).to(DEV)
    kc = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    pk.kv_write_fused_k_norm_rope_bf16(w.key.to(DEV), wt.to(DEV), pos.to(DEV), kc, slots, n, H, D,
                                       rotary_dim, bs, eps, theta)
    kr = np.full((nb, bs, H, D), kvgen.BF16_NAN, np.uint16)
    oracle.write_fused_k_norm_rope_bf16(u16(w.key), u16(wt), np.ascontiguousarray(pos.cpu().numpy()), kr,
                                        slots_ref, n, H, D, rotary_dim, bs, eps, theta)
    got = u16(kc)
    d = np.abs(ordered(got) - ordered(kr))
    return int(d.max()), int((d == 1).sum()), d.size


def test_fused_write_full_workload_within_one_ulp():
    w = kvgen.fused_write()
    worst, ones, total = _fused_check(w, 128, 1e6, 1e-6)
    print(f"fused write: max {worst} ulp, {ones} of {total} elements at 1 ulp")
    assert worst <= 1


@pytest.mark.parametrize("D,R,theta", [(64, 64, 1e4), (128, 64, 1e6), (256, 256, 5e5), (128, 8, 1e4),
                                       (256, 128, 1e6)])
def test_fused_write_shapes(D, R, theta):
    w = kvgen.custom(50 + D + R, seq_lens=[33, 70, 1], num_q_heads=4, num_kv_heads=4, head_dim=D,
                     block_size=16, key_sigma=4.0)
    worst, _, _ = _fused_check(w, R, theta, 1e-5)
    assert worst <= 1


def test_fused_write_large_positions_and_padding():
    w = kvgen.custom(77, seq_lens=[200, 57], num_q_heads=8, num_kv_heads=8, head_dim=128, block_size=16,
                     key_sigma=18.0)
    g = torch.Generator().manual_seed(8)
    pos = torch.cat([torch.randint(0, 1 << 20, (100,), generator=g), torch.arange(65530, 65630),
                     torch.randint(0, 2000, (57,), generator=g)]).to(torch.int32)
    slots_ref = oracle_slots(w)
    slots_ref[::7] = -3
    worst, _, _ = _fused_check(w, 128, 1e6, 1e-6, positions=pos, slots_ref=slots_ref)
    assert worst <= 1


def _norm_weight(D):
    return (torch.rand(D, generator=torch.Generator().manual_seed(D)) + 0.5).to(torch.bfloat16)


def _mrope_check(w, rotary_dim, theta, eps, pos3):
    H, D, bs, nb, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.num_tokens
    wt = _norm_weight(D)
    slots_ref = oracle_slots(w)
    slots = torch.from_numpy(slots_ref).to(DEV)
    kc = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    pt, ph, pw = (p.to(DEV) for p in pos3)
    pk.kv_write_fused_k_norm_rope_bf16_mrope(w.key.to(DEV), wt.to(DEV), pt, ph, pw, kc, slots, n, H, D,
                                             rotary_dim, bs, eps, theta)
    kr = np.full((nb, bs, H, D), kvgen.BF16_NAN, np.uint16)
    oracle.write_fused_k_norm_rope_bf16_mrope(u16(w.key), u16(wt), *(np.ascontiguousarray(p.numpy()) for p in pos3),
                                              kr, slots_ref, n, H, D, rotary_dim, bs, eps, theta)
    got = u16(kc)
    return int(np.abs(ordered(got) - ordered(kr)).max()), got


@pytest.mark.parametrize("D,R,theta", [(128, 128, 1e6), (128, 64, 1e4), (64, 48, 1e4), (256, 256, 5e5)])
def test_mrope_write_within_one_ulp(D, R, theta):
    w = kvgen.custom(90 + D + R, seq_lens=[300, 41, 1], num_q_heads=8, num_kv_heads=4, head_dim=D,
                     block_size=16, key_sigma=4.0)
    g = torch.Generator().manual_seed(R)
    n = w.num_tokens
    # text-like runs (t = h = w) next to image-like tokens with spread h/w and
    # a few positions past 2^16
    pt = torch.randint(0, 4096, (n,), generator=g).to(torch.int32)
    ph = torch.where(torch.arange(n) % 3 == 0, pt, torch.randint(0, 1 << 17, (n,), generator=g).to(torch.int32))
    pw = torch.randint(0, 512, (n,), generator=g).to(torch.int32)
    worst, _ = _mrope_check(w, R, theta, 1e-6, (pt, ph, pw))
    assert worst <= 1


def test_mrope_with_equal_positions_is_bit_identical_to_plain_fused_write():
    w = kvgen.custom(4242, seq_lens=[500, 12], num_q_heads=8, num_kv_heads=8, head_dim=128, block_size=16,
                     key_sigma=6.0)
    H, D, bs, nb, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.num_tokens
    pos = torch.randint(0, 1 << 20, (n,), generator=torch.Generator().manual_seed(5)).to(torch.int32)
    _, got = _mrope_check(w, 128, 1e6, 1e-6, (pos, pos, pos))
    wt = _norm_weight(D).to(DEV)
    kc = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    pk.kv_write_fused_k_norm_rope_bf16(w.key.to(DEV), wt, pos.to(DEV), kc, torch.from_numpy(oracle_slots(w)).to(DEV),
                                       n, H, D, 128, bs, 1e-6, 1e6)
    assert np.array_equal(got, u16(kc))


def _fp8_fused_check(w, rotary_dim, theta, eps, inv_scale, slots_ref=None):
    """Codes must equal the oracle's, except where the exact scaled value lies
    within a relative 2^-19 of the midpoint between the two codes (the kernel
    works in binary32 and its reciprocal square root is not correctly
    rounded); there the other neighbour is accepted. Returns the number of
    such accepted differences."""
    H, D, bs, nb, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.num_tokens
    wt = _norm_weight(D)
    if slots_ref is None:
        slots_ref = oracle_slots(w)
    kc = kvgen.poisoned_pool(nb, bs, H, D, "fp8", DEV)
    pk.kv_write_fused_k_norm_rope_fp8(w.key.to(DEV), wt.to(DEV), w.positions.to(DEV), kc,
                                      torch.from_numpy(slots_ref).to(DEV), n, H, D, rotary_dim, bs, eps, theta,
                                      inv_scale)
    kr = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    k16, w16, pos = u16(w.key), u16(wt), np.ascontiguousarray(w.positions.numpy())
    oracle.write_fused_k_norm_rope_fp8(k16, w16, pos, kr, slots_ref, n, H, D, rotary_dim, bs, eps, theta,
                                       inv_scale)
    got = kc.cpu().numpy()
    bad = np.argwhere(got != kr)
    if len(bad) == 0:
        return 0
    token_of_slot = {int(s): t for t, s in enumerate(slots_ref) if s >= 0}
    exact_rows = {}
    for blk, off, h, d in bad:
        t = token_of_slot.get(int(blk) * bs + int(off))
        assert t is not None, "a slot no token maps to was written"
        if (t, h) not in exact_rows:
            exact_rows[(t, h)] = oracle.fused_k_row_f64(k16, w16, pos, t, h, H, D, rotary_dim, eps, theta)
        v = exact_rows[(t, h)][d] * np.float64(np.float32(inv_scale))
        a, b = oracle.e4m3_to_f64(np.array([got[blk, off, h, d], kr[blk, off, h, d]], np.uint8))
        mid = 0.5 * (a + b)
        assert abs(int(got[blk, off, h, d] & 0x7F) - int(kr[blk, off, h, d] & 0x7F)) == 1, (v, a, b)
        assert abs(v - mid) <= abs(mid) * 2.0 ** -19, (v, a, b)
    return len(bad)


def test_fp8_fused_write_full_workload():
    w = kvgen.fused_write()
    # the FP8-K decode's scale rule: the largest |K| after norm and rotation
    # maps near the top of the E4M3 range
    ties = _fp8_fused_check(w, 128, 1e6, 1e-6, inv_scale=448.0 / 6.0)
    print(f"fused FP8 write: {ties} codes at a rounding midpoint")
    assert ties <= w.num_tokens * w.num_kv_heads * w.head_dim * 1e-4


@pytest.mark.parametrize("D,R,inv_scale", [(64, 64, 30.0), (128, 32, 100.0), (256, 256, 1.0), (128, 128, 1e4)])
def test_fp8_fused_write_shapes_scales_and_saturation(D, R, inv_scale):
    # inv_scale 1e4 drives most codes into saturation (+-448); 1.0 leaves many
    # in the subnormal range
    w = kvgen.custom(60 + D + R, seq_lens=[65, 3], num_q_heads=4, num_kv_heads=2, head_dim=D, block_size=16,
                     key_sigma=3.0)
    slots_ref = oracle_slots(w)
    slots_ref[5::9] = -1
    _fp8_fused_check(w, R, 1e4, 1e-5, inv_scale, slots_ref=slots_ref)


# ---------------------------------------------------------------------------
# paged decode
# ---------------------------------------------------------------------------
def _caches(w, fp8):
    """The same cache on both sides: the GPU write kernels fill the device
    pools, the oracle's writes fill host pools. fp8: False (BF16 K and V),
    True (FP8 K, BF16 V) or "kv" (FP8 K and V)."""
    H, D, bs, nb, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.num_tokens
    slots_ref = oracle_slots(w)
    slots = gpu_slots(w)
    if fp8 == "kv":
        kc, vc = (kvgen.poisoned_pool(nb, bs, H, D, "fp8", DEV) for _ in range(2))
        kr, vr = (np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8) for _ in range(2))
        if n:
            pk.kv_write_fp8(w.key.to(DEV), w.value.to(DEV), kc, vc, slots, n, H, D, bs, w.k_scale, w.v_scale,
                            H * D, H * D)
            oracle.write_fp8(u16(w.key), u16(w.value), kr, vr, slots_ref, n, H, D, bs, w.k_scale, w.v_scale,
                             H * D, H * D)
            assert np.array_equal(kc.cpu().numpy(), kr) and np.array_equal(vc.cpu().numpy(), vr)
        return kc, vc, kr, vr
    vc = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    vr = np.full((nb, bs, H, D), kvgen.BF16_NAN, np.uint16)
    if fp8:
        kc = kvgen.poisoned_pool(nb, bs, H, D, "fp8", DEV)
        kr = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
        if n:
            pk.kv_write_fp8k(w.key.to(DEV), w.value.to(DEV), kc, vc, slots, n, H, D, bs, H * D, H * D,
                             w.k_scale)
            oracle.write_fp8k(u16(w.key), u16(w.value), kr, vr, slots_ref, n, H, D, bs, H * D, H * D,
                              w.k_scale)
    else:
        kc = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
        kr = np.full((nb, bs, H, D), kvgen.BF16_NAN, np.uint16)
        if n:
            pk.kv_write_bf16(w.key.to(DEV), w.value.to(DEV), kc, vc, slots, n, H, D, bs, H * D, H * D)
            oracle.write_bf16(u16(w.key), u16(w.value), kr, vr, slots_ref, n, H, D, bs, H * D, H * D)
    return kc, vc, kr, vr


def _decode_gpu(w, kc, vc, window, fp8, q=None, q_stride=None):
    q = w.q if q is None else q
    q_stride = q_stride or w.num_q_heads * w.head_dim
    out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"), device=DEV)
    args = (w.block_tables.to(DEV), w.seq_lens.to(DEV), w.max_blocks_per_seq, w.num_seqs, w.num_q_heads,
            w.num_kv_heads, w.head_dim, w.block_size, w.inv_sqrt_d)
    if fp8 == "kv":
        pk.paged_decode_attn_fp8(q.to(DEV), kc, vc, out, *args, w.k_scale, w.v_scale, q_stride, window)
    elif fp8:
        pk.paged_decode_attn_fp8k(q.to(DEV), kc, vc, out, *args, w.k_scale, q_stride, window)
    else:
        pk.paged_decode_attn_bf16(q.to(DEV), kc, vc, out, *args, q_stride, window)
    return out.cpu().numpy()


def _decode_ref(w, kr, vr, window, fp8, q=None, q_stride=None):
    q = w.q if q is None else q
    q_stride = q_stride or w.num_q_heads * w.head_dim
    args = (w.block_tables.numpy(), w.seq_lens.numpy(), w.max_blocks_per_seq, w.num_seqs, w.num_q_heads,
            w.num_kv_heads, w.head_dim, w.block_size, w.inv_sqrt_d)
    if fp8 == "kv":
        return oracle.paged_decode_attn_fp8(u16(q), kr, vr, *args, w.k_scale, w.v_scale, q_stride, window)
    if fp8:
        return oracle.paged_decode_attn_fp8k(u16(q), kr, vr, *args, w.k_scale, q_stride, window)
    return oracle.paged_decode_attn_bf16(u16(q), kr, vr, *args, q_stride, window)


@pytest.mark.parametrize("split", [False, True])
def test_decode_tiny_workload(split):
    w = kvgen.tiny()
    kc, vc, kr, vr = _caches(w, False)
    with_workspace(w, split)
    assert_decode_close(_decode_gpu(w, kc, vc, 0, False), _decode_ref(w, kr, vr, 0, False), "tiny")
    assert pk.kv_get_device_error() == 0


CASES = [
    # (seq_lens, Hq, H, D, bs, windows)
    ([1, 15, 16, 17, 31, 33, 100, 0], 8, 2, 128, 16, (0, 1, 16, 17, 40)),
    ([700, 1000, 2049, 5], 32, 8, 128, 16, (0, 100, 1024)),
    ([333, 64, 65, 1], 64, 8, 128, 64, (0, 63, 200)),
    ([500, 129, 40], 16, 16, 64, 32, (0, 7)),
    ([260, 1000], 16, 1, 256, 128, (0, 300)),
    ([300, 77], 12, 1, 128, 256, (0, 50)),
    ([400, 90, 3], 6, 3, 64, 16, (0, 33)),
    ([129, 1500, 16], 32, 2, 128, 16, (0, 200)),     # the largest group (16): two 8-head tiles per KV head
    ([129, 900, 17, 2000], 32, 2, 64, 16, (0, 100)),  # head_dim 64 with two 8-head tiles per KV head
]


@pytest.mark.parametrize("fp8", [False, True, "kv"])
@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("split", [False, True])
def test_decode_cases(fp8, case, split):
    lens, Hq, H, D, bs, windows = CASES[case]
    w = kvgen.custom(100 + case, seq_lens=lens, num_q_heads=Hq, num_kv_heads=H, head_dim=D, block_size=bs,
                     fp8=bool(fp8))
    kc, vc, kr, vr = _caches(w, fp8)
    with_workspace(w, split)
    for win in windows:
        got = _decode_gpu(w, kc, vc, win, fp8)
        ref = _decode_ref(w, kr, vr, win, fp8)
        assert_decode_close(got, ref, f"case {case} window {win}")
    assert pk.kv_get_device_error() == 0


def test_decode_padded_q_stride_and_determinism():
    w = kvgen.custom(7, seq_lens=[3000, 17, 900], num_q_heads=32, num_kv_heads=8, head_dim=128,
                     block_size=16)
    kc, vc, kr, vr = _caches(w, False)
    with_workspace(w, True)
    stride = 32 * 128 + 3 * 128 + 64
    qpad = torch.zeros((w.num_seqs, stride), dtype=torch.bfloat16)
    qpad[:, :32 * 128] = w.q
    got1 = _decode_gpu(w, kc, vc, 0, False, q=qpad, q_stride=stride)
    got2 = _decode_gpu(w, kc, vc, 0, False, q=qpad, q_stride=stride)
    assert np.array_equal(got1, got2)
    assert_decode_close(got1, _decode_ref(w, kr, vr, 0, False, q=qpad, q_stride=stride))


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_stream_chunks(fp8):
    """Split-KV cuts the tiles of all (sequence, head group) pairs, taken in
    sequence order, into equal chunks. Here: sequences that straddle chunk
    boundaries, empty sequences between them (their rows are written as
    zeros by the combine), two head groups per sequence (16 KV heads), and
    the same decode with workspaces that hold only 3 and 2 pieces per
    sequence (longer chunks); every output against the oracle, and repeats
    bit-identical."""
    lens = [0, 5000, 3, 0, 777, 16, 17, 12000, 0, 1, 4097, 300]
    Hq, H, D, bs = 64, 16, 128, 16
    w = kvgen.custom(31, seq_lens=lens, num_q_heads=Hq, num_kv_heads=H, head_dim=D, block_size=bs, fp8=fp8)
    kc, vc, kr, vr = _caches(w, fp8)
    ref = _decode_ref(w, kr, vr, 0, fp8)
    full = pk.kv_decode_workspace_bytes(w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs)
    counts = -(-w.num_seqs * H * 4 // 256) * 256
    per_piece = w.num_seqs * Hq * (D + 2) * 4
    for pieces in (None, 3, 2):
        _WORKSPACE.clear()
        ws = torch.empty(full if pieces is None else 256 + counts + pieces * per_piece, dtype=torch.uint8,
                         device=DEV)
        pk.kv_set_decode_workspace(ws)
        _WORKSPACE.append(ws)
        got = _decode_gpu(w, kc, vc, 0, fp8)
        assert_decode_close(got, ref, f"pieces {pieces}")
        assert np.array_equal(got, _decode_gpu(w, kc, vc, 0, fp8)), f"pieces {pieces}: not deterministic"
    for win in (1, 100, 4096):
        assert_decode_close(_decode_gpu(w, kc, vc, win, fp8), _decode_ref(w, kr, vr, win, fp8), f"window {win}")
    assert pk.kv_get_device_error() == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_many_short_sequences(fp8):
    """700 sequences of 0..60 positions (about one in six empty): each chunk
    of the tile stream spans dozens of sequences, the producer's walk scans
    sequence counts 32 at a time many times over, and the empty sequences'
    rows are written as zeros; with and without split-KV and a window."""
    g = np.random.default_rng(77)
    lens = [int(x) if x > 9 else 0 for x in g.integers(0, 61, 700)]
    w = kvgen.custom(32, seq_lens=lens, num_q_heads=16, num_kv_heads=4, head_dim=128, block_size=16, fp8=fp8)
    kc, vc, kr, vr = _caches(w, fp8)
    for split in (True, False):
        with_workspace(w, split)
        for win in (0, 7):
            assert_decode_close(_decode_gpu(w, kc, vc, win, fp8), _decode_ref(w, kr, vr, win, fp8),
                                f"split {split} window {win}")
    assert pk.kv_get_device_error() == 0


def test_decode_clamps_overlong_sequence_and_flags_it():
    w = kvgen.custom(8, seq_lens=[40], num_q_heads=4, num_kv_heads=2, head_dim=128, block_size=16)
    kc, vc, kr, vr = _caches(w, False)
    long = kvgen.Workload(**{**w.__dict__, "seq_lens": torch.tensor([10_000], dtype=torch.int32)})
    pk.kv_get_device_error()
    got = _decode_gpu(long, kc, vc, 0, False)
    assert pk.kv_get_device_error() & 2
    # clamped to the table's 3 blocks = 48 positions, 8 of which hold NaN poison in
    # the last block: the clamp must not read past the table, and the output is
    # finite where the clamped range holds data only; here it does not
    assert got.shape == (1, 4, 128)


# ---------------------------------------------------------------------------
# multi-token (chunked-prefill) paged attention
# ---------------------------------------------------------------------------
def _prefill_gpu(w, kc, vc, qsl, window, fp8, q_stride=None):
    n_q = int(qsl[-1])
    q_stride = q_stride or w.num_q_heads * w.head_dim
    out = torch.full((max(n_q, 1), w.num_q_heads, w.head_dim), float("nan"), device=DEV)
    args = (w.block_tables.to(DEV), w.seq_lens.to(DEV), torch.from_numpy(qsl).to(DEV), w.max_blocks_per_seq,
            w.num_seqs, n_q, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.inv_sqrt_d)
    q = w.q.to(DEV)
    if fp8 == "kv":
        pk.paged_prefill_attn_fp8(q, kc, vc, out, *args, w.k_scale, w.v_scale, q_stride, window)
    elif fp8:
        pk.paged_prefill_attn_fp8k(q, kc, vc, out, *args, w.k_scale, q_stride, window)
    else:
        pk.paged_prefill_attn_bf16(q, kc, vc, out, *args, q_stride, window)
    return out[:n_q].cpu().numpy()


def _prefill_ref(w, kr, vr, qsl, window, fp8):
    kv = fp8 == "kv"
    return oracle.paged_prefill_attn(u16(w.q), None if fp8 else kr, kr if fp8 else None, None if kv else vr,
                                     w.block_tables.numpy(), w.seq_lens.numpy(), qsl, w.max_blocks_per_seq,
                                     w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                     w.inv_sqrt_d, w.k_scale, w.num_q_heads * w.head_dim, window,
                                     v_cache_fp8=vr if kv else None, v_scale=w.v_scale)


PREFILL_CASES = [
    # (seq_lens, query tokens per sequence, Hq, H, D, bs, windows)
    ([37, 100, 1, 16, 300, 65], [37, 20, 1, 16, 129, 1], 8, 2, 128, 16, (0, 1, 17, 100)),
    ([700, 1000, 2049, 5], [700, 64, 333, 5], 32, 8, 128, 16, (0, 256)),
    ([333, 64, 129], [100, 64, 3], 64, 8, 128, 64, (0, 63)),
    ([500, 129, 40], [77, 129, 40], 16, 16, 64, 32, (0, 7)),
    ([260, 1000], [260, 50], 16, 1, 128, 128, (0, 300)),
    ([300, 77, 90], [31, 77, 90], 12, 4, 64, 256, (0, 50)),
    ([3, 10, 0, 50], [5, 2, 0, 50], 8, 2, 128, 16, (0, 4)),      # more queries than positions; an empty sequence
]


@pytest.mark.parametrize("fp8", [False, True, "kv"])
@pytest.mark.parametrize("case", range(len(PREFILL_CASES)))
def test_prefill_cases(fp8, case):
    lens, qlens, Hq, H, D, bs, windows = PREFILL_CASES[case]
    w = kvgen.custom(200 + case, seq_lens=lens, num_q_heads=Hq, num_kv_heads=H, head_dim=D, block_size=bs,
                     fp8=fp8, q_rows=max(sum(qlens), 1))
    kc, vc, kr, vr = _caches(w, fp8)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    for win in windows:
        got = _prefill_gpu(w, kc, vc, qsl, win, fp8)
        ref = _prefill_ref(w, kr, vr, qsl, win, fp8)
        assert_decode_close(got, ref, f"prefill case {case} window {win}")
    assert pk.kv_get_device_error() == 0


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("log2_scale", [20, -12])
def test_prefill_bf16_v_range(fp8, log2_scale):
    """BF16 V enters the chunked prefill's PV product as v * 2^-8 rounded to
    f16: exact for 2^-6 <= |v| < 2^24, within 2^-17 (absolute) below. V
    scaled by 2^20 (|v| up to ~2^22.5) must give the unit-scale result
    times 2^20 within the usual bound; V scaled by 2^-12 (every |v| below
    2^-6) must stay within 2^-17 per value plus the weights' f16 rounding
    (2^-11 relative) of the oracle's output."""
    lens, qlens, Hq, H, D, bs, _ = PREFILL_CASES[1]
    w = kvgen.custom(240 + (log2_scale > 0), seq_lens=lens, num_q_heads=Hq, num_kv_heads=H, head_dim=D,
                     block_size=bs, fp8=fp8, q_rows=sum(qlens))
    scale = 2.0 ** log2_scale
    w.value = (w.value.float() * scale).to(torch.bfloat16)   # exact: a power of two
    vmax = float(w.value.float().abs().max())
    assert (vmax < 2.0 ** 24) if log2_scale > 0 else (vmax < 2.0 ** -6)
    kc, vc, kr, vr = _caches(w, fp8)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    for win in (0, 256):
        got = _prefill_gpu(w, kc, vc, qsl, win, fp8)
        ref = _prefill_ref(w, kr, vr, qsl, win, fp8)
        if log2_scale > 0:
            assert_decode_close(got / scale, ref / scale, f"V x 2^{log2_scale}, window {win}")
        else:
            assert np.isfinite(got).all()
            err = np.abs(got.astype(np.float64) - ref)
            assert err.max() <= 2.0 ** -17 + 2.0 ** -11 * vmax, f"V x 2^{log2_scale}: max abs err {err.max():.3e}"
    assert pk.kv_get_device_error() == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_prefill_many_sequences_of_spread_lengths(fp8):
    """120 sequences with lengths log-uniform in [1, 3000] and 1..32 queries
    each (GQA 4: single-Q-tile items, the last tile of most), so that the
    items spread over many length classes and the kernel's longest-first
    order across sequences must still reach every item once; with and
    without a window."""
    rng = np.random.default_rng(77)
    lens = np.maximum(1, np.round(np.exp(rng.uniform(0, np.log(3000), 120)))).astype(int).tolist()
    qlens = [int(min(L, rng.integers(1, 33))) for L in lens]
    w = kvgen.custom(250 + bool(fp8), seq_lens=lens, num_q_heads=16, num_kv_heads=4, head_dim=128,
                     block_size=16, fp8=fp8, q_rows=sum(qlens))
    kc, vc, kr, vr = _caches(w, fp8)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    for win in (0, 100):
        got = _prefill_gpu(w, kc, vc, qsl, win, fp8)
        ref = _prefill_ref(w, kr, vr, qsl, win, fp8)
        assert_decode_close(got, ref, f"many sequences, window {win}")
    assert pk.kv_get_device_error() == 0


def test_prefill_one_query_per_sequence_matches_the_decode():
    w = kvgen.custom(230, seq_lens=[4000, 17, 900, 1], num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16)
    kc, vc, kr, vr = _caches(w, False)
    qsl = np.arange(w.num_seqs + 1, dtype=np.int32)
    with_workspace(w, True)
    dec = _decode_gpu(w, kc, vc, 0, False)
    pre = _prefill_gpu(w, kc, vc, qsl, 0, False)
    assert_decode_close(pre, dec, "prefill of one token vs decode")
    assert_decode_close(pre, _decode_ref(w, kr, vr, 0, False), "prefill of one token vs oracle decode")


def test_prefill_flags_a_decreasing_query_layout():
    w = kvgen.custom(231, seq_lens=[40, 40], num_q_heads=4, num_kv_heads=2, head_dim=128, block_size=16,
                     q_rows=10)
    kc, vc, _, _ = _caches(w, False)
    pk.kv_get_device_error()
    qsl = np.array([0, 8, 4], np.int32)          # the second sequence would have -4 queries
    out = torch.zeros((10, 4, 128), device=DEV)
    pk.paged_prefill_attn_bf16(w.q.to(DEV), kc, vc, out, w.block_tables.to(DEV), w.seq_lens.to(DEV),
                               torch.from_numpy(qsl).to(DEV), w.max_blocks_per_seq, 2, 10, 4, 2, 128, 16,
                               w.inv_sqrt_d, 4 * 128, 0)
    assert pk.kv_get_device_error() & 4
    assert torch.isfinite(out).all()


# ---------------------------------------------------------------------------
# full-size workloads, sampled outputs, in the benchmark's launch configuration
# ---------------------------------------------------------------------------
def _sampled_reference(w, rows, q_cpu, seqs, heads, window, fp8):
    """Oracle outputs for the sampled sequences: the oracle writes just those
    sequences' tokens into a compact host pool (blocks renumbered in table
    order) and decodes from it."""
    bs, H, D = w.block_size, w.num_kv_heads, w.head_dim
    lens = w.seq_lens.cpu().numpy()
    nblk = [-(-int(lens[s]) // bs) for s in seqs]
    mb = max(max(nblk), 1)
    table = np.full((len(seqs), mb), -1, np.int32)
    cursor = 0
    for i, nb in enumerate(nblk):
        table[i, :nb] = np.arange(cursor, cursor + nb, dtype=np.int32)
        cursor += nb
    pool_blocks = max(cursor, 1)
    if fp8 == "kv":
        vr = np.full((pool_blocks, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    else:
        vr = np.full((pool_blocks, bs, H, D), kvgen.BF16_NAN, np.uint16)
    kr = np.full((pool_blocks, bs, H, D), kvgen.E4M3_NAN if fp8 else kvgen.BF16_NAN,
                 np.uint8 if fp8 else np.uint16)
    for i, s in enumerate(seqs):
        L = int(lens[s])
        if L == 0:
            continue
        sl = oracle.fill_slots(table[i], 0, L, bs)
        kk, vv = u16(rows[s][0]), u16(rows[s][1])
        if fp8 == "kv":
            oracle.write_fp8(kk, vv, kr, vr, sl, L, H, D, bs, w.k_scale, w.v_scale, H * D, H * D)
        elif fp8:
            oracle.write_fp8k(kk, vv, kr, vr, sl, L, H, D, bs, H * D, H * D, w.k_scale)
        else:
            oracle.write_bf16(kk, vv, kr, vr, sl, L, H, D, bs, H * D, H * D)
    qs = u16(q_cpu[list(seqs)])
    sub_lens = np.ascontiguousarray(lens[list(seqs)].astype(np.int32))
    fp8_v = fp8 == "kv"

    def one(job):
        i, h = job
        return oracle.decode_one(qs, None if fp8 else kr, kr if fp8 else None, None if fp8_v else vr, table,
                                 sub_lens, mb, w.num_q_heads, H, D, bs, w.inv_sqrt_d, w.k_scale,
                                 w.num_q_heads * D, window, i, h, v_cache_fp8=vr if fp8_v else None,
                                 v_scale=w.v_scale)
    # the oracle's C calls release the GIL and share no state: threads run
    # them side by side (no process is forked after the GPU calls)
    jobs = [(i, h) for i in range(len(seqs)) for h in heads]
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as pool:
        results = list(pool.map(one, jobs))
    return {(seqs[i], h): r for (i, h), r in zip(jobs, results)}


def _check_pool_sample(w, fp8, kc, vc, lens, starts):
    """The written pools on a seeded stratified sample of tokens: every
    sequence's first and last token and every 97th (offset by the sequence
    index), bit-exact against the oracle's encoding of the same rows at the
    slots the oracle computes from the block tables."""
    H, D, bs = w.num_kv_heads, w.head_dim, w.block_size
    toks, slot_rows = [], []
    tables = w.block_tables.cpu().numpy()
    for s in range(w.num_seqs):
        L = int(lens[s])
        if L == 0:
            continue
        js = sorted({0, L - 1} | set(range(s % 97, L, 97)))
        sl = oracle.fill_slots(tables[s], 0, L, bs)
        toks += [int(starts[s]) + j for j in js]
        slot_rows += [int(sl[j]) for j in js]
    toks_t = torch.tensor(toks, dtype=torch.int64, device=DEV)
    rows_t = torch.tensor(slot_rows, dtype=torch.int64, device=DEV)
    m = len(toks)
    key, value = u16(w.key[toks_t]), u16(w.value[toks_t])
    k8, v8 = bool(fp8), fp8 == "kv"
    kr = np.full((m, 1, H, D), kvgen.E4M3_NAN if k8 else kvgen.BF16_NAN, np.uint8 if k8 else np.uint16)
    vr = np.full((m, 1, H, D), kvgen.E4M3_NAN if v8 else kvgen.BF16_NAN, np.uint8 if v8 else np.uint16)
    compact = np.arange(m, dtype=np.int64)
    if v8:
        oracle.write_fp8(key, value, kr, vr, compact, m, H, D, 1, w.k_scale, w.v_scale, H * D, H * D)
    elif k8:
        oracle.write_fp8k(key, value, kr, vr, compact, m, H, D, 1, H * D, H * D, w.k_scale)
    else:
        oracle.write_bf16(key, value, kr, vr, compact, m, H, D, 1, H * D, H * D)

    def gathered(pool):
        flat = pool.view(-1, H * D)[rows_t]
        return flat.cpu().numpy() if pool.dtype == torch.uint8 else u16(flat)
    assert np.array_equal(gathered(kc), kr.reshape(m, H * D)), f"{w.name}: K pool sample differs"
    assert np.array_equal(gathered(vc), vr.reshape(m, H * D)), f"{w.name}: V pool sample differs"


def _stratified(lens, k, seed):
    """k sequences: the longest, the shortest and a seeded spread of the rest."""
    rng = np.random.default_rng(seed)
    pick = {int(lens.argmax()), int(lens.argmin())}
    rest = [s for s in range(len(lens)) if s not in pick]
    pick |= set(int(x) for x in rng.choice(rest, size=min(k - len(pick), len(rest)), replace=False))
    return sorted(pick)


def _full_size(w, fp8, windows, sample_seqs, heads):
    H, D, bs, nb, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.num_tokens
    slots = gpu_slots(w)
    vc = kvgen.poisoned_pool(nb, bs, H, D, "fp8" if fp8 == "kv" else "bf16", DEV)
    kc = kvgen.poisoned_pool(nb, bs, H, D, "fp8" if fp8 else "bf16", DEV)
    chunk = 262144
    for t0 in range(0, n, chunk):
        t1 = min(n, t0 + chunk)
        if fp8 == "kv":
            pk.kv_write_fp8(w.key[t0:t1], w.value[t0:t1], kc, vc, slots[t0:t1], t1 - t0, H, D, bs, w.k_scale,
                            w.v_scale, H * D, H * D)
        elif fp8:
            pk.kv_write_fp8k(w.key[t0:t1], w.value[t0:t1], kc, vc, slots[t0:t1], t1 - t0, H, D, bs, H * D,
                             H * D, w.k_scale)
        else:
            pk.kv_write_bf16(w.key[t0:t1], w.value[t0:t1], kc, vc, slots[t0:t1], t1 - t0, H, D, bs, H * D,
                             H * D)
    with_workspace(w, True)
    lens = w.seq_lens.cpu().numpy()
    starts = np.concatenate([[0], np.cumsum(lens.astype(np.int64))])
    _check_pool_sample(w, fp8, kc, vc, lens, starts)
    # copy just the sampled sequences' rows to the host
    rows = {s: (w.key[starts[s]:starts[s + 1]].cpu(), w.value[starts[s]:starts[s + 1]].cpu())
            for s in sample_seqs}
    q_cpu = w.q.cpu()
    for win in windows:
        got = _decode_gpu(w, kc, vc, win, fp8)
        ref = _sampled_reference(w, rows, q_cpu, sample_seqs, heads, win, fp8)
        g = np.stack([got[s, h] for (s, h) in ref])
        r = np.stack(list(ref.values()))
        assert_decode_close(g, r, f"{w.name} window {win}")
        assert np.isfinite(got).all()
    assert pk.kv_get_device_error() == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_one_very_long_sequence_every_head(fp8):
    """A 262,144-position sequence beside a one-position one: the long one
    is cut into a piece per SM (~150 split-KV partials per query head), the
    pool written in the benchmark's 262,144-token chunks; every query head,
    with and without a window."""
    w = kvgen.custom(240, device=DEV, seq_lens=[262144, 1], num_q_heads=32, num_kv_heads=8, head_dim=128,
                     block_size=16, fp8=fp8)
    _full_size(w, fp8, (0, 5000), [0, 1], tuple(range(32)))


def test_full_bf16_gqa4_every_output():
    """The BF16 decode workload in full: every (sequence, query head)."""
    w = kvgen.bf16_gqa4(device=DEV)
    _full_size(w, False, (0,), list(range(w.num_seqs)), tuple(range(w.num_q_heads)))


def test_full_fp8k_long_sampled():
    """Every query head of 16 stratified sequences, W = 0 and 4096."""
    w = kvgen.fp8k_long(device=DEV)
    _full_size(w, True, (0, 4096), _stratified(w.seq_lens.cpu().numpy(), 16, 4),
               tuple(range(w.num_q_heads)))


def test_full_fp8k_mixed_sampled():
    w = kvgen.fp8k_mixed(device=DEV)
    _full_size(w, True, (0,), _stratified(w.seq_lens.cpu().numpy(), 16, 5), tuple(range(w.num_q_heads)))


def test_full_fp8_kv_long_sampled():
    w = kvgen.fp8k_long(device=DEV)
    _full_size(w, "kv", (0, 4096), _stratified(w.seq_lens.cpu().numpy(), 16, 6), tuple(range(w.num_q_heads)))


def test_full_fp8_kv_mixed_sampled():
    w = kvgen.fp8k_mixed(device=DEV)
    _full_size(w, "kv", (0,), _stratified(w.seq_lens.cpu().numpy(), 16, 7), tuple(range(w.num_q_heads)))


def _full_prefill_sampled(w, fp8, chunk, seqs, rows_per_seq=3):
    """The benchmark's chunked prefill (the last min(chunk, L) positions of
    every sequence as causal queries) over the full-size cache, on the GPU;
    for each sampled sequence, its first, middle and last query rows from the
    oracle, which runs just those queries over the same sequence (cache rows
    written by the oracle's own write into a compact host pool)."""
    H, D, bs, Hq, nb, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_q_heads, w.num_blocks, w.num_tokens
    kv = fp8 == "kv"
    slots = gpu_slots(w)
    vc = kvgen.poisoned_pool(nb, bs, H, D, "fp8" if kv else "bf16", DEV)
    kc = kvgen.poisoned_pool(nb, bs, H, D, "fp8" if fp8 else "bf16", DEV)
    for t0 in range(0, n, 262144):
        t1 = min(n, t0 + 262144)
        if kv:
            pk.kv_write_fp8(w.key[t0:t1], w.value[t0:t1], kc, vc, slots[t0:t1], t1 - t0, H, D, bs, w.k_scale,
                            w.v_scale, H * D, H * D)
        elif fp8:
            pk.kv_write_fp8k(w.key[t0:t1], w.value[t0:t1], kc, vc, slots[t0:t1], t1 - t0, H, D, bs, H * D, H * D,
                             w.k_scale)
        else:
            pk.kv_write_bf16(w.key[t0:t1], w.value[t0:t1], kc, vc, slots[t0:t1], t1 - t0, H, D, bs, H * D, H * D)
    lens = w.seq_lens.cpu().numpy()
    q_lens = [min(chunk, int(L)) for L in lens]
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    n_q = int(qsl[-1])
    q = torch.randn((n_q, Hq * D), generator=torch.Generator().manual_seed(77)).to(torch.bfloat16)
    out = torch.full((n_q, Hq, D), float("nan"), device=DEV)
    args = (w.block_tables.to(DEV), w.seq_lens.to(DEV), torch.from_numpy(qsl).to(DEV), w.max_blocks_per_seq,
            w.num_seqs, n_q, Hq, H, D, bs, w.inv_sqrt_d)
    if kv:
        pk.paged_prefill_attn_fp8(q.to(DEV), kc, vc, out, *args, w.k_scale, w.v_scale, Hq * D, 0)
    elif fp8:
        pk.paged_prefill_attn_fp8k(q.to(DEV), kc, vc, out, *args, w.k_scale, Hq * D, 0)
    else:
        pk.paged_prefill_attn_bf16(q.to(DEV), kc, vc, out, *args, Hq * D, 0)
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    starts = np.concatenate([[0], np.cumsum(lens.astype(np.int64))])
    for s in seqs:
        L = int(lens[s])
        nq = q_lens[s]
        js = sorted({0, nq // 2, nq - 1})[:rows_per_seq]
        # compact host cache of sequence s
        nblk = -(-L // bs)
        table = np.arange(nblk, dtype=np.int32)[None]
        kr = np.full((nblk, bs, H, D), kvgen.E4M3_NAN if fp8 else kvgen.BF16_NAN, np.uint8 if fp8 else np.uint16)
        vr = (np.full((nblk, bs, H, D), kvgen.E4M3_NAN, np.uint8) if kv
              else np.full((nblk, bs, H, D), kvgen.BF16_NAN, np.uint16))
        sl = oracle.fill_slots(table[0], 0, L, bs)
        kk, vv = u16(w.key[starts[s]:starts[s + 1]].cpu()), u16(w.value[starts[s]:starts[s + 1]].cpu())
        if kv:
            oracle.write_fp8(kk, vv, kr, vr, sl, L, H, D, bs, w.k_scale, w.v_scale, H * D, H * D)
        elif fp8:
            oracle.write_fp8k(kk, vv, kr, vr, sl, L, H, D, bs, H * D, H * D, w.k_scale)
        else:
            oracle.write_bf16(kk, vv, kr, vr, sl, L, H, D, bs, H * D, H * D)
        for j in js:
            # one query at position L - nq + j: a sequence cut to that length + 1
            qrow = np.ascontiguousarray(u16(q[qsl[s] + j][None]))
            ref = oracle.paged_prefill_attn(qrow, None if fp8 else kr, kr if fp8 else None, None if kv else vr,
                                            table, np.array([L - nq + j + 1], np.int32), np.array([0, 1], np.int32),
                                            nblk, 1, Hq, H, D, bs, w.inv_sqrt_d, w.k_scale, Hq * D, 0,
                                            v_cache_fp8=vr if kv else None, v_scale=w.v_scale)
            assert_decode_close(got[qsl[s] + j][None], ref, f"{w.name} seq {s} query {j}")
    assert pk.kv_get_device_error() == 0


def test_full_bf16_chunked_prefill_sampled():
    w = kvgen.bf16_gqa4(device=DEV)
    lens = w.seq_lens.cpu().numpy()
    _full_prefill_sampled(w, False, 256, sorted({int(lens.argmax()), int(lens.argmin()), 0, 63}))


def test_full_fp8k_chunked_prefill_sampled():
    w = kvgen.fp8k_mixed(device=DEV)
    lens = w.seq_lens.cpu().numpy()[:32]
    _full_prefill_sampled(w, True, 256, sorted({int(lens.argmax()), int(lens.argmin()), 5}))


def test_full_fp8_kv_chunked_prefill_sampled():
    w = kvgen.fp8k_mixed(device=DEV)
    lens = w.seq_lens.cpu().numpy()
    _full_prefill_sampled(w, "kv", 256, sorted({int(lens.argmax()), int(lens.argmin()), 11, len(lens) - 1}))
