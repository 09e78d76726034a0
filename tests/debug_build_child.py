"""Child process of tests/test_debug_build_gpu.py: loads the bounds-checking
library (libpagedkv_debug.so) alone, runs one case and prints its findings as
one JSON line. Run: python tests/debug_build_child.py <case> <library path>

Cases:
  timeout  FP8-K decodes with the pipeline wait limit cut to 1 ns until one
           of them reports a wait that ran out (bit 0), then the default limit
           again and a decode checked against the oracle.
  bounds   a block table holding one block id outside the pool and the slots
           it gives: slot filling, the BF16, FP8-K and fused K writes, the
           BF16 decode and the BF16 chunked prefill, each checked against the
           oracle on everything the bad index does not touch.
"""
import ctypes
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import kvgen  # noqa: E402
import oracle  # noqa: E402
import paged_kv_cache_fill_gb300 as pk  # noqa: E402

DEV = torch.device("cuda")


def u16(t):
    return np.ascontiguousarray(t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16))


def ordered(bits):
    b = bits.astype(np.int64) & 0xFFFF
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


def decode_err(got, ref):
    """(max abs error, max relative error where |ref| >= 0.2), the decode
    parity measures."""
    err = np.abs(got.astype(np.float64) - ref)
    big = np.abs(ref) >= 0.2
    return float(err.max()), float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0


def device_error_status():
    bits = ctypes.c_uint32(0)
    status = pk.lib().kv_get_device_error(ctypes.byref(bits))
    return int(status), int(bits.value)


def oracle_slots(w):
    return np.concatenate([oracle.fill_slots(w.block_tables[s].numpy(), 0, int(L), w.block_size)
                           for s, L in enumerate(w.seq_lens.tolist())])


def case_timeout():
    w = kvgen.custom(606, seq_lens=[6000, 3000, 9000, 100, 4500], num_q_heads=32, num_kv_heads=8, head_dim=128,
                     block_size=16, fp8=True)
    H, D, bs, Hq, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_q_heads, w.num_tokens
    slots_ref = oracle_slots(w)
    tables, lens, q = w.block_tables.to(DEV), w.seq_lens.to(DEV), w.q.to(DEV)
    kc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "fp8", DEV)
    vc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "bf16", DEV)
    pk.kv_write_fp8k(w.key.to(DEV), w.value.to(DEV), kc, vc, torch.from_numpy(slots_ref).to(DEV), n, H, D, bs,
                     H * D, H * D, w.k_scale)
    ws = torch.empty(pk.kv_decode_workspace_bytes(w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs),
                     dtype=torch.uint8, device=DEV)
    pk.kv_set_decode_workspace(ws)
    out = torch.empty((w.num_seqs, Hq, D), dtype=torch.float32, device=DEV)

    def decode():
        pk.paged_decode_attn_fp8k(q, kc, vc, out, tables, lens, w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs,
                                  w.inv_sqrt_d, w.k_scale, Hq * D, 0)

    res = {"before": device_error_status()}
    pk.kv_debug_set_wait_limit(1)
    seen, attempts = [], 0
    while attempts < 8:
        attempts += 1
        decode()
        st = device_error_status()  # synchronises: every decode CTA has returned
        seen.append(st)
        if st[1] & 1:
            break
    res.update(attempts=attempts, seen=seen)
    pk.kv_debug_set_wait_limit(0)
    decode()  # same workspace, no re-registration: its counters were reset by the last CTA
    res["after"] = device_error_status()
    kr = np.full((w.num_blocks, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    vr = np.full((w.num_blocks, bs, H, D), kvgen.BF16_NAN, np.uint16)
    oracle.write_fp8k(u16(w.key), u16(w.value), kr, vr, slots_ref, n, H, D, bs, H * D, H * D, w.k_scale)
    ref = oracle.paged_decode_attn_fp8k(u16(w.q), kr, vr, w.block_tables.numpy(), w.seq_lens.numpy(),
                                        w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs, w.inv_sqrt_d, w.k_scale,
                                        Hq * D, 0)
    got = out.cpu().numpy()
    res["finite"] = bool(np.isfinite(got).all())
    res["abs_err"], res["rel_err"] = decode_err(got, ref)
    pk.kv_set_decode_workspace(None)
    return res


def case_bounds():
    w = kvgen.custom(707, seq_lens=[200, 57, 130], num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                     key_sigma=4.0)
    H, D, bs, Hq, nb, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_q_heads, w.num_blocks, w.num_tokens
    pk.kv_debug_set_pool(nb, bs)
    res = {"clean": device_error_status()}
    # sequence 0's logical block 1 (positions 16..31) names a block past the pool
    bad_tables = w.block_tables.clone()
    bad_tables[0, 1] = nb + 5
    good_slots = oracle_slots(w)
    bad_rows = np.arange(16, 32)                 # token rows of positions 16..31 of sequence 0
    slots = torch.empty(n, dtype=torch.int64, device=DEV)
    off = 0
    for s, L in enumerate(w.seq_lens.tolist()):
        pk.kv_fill_slots(slots[off:off + L], bad_tables[s].to(DEV), 0, L, bs)
        off += L
    res["fill"] = device_error_status()
    got_slots = slots.cpu().numpy()
    want_slots = good_slots.copy()
    want_slots[bad_rows] = (nb + 5) * bs + np.arange(16)
    res["fill_slots_equal"] = bool(np.array_equal(got_slots, want_slots))
    skip = good_slots.copy()
    skip[bad_rows] = -1                          # the rows the kernels must leave out
    k16, v16 = u16(w.key), u16(w.value)

    # BF16 write
    kc = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    vc = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    pk.kv_write_bf16(w.key.to(DEV), w.value.to(DEV), kc, vc, slots, n, H, D, bs, H * D, H * D)
    res["write_bf16"] = device_error_status()
    kr = np.full((nb, bs, H, D), kvgen.BF16_NAN, np.uint16)
    vr = kr.copy()
    oracle.write_bf16(k16, v16, kr, vr, skip, n, H, D, bs, H * D, H * D)
    res["write_bf16_equal"] = bool(np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr))

    # FP8-K write
    k_scale = kvgen.amax_scale(w.key)
    kc8 = kvgen.poisoned_pool(nb, bs, H, D, "fp8", DEV)
    vcb = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    pk.kv_write_fp8k(w.key.to(DEV), w.value.to(DEV), kc8, vcb, slots, n, H, D, bs, H * D, H * D, k_scale)
    res["write_fp8k"] = device_error_status()
    kr8 = np.full((nb, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    vrb = np.full((nb, bs, H, D), kvgen.BF16_NAN, np.uint16)
    oracle.write_fp8k(k16, v16, kr8, vrb, skip, n, H, D, bs, H * D, H * D, k_scale)
    res["write_fp8k_equal"] = bool(np.array_equal(kc8.cpu().numpy(), kr8) and np.array_equal(u16(vcb), vrb))

    # fused K write (within 1 BF16 ulp of the oracle; skipped rows untouched)
    wt = (torch.rand(D, generator=torch.Generator().manual_seed(3)) + 0.5).to(torch.bfloat16)
    pos = torch.randint(0, 4096, (n,), generator=torch.Generator().manual_seed(4)).to(torch.int32)
    kf = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    pk.kv_write_fused_k_norm_rope_bf16(w.key.to(DEV), wt.to(DEV), pos.to(DEV), kf, slots, n, H, D, 128, bs, 1e-6,
                                       1e6)
    res["write_fused"] = device_error_status()
    kfr = np.full((nb, bs, H, D), kvgen.BF16_NAN, np.uint16)
    oracle.write_fused_k_norm_rope_bf16(k16, u16(wt), pos.numpy(), kfr, skip, n, H, D, 128, bs, 1e-6, 1e6)
    res["write_fused_ulp"] = int(np.abs(ordered(u16(kf)) - ordered(kfr)).max())

    # BF16 decode over the caches of the good slots, with the bad table: the
    # kernel reads block 0 in place of the bad id (sequence 0 only)
    kg = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    vg = kvgen.poisoned_pool(nb, bs, H, D, "bf16", DEV)
    pk.kv_write_bf16(w.key.to(DEV), w.value.to(DEV), kg, vg, torch.from_numpy(good_slots).to(DEV), n, H, D, bs,
                     H * D, H * D)
    res["write_good"] = device_error_status()
    krg = np.full((nb, bs, H, D), kvgen.BF16_NAN, np.uint16)
    vrg = krg.copy()
    oracle.write_bf16(k16, v16, krg, vrg, good_slots, n, H, D, bs, H * D, H * D)
    out = torch.empty((w.num_seqs, Hq, D), dtype=torch.float32, device=DEV)
    pk.paged_decode_attn_bf16(w.q.to(DEV), kg, vg, out, bad_tables.to(DEV), w.seq_lens.to(DEV), w.max_blocks_per_seq,
                              w.num_seqs, Hq, H, D, bs, w.inv_sqrt_d, Hq * D, 0)
    res["decode"] = device_error_status()
    ref = oracle.paged_decode_attn_bf16(u16(w.q), krg, vrg, w.block_tables.numpy(), w.seq_lens.numpy(),
                                        w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs, w.inv_sqrt_d, Hq * D, 0)
    got = out.cpu().numpy()
    res["decode_untouched_finite"] = bool(np.isfinite(got[1:]).all())
    res["decode_untouched_abs_err"], res["decode_untouched_rel_err"] = decode_err(got[1:], ref[1:])

    # BF16 chunked prefill over the same caches and the bad table: each
    # sequence's last positions as queries; sequence 0's rows read block 0
    # in place of the bad id, the others must match the oracle
    qlens = [40, 20, 30]
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    n_q = int(qsl[-1])
    qp = torch.randn((n_q, Hq * D), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    outp = torch.empty((n_q, Hq, D), dtype=torch.float32, device=DEV)
    pk.paged_prefill_attn_bf16(qp.to(DEV), kg, vg, outp, bad_tables.to(DEV), w.seq_lens.to(DEV),
                               torch.from_numpy(qsl).to(DEV), w.max_blocks_per_seq, w.num_seqs, n_q, Hq, H, D, bs,
                               w.inv_sqrt_d, Hq * D, 0)
    res["prefill"] = device_error_status()
    refp = oracle.paged_prefill_attn(u16(qp), krg, None, vrg, w.block_tables.numpy(), w.seq_lens.numpy(), qsl,
                                     w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs, w.inv_sqrt_d, 1.0, Hq * D, 0)
    gotp = outp.cpu().numpy()
    res["prefill_untouched_finite"] = bool(np.isfinite(gotp[qlens[0]:]).all())
    res["prefill_untouched_abs_err"], res["prefill_untouched_rel_err"] = decode_err(gotp[qlens[0]:],
                                                                                    refp[qlens[0]:])
    pk.kv_debug_set_pool(0, 0)
    return res


def main():
    case, library = sys.argv[1], sys.argv[2]
    pk.use_library(library)
    torch.cuda.set_device(0)
    res = {"timeout": case_timeout, "bounds": case_bounds}[case]()
    print(json.dumps(res))


if __name__ == "__main__":
    main()
