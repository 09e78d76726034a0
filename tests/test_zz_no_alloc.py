"""The FP8-K decode that needs no caller memory
(paged_decode_attn_fp8k_static_scratch), against the CPU oracle and against
the regular FP8-K decode.

That entry point is for callers that cannot give the library a device
allocation: an application whose device memory all belongs to another
allocator (a framework memory pool, a serving engine that reserves all of HBM
for its KV cache) cannot set a raw buffer aside for a library. Its split-KV
scratch is a fixed 64 MiB array inside the library instead. Here it is called
through the C ABI twice in a row per window on a workload that needs split-KV;
each result is held to the decode parity tolerance against the fp64 oracle and
against paged_decode_attn_fp8k with a caller-registered workspace. This file
sorts last so that a run stopping at its first failure has run everything
else.
"""
import ctypes

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
STATIC_SCRATCH_BYTES = 64 << 20


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    pk.kv_set_decode_workspace(None)


def _close(got, ref):
    assert np.isfinite(got).all()
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert err.max() <= ABS_TOL, err.max()
    big = np.abs(ref) >= REL_FLOOR
    assert (err[big] / np.abs(ref[big])).max() <= REL_TOL


def _u16(t):
    return np.ascontiguousarray(t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16))


def _static_decode(lib, q, kc, vc, out, tables, lens, w, window, stream):
    return lib.paged_decode_attn_fp8k_static_scratch(
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), out.data_ptr(), tables.data_ptr(), lens.data_ptr(),
        w.max_blocks_per_seq, w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.inv_sqrt_d,
        w.k_scale, w.num_q_heads * w.head_dim, window, stream)


def test_static_scratch_decode_matches_the_oracle_and_the_registered_workspace_decode():
    w = kvgen.custom(31337, seq_lens=[4000, 1, 2500, 700, 3999, 128, 0, 1500], num_q_heads=32,
                     num_kv_heads=8, head_dim=128, block_size=16, fp8=True)
    H, D, bs, Hq, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_q_heads, w.num_tokens
    # the cache, written by the library's FP8-K write (bit-exact to the
    # oracle's write, tested elsewhere) and by the oracle for its reference
    slots_ref = np.concatenate([oracle.fill_slots(w.block_tables[s].numpy(), 0, int(L), bs)
                                for s, L in enumerate(w.seq_lens.tolist())])
    tables = w.block_tables.to(DEV)
    slots = torch.from_numpy(slots_ref).to(DEV)
    kc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "fp8", DEV)
    vc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "bf16", DEV)
    pk.kv_write_fp8k(w.key.to(DEV), w.value.to(DEV), kc, vc, slots, n, H, D, bs, H * D, H * D, w.k_scale)
    kr = np.full((w.num_blocks, bs, H, D), kvgen.E4M3_NAN, np.uint8)
    vr = np.full((w.num_blocks, bs, H, D), kvgen.BF16_NAN, np.uint16)
    oracle.write_fp8k(_u16(w.key), _u16(w.value), kr, vr, slots_ref, n, H, D, bs, H * D, H * D, w.k_scale)
    q, lens = w.q.to(DEV), w.seq_lens.to(DEV)
    assert pk.kv_decode_workspace_bytes(w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs) <= STATIC_SCRATCH_BYTES

    lib = pk.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for window in (0, 1000):
        want = oracle.paged_decode_attn_fp8k(_u16(w.q), kr, vr, w.block_tables.numpy(), w.seq_lens.numpy(),
                                             w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs, w.inv_sqrt_d,
                                             w.k_scale, Hq * D, window)
        # the regular entry point with a workspace the caller allocated
        ws = torch.empty(pk.kv_decode_workspace_bytes(w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs),
                         dtype=torch.uint8, device=DEV)
        pk.kv_set_decode_workspace(ws)
        ref_out = torch.empty((w.num_seqs, Hq, D), dtype=torch.float32, device=DEV)
        pk.paged_decode_attn_fp8k(q, kc, vc, ref_out, tables, lens, w.max_blocks_per_seq, w.num_seqs, Hq, H, D,
                                  bs, w.inv_sqrt_d, w.k_scale, Hq * D, window)
        ref = ref_out.cpu().numpy()
        pk.kv_set_decode_workspace(None)
        _close(ref, want)
        # the no-allocation entry point, straight through the C ABI, twice in a row
        for _ in range(2):
            out = torch.full((w.num_seqs, Hq, D), float("nan"), device=DEV)
            status = _static_decode(lib, q, kc, vc, out, tables, lens, w, window, stream)
            assert status == pk.KV_OK, status
            got = out.cpu().numpy()
            _close(got, want)
            _close(got, ref)
    assert pk.kv_get_device_error() == 0


def test_static_scratch_refuses_a_shape_larger_than_its_array():
    # 64 sequences whose tables hold 65,536 positions each could need 274 MB
    # of split-KV scratch: refused before anything is launched. Every buffer
    # is real and the lengths are zero, so that even a launch would only
    # write zeros to `out`.
    num_seqs, mbps, Hq, H, D, bs = 64, 4096, 32, 8, 128, 16
    assert pk.kv_decode_workspace_bytes(mbps, num_seqs, Hq, H, D, bs) > STATIC_SCRATCH_BYTES
    tables = torch.zeros((num_seqs, mbps), dtype=torch.int32, device=DEV)
    lens = torch.zeros(num_seqs, dtype=torch.int32, device=DEV)
    q = torch.zeros((num_seqs, Hq * D), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((1, bs, H, D), dtype=torch.uint8, device=DEV)
    vc = torch.zeros((1, bs, H, D), dtype=torch.bfloat16, device=DEV)
    out = torch.full((num_seqs, Hq, D), 7.0, device=DEV)
    status = pk.lib().paged_decode_attn_fp8k_static_scratch(
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), out.data_ptr(), tables.data_ptr(), lens.data_ptr(),
        mbps, num_seqs, Hq, H, D, bs, 0.088, 0.04, Hq * D, 0, None)
    assert status == pk.KV_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a refused call wrote its output"
