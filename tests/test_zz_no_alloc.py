"""The FP8-K decode that needs no caller memory
(paged_decode_attn_fp8k_static_scratch) against the regular FP8-K decode.

That entry point is for callers that cannot give the library a device
allocation (for example host code running in a CUDA host-function callback,
where the CUDA API may not be called, or an application whose device memory
all belongs to another allocator); its split-KV scratch is a fixed 64 MiB
array inside the library. Here it is called through the C ABI twice in a
row on a workload that needs split-KV, and each result is held to the same
tolerance as every decode parity test against the output of
paged_decode_attn_fp8k with a caller-registered workspace. This file sorts
last so that a run stopping at its first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import kvgen
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


def _close(got, ref):
    assert np.isfinite(got).all()
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert err.max() <= ABS_TOL, err.max()
    big = np.abs(ref) >= REL_FLOOR
    assert (err[big] / np.abs(ref[big])).max() <= REL_TOL


def test_static_scratch_decode_matches_registered_workspace_decode():
    w = kvgen.custom(31337, seq_lens=[4000, 1, 2500, 700, 3999, 128, 0, 1500], num_q_heads=32,
                     num_kv_heads=8, head_dim=128, block_size=16, fp8=True)
    H, D, bs, Hq, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_q_heads, w.num_tokens
    # the cache, written by the library's FP8-K write
    tables = w.block_tables.to(DEV)
    slots = torch.empty(n, dtype=torch.int64, device=DEV)
    off = 0
    for s, L in enumerate(w.seq_lens.tolist()):
        pk.kv_fill_slots(slots[off:off + L], tables[s], 0, L, bs)
        off += L
    kc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "fp8", DEV)
    vc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "bf16", DEV)
    pk.kv_write_fp8k(w.key.to(DEV), w.value.to(DEV), kc, vc, slots, n, H, D, bs, H * D, H * D, w.k_scale)
    q, lens = w.q.to(DEV), w.seq_lens.to(DEV)
    args = (tables, lens, w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs, w.inv_sqrt_d, w.k_scale, Hq * D, 0)

    # reference: the regular entry point with a workspace the caller allocated
    ws = torch.empty(pk.kv_decode_workspace_bytes(w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs),
                     dtype=torch.uint8, device=DEV)
    pk.kv_set_decode_workspace(ws)
    ref_out = torch.empty((w.num_seqs, Hq, D), dtype=torch.float32, device=DEV)
    pk.paged_decode_attn_fp8k(q, kc, vc, ref_out, *args)
    ref = ref_out.cpu().numpy()
    pk.kv_set_decode_workspace(None)

    # the no-allocation entry point, straight through the C ABI, twice in a row
    lib = pk.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full((w.num_seqs, Hq, D), float("nan"), device=DEV)
        status = lib.paged_decode_attn_fp8k_static_scratch(
            q.data_ptr(), kc.data_ptr(), vc.data_ptr(), out.data_ptr(), tables.data_ptr(), lens.data_ptr(),
            w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs, w.inv_sqrt_d, w.k_scale, Hq * D, 0, stream)
        assert status == pk.KV_OK, status
        _close(out.cpu().numpy(), ref)
    assert pk.kv_get_device_error() == 0


def test_static_scratch_rejects_a_shape_larger_than_its_array():
    # 4096 sequences of up to 65536 positions would need far more than 64 MiB
    # of split-KV scratch: refused before anything is launched
    lib = pk.lib()
    fake = ctypes.c_void_p(0x100000)
    status = lib.paged_decode_attn_fp8k_static_scratch(
        fake, fake, fake, fake, fake, fake, 4096, 4096, 32, 8, 128, 16, 0.088, 0.04, 32 * 128, 0, None)
    assert status == pk.KV_ERR_UNSUPPORTED
