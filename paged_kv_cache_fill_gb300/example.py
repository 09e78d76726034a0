"""A first call sequence through the Python binding (needs a GB300):
slot filling, a BF16 cache write, a paged decode with split-KV and a chunked
prefill over the same cache. PyTorch supplies the device memory; every array
is a contiguous CUDA tensor and every size is passed explicitly.

Run: python -m paged_kv_cache_fill_gb300.example
"""
import torch

import paged_kv_cache_fill_gb300 as pk


def main() -> None:
    dev, H, Hq, D, bs, nb, mbps = "cuda", 8, 32, 128, 16, 1024, 64
    seq_lens = torch.tensor([37, 100], dtype=torch.int32, device=dev)
    block_tables = torch.randperm(nb, device=dev)[:2 * mbps].view(2, mbps).to(torch.int32)
    k_cache = torch.empty((nb, bs, H, D), dtype=torch.bfloat16, device=dev)
    v_cache = torch.empty_like(k_cache)

    # write every position's K and V through its slot
    n = int(seq_lens.sum())
    slots = torch.empty(n, dtype=torch.int64, device=dev)
    off = 0
    for s, L in enumerate(seq_lens.tolist()):
        pk.kv_fill_slots(slots[off:off + L], block_tables[s], 0, L, bs)
        off += L
    key = torch.randn(n, H * D, device=dev).to(torch.bfloat16)
    value = torch.randn(n, H * D, device=dev).to(torch.bfloat16)
    pk.kv_write_bf16(key, value, k_cache, v_cache, slots, n, H, D, bs, H * D, H * D)

    # decode one query token per sequence (a registered workspace enables split-KV)
    pk.kv_set_decode_workspace(torch.empty(pk.kv_decode_workspace_bytes(mbps, 2, Hq, H, D, bs),
                                           dtype=torch.uint8, device=dev))
    q = torch.randn(2, Hq * D, device=dev).to(torch.bfloat16)
    out = torch.empty(2, Hq, D, device=dev)
    pk.paged_decode_attn_bf16(q, k_cache, v_cache, out, block_tables, seq_lens, mbps, 2, Hq, H, D, bs,
                              D ** -0.5, Hq * D, 0)

    # or attend the last 5 and 20 positions as a causal chunk of query tokens
    qsl = torch.tensor([0, 5, 25], dtype=torch.int32, device=dev)
    qp = torch.randn(25, Hq * D, device=dev).to(torch.bfloat16)
    outp = torch.empty(25, Hq, D, device=dev)
    pk.paged_prefill_attn_bf16(qp, k_cache, v_cache, outp, block_tables, seq_lens, qsl, mbps, 2, 25, Hq, H, D,
                               bs, D ** -0.5, Hq * D, 0)
    assert pk.kv_get_device_error() == 0   # synchronises; nonzero bits name a fault
    pk.kv_set_decode_workspace(None)
    print("decode output", tuple(out.shape), "prefill output", tuple(outp.shape))


if __name__ == "__main__":
    main()
