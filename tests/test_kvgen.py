"""The seeded input generators, on CPU: every input of the oracle and of the
CUDA path comes from kvgen, so its recipe (shapes, length ranges, the block
hand-out, the FP8-K outliers and scales) is checked here directly, on the
workloads shrunk through their size arguments."""
import math
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import kvgen  # noqa: E402

SMALL = {
    "tiny": lambda: kvgen.tiny(),
    "fused_write": lambda: kvgen.fused_write(seqs=3, tokens_per_seq=100),
    "bf16_gqa4": lambda: kvgen.bf16_gqa4(num_seqs=6, max_len=1500, num_blocks=1000),
    "fp8k_long": lambda: kvgen.fp8k_long(num_seqs=2, seq_len=300),
    "fp8k_mixed": lambda: kvgen.fp8k_mixed(num_seqs=12, max_len=4096),
}


def _tensors(w):
    return {k: v for k, v in vars(w).items() if isinstance(v, torch.Tensor)}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_same_seed_same_bytes(name):
    a, b = SMALL[name](), SMALL[name]()
    ta, tb = _tensors(a), _tensors(b)
    assert ta.keys() == tb.keys()
    for k in ta:
        assert torch.equal(ta[k].view(torch.uint8) if ta[k].dtype == torch.bfloat16 else ta[k],
                           tb[k].view(torch.uint8) if tb[k].dtype == torch.bfloat16 else tb[k]), k
    assert a.k_scale == b.k_scale and a.v_scale == b.v_scale


def test_workloads_differ_from_one_another():
    # distinct seeds: the first query rows of the two decode workloads differ
    assert not torch.equal(SMALL["bf16_gqa4"]().q[0], SMALL["fp8k_long"]().q[0])


@pytest.mark.parametrize("name", sorted(SMALL))
def test_block_tables_hand_out_distinct_pool_blocks(name):
    w = SMALL[name]()
    t, lens = w.block_tables, w.seq_lens.tolist()
    assert t.dtype == torch.int32 and tuple(t.shape) == (w.num_seqs, w.max_blocks_per_seq)
    used = []
    for s, L in enumerate(lens):
        nb = -(-L // w.block_size)
        assert nb <= w.max_blocks_per_seq
        row = t[s].tolist()
        assert all(0 <= b < w.num_blocks for b in row[:nb])
        assert all(b == -1 for b in row[nb:])
        used += row[:nb]
    assert len(set(used)) == len(used)        # no block shared between sequences


@pytest.mark.parametrize("name", sorted(SMALL))
def test_prefill_token_index(name):
    w = SMALL[name]()
    lens = w.seq_lens.tolist()
    assert w.num_tokens == sum(lens)
    assert w.positions.tolist() == [p for L in lens for p in range(L)]
    assert w.token_seq.tolist() == [s for s, L in enumerate(lens) for _ in range(L)]
    assert tuple(w.key.shape) == (sum(lens), w.num_kv_heads * w.head_dim)
    assert w.key.dtype == torch.bfloat16 and w.value.dtype == torch.bfloat16


def test_shapes_of_the_named_workloads():
    t = kvgen.tiny()
    assert (t.seq_lens.tolist(), t.num_q_heads, t.num_kv_heads, t.head_dim, t.block_size, t.num_blocks) == \
        ([37, 100], 4, 2, 64, 16, 16)
    assert t.inv_sqrt_d == 1.0 / 8.0
    f = SMALL["fused_write"]()
    assert (f.num_kv_heads, f.head_dim, f.block_size) == (8, 128, 16)
    assert f.extra["rotary_dim"] == 128 and f.extra["theta"] == 1e6 and f.extra["rms_eps"] == 1e-6
    assert set(f.extra["sigma"].tolist()) <= {1.0, 4.0, 18.0}
    wt = f.extra["k_norm_weight"].float()
    assert (wt >= 0.5).all() and (wt <= 1.5).all()
    g = SMALL["bf16_gqa4"]()
    assert (g.num_q_heads, g.num_kv_heads, g.head_dim, g.block_size) == (32, 8, 128, 16)
    m = SMALL["fp8k_mixed"]()
    assert (m.num_q_heads, m.num_kv_heads, m.head_dim, m.block_size) == (64, 8, 128, 64)
    needed = sum(-(-L // 64) for L in m.seq_lens.tolist())
    assert m.num_blocks == math.ceil(1.25 * needed)


def test_length_ranges():
    g = kvgen.bf16_gqa4(num_seqs=16, max_len=2000, num_blocks=4000)
    lens = g.seq_lens.tolist()
    assert all(512 <= L <= 2000 for L in lens) and len(set(lens)) > 1
    m = kvgen.fp8k_mixed(num_seqs=40, max_len=4096)
    lens = m.seq_lens.tolist()
    assert all(128 <= L <= 4096 for L in lens)
    # log-uniform: about as many lengths below the geometric midpoint as above
    mid = math.sqrt(128 * 4096)
    assert 8 <= sum(L < mid for L in lens) <= 32


def test_fp8k_keys_outliers_and_scales():
    w = kvgen.fp8k_long(num_seqs=1, seq_len=4096)
    k = w.key.float()
    n = k.numel()
    outliers = int((k.abs() == 20.0).sum())
    # 0.1% of the elements set to +-20, both signs drawn
    assert abs(outliers - n * 1e-3) < 6 * math.sqrt(n * 1e-3)
    assert int((k == 20.0).sum()) > 0 and int((k == -20.0).sum()) > 0
    # the rest is N(0, 2): its standard deviation, and no other value as large
    rest = k[k.abs() != 20.0]
    assert abs(float(rest.std()) - 2.0) < 0.02
    assert float(k.abs().max()) == 20.0
    # per-tensor scales max|x| / 448 in float32
    assert w.k_scale == float(torch.tensor(20.0 / 448.0, dtype=torch.float32))
    vmax = float(w.value.float().abs().max())
    assert w.v_scale == float(torch.tensor(vmax / 448.0, dtype=torch.float32))


def test_poisoned_pools_hold_the_nan_patterns():
    b = kvgen.poisoned_pool(3, 16, 2, 64, "bf16")
    e = kvgen.poisoned_pool(3, 16, 2, 64, "fp8")
    assert tuple(b.shape) == (3, 16, 2, 64) and b.dtype == torch.bfloat16
    assert (b.view(torch.int16) == kvgen.BF16_NAN).all() and torch.isnan(b.float()).all()
    assert e.dtype == torch.uint8 and (e == kvgen.E4M3_NAN).all()
