"""Seeded synthetic inputs for the paged KV-cache path.

This module only draws random inputs and lays out block tables; it holds none
of the method's arithmetic (no slot computation, no cache write, no
attention). Both the CUDA path and the CPU oracle consume what it returns, so
the two sides always see the same bytes.

Workloads (shapes and distributions of the paged KV-cache decode server):
  tiny        2 sequences (37 and 100 tokens), 4 query / 2 KV heads, head_dim 64,
              block_size 16, a 16-block pool in seeded permuted order.
  fused_write 4 sequences x 1024 tokens, 8 KV heads, head_dim 128, rotary 128,
              theta 1e6, rms_eps 1e-6, block_size 16, 256-block shuffled pool;
              K ~ N(0, sigma_h) with sigma_h per head from {1, 4, 18},
              V ~ N(0, 1), k_norm_weight ~ U(0.5, 1.5).
  bf16_gqa4   64 sequences, lengths uniform in [512, 8192], 32 query / 8 KV
              heads, head_dim 128, block_size 16, 40000-block permuted pool.
  fp8k_long   128 sequences of 32768 tokens, 32 query / 8 KV heads, head_dim
              128, block_size 16, 262144-block permuted pool; K ~ N(0, 2) with
              0.1% of elements set to +-20, k_scale = max|K| / 448.
  fp8k_mixed  256 sequences, lengths log-uniform in [128, 65536], 64 query / 8
              KV heads, head_dim 128, block_size 64, pool of 1.25 x the blocks
              needed, shuffled; K as in fp8k_long.

All tensors are torch tensors on the requested device. BF16 values are drawn
in float32 and converted with torch's round-to-nearest-even. Unused pool
blocks and the tail rows of partly filled blocks hold NaN patterns (BF16
0x7FC0, E4M3 0x7F) so that any read outside the attended positions shows up.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    seq_lens: torch.Tensor          # int32 [num_seqs]
    block_tables: torch.Tensor      # int32 [num_seqs, max_blocks_per_seq]
    key: torch.Tensor | None        # bf16 [num_tokens, num_kv_heads * head_dim] prefill K
    value: torch.Tensor | None      # bf16 [num_tokens, num_kv_heads * head_dim] prefill V
    q: torch.Tensor | None          # bf16 [num_seqs, num_q_heads * head_dim]
    positions: torch.Tensor | None  # int32 [num_tokens], position of each prefill token
    token_seq: torch.Tensor | None  # int32 [num_tokens], sequence of each prefill token
    inv_sqrt_d: float = 0.0
    k_scale: float = 1.0
    v_scale: float = 1.0
    sliding_windows: tuple = (0,)
    extra: dict = field(default_factory=dict)

    @property
    def num_tokens(self) -> int:
        return int(self.seq_lens.to(torch.int64).sum().item())

    @property
    def kv_row(self) -> int:
        return self.num_kv_heads * self.head_dim


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


# Large tensors are drawn in row chunks of this many elements (at most), so
# no full-size float32 temporary is ever materialised; the chunking is part of
# the recipe (the same seed and shape always give the same bytes).
CHUNK_ELEMS = 1 << 26


def _rows_per_chunk(row: int) -> int:
    return max(1, CHUNK_ELEMS // max(row, 1))


def _normal_bf16(shape, sigma, g, device) -> torch.Tensor:
    """N(0, sigma) drawn in float32, rounded to BF16 (RNE), row chunk by row chunk."""
    rows, row = (shape[0], int(torch.tensor(shape[1:]).prod().item()) if len(shape) > 1 else 1)
    out = torch.empty((rows, row), dtype=torch.bfloat16, device=device)
    step = _rows_per_chunk(row)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = torch.randn((r1 - r0, row), generator=g, device=device, dtype=torch.float32)
        if not isinstance(sigma, (int, float)) or sigma != 1:
            x = x * sigma
        out[r0:r1] = x.to(torch.bfloat16)
    return out.reshape(shape)


def block_tables_from_pool(seq_lens: torch.Tensor, block_size: int, num_blocks: int,
                           max_blocks_per_seq: int, g: torch.Generator,
                           fill: int = -1) -> torch.Tensor:
    """A seeded permutation of the pool's block ids, handed out to the
    sequences in consecutive chunks of ceil(len / block_size) blocks. Table
    entries past a sequence's blocks hold `fill`."""
    perm = torch.randperm(num_blocks, generator=g, device=g.device).to(torch.int32).cpu()
    lens = seq_lens.cpu().tolist()
    tables = torch.full((len(lens), max_blocks_per_seq), fill, dtype=torch.int32)
    cursor = 0
    for s, L in enumerate(lens):
        nb = -(-int(L) // block_size)
        if nb > max_blocks_per_seq or cursor + nb > num_blocks:
            raise ValueError("pool too small for the requested lengths")
        tables[s, :nb] = perm[cursor:cursor + nb]
        cursor += nb
    return tables.to(seq_lens.device)


def _prefill_token_index(seq_lens: torch.Tensor):
    """Sequence id and position of every prefill token, sequences in order."""
    lens = seq_lens.to(torch.int64).cpu()
    token_seq = torch.repeat_interleave(torch.arange(len(lens), dtype=torch.int32), lens)
    starts = torch.cumsum(lens, 0) - lens
    positions = (torch.arange(int(lens.sum()), dtype=torch.int64)
                 - torch.repeat_interleave(starts, lens)).to(torch.int32)
    return token_seq.to(seq_lens.device), positions.to(seq_lens.device)


def fp8k_keys(num_tokens: int, row: int, g: torch.Generator, device) -> tuple[torch.Tensor, float]:
    """K ~ N(0, 2) with 0.1% of the elements set to +-20 (random sign), and
    the per-tensor scale max|K| / 448 of the resulting tensor (in float32)."""
    out = torch.empty((num_tokens, row), dtype=torch.bfloat16, device=device)
    step = _rows_per_chunk(row)
    amax = torch.zeros((), dtype=torch.float32, device=device)
    for r0 in range(0, num_tokens, step):
        r1 = min(num_tokens, r0 + step)
        k = torch.randn((r1 - r0, row), generator=g, device=device, dtype=torch.float32) * 2.0
        outlier = torch.rand((r1 - r0, row), generator=g, device=device) < 1e-3
        sign = torch.randint(0, 2, (r1 - r0, row), generator=g, device=device,
                             dtype=torch.int8).to(torch.float32) * 2 - 1
        kb = torch.where(outlier, 20.0 * sign, k).to(torch.bfloat16)
        out[r0:r1] = kb
        amax = torch.maximum(amax, kb.abs().max().float())
    k_scale = float(amax.item()) / 448.0
    return out, float(torch.tensor(k_scale, dtype=torch.float32).item())


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------
def tiny(seed: int = 1001, device="cpu") -> Workload:
    g = _gen(seed, device)
    seq_lens = torch.tensor([37, 100], dtype=torch.int32, device=device)
    H, Hq, D, bs, nb = 2, 4, 64, 16, 16
    mbps = 8
    tables = block_tables_from_pool(seq_lens, bs, nb, mbps, g)
    n = int(seq_lens.sum())
    key = _normal_bf16((n, H * D), 1.0, g, device)
    value = _normal_bf16((n, H * D), 1.0, g, device)
    q = _normal_bf16((2, Hq * D), 1.0, g, device)
    token_seq, positions = _prefill_token_index(seq_lens)
    return Workload("tiny", 2, Hq, H, D, bs, nb, mbps, seq_lens, tables, key, value, q,
                    positions, token_seq, inv_sqrt_d=1.0 / 8.0)


def fused_write(seed: int = 1002, device="cpu", seqs: int = 4, tokens_per_seq: int = 1024) -> Workload:
    g = _gen(seed, device)
    H, D, bs = 8, 128, 16
    seq_lens = torch.full((seqs,), tokens_per_seq, dtype=torch.int32, device=device)
    mbps = -(-tokens_per_seq // bs)
    nb = seqs * mbps
    tables = block_tables_from_pool(seq_lens, bs, nb, mbps, g)
    n = seqs * tokens_per_seq
    choices = torch.tensor([1.0, 4.0, 18.0], device=device)
    sigma = choices[torch.randint(0, 3, (H,), generator=g, device=device)]
    key = (torch.randn((n, H, D), generator=g, device=device, dtype=torch.float32)
           * sigma[None, :, None]).to(torch.bfloat16).reshape(n, H * D)
    value = _normal_bf16((n, H * D), 1.0, g, device)
    weight = (torch.rand((D,), generator=g, device=device, dtype=torch.float32) + 0.5).to(torch.bfloat16)
    token_seq, positions = _prefill_token_index(seq_lens)
    return Workload("fused_write", seqs, H, H, D, bs, nb, mbps, seq_lens, tables, key, value, None,
                    positions, token_seq,
                    extra=dict(k_norm_weight=weight, rotary_dim=128, theta=1e6, rms_eps=1e-6,
                               sigma=sigma))


def bf16_gqa4(seed: int = 1003, device="cpu", num_seqs: int = 64, min_len: int = 512,
              max_len: int = 8192, num_blocks: int = 40000) -> Workload:
    g = _gen(seed, device)
    Hq, H, D, bs = 32, 8, 128, 16
    seq_lens = torch.randint(min_len, max_len + 1, (num_seqs,), generator=g, device=device,
                             dtype=torch.int64).to(torch.int32)
    mbps = -(-max_len // bs)
    tables = block_tables_from_pool(seq_lens, bs, num_blocks, mbps, g)
    n = int(seq_lens.sum())
    key = _normal_bf16((n, H * D), 1.0, g, device)
    value = _normal_bf16((n, H * D), 1.0, g, device)
    q = _normal_bf16((num_seqs, Hq * D), 1.0, g, device)
    token_seq, positions = _prefill_token_index(seq_lens)
    return Workload("bf16_gqa4", num_seqs, Hq, H, D, bs, num_blocks, mbps, seq_lens, tables, key,
                    value, q, positions, token_seq, inv_sqrt_d=1.0 / math.sqrt(D))


def fp8k_long(seed: int = 1004, device="cpu", num_seqs: int = 128, seq_len: int = 32768) -> Workload:
    g = _gen(seed, device)
    Hq, H, D, bs = 32, 8, 128, 16
    seq_lens = torch.full((num_seqs,), seq_len, dtype=torch.int32, device=device)
    mbps = -(-seq_len // bs)
    nb = num_seqs * mbps
    tables = block_tables_from_pool(seq_lens, bs, nb, mbps, g)
    n = num_seqs * seq_len
    key, k_scale = fp8k_keys(n, H * D, g, device)
    value = _normal_bf16((n, H * D), 1.0, g, device)
    q = _normal_bf16((num_seqs, Hq * D), 1.0, g, device)
    token_seq, positions = _prefill_token_index(seq_lens)
    return Workload("fp8k_long", num_seqs, Hq, H, D, bs, nb, mbps, seq_lens, tables, key, value, q,
                    positions, token_seq, inv_sqrt_d=1.0 / math.sqrt(D), k_scale=k_scale,
                    v_scale=amax_scale(value),
                    sliding_windows=(0, 4096))


def fp8k_mixed(seed: int = 1005, device="cpu", num_seqs: int = 256, min_len: int = 128,
               max_len: int = 65536) -> Workload:
    g = _gen(seed, device)
    Hq, H, D, bs = 64, 8, 128, 64
    u = torch.rand((num_seqs,), generator=g, device=device, dtype=torch.float64)
    lens = torch.exp(math.log(min_len) + u * (math.log(max_len) - math.log(min_len)))
    seq_lens = torch.round(lens).clamp(min_len, max_len).to(torch.int32)
    needed = int((-(-seq_lens.to(torch.int64) // bs)).sum())
    nb = int(math.ceil(1.25 * needed))
    mbps = -(-max_len // bs)
    tables = block_tables_from_pool(seq_lens, bs, nb, mbps, g)
    n = int(seq_lens.sum())
    key, k_scale = fp8k_keys(n, H * D, g, device)
    value = _normal_bf16((n, H * D), 1.0, g, device)
    q = _normal_bf16((num_seqs, Hq * D), 1.0, g, device)
    token_seq, positions = _prefill_token_index(seq_lens)
    return Workload("fp8k_mixed", num_seqs, Hq, H, D, bs, nb, mbps, seq_lens, tables, key, value, q,
                    positions, token_seq, inv_sqrt_d=1.0 / math.sqrt(D), k_scale=k_scale,
                    v_scale=amax_scale(value))


WORKLOADS = {
    "tiny": tiny,
    "fused_write": fused_write,
    "bf16_gqa4": bf16_gqa4,
    "fp8k_long": fp8k_long,
    "fp8k_mixed": fp8k_mixed,
}


def custom(seed: int, device="cpu", *, seq_lens, num_q_heads, num_kv_heads, head_dim, block_size,
           num_blocks=None, max_blocks_per_seq=None, key_sigma=1.0, fp8=False, q_rows=None) -> Workload:
    """A small workload of any shape, for edge-case tests: given lengths, a
    permuted pool with spare blocks, N(0, key_sigma) K (or fp8k_keys when
    fp8), N(0, 1) V and Q. v_scale is max|V| / 448 (float32), the scale an
    E4M3 V cache of these rows would use."""
    g = _gen(seed, device)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32).to(device)
    need = [-(-int(L) // block_size) for L in seq_lens.tolist()]
    mbps = max_blocks_per_seq or max(max(need), 1)
    nb = num_blocks or max(sum(need) + 3, 1)
    tables = block_tables_from_pool(seq_lens, block_size, nb, mbps, g)
    n = int(seq_lens.to(torch.int64).sum())
    row = num_kv_heads * head_dim
    k_scale = 1.0
    if fp8:
        key, k_scale = fp8k_keys(max(n, 1), row, g, device)
        key = key[:n]
    else:
        key = _normal_bf16((n, row), key_sigma, g, device)
    value = _normal_bf16((n, row), 1.0, g, device)
    q = _normal_bf16((q_rows or len(seq_lens), num_q_heads * head_dim), 1.0, g, device)
    token_seq, positions = _prefill_token_index(seq_lens)
    return Workload("custom", len(seq_lens), num_q_heads, num_kv_heads, head_dim, block_size, nb,
                    mbps, seq_lens, tables, key, value, q, positions, token_seq,
                    inv_sqrt_d=1.0 / math.sqrt(head_dim), k_scale=k_scale, v_scale=amax_scale(value))


def amax_scale(x: torch.Tensor) -> float:
    """Per-tensor E4M3 scale max|x| / 448, in float32 (1.0 for an empty or
    all-zero tensor). Rows are scanned in chunks, so no full-size temporary
    is made."""
    if x.numel() == 0:
        return 1.0
    step = _rows_per_chunk(x.shape[-1]) if x.dim() == 2 else x.shape[0]
    amax = 0.0
    for r0 in range(0, x.shape[0], step):
        amax = max(amax, float(x[r0:r0 + step].abs().max().float().item()))
    return float(torch.tensor(amax / 448.0, dtype=torch.float32).item()) if amax > 0 else 1.0


def poisoned_pool(num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                  dtype: str, device="cpu") -> torch.Tensor:
    """A cache pool [num_blocks, block_size, num_kv_heads, head_dim] filled
    with the NaN pattern of its format: bf16 pools as int16 0x7FC0 viewed as
    bfloat16, fp8 pools as uint8 0x7F."""
    shape = (num_blocks, block_size, num_kv_heads, head_dim)
    if dtype == "bf16":
        return torch.full(shape, BF16_NAN, dtype=torch.int16, device=device).view(torch.bfloat16)
    if dtype == "fp8":
        return torch.full(shape, E4M3_NAN, dtype=torch.uint8, device=device)
    raise ValueError(dtype)
