"""CPU oracle for the paged KV-cache path (test infrastructure only).

A plain, slow, single-threaded C restatement (``oracle.c``) of the library's
calls, loaded with ctypes. Only the tests, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import this package; the product
path (``paged_kv_cache_fill_gb300``) never does, and the two share no code.

Every array argument is a C-contiguous numpy array with the dtype named in the
signature; BF16 tensors travel as their uint16 bit patterns and FP8 E4M3 as
uint8 codes. Functions that write a cache modify the given pool in place.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
# The mutation test points this at a deliberately broken build of oracle.c.
_OVERRIDE = os.environ.get("PAGEDKV_ORACLE_LIB")
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def compile_to(src: str, out: str) -> None:
    subprocess.run(["gcc", *CFLAGS, "-o", out, src, "-lm"], check=True)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, host architecture)."""
    if _OVERRIDE:
        return _OVERRIDE
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        compile_to(_SRC, tmp)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _u32(x):
    return ctypes.c_uint32(int(x))


def _f32(x):
    return ctypes.c_float(float(x))


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.oracle_bf16_to_f64.restype = ctypes.c_double
        _lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        _lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        _lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        _lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        _lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        _lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        _lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    return _lib


def _check(a: np.ndarray, dtype, name: str) -> np.ndarray:
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"{name}: expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    bits = _check(np.asarray(bits), np.uint16, "bits")
    out = np.empty(bits.shape, np.float64)
    lib().oracle_bf16_to_f64_array(_ptr(bits), _ptr(out), ctypes.c_int64(bits.size))
    return out


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    x = _check(np.asarray(x, np.float64), np.float64, "x")
    out = np.empty(x.shape, np.uint16)
    lib().oracle_f64_to_bf16_array(_ptr(x), _ptr(out), ctypes.c_int64(x.size))
    return out


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    codes = _check(np.asarray(codes), np.uint8, "codes")
    out = np.empty(codes.shape, np.float64)
    lib().oracle_e4m3_to_f64_array(_ptr(codes), _ptr(out), ctypes.c_int64(codes.size))
    return out


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    x = _check(np.asarray(x, np.float32), np.float32, "x")
    out = np.empty(x.shape, np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(x), _ptr(out), ctypes.c_int64(x.size))
    return out


def e4m3_encode_f64(x: np.ndarray) -> np.ndarray:
    x = _check(np.asarray(x, np.float64), np.float64, "x")
    out = np.empty(x.shape, np.uint8)
    lib().oracle_e4m3_encode_f64_array(_ptr(x), _ptr(out), ctypes.c_int64(x.size))
    return out


# --------------------------------------------------------------------------
# the seven calls
# --------------------------------------------------------------------------
def fill_slots(block_table: np.ndarray, start_pos: int, count: int, block_size: int) -> np.ndarray:
    block_table = _check(block_table, np.int32, "block_table")
    slots = np.empty(int(count), np.int64)
    lib().oracle_fill_slots(_ptr(slots), _ptr(block_table), _u32(start_pos), _u32(count),
                            _u32(block_size))
    return slots


def write_bf16(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
               block_size, key_stride, value_stride) -> None:
    for a, n in ((key, "key"), (value, "value"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(a, np.uint16, n)
    _check(slot_mapping, np.int64, "slot_mapping")
    lib().oracle_write_bf16(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                            _ptr(slot_mapping), _u32(num_tokens), _u32(num_kv_heads),
                            _u32(head_dim), _u32(block_size), _u32(key_stride),
                            _u32(value_stride))


def write_v_only(value, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim, block_size,
                 value_stride) -> None:
    _check(value, np.uint16, "value")
    _check(v_cache, np.uint16, "v_cache")
    _check(slot_mapping, np.int64, "slot_mapping")
    lib().oracle_write_v_only(_ptr(value), _ptr(v_cache), _ptr(slot_mapping), _u32(num_tokens),
                              _u32(num_kv_heads), _u32(head_dim), _u32(block_size),
                              _u32(value_stride))


def write_fp8k(key, value, k_cache_fp8, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
               block_size, key_stride, value_stride, k_scale) -> None:
    _check(key, np.uint16, "key")
    _check(value, np.uint16, "value")
    _check(k_cache_fp8, np.uint8, "k_cache_fp8")
    _check(v_cache, np.uint16, "v_cache")
    _check(slot_mapping, np.int64, "slot_mapping")
    lib().oracle_write_fp8k(_ptr(key), _ptr(value), _ptr(k_cache_fp8), _ptr(v_cache),
                            _ptr(slot_mapping), _u32(num_tokens), _u32(num_kv_heads),
                            _u32(head_dim), _u32(block_size), _u32(key_stride),
                            _u32(value_stride), _f32(k_scale))


def write_fp8(key, value, k_cache_fp8, v_cache_fp8, slot_mapping, num_tokens, num_kv_heads, head_dim,
              block_size, k_scale, v_scale, key_stride, value_stride) -> None:
    _check(key, np.uint16, "key")
    _check(value, np.uint16, "value")
    _check(k_cache_fp8, np.uint8, "k_cache_fp8")
    _check(v_cache_fp8, np.uint8, "v_cache_fp8")
    _check(slot_mapping, np.int64, "slot_mapping")
    lib().oracle_write_fp8(_ptr(key), _ptr(value), _ptr(k_cache_fp8), _ptr(v_cache_fp8),
                           _ptr(slot_mapping), _u32(num_tokens), _u32(num_kv_heads),
                           _u32(head_dim), _u32(block_size), _f32(k_scale), _f32(v_scale),
                           _u32(key_stride), _u32(value_stride))


def write_fused_k_norm_rope_bf16(k_in, k_norm_weight, positions, k_cache, slot_mapping,
                                 num_tokens, num_kv_heads, head_dim, rotary_dim, block_size,
                                 rms_eps, theta) -> None:
    _check(k_in, np.uint16, "k_in")
    _check(k_norm_weight, np.uint16, "k_norm_weight")
    _check(positions, np.int32, "positions")
    _check(k_cache, np.uint16, "k_cache")
    _check(slot_mapping, np.int64, "slot_mapping")
    if head_dim > 1024:
        raise ValueError("oracle supports head_dim <= 1024")
    lib().oracle_write_fused_k_norm_rope_bf16(
        _ptr(k_in), _ptr(k_norm_weight), _ptr(positions), _ptr(k_cache), _ptr(slot_mapping),
        _u32(num_tokens), _u32(num_kv_heads), _u32(head_dim), _u32(rotary_dim),
        _u32(block_size), _f32(rms_eps), _f32(theta))


def write_fused_k_norm_rope_bf16_mrope(k_in, k_norm_weight, pos_t, pos_h, pos_w, k_cache,
                                       slot_mapping, num_tokens, num_kv_heads, head_dim, rotary_dim,
                                       block_size, rms_eps, theta) -> None:
    _check(k_in, np.uint16, "k_in")
    _check(k_norm_weight, np.uint16, "k_norm_weight")
    for a, n in ((pos_t, "pos_t"), (pos_h, "pos_h"), (pos_w, "pos_w")):
        _check(a, np.int32, n)
    _check(k_cache, np.uint16, "k_cache")
    _check(slot_mapping, np.int64, "slot_mapping")
    lib().oracle_write_fused_k_norm_rope_bf16_mrope(
        _ptr(k_in), _ptr(k_norm_weight), _ptr(pos_t), _ptr(pos_h), _ptr(pos_w), _ptr(k_cache),
        _ptr(slot_mapping), _u32(num_tokens), _u32(num_kv_heads), _u32(head_dim), _u32(rotary_dim),
        _u32(block_size), _f32(rms_eps), _f32(theta))


def write_fused_k_norm_rope_fp8(k_in, k_norm_weight, positions, k_cache_fp8, slot_mapping, num_tokens,
                                num_kv_heads, head_dim, rotary_dim, block_size, rms_eps, theta,
                                inv_scale) -> None:
    _check(k_in, np.uint16, "k_in")
    _check(k_norm_weight, np.uint16, "k_norm_weight")
    _check(positions, np.int32, "positions")
    _check(k_cache_fp8, np.uint8, "k_cache_fp8")
    _check(slot_mapping, np.int64, "slot_mapping")
    lib().oracle_write_fused_k_norm_rope_fp8(
        _ptr(k_in), _ptr(k_norm_weight), _ptr(positions), _ptr(k_cache_fp8), _ptr(slot_mapping),
        _u32(num_tokens), _u32(num_kv_heads), _u32(head_dim), _u32(rotary_dim), _u32(block_size),
        _f32(rms_eps), _f32(theta), _f32(inv_scale))


def rope_row_mrope(y: np.ndarray, rotary_dim: int, pos3, theta: float) -> np.ndarray:
    y = _check(np.asarray(y, np.float64), np.float64, "y")
    p3 = np.ascontiguousarray(np.asarray(pos3, np.float64))
    out = np.empty_like(y)
    lib().oracle_rope_row_mrope(_ptr(y), _u32(y.size), _u32(rotary_dim), _ptr(p3), ctypes.c_double(theta),
                                _ptr(out))
    return out


def fused_k_row_f64_mrope(k_in, k_norm_weight, pos_t, pos_h, pos_w, t, h, num_kv_heads, head_dim,
                          rotary_dim, rms_eps, theta) -> np.ndarray:
    out = np.empty(int(head_dim), np.float64)
    lib().oracle_fused_k_row_f64_mrope(
        _ptr(_check(k_in, np.uint16, "k_in")), _ptr(_check(k_norm_weight, np.uint16, "w")),
        _ptr(_check(pos_t, np.int32, "pos_t")), _ptr(_check(pos_h, np.int32, "pos_h")),
        _ptr(_check(pos_w, np.int32, "pos_w")), _u32(t), _u32(h), _u32(num_kv_heads), _u32(head_dim),
        _u32(rotary_dim), _f32(rms_eps), _f32(theta), _ptr(out))
    return out


def rmsnorm_row(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x = _check(np.asarray(x, np.float64), np.float64, "x")
    w = _check(np.asarray(w, np.float64), np.float64, "w")
    y = np.empty_like(x)
    lib().oracle_rmsnorm_row(_ptr(x), _ptr(w), _u32(x.size), ctypes.c_double(eps), _ptr(y))
    return y


def rope_row(y: np.ndarray, rotary_dim: int, pos: float, theta: float) -> np.ndarray:
    y = _check(np.asarray(y, np.float64), np.float64, "y")
    out = np.empty_like(y)
    lib().oracle_rope_row(_ptr(y), _u32(y.size), _u32(rotary_dim), ctypes.c_double(pos),
                          ctypes.c_double(theta), _ptr(out))
    return out


def fused_k_row_f64(k_in, k_norm_weight, positions, t, h, num_kv_heads, head_dim, rotary_dim,
                    rms_eps, theta) -> np.ndarray:
    out = np.empty(int(head_dim), np.float64)
    lib().oracle_fused_k_row_f64(_ptr(_check(k_in, np.uint16, "k_in")),
                                 _ptr(_check(k_norm_weight, np.uint16, "w")),
                                 _ptr(_check(positions, np.int32, "positions")), _u32(t), _u32(h),
                                 _u32(num_kv_heads), _u32(head_dim), _u32(rotary_dim),
                                 _f32(rms_eps), _f32(theta), _ptr(out))
    return out


def decode_one(q, k_cache_bf16, k_cache_fp8, v_cache, block_tables, seq_lens, max_blocks_per_seq,
               num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d, k_scale, q_stride,
               sliding_window, s, h, want_weights=False, v_cache_fp8=None, v_scale=1.0):
    """Output (float64[head_dim]) and optionally the softmax weights by position
    for one (sequence, query head). v_cache_fp8 (with v_scale) in place of
    v_cache selects an E4M3 V cache."""
    _check(q, np.uint16, "q")
    if v_cache_fp8 is None:
        _check(v_cache, np.uint16, "v_cache")
    else:
        _check(v_cache_fp8, np.uint8, "v_cache_fp8")
        v_cache = None
    _check(block_tables, np.int32, "block_tables")
    _check(seq_lens, np.int32, "seq_lens")
    if head_dim > 1024:
        raise ValueError("oracle supports head_dim <= 1024")
    out = np.empty(int(head_dim), np.float64)
    weights = np.empty(max(int(seq_lens[s]), 1), np.float64) if want_weights else None
    lib().oracle_decode_one(
        _ptr(q), _ptr(k_cache_bf16), _ptr(k_cache_fp8), _ptr(v_cache), _ptr(v_cache_fp8),
        _ptr(block_tables), _ptr(seq_lens), _u32(max_blocks_per_seq), _u32(num_q_heads),
        _u32(num_kv_heads), _u32(head_dim), _u32(block_size), _f32(inv_sqrt_d), _f32(k_scale),
        _f32(v_scale), _u32(q_stride), _u32(sliding_window), _u32(s), _u32(h), _ptr(out),
        _ptr(weights))
    if want_weights:
        return out, weights[: int(seq_lens[s])]
    return out


def paged_decode_attn_bf16(q, k_cache, v_cache, block_tables, seq_lens, max_blocks_per_seq,
                           num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d,
                           q_stride, sliding_window) -> np.ndarray:
    for a, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(a, np.uint16, n)
    _check(block_tables, np.int32, "block_tables")
    _check(seq_lens, np.int32, "seq_lens")
    out = np.empty((int(num_seqs), int(num_q_heads), int(head_dim)), np.float32)
    lib().oracle_paged_decode_attn_bf16(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(block_tables), _ptr(seq_lens),
        _u32(max_blocks_per_seq), _u32(num_seqs), _u32(num_q_heads), _u32(num_kv_heads),
        _u32(head_dim), _u32(block_size), _f32(inv_sqrt_d), _u32(q_stride), _u32(sliding_window))
    return out


def paged_decode_attn_fp8k(q, k_cache_fp8, v_cache, block_tables, seq_lens, max_blocks_per_seq,
                           num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d,
                           k_scale, q_stride, sliding_window) -> np.ndarray:
    _check(q, np.uint16, "q")
    _check(k_cache_fp8, np.uint8, "k_cache_fp8")
    _check(v_cache, np.uint16, "v_cache")
    _check(block_tables, np.int32, "block_tables")
    _check(seq_lens, np.int32, "seq_lens")
    out = np.empty((int(num_seqs), int(num_q_heads), int(head_dim)), np.float32)
    lib().oracle_paged_decode_attn_fp8k(
        _ptr(q), _ptr(k_cache_fp8), _ptr(v_cache), _ptr(out), _ptr(block_tables), _ptr(seq_lens),
        _u32(max_blocks_per_seq), _u32(num_seqs), _u32(num_q_heads), _u32(num_kv_heads),
        _u32(head_dim), _u32(block_size), _f32(inv_sqrt_d), _f32(k_scale), _u32(q_stride),
        _u32(sliding_window))
    return out


def paged_decode_attn_fp8(q, k_cache_fp8, v_cache_fp8, block_tables, seq_lens, max_blocks_per_seq,
                          num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d,
                          k_scale, v_scale, q_stride, sliding_window) -> np.ndarray:
    _check(q, np.uint16, "q")
    _check(k_cache_fp8, np.uint8, "k_cache_fp8")
    _check(v_cache_fp8, np.uint8, "v_cache_fp8")
    _check(block_tables, np.int32, "block_tables")
    _check(seq_lens, np.int32, "seq_lens")
    out = np.empty((int(num_seqs), int(num_q_heads), int(head_dim)), np.float32)
    lib().oracle_paged_decode_attn_fp8(
        _ptr(q), _ptr(k_cache_fp8), _ptr(v_cache_fp8), _ptr(out), _ptr(block_tables), _ptr(seq_lens),
        _u32(max_blocks_per_seq), _u32(num_seqs), _u32(num_q_heads), _u32(num_kv_heads),
        _u32(head_dim), _u32(block_size), _f32(inv_sqrt_d), _f32(k_scale), _f32(v_scale),
        _u32(q_stride), _u32(sliding_window))
    return out


def paged_prefill_attn(q, k_cache_bf16, k_cache_fp8, v_cache, block_tables, seq_lens, query_start_loc,
                       max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       inv_sqrt_d, k_scale, q_stride, sliding_window, v_cache_fp8=None,
                       v_scale=1.0) -> np.ndarray:
    """Multi-token paged attention; pass k_cache_fp8 (and k_scale) or
    k_cache_bf16, the other None; v_cache_fp8 (with v_scale) in place of
    v_cache selects an E4M3 V cache. Returns float32 [num_q_tokens, Hq, D]."""
    _check(q, np.uint16, "q")
    if k_cache_fp8 is None:
        _check(k_cache_bf16, np.uint16, "k_cache_bf16")
    else:
        _check(k_cache_fp8, np.uint8, "k_cache_fp8")
    if v_cache_fp8 is None:
        _check(v_cache, np.uint16, "v_cache")
    else:
        _check(v_cache_fp8, np.uint8, "v_cache_fp8")
        v_cache = None
    _check(block_tables, np.int32, "block_tables")
    _check(seq_lens, np.int32, "seq_lens")
    _check(query_start_loc, np.int32, "query_start_loc")
    n_q = int(query_start_loc[int(num_seqs)])
    out = np.empty((n_q, int(num_q_heads), int(head_dim)), np.float32)
    lib().oracle_paged_prefill_attn(
        _ptr(q), _ptr(k_cache_bf16), _ptr(k_cache_fp8), _ptr(v_cache), _ptr(v_cache_fp8), _ptr(out),
        _ptr(block_tables), _ptr(seq_lens), _ptr(query_start_loc), _u32(max_blocks_per_seq), _u32(num_seqs),
        _u32(num_q_heads), _u32(num_kv_heads), _u32(head_dim), _u32(block_size), _f32(inv_sqrt_d), _f32(k_scale),
        _f32(v_scale), _u32(q_stride), _u32(sliding_window))
    return out
