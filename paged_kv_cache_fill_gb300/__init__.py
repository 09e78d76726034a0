"""Python binding of libpagedkv (the paged KV-cache C ABI, include/pagedkv.h).

Argument marshalling only: every function passes its tensors' device
pointers and its scalars straight to the C entry point of the same name and
raises PagedKVError on a non-zero status. All work runs in the library's
CUDA kernels; there is no other implementation to fall back on, so a missing
library is an error.

Tensors must be contiguous and live on the current CUDA device (checked
here; the C entry points take raw pointers). BF16 data are torch.bfloat16
(or int16/uint16 bit patterns), FP8 caches torch.uint8 or
torch.float8_e4m3fn. `stream` is a torch.cuda.Stream, a raw cudaStream_t
integer, or None for torch's current stream.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "PagedKVError", "library_path", "kv_fill_slots", "kv_write_bf16", "kv_write_fp8k", "kv_write_fp8",
    "kv_write_fused_k_norm_rope_bf16", "kv_write_fused_k_norm_rope_bf16_mrope",
    "kv_write_fused_k_norm_rope_fp8", "kv_write_v_only", "paged_decode_attn_bf16",
    "paged_decode_attn_fp8k", "paged_decode_attn_fp8", "paged_prefill_attn_bf16", "paged_prefill_attn_fp8k",
    "paged_prefill_attn_fp8", "paged_decode_attn_fp8k_static_scratch",
    "kv_decode_workspace_bytes",
    "kv_set_decode_workspace", "kv_get_device_error", "kv_device_info", "kv_debug_set_pool",
    "kv_debug_set_wait_limit", "use_library",
    "KV_OK", "KV_ERR_INVALID_ARG",
    "KV_ERR_UNSUPPORTED", "KV_ERR_CUDA", "KV_ERR_DEVICE",
]

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_UNSUPPORTED, KV_ERR_CUDA, KV_ERR_DEVICE = 0, 1, 2, 3, 4

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpagedkv.so")
_lib = None
_workspace_keepalive: dict[int, torch.Tensor] = {}

_P, _U32, _F32, _SZ = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t
_SIGNATURES = {
    "kv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kv_fill_slots": (ctypes.c_int, [_P, _P, _U32, _U32, _U32, _P]),
    "kv_write_bf16": (ctypes.c_int, [_P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _U32, _P]),
    "kv_write_fp8k": (ctypes.c_int, [_P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _U32, _F32, _P]),
    "kv_write_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _F32, _F32, _U32, _U32, _P]),
    "kv_write_fused_k_norm_rope_bf16": (
        ctypes.c_int, [_P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _F32, _F32, _P]),
    "kv_write_fused_k_norm_rope_bf16_mrope": (
        ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _F32, _F32, _P]),
    "kv_write_fused_k_norm_rope_fp8": (
        ctypes.c_int, [_P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _F32, _F32, _F32, _P]),
    "kv_write_v_only": (ctypes.c_int, [_P, _P, _P, _U32, _U32, _U32, _U32, _U32, _P]),
    "paged_decode_attn_bf16": (
        ctypes.c_int, [_P, _P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _U32, _F32, _U32, _U32, _P]),
    "paged_decode_attn_fp8k": (
        ctypes.c_int,
        [_P, _P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _U32, _F32, _F32, _U32, _U32, _P]),
    "paged_decode_attn_fp8": (
        ctypes.c_int,
        [_P, _P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _U32, _F32, _F32, _F32, _U32, _U32, _P]),
    "paged_prefill_attn_bf16": (
        ctypes.c_int,
        [_P, _P, _P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _U32, _U32, _F32, _U32, _U32, _P]),
    "paged_prefill_attn_fp8k": (
        ctypes.c_int,
        [_P, _P, _P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _U32, _U32, _F32, _F32, _U32, _U32, _P]),
    "paged_prefill_attn_fp8": (
        ctypes.c_int,
        [_P, _P, _P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _U32, _U32, _F32, _F32, _F32, _U32, _U32, _P]),
    "paged_decode_attn_fp8k_static_scratch": (
        ctypes.c_int,
        [_P, _P, _P, _P, _P, _P, _U32, _U32, _U32, _U32, _U32, _U32, _F32, _F32, _U32, _U32, _P]),
    "kv_decode_workspace_bytes": (_SZ, [_U32, _U32, _U32, _U32, _U32, _U32]),
    "kv_set_decode_workspace": (ctypes.c_int, [_P, _SZ]),
    "kv_get_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "kv_device_info": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "kv_debug_set_pool": (ctypes.c_int, [_U32, _U32]),
    "kv_debug_set_wait_limit": (ctypes.c_int, [ctypes.c_uint64]),
}


class PagedKVError(RuntimeError):
    def __init__(self, name: str, status: int):
        self.status = status
        super().__init__(f"{name}: status {status} ({_status_text(status)})")


def use_library(path: str) -> None:
    """Load the library from `path` instead of the default build, e.g. the
    bounds-checking libpagedkv_debug.so (`_build.build(debug=True)`). Only
    before the first call: the library in use cannot be swapped."""
    global library_path
    if _lib is not None:
        raise RuntimeError(f"{library_path} is already loaded")
    library_path = os.path.abspath(path)


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(
                f"{library_path} is missing: build it with `python -c \"import __graft_entry__ as g; "
                f"g.build()\"` (nvcc, sm_103a)")
        handle = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype, fn.argtypes = res, args
        _lib = handle
    return _lib


def _status_text(status: int) -> str:
    try:
        return lib().kv_status_string(status).decode()
    except Exception:  # noqa: BLE001 - only used to format an error
        return "?"


def _check(name: str, status: int) -> None:
    if status != KV_OK:
        raise PagedKVError(name, status)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if t.numel():
        if not t.is_cuda:
            raise ValueError("tensor must be on a CUDA device")
        if t.get_device() != torch.cuda.current_device():
            raise ValueError(f"tensor is on cuda:{t.get_device()}, the current device is "
                             f"cuda:{torch.cuda.current_device()}")
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous (the library reads rows at the strides it is given)")
    return t.data_ptr() or None


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def kv_fill_slots(slots, block_table, start_pos, count, block_size, stream=None):
    _check("kv_fill_slots", lib().kv_fill_slots(
        _ptr(slots), _ptr(block_table), start_pos, count, block_size, _stream(stream)))


def kv_write_bf16(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
                  block_size, key_stride, value_stride, stream=None):
    _check("kv_write_bf16", lib().kv_write_bf16(
        _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), num_tokens,
        num_kv_heads, head_dim, block_size, key_stride, value_stride, _stream(stream)))


def kv_write_fp8k(key, value, k_cache_fp8, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
                  block_size, key_stride, value_stride, k_scale, stream=None):
    _check("kv_write_fp8k", lib().kv_write_fp8k(
        _ptr(key), _ptr(value), _ptr(k_cache_fp8), _ptr(v_cache), _ptr(slot_mapping), num_tokens,
        num_kv_heads, head_dim, block_size, key_stride, value_stride, k_scale, _stream(stream)))


def kv_write_fp8(key, value, k_cache_fp8, v_cache_fp8, slot_mapping, num_tokens, num_kv_heads, head_dim,
                 block_size, k_scale, v_scale, key_stride, value_stride, stream=None):
    _check("kv_write_fp8", lib().kv_write_fp8(
        _ptr(key), _ptr(value), _ptr(k_cache_fp8), _ptr(v_cache_fp8), _ptr(slot_mapping), num_tokens,
        num_kv_heads, head_dim, block_size, k_scale, v_scale, key_stride, value_stride, _stream(stream)))


def kv_write_fused_k_norm_rope_bf16(k_in, k_norm_weight, positions, k_cache, slot_mapping, num_tokens,
                                    num_kv_heads, head_dim, rotary_dim, block_size, rms_eps, theta,
                                    stream=None):
    _check("kv_write_fused_k_norm_rope_bf16", lib().kv_write_fused_k_norm_rope_bf16(
        _ptr(k_in), _ptr(k_norm_weight), _ptr(positions), _ptr(k_cache), _ptr(slot_mapping),
        num_tokens, num_kv_heads, head_dim, rotary_dim, block_size, rms_eps, theta, _stream(stream)))


def kv_write_fused_k_norm_rope_bf16_mrope(k_in, k_norm_weight, pos_t, pos_h, pos_w, k_cache, slot_mapping,
                                          num_tokens, num_kv_heads, head_dim, rotary_dim, block_size, rms_eps,
                                          theta, stream=None):
    _check("kv_write_fused_k_norm_rope_bf16_mrope", lib().kv_write_fused_k_norm_rope_bf16_mrope(
        _ptr(k_in), _ptr(k_norm_weight), _ptr(pos_t), _ptr(pos_h), _ptr(pos_w), _ptr(k_cache),
        _ptr(slot_mapping), num_tokens, num_kv_heads, head_dim, rotary_dim, block_size, rms_eps, theta,
        _stream(stream)))


def kv_write_fused_k_norm_rope_fp8(k_in, k_norm_weight, positions, k_cache_fp8, slot_mapping, num_tokens,
                                   num_kv_heads, head_dim, rotary_dim, block_size, rms_eps, theta, inv_scale,
                                   stream=None):
    _check("kv_write_fused_k_norm_rope_fp8", lib().kv_write_fused_k_norm_rope_fp8(
        _ptr(k_in), _ptr(k_norm_weight), _ptr(positions), _ptr(k_cache_fp8), _ptr(slot_mapping), num_tokens,
        num_kv_heads, head_dim, rotary_dim, block_size, rms_eps, theta, inv_scale, _stream(stream)))


def kv_write_v_only(value, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim, block_size,
                    value_stride, stream=None):
    _check("kv_write_v_only", lib().kv_write_v_only(
        _ptr(value), _ptr(v_cache), _ptr(slot_mapping), num_tokens, num_kv_heads, head_dim,
        block_size, value_stride, _stream(stream)))


def paged_decode_attn_bf16(q, k_cache, v_cache, output, block_tables, seq_lens, max_blocks_per_seq,
                           num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d,
                           q_stride, sliding_window, stream=None):
    _check("paged_decode_attn_bf16", lib().paged_decode_attn_bf16(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(output), _ptr(block_tables), _ptr(seq_lens),
        max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d,
        q_stride, sliding_window, _stream(stream)))


def paged_decode_attn_fp8k(q, k_cache_fp8, v_cache, output, block_tables, seq_lens, max_blocks_per_seq,
                           num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d,
                           k_scale, q_stride, sliding_window, stream=None):
    _check("paged_decode_attn_fp8k", lib().paged_decode_attn_fp8k(
        _ptr(q), _ptr(k_cache_fp8), _ptr(v_cache), _ptr(output), _ptr(block_tables), _ptr(seq_lens),
        max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d,
        k_scale, q_stride, sliding_window, _stream(stream)))


def paged_decode_attn_fp8(q, k_cache_fp8, v_cache_fp8, output, block_tables, seq_lens, max_blocks_per_seq,
                          num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d, k_scale, v_scale,
                          q_stride, sliding_window, stream=None):
    _check("paged_decode_attn_fp8", lib().paged_decode_attn_fp8(
        _ptr(q), _ptr(k_cache_fp8), _ptr(v_cache_fp8), _ptr(output), _ptr(block_tables), _ptr(seq_lens),
        max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d,
        k_scale, v_scale, q_stride, sliding_window, _stream(stream)))


def paged_prefill_attn_bf16(q, k_cache, v_cache, output, block_tables, seq_lens, query_start_loc,
                            max_blocks_per_seq, num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
                            block_size, inv_sqrt_d, q_stride, sliding_window, stream=None):
    _check("paged_prefill_attn_bf16", lib().paged_prefill_attn_bf16(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(output), _ptr(block_tables), _ptr(seq_lens),
        _ptr(query_start_loc), max_blocks_per_seq, num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
        block_size, inv_sqrt_d, q_stride, sliding_window, _stream(stream)))


def paged_prefill_attn_fp8k(q, k_cache_fp8, v_cache, output, block_tables, seq_lens, query_start_loc,
                            max_blocks_per_seq, num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
                            block_size, inv_sqrt_d, k_scale, q_stride, sliding_window, stream=None):
    _check("paged_prefill_attn_fp8k", lib().paged_prefill_attn_fp8k(
        _ptr(q), _ptr(k_cache_fp8), _ptr(v_cache), _ptr(output), _ptr(block_tables), _ptr(seq_lens),
        _ptr(query_start_loc), max_blocks_per_seq, num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
        block_size, inv_sqrt_d, k_scale, q_stride, sliding_window, _stream(stream)))


def paged_prefill_attn_fp8(q, k_cache_fp8, v_cache_fp8, output, block_tables, seq_lens, query_start_loc,
                           max_blocks_per_seq, num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
                           block_size, inv_sqrt_d, k_scale, v_scale, q_stride, sliding_window, stream=None):
    _check("paged_prefill_attn_fp8", lib().paged_prefill_attn_fp8(
        _ptr(q), _ptr(k_cache_fp8), _ptr(v_cache_fp8), _ptr(output), _ptr(block_tables), _ptr(seq_lens),
        _ptr(query_start_loc), max_blocks_per_seq, num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
        block_size, inv_sqrt_d, k_scale, v_scale, q_stride, sliding_window, _stream(stream)))


def paged_decode_attn_fp8k_static_scratch(q, k_cache_fp8, v_cache, output, block_tables, seq_lens,
                                          max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                          block_size, inv_sqrt_d, k_scale, q_stride, sliding_window, stream=None):
    """paged_decode_attn_fp8k without any caller-provided memory: the split-KV
    scratch is a fixed 64 MiB array inside the library (for callers that
    cannot allocate device memory or register a workspace). Calls share that
    array, so calls that may overlap on the GPU must be ordered."""
    _check("paged_decode_attn_fp8k_static_scratch", lib().paged_decode_attn_fp8k_static_scratch(
        _ptr(q), _ptr(k_cache_fp8), _ptr(v_cache), _ptr(output), _ptr(block_tables), _ptr(seq_lens),
        max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d,
        k_scale, q_stride, sliding_window, _stream(stream)))


def kv_decode_workspace_bytes(max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim,
                              block_size) -> int:
    return int(lib().kv_decode_workspace_bytes(max_blocks_per_seq, num_seqs, num_q_heads,
                                               num_kv_heads, head_dim, block_size))


def kv_set_decode_workspace(workspace: torch.Tensor | None) -> None:
    """Register (or, with None, unregister) the split-KV workspace of the
    current device. The tensor is kept alive until it is replaced."""
    dev = torch.cuda.current_device()
    if workspace is None:
        _check("kv_set_decode_workspace", lib().kv_set_decode_workspace(None, 0))
        _workspace_keepalive.pop(dev, None)
        return
    nbytes = workspace.numel() * workspace.element_size()
    _check("kv_set_decode_workspace", lib().kv_set_decode_workspace(_ptr(workspace), nbytes))
    _workspace_keepalive[dev] = workspace


def kv_debug_set_pool(num_blocks: int, block_size: int) -> None:
    """Bounds-checking build only: check every slot and block id against a
    pool of num_blocks blocks of block_size slots (0 blocks: unchecked) on
    the current device; an index outside it sets 8 in kv_get_device_error's
    bits. Raises PagedKVError (KV_ERR_UNSUPPORTED) on the product build."""
    _check("kv_debug_set_pool", lib().kv_debug_set_pool(num_blocks, block_size))


def kv_debug_set_wait_limit(nanoseconds: int) -> None:
    """Bounds-checking build only: the paged decode's pipeline wait limit on
    the current device (0 restores the default 2 s). Raises PagedKVError
    (KV_ERR_UNSUPPORTED) on the product build."""
    _check("kv_debug_set_wait_limit", lib().kv_debug_set_wait_limit(nanoseconds))


def kv_get_device_error() -> int:
    """Synchronise the current device and return (and clear) the kernels'
    fault bits: 1 = a pipeline wait timed out, 2 = a sequence length was
    clamped to its block table, 4 = a prefill's query_start_loc was
    decreasing, negative or past num_q_tokens (that sequence skipped),
    8 = (bounds-checking build) a slot or block id outside the pool."""
    bits = ctypes.c_uint32(0)
    status = lib().kv_get_device_error(ctypes.byref(bits))
    if status != KV_ERR_DEVICE:  # KV_ERR_DEVICE only says that some bit was set
        _check("kv_get_device_error", status)
    return int(bits.value)


def kv_device_info() -> tuple[int, int]:
    sms, ctas = ctypes.c_int(0), ctypes.c_int(0)
    _check("kv_device_info", lib().kv_device_info(ctypes.byref(sms), ctypes.byref(ctas)))
    return int(sms.value), int(ctas.value)
