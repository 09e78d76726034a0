"""C-ABI contract checks that need no GPU: the library builds and loads, it
exports every entry point include/pagedkv.h declares (and the binding wraps
each of them), and argument validation returns the documented status before
any CUDA call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_fill_gb300 import _build
    _build.build()
    import paged_kv_cache_fill_gb300 as pk
    pk.lib()
    return pk


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^PAGEDKV_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)


def test_header_declares_the_seven_calls():
    names = set(declared_functions())
    for n in ["kv_fill_slots", "kv_write_bf16", "kv_write_fp8k", "kv_write_fused_k_norm_rope_bf16",
              "kv_write_v_only", "paged_decode_attn_bf16", "paged_decode_attn_fp8k"]:
        assert n in names


def test_library_exports_every_declared_symbol(pk):
    for name in declared_functions():
        assert hasattr(pk.lib(), name), name


def test_binding_argument_counts_match_header(pk):
    text = open(HEADER).read()
    for name in declared_functions():
        m = re.search(r"^PAGEDKV_API[^;]*?\b" + name + r"\s*\(([^)]*)\)", text, re.S | re.M)
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(pk._SIGNATURES[name][1]) == len(params), name


def test_only_declared_symbols_are_exported(pk):
    lib = pk.lib()
    # a few internal names that must stay hidden
    for hidden in ["launch_decode", "device_info", "_ZN7pagedkv13launch_decodeERKNS_10DecodeArgsEP11CUstream_st"]:
        with pytest.raises(AttributeError):
            getattr(lib, hidden)


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: validation fails first


def test_zero_work_is_ok_and_launches_nothing(pk):
    L = pk.lib()
    assert L.kv_fill_slots(None, None, 0, 0, 16, None) == pk.KV_OK
    assert L.kv_write_bf16(None, None, None, None, None, 0, 8, 128, 16, 1024, 1024, None) == pk.KV_OK
    assert L.kv_write_v_only(None, None, None, 0, 8, 128, 16, 1024, None) == pk.KV_OK
    assert L.kv_write_fp8k(None, None, None, None, None, 0, 8, 128, 16, 1024, 1024, 1.0, None) == pk.KV_OK
    assert L.kv_write_fused_k_norm_rope_bf16(None, None, None, None, None, 0, 8, 128, 128, 16, 1e-6, 1e6,
                                             None) == pk.KV_OK
    assert L.paged_decode_attn_bf16(None, None, None, None, None, None, 4, 0, 32, 8, 128, 16, 0.1, 4096, 0,
                                    None) == pk.KV_OK
    assert L.paged_decode_attn_fp8k(None, None, None, None, None, None, 4, 0, 32, 8, 128, 16, 0.1, 1.0, 4096,
                                    0, None) == pk.KV_OK


def test_invalid_arguments(pk):
    L, INV = pk.lib(), pk.KV_ERR_INVALID_ARG
    assert L.kv_fill_slots(None, FAKE, 0, 5, 16, None) == INV
    assert L.kv_fill_slots(FAKE, FAKE, 0, 5, 0, None) == INV
    assert L.kv_write_bf16(FAKE, FAKE, FAKE, FAKE, None, 3, 8, 128, 16, 1024, 1024, None) == INV
    assert L.kv_write_bf16(FAKE, FAKE, FAKE, FAKE, FAKE, 3, 8, 128, 16, 1000, 1024, None) == INV  # stride
    assert L.kv_write_bf16(FAKE, FAKE, FAKE, FAKE, FAKE, 3, 8, 128, 0, 1024, 1024, None) == INV
    assert L.kv_write_v_only(FAKE, FAKE, FAKE, 3, 0, 128, 16, 1024, None) == INV
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        assert L.kv_write_fp8k(FAKE, FAKE, FAKE, FAKE, FAKE, 3, 8, 128, 16, 1024, 1024, bad, None) == INV
    fused = lambda **kw: L.kv_write_fused_k_norm_rope_bf16(  # noqa: E731
        FAKE, FAKE, FAKE, FAKE, FAKE, 3, 8, kw.get("D", 128), kw.get("R", 128), 16, kw.get("eps", 1e-6),
        kw.get("theta", 1e6), None)
    assert fused(R=127) == INV and fused(R=0) == INV and fused(R=256) == INV
    assert fused(eps=-1.0) == INV and fused(theta=0.0) == INV and fused(theta=float("nan")) == INV
    dec = lambda **kw: L.paged_decode_attn_fp8k(  # noqa: E731
        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, kw.get("Hq", 32), kw.get("H", 8), 128, 16, 0.1,
        kw.get("k_scale", 1.0), kw.get("q_stride", 4096), 0, None)
    assert dec(Hq=30) == INV and dec(H=0) == INV and dec(q_stride=100) == INV
    assert dec(k_scale=0.0) == INV and dec(k_scale=float("nan")) == INV


def test_unsupported_shapes(pk):
    L, UNS = pk.lib(), pk.KV_ERR_UNSUPPORTED
    assert L.kv_write_fused_k_norm_rope_bf16(FAKE, FAKE, FAKE, FAKE, FAKE, 3, 8, 96, 96, 16, 1e-6, 1e6,
                                             None) == UNS
    assert L.kv_write_fused_k_norm_rope_bf16(FAKE, FAKE, FAKE, FAKE, FAKE, 3, 8, 128, 100, 16, 1e-6, 1e6,
                                             None) == UNS
    base = dict(mbps=4, D=128, bs=16, Hq=32, H=8)

    def dec(fp8=False, **kw):
        a = dict(base, **kw)
        if fp8:
            return L.paged_decode_attn_fp8k(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["mbps"], 2, a["Hq"], a["H"],
                                            a["D"], a["bs"], 0.1, 1.0, a["Hq"] * a["D"], 0, None)
        return L.paged_decode_attn_bf16(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["mbps"], 2, a["Hq"], a["H"],
                                        a["D"], a["bs"], 0.1, a["Hq"] * a["D"], 0, None)
    assert dec(D=96) == UNS and dec(fp8=True, D=96) == UNS and dec(fp8=True, D=512) == UNS
    assert dec(bs=8) == UNS and dec(bs=24) == UNS and dec(bs=512) == UNS
    assert dec(Hq=64, H=2) == UNS            # group of 32 query heads
    misaligned = ctypes.c_void_p(0x10008)
    assert L.paged_decode_attn_bf16(misaligned, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 32, 8, 128, 16, 0.1,
                                    4096, 0, None) == UNS


def _prefill(L, kind, **kw):
    """One prefill call of `kind` ("bf16", "fp8k", "fp8") on fake pointers;
    every case below must fail validation before any device work."""
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, mbps=4, ns=2, nq=10, Hq=32, H=8, D=128, bs=16, isd=0.1,
             k_scale=1.0, v_scale=1.0, q_stride=4096, win=0)
    a.update(kw)
    head = (a["q"], a["k"], a["v"], a["out"], FAKE, FAKE, FAKE, a["mbps"], a["ns"], a["nq"], a["Hq"], a["H"],
            a["D"], a["bs"], a["isd"])
    if kind == "bf16":
        return L.paged_prefill_attn_bf16(*head, a["q_stride"], a["win"], None)
    if kind == "fp8k":
        return L.paged_prefill_attn_fp8k(*head, a["k_scale"], a["q_stride"], a["win"], None)
    return L.paged_prefill_attn_fp8(*head, a["k_scale"], a["v_scale"], a["q_stride"], a["win"], None)


@pytest.mark.parametrize("kind", ["bf16", "fp8k", "fp8"])
def test_prefill_zero_work_and_invalid_arguments(pk, kind):
    L, INV = pk.lib(), pk.KV_ERR_INVALID_ARG
    none = dict(q=None, k=None, v=None, out=None)
    assert _prefill(L, kind, ns=0, **none) == pk.KV_OK
    assert _prefill(L, kind, nq=0, **none) == pk.KV_OK
    assert _prefill(L, kind, out=None) == INV and _prefill(L, kind, v=None) == INV
    assert _prefill(L, kind, Hq=30) == INV and _prefill(L, kind, H=0) == INV
    assert _prefill(L, kind, q_stride=100) == INV and _prefill(L, kind, isd=float("nan")) == INV
    assert _prefill(L, kind, bs=0) == INV and _prefill(L, kind, D=0) == INV
    if kind != "bf16":
        for bad in (0.0, -1.0, float("inf"), float("nan")):
            assert _prefill(L, kind, k_scale=bad) == INV
    if kind == "fp8":
        for bad in (0.0, -1.0, float("inf"), float("nan")):
            assert _prefill(L, kind, v_scale=bad) == INV


@pytest.mark.parametrize("kind", ["bf16", "fp8k", "fp8"])
def test_prefill_unsupported_shapes(pk, kind):
    L, UNS = pk.lib(), pk.KV_ERR_UNSUPPORTED
    assert _prefill(L, kind, D=96, q_stride=32 * 96) == UNS
    assert _prefill(L, kind, D=256, q_stride=32 * 256) == UNS    # the prefills take head_dim 64 and 128
    assert _prefill(L, kind, bs=8) == UNS and _prefill(L, kind, bs=24) == UNS and _prefill(L, kind, bs=512) == UNS
    misaligned = ctypes.c_void_p(0x10008)
    assert _prefill(L, kind, q=misaligned) == UNS and _prefill(L, kind, out=misaligned) == UNS
    assert _prefill(L, kind, v=misaligned) == UNS
    assert _prefill(L, kind, q_stride=4097) == UNS                 # q rows must start on 16 bytes
    assert _prefill(L, kind, mbps=1 << 27, bs=16) == UNS           # 2^31 positions per sequence


def test_example_calls_match_the_binding(pk):
    """The example call sequence (paged_kv_cache_fill_gb300/example.py) needs
    a GPU to run; parse it instead and bind every pk.* call to the binding's
    signature."""
    import ast
    import inspect
    tree = ast.parse(open(os.path.join(ROOT, "paged_kv_cache_fill_gb300", "example.py")).read())
    calls = [n for n in ast.walk(tree) if isinstance(n, ast.Call) and isinstance(n.func, ast.Attribute)
             and isinstance(n.func.value, ast.Name) and n.func.value.id == "pk"]
    assert len(calls) >= 5
    for c in calls:
        name = c.func.attr
        assert name in pk.__all__, name
        sig = inspect.signature(getattr(pk, name))
        sig.bind(*[None] * len(c.args), **{k.arg: None for k in c.keywords})
        required = [q for q in sig.parameters.values() if q.default is inspect.Parameter.empty]
        assert len(c.args) == len(required), f"{name}: {len(c.args)} positional, {len(required)} required"


def test_product_build_has_no_bounds_checks(pk):
    assert pk.lib().kv_debug_set_pool(16, 16) == pk.KV_ERR_UNSUPPORTED
    assert pk.lib().kv_debug_set_wait_limit(1000) == pk.KV_ERR_UNSUPPORTED


def test_bounds_checking_build(pk):
    """The PAGEDKV_DEBUG_BOUNDS build compiles, exports exactly the header's
    calls, and takes kv_debug_set_pool (checked in a child process, which
    loads that library alone)."""
    import subprocess
    import sys
    sys.path.insert(0, os.path.join(ROOT, "paged_kv_cache_fill_gb300"))
    import _build
    path = _build.build(debug=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(declared_functions())
    code = (
        "import ctypes, sys\n"
        "L = ctypes.CDLL(sys.argv[1])\n"
        "f = L.kv_debug_set_pool\n"
        "f.restype, f.argtypes = ctypes.c_int, [ctypes.c_uint32, ctypes.c_uint32]\n"
        "print(f(16, 0), f(16, 16))\n")
    r = subprocess.run([sys.executable, "-c", code, path], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    bad_block_size, ok_or_no_device = map(int, r.stdout.split())
    assert bad_block_size == pk.KV_ERR_INVALID_ARG
    assert ok_or_no_device in (pk.KV_OK, pk.KV_ERR_CUDA)   # KV_OK where a GPU is present


def test_workspace_size_formula(pk):
    # header + piece counts (num_seqs * num_kv_heads words, in 256-byte
    # units) + num_seqs * P pieces * Hq * (D + 2) floats, where a sequence of
    # T = ceil(mbps * bs / 16) tiles cut by 16-tile chunks makes at most
    # P = (T - 2) // 16 + 2 pieces (T > 1)
    got = pk.kv_decode_workspace_bytes(512, 64, 32, 8, 128, 16)
    assert got == 256 + 2048 + 64 * 33 * 32 * 130 * 4
    assert pk.kv_decode_workspace_bytes(1, 1, 4, 2, 64, 16) == 256 + 256 + 1 * 1 * 4 * 66 * 4
    # the table geometry, not the lengths, sets the piece count: 19 blocks of
    # 16 positions (19 tiles) can meet 3 chunks of 16 tiles
    assert pk.kv_decode_workspace_bytes(19, 3, 8, 2, 128, 16) == 256 + 256 + 3 * 3 * 8 * 130 * 4
    # 64-position blocks: 4 tiles each
    assert pk.kv_decode_workspace_bytes(8, 100, 64, 8, 128, 64) == 256 + 3328 + 100 * 3 * 64 * 130 * 4


def max_pieces(tiles, chunk):
    """The most chunks of `chunk` tiles a run of `tiles` consecutive tiles,
    starting anywhere, can meet (brute force over the start offset)."""
    return max(((a + tiles - 1) // chunk - a // chunk + 1) if tiles else 0 for a in range(chunk))


def test_piece_bound_is_tight():
    # the workspace formula's P is the exact worst case of the chunk cut
    for tiles in range(0, 200):
        p = tiles if tiles <= 1 else (tiles - 2) // 16 + 2
        assert p == max_pieces(tiles, 16), tiles


def test_status_strings(pk):
    for s in range(5):
        assert pk.lib().kv_status_string(s)
    assert b"unknown" in pk.lib().kv_status_string(99)
