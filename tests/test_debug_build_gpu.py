"""The bounds-checking build (libpagedkv_debug.so) on the GPU, each case in a
child process that loads that library alone (tests/debug_build_child.py).

- A decode wait that runs out: with the pipeline wait limit cut to 1 ns, an
  FP8-K decode gives up, the call returns, the fault word shows bit 0 (and
  kv_get_device_error returns KV_ERR_DEVICE); every copy the kernel issued
  was drained before its CTAs exited, so with the default limit back the
  next decode on the same context matches the oracle and reports nothing.
- Indices outside the pool: a block table with one block id past the pool
  and the slots it gives. Slot filling flags it; the BF16, FP8-K and fused K
  writes skip those rows (every other pool byte equals the oracle's write of
  the remaining rows); the decode reads block 0 in place of the bad id, and
  the sequences that do not use it match the oracle, and so does the BF16
  chunked prefill's. Each step sets bit 3.
Nothing here faults, traps or hangs a GPU: every wait is bounded, and no
access leaves the buffers.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KV_OK, KV_ERR_DEVICE = 0, 4
BIT_TIMEOUT, BIT_OUT_OF_POOL = 1, 8


@pytest.fixture(scope="module")
def debug_library():
    sys.path.insert(0, os.path.join(ROOT, "paged_kv_cache_fill_gb300"))
    import _build
    import __graft_entry__
    __graft_entry__.build()  # the oracle, which the child uses
    return _build.build(debug=True)


def run_child(case, library):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_build_child.py"), case, library],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_decode_wait_timeout_returns_flags_and_drains(debug_library):
    res = run_child("timeout", debug_library)
    assert res["before"] == [KV_OK, 0]
    status, bits = res["seen"][-1]
    assert bits & BIT_TIMEOUT, res["seen"]
    assert status == KV_ERR_DEVICE
    # the default limit again: a clean decode on the same context
    assert res["after"] == [KV_OK, 0]
    assert res["finite"]
    assert res["abs_err"] <= 2e-3 and res["rel_err"] <= 1e-2, res


def test_out_of_pool_indices_are_flagged_and_skipped(debug_library):
    res = run_child("bounds", debug_library)
    assert res["clean"] == [KV_OK, 0]
    for step in ("fill", "write_bf16", "write_fp8k", "write_fused", "decode", "prefill"):
        assert res[step] == [KV_ERR_DEVICE, BIT_OUT_OF_POOL], (step, res[step])
    assert res["write_good"] == [KV_OK, 0]
    assert res["fill_slots_equal"]
    assert res["write_bf16_equal"] and res["write_fp8k_equal"]
    assert res["write_fused_ulp"] <= 1
    assert res["decode_untouched_finite"]
    assert res["decode_untouched_abs_err"] <= 2e-3 and res["decode_untouched_rel_err"] <= 1e-2, res
    assert res["prefill_untouched_finite"]
    assert res["prefill_untouched_abs_err"] <= 2e-3 and res["prefill_untouched_rel_err"] <= 1e-2, res
