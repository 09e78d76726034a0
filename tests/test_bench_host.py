"""bench.py's host-side accounting, on CPU: the algorithmic bytes and flops
every reported rate divides by, the clock-sample parsing that decides
whether a run is kept, and the bounded oracle sample behind the CPU
baseline."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_write_bytes_per_token_counts_each_row_once():
    row = 8 * 128
    # BF16 write: K and V read (2 B) and written (2 B), and the int64 slot
    assert bench.write_bytes_per_token(row, 2) == 4 * 2 * row + 8 == 8200
    # FP8-K: K written as 1 B codes
    assert bench.write_bytes_per_token(row, 1) == 7176
    # FP8 K and V
    assert bench.write_bytes_per_token(row, 1, 1) == 6152


def test_decode_bytes_by_hand():
    # two sequences (100 and 7 positions), 2 KV heads of 64 dims, BF16 K and V,
    # 4 query heads: KV of every attended position once, Q in (bf16), the
    # float32 output and one int32 length per sequence
    kv = (100 + 7) * 2 * 64 * (2 + 2)
    q = 2 * 4 * 64 * 2
    out = 2 * 4 * 64 * 4
    assert bench.decode_bytes([100, 7], 0, 2, 64, 2, 2, 4, 16) == kv + q + out + 2 * 4
    # a window of 10 attends min(L, 10) positions; FP8 K is 1 B
    kv_w = (10 + 7) * 2 * 64 * (1 + 2)
    assert bench.decode_bytes([100, 7], 10, 2, 64, 1, 2, 4, 16) == kv_w + q + out + 2 * 4
    # FP8 K and V
    assert bench.decode_bytes([100, 7], 0, 2, 64, 1, 2, 4, 16, v_bytes=1) == (107 * 2 * 64 * 2) + q + out + 8


def test_prefill_flops_counts_causal_pairs():
    # L = 5 cached positions, the last 3 as queries: positions 2, 3, 4 attend
    # 3, 4 and 5 keys -> 12 pairs; 4 * Hq * D flops per pair
    assert bench.prefill_flops([5], [3], 0, 8, 128) == 4 * 8 * 128 * 12
    # a window of 2 caps each query at 2 keys
    assert bench.prefill_flops([5], [3], 2, 8, 128) == 4 * 8 * 128 * 6
    # more queries than positions: the first ones sit before position 0
    assert bench.prefill_flops([2], [4], 0, 1, 64) == 4 * 64 * (1 + 2)
    # several sequences add up
    assert bench.prefill_flops([5, 2], [3, 4], 0, 1, 64) == 4 * 64 * (12 + 3)


def test_clock_samples_parse_median_and_reasons(tmp_path):
    c = bench.Clocks(0)
    c.path = str(tmp_path / "clocks.csv")
    lines = [
        "0, 2070 MHz, 2070 MHz, 900.00 W, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2055 MHz, 2070 MHz, 1100.00 W, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070 MHz, 2070 MHz, 1000.00 W, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    with open(c.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    c.proc = object()  # a sampler ran
    s = c.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_without_a_sampler_says_so():
    c = bench.Clocks(0)
    c.proc = None
    assert c.summary()["reasons"] == ["unavailable"]


def test_oracle_sample_is_bounded_by_its_budget():
    nbytes, secs, what = bench.oracle_sample(0.5)
    assert nbytes > 0 and secs > 0
    # the budget bounds the decodes; one decode of the longest sample length
    # can overshoot it, not more
    assert secs < 0.5 + 5.0
    assert "decodes" in what


def _run_bench(args, env_extra=None):
    import json
    import subprocess
    env = dict(os.environ, **(env_extra or {}))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return [json.loads(ln) for ln in lines]


def test_reference_arm_prints_the_contract_line():
    (line,) = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0", "--cpu-budget", "2"])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["warmup"] == 0
    assert line["config"] == bench.bench_config(1)          # the GPU arm's workload, sampled
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] == line["value"] and cpu["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    assert _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0"],
                      {"RANK": "1", "WORLD_SIZE": "2"}) == []
