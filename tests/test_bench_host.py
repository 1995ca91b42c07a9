"""Host-side arithmetic of bench.py (CPU only): the algorithmic work behind
the roofline figures, the traffic table's source check and the clock summary."""
import os
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from sparse_latent_attention_02_gb300 import inputs as I  # noqa: E402


def test_decode_algorithmic_bytes():
    """64 queries x (640 rows x 1 KiB + q 64 KiB + bf16 out 64 KiB + 640 int32
    indices) + the 256-byte sink = 50,495,744 bytes; flops 4*64*512 per
    (query, row) pair."""
    wl = I.WORKLOADS["decode"]
    x = I.make_inputs(wl, seed=0)
    a = bench.algorithmic(wl, x["idx"])
    assert a["pairs"] == 64 * 640
    assert a["bytes"] == 64 * (640 * 1024 + 65536 + 65536 + 640 * 4) + 256 == 50_495_744
    assert a["flops"] == 4 * 64 * 512 * 64 * 640


def test_prefill_flops_count_valid_pairs_only():
    wl = I.WORKLOADS["prefill"]
    x = I.make_inputs(wl, seed=0)
    a = bench.algorithmic(wl, x["idx"])
    assert a["pairs"] == int((x["idx"] >= 0).sum()) == 4_972_096
    assert a["flops"] == 4 * 64 * 512 * 4_972_096


def test_skipped_entries_are_not_counted():
    wl = I.WORKLOADS["decode"]
    x = I.make_inputs(wl, seed=0)
    idx = x["idx"].clone()
    idx[:, :, ::2] = -1
    a, b = bench.algorithmic(wl, x["idx"]), bench.algorithmic(wl, idx)
    assert b["pairs"] == a["pairs"] // 2
    assert a["bytes"] - b["bytes"] == (a["pairs"] - b["pairs"]) * 1024


def test_traffic_table_is_keyed_to_the_kernel_source(tmp_path, monkeypatch):
    """A measured traffic figure is reported only for the kernel source it was
    captured on."""
    assert bench.measured_traffic("no such workload") is None
    for w in bench.MEASURED_TRAFFIC:
        assert w in bench.TRAFFIC_SOURCES
    if bench.measured_traffic("fused_tail") is not None and bench.measured_traffic("decode") is not None:
        # a changed GEMM drops the tails' figures, not the attention-only ones
        changed = tmp_path / "sa_gemm.cu"
        changed.write_text(open(bench.GEMM_SRC).read() + "\n// changed\n")
        monkeypatch.setattr(bench, "GEMM_SRC", str(changed))
        assert bench.measured_traffic("fused_tail") is None
        assert bench.measured_traffic("decode") is not None
    if bench.measured_traffic("decode") is not None:
        changed = tmp_path / "sa_attn.cu"
        changed.write_text(open(bench.KERNEL_SRC).read() + "\n// changed\n")
        monkeypatch.setattr(bench, "KERNEL_SRC", str(changed))
        assert bench.measured_traffic("decode") is None


def test_clock_summary_inside_window_and_reasons():
    s = bench.ClockSampler(0)
    t = time.time()
    row = lambda mhz, hw="Not Active": [str(mhz), "2070", "900.0", "0x0", hw, "Not Active", "Not Active",
                                        "Not Active"]
    s.samples = [(t - 1.0, row(1000)), (t + 0.01, row(2070)), (t + 0.03, row(2055)),
                 (t + 0.05, row(2070, "Active")), (t + 2.0, row(500))]
    out = s.summary(t, t + 0.06)
    assert out["samples"] == 3 and out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["hw_slowdown"]
    assert "note" not in out
    # a window with no sample inside falls back to the nearest ones, and says so
    near = s.summary(t + 0.5, t + 0.51)
    assert near["samples"] == 3 and "note" in near


def test_launch_counts_per_call():
    assert bench.launches_per_call(I.WORKLOADS["decode"], 148) == 1
    assert bench.launches_per_call(I.WORKLOADS["fused_tail"], 148) == 2
    assert bench.launches_per_call(I.WORKLOADS["block_tail"], 148) == 3


def _bench(env_extra, *args):
    import json
    import subprocess
    env = dict(os.environ, OMP_NUM_THREADS="4", **env_extra)
    p = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), *args], cwd=bench.ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(x) for x in p.stdout.splitlines() if x.startswith("{")]
    return lines


def test_reference_arm_prints_one_line_on_rank_zero_only():
    """The oracle arm: one JSON line from rank 0 with the contract's keys, on
    the headline workload; any other rank of a launch exits at once, silent."""
    ranks = dict(WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT="29599")
    args = ("--impl", "reference", "--steps", "1", "--warmup", "1")
    assert _bench(dict(ranks, RANK="1", LOCAL_RANK="1"), *args) == []
    (line,) = _bench(dict(ranks, RANK="0", LOCAL_RANK="0"), *args)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "queries/s" and line["value"] > 0
    assert line["steps"] == 1 and line["warmup"] == 3          # raised to the minimum of three
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"].startswith("decode: B=64 T=1")


def test_tensor_peak_is_burst_for_short_regions():
    pk = {"hbm_gbs": 6784.8, "bf16_tflops": 1890.6, "bf16_tflops_sustained": 1687.3, "source": "measured"}
    assert bench.tensor_peak(pk, 0.03)[0] == 1890.6 and "burst" in bench.tensor_peak(pk, 0.03)[1]
    assert bench.tensor_peak(pk, 4.0)[0] == 1687.3 and "sustained" in bench.tensor_peak(pk, 4.0)[1]


def test_printed_line_rounding_and_entries():
    assert bench.sig({"a": 1234.5678, "b": [0.000123456, 7], "c": "x"}) == {"a": 1235.0, "b": [0.0001235, 7], "c": "x"}
    r = {"ms_per_step": 1.2345678, "queries_per_s": 6.5e6, "cpu": {"value": 530.0},
         "roofline": {"bound": "tensor", "achieved": 500.0, "peak": 1890.6, "frac": 0.2645, "traffic": None,
                      "peak_note": "measured burst bf16"}}
    e = bench._entry(r)
    assert e == {"ms": 1.2345678, "qps": 6.5e6, "bound": "tensor", "ach": 500.0, "peak": 1890.6, "frac": 0.2645,
                 "traffic": None, "peak_kind": "burst", "cpu": 530.0}


def test_oracle_rate_scales_a_block_by_flops():
    """The per-workload oracle baseline: whole calls for decode, a block of
    queries scaled by algorithmic flops otherwise (a positive rate, its sample
    stated)."""
    wl = I.scaled(I.WORKLOADS["prefill"], T=1100)
    I.WORKLOADS["_tiny_prefill"] = wl
    try:
        x = I.make_inputs(wl, seed=0)
        r = bench.cpu_rate("_tiny_prefill", x, 1.0)
        assert r["value"] > 0 and r["kind"] == "oracle" and "scaled by flops" in r["sample"]
        assert r["sample"].startswith("512 queries (t 550..1061)")
    finally:
        del I.WORKLOADS["_tiny_prefill"]
