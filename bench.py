"""Benchmark of the sparse latent attention path on one GB300.

Default (our arm): the decode workload (B=64 queries, 640-entry index lists,
8192-token context at ratio 2 -> 4224 latent rows per batch row), timed as one
`sa_sparse_attn` call per step over rotating input sets whose total size
exceeds L2, replayed from a CUDA graph.  Prints ONE compact JSON line (floats
to four significant digits, the per-workload entries last).  Besides the
contract's keys it carries, under "workloads", the other lines: long-context
decode, prefill, the fused tail (attention, inverse RoPE, grouped wo_a), the
block tail (plus wo_b), the top-k selection (8192 rows x 4096 scores -> 512),
decode with fp4 compressed rows, the fused tail with an fp8 wo_a and the fp4
quantization of the decode workload's compressed cache.  Each entry: "ms" per
call, "qps" (queries/s; "rows_per_s" for top-k and the quantization), the roofline
("bound" hbm or tensor; "ach" achieved, GB/s or TFLOP/s; "peak"; "frac";
"traffic", measured DRAM bytes per launch of the dominant kernel, or null;
"peak_kind" burst or sustained for tensor-bound lines) and "cpu", the fp64
oracle's queries/s (rows/s) on the host cores on the same inputs (whole calls
for decode, else a block of queries scaled by flops).  A tensor-bound line is
divided by the burst bf16 peak when its timed region is under a second, by
the sustained one otherwise.  --extra NAME times one additional line alone.

--impl reference: the fp64 CPU oracle, timed as it stands on the host cores
on a bounded sample of the same workload (the only reference this path has).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_latent_attention_02_gb300 import inputs as I  # noqa: E402

METRIC = "sparse_attn queries/s; decode gathered-KV GB/s & prefill TFLOP/s vs GB300 roofline"
HEADLINE = "decode"

# DRAM bytes (read + write) per call -- every kernel the call launches -- from one
# ncu capture of the workload (the commands are in profiles/), keyed by the SHA-256
# of the kernel sources the call runs: a changed kernel reports null until it is
# captured again.  The long-decode figure was captured with 8192 compressed rows per
# batch row instead of 65536 (the same 640-entry lists, each query gathering from
# its own batch row, so the same rows move per call).
CSRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "sparse_latent_attention_02_gb300", "csrc")
KERNEL_SRC = os.path.join(CSRC, "sa_attn.cu")
GEMM_SRC = os.path.join(CSRC, "sa_gemm.cu")
TOPK_SRC = os.path.join(CSRC, "sa_topk.cu")
QUANT_SRC = os.path.join(CSRC, "sa_quant.cu")
TRAFFIC_SOURCES = {
    "decode": ("attn",), "long_decode": ("attn",), "prefill": ("attn",),
    "fused_tail": ("attn", "gemm"), "block_tail": ("attn", "gemm"), "topk": ("topk",),
    "decode_fp4": ("attn",), "fused_tail_fp8": ("attn", "gemm"), "fp4_quant": ("quant",),
}
MEASURED_TRAFFIC = {
    "decode": ("c0695bcb20121647378ec988ff00bb0b07cf9cfc3132e85185b188a1f781abfc", 46_600_903),
    "long_decode": ("c0695bcb20121647378ec988ff00bb0b07cf9cfc3132e85185b188a1f781abfc", 87_575_723),
    "prefill": ("c0695bcb20121647378ec988ff00bb0b07cf9cfc3132e85185b188a1f781abfc", 1_055_305_024),
    "fused_tail": ("3b0734421b6a018e03d32c19911824853d9a61784666510c0d992da5241889ec", 1_789_614_368),
    "block_tail": ("3b0734421b6a018e03d32c19911824853d9a61784666510c0d992da5241889ec", 2_776_463_264),
    "topk": ("2880efe58a9e4df996f9bd0d61bcf6571513ce84b62392e3fb99bc4054c3dce8", 139_115_691),
    "decode_fp4": ("c0695bcb20121647378ec988ff00bb0b07cf9cfc3132e85185b188a1f781abfc", 25_186_662),
    "fused_tail_fp8": ("3b0734421b6a018e03d32c19911824853d9a61784666510c0d992da5241889ec", 1_831_613_824),
    "fp4_quant": ("9f2f2da73bfacbbf925cdb6048855baab90b28aabf06e44c25fa463666b8b2a5", 323_808_544),
}


def measured_traffic(workload):
    import hashlib
    entry = MEASURED_TRAFFIC.get(workload)
    if entry is None:
        return None
    paths = {"attn": KERNEL_SRC, "gemm": GEMM_SRC, "topk": TOPK_SRC, "quant": QUANT_SRC}
    digest = hashlib.sha256()
    for key in TRAFFIC_SOURCES[workload]:
        with open(paths[key], "rb") as f:
            digest.update(f.read())
    return entry[1] if digest.hexdigest() == entry[0] else None


# ------------------------------------------------------------------ algorithmic work

def algorithmic(wl: I.Workload, idx: torch.Tensor) -> dict:
    """Bytes and flops the method must move / do for one call on these lists.

    bytes: every valid gathered row (D bf16), q, the output, the index lists
    and the sink; flops: 4 * H * D per valid (query, row) pair (QK^T and PV).
    """
    pairs = int((idx >= 0).sum().item())
    out_bytes = 4 if wl.out_f32 else 2
    nbytes = (pairs * wl.D * 2 + wl.n_queries * wl.H * wl.D * (2 + out_bytes)
              + idx.numel() * 4 + wl.H * 4)
    flops = 4 * wl.H * wl.D * pairs
    if wl.tail:
        din = wl.H * wl.D // wl.G
        flops += 2 * wl.n_queries * wl.G * wl.R * din
        nbytes += wl.G * wl.R * din * 2 + wl.n_queries * wl.G * wl.R * 2 - wl.n_queries * wl.H * wl.D * 2
    if wl.wo_b:
        flops += 2 * wl.n_queries * wl.G * wl.R * wl.dim
        nbytes += wl.dim * wl.G * wl.R * 2 + wl.n_queries * (wl.dim - wl.G * wl.R) * 2
    return {"pairs": pairs, "bytes": nbytes, "flops": flops}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (every 20 ms) of SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = None
        if not inside:
            # the timed region was shorter than the sampling interval: use the
            # samples nearest to it
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            inside = [p for (_, p) in near]
            note = "timed region shorter than the sampling interval; nearest samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[4 + i].lower().startswith("active")})
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
               "samples": len(inside)}
        if note:
            out["note"] = note
        return out


# ------------------------------------------------------------------ helpers

def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def tensor_peak(pk: dict, timed_s: float):
    """The bf16 peak a tensor-bound line is divided by: the burst figure for a
    timed region under a second (a kernel timed alone), the sustained one for a
    longer region (a kernel running under the power cap)."""
    if timed_s < 1.0:
        return pk["bf16_tflops"], f"{pk['source']} burst bf16"
    return pk["bf16_tflops_sustained"], f"{pk['source']} sustained bf16"


def sig(x, digits=4):
    """Round every float in a JSON-able structure to `digits` significant digits."""
    if isinstance(x, float):
        return float(f"{x:.{digits}g}")
    if isinstance(x, dict):
        return {k: sig(v, digits) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [sig(v, digits) for v in x]
    return x


def l2_bytes() -> int:
    try:
        return int(torch.cuda.get_device_properties(0).L2_cache_size)
    except Exception:
        return 129 * 2 ** 20


def make_sets(wl: I.Workload, n_sets: int, seed: int, dev) -> list:
    return [I.make_inputs(wl, seed=seed + 17 * i, device=dev) for i in range(n_sets)]


def sets_for(wl: I.Workload, dev, seed=0, min_sets=2, n_sets=None) -> list:
    """Enough independent input sets that one rotation touches > 2x L2."""
    probe = I.make_inputs(wl, seed=seed, device=dev)
    a = algorithmic(wl, probe["idx"])
    n = max(min_sets, int(np.ceil(2.5 * l2_bytes() / max(a["bytes"], 1))))
    n = min(n, 8) if n_sets is None else n_sets
    return [probe] + make_sets(wl, n - 1, seed + 1, dev)


# ------------------------------------------------------------------ ranks

def dist_env():
    """(rank, world, local_rank) from the torchrun environment (1 process if unset)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate_over_ranks(local_seconds: float, local_units: float):
    """Whole-job throughput of independent replicas: the slowest rank's time
    (max over ranks) and the units all ranks processed (sum)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local_seconds, local_units
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def time_graph_steps(step_fns, steps: int, warmup: int):
    """Capture `steps` calls (rotating over step_fns) into one CUDA graph, warm
    up with a `warmup`-step graph, then time one replay with CUDA events on
    the capturing stream, between barriers across ranks.  Returns seconds for
    the `steps` calls."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for f in step_fns:          # one eager pass (library attributes, allocations)
            f()
    torch.cuda.synchronize()
    gw = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gw, stream=s):
        for i in range(warmup):
            step_fns[i % len(step_fns)]()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(steps):
            step_fns[i % len(step_fns)]()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        gw.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier()
        t0 = time.time()
        e0.record(s)
        g.replay()
        e1.record(s)
        e1.synchronize()
        torch.cuda.synchronize()
        barrier()
        t1 = time.time()
    return e0.elapsed_time(e1) / 1e3, (t0, t1)


# ------------------------------------------------------------------ our arm

def launches_per_call(wl: I.Workload, num_sms: int) -> int:
    """Kernels one call enqueues: the attention kernel (the list pieces of a
    query merge inside their cluster, with no second kernel), plus the grouped
    GEMM of the tail, plus the wo_b GEMM of the block tail."""
    del num_sms
    return 1 + (1 if wl.tail else 0) + (1 if wl.wo_b else 0)


def bench_workload(name: str, steps: int, warmup: int, dev, with_e2e: bool, n_sets=None, cpu_s: float = 0.0,
                   wl: I.Workload = None):
    import sparse_latent_attention_02_gb300 as sa
    wl = I.WORKLOADS[name] if wl is None else wl
    sets = sets_for(wl, dev, n_sets=n_sets)
    outs = []
    fns = []
    if wl.wo_b:
        rope = sa.rope_table(wl.theta, 0, wl.T, wl.rope_dim).to(dev)
        for x in sets:
            z = torch.empty((wl.B, wl.T, wl.dim), dtype=torch.bfloat16, device=dev)
            ws = torch.zeros(sa.block_tail_workspace_size(wl.B, wl.T, wl.K, wl.G, wl.R),
                             dtype=torch.uint8, device=dev)
            outs.append((z, ws))
            fns.append(lambda x=x, z=z, ws=ws: sa.sparse_attn_block_tail(
                x["q"], x["kv"], x["sink"], x["idx"], wl.scale, rope, x["wo_a"], x["wo_b"], out=z,
                workspace=ws))
    elif wl.tail:
        rope = sa.rope_table(wl.theta, 0, wl.T, wl.rope_dim).to(dev)
        for x in sets:
            y = torch.empty((wl.B, wl.T, wl.G * wl.R), dtype=torch.bfloat16, device=dev)
            ws = torch.zeros(sa.fused_workspace_size(wl.B, wl.T, wl.K, wl.G, wl.R),
                             dtype=torch.uint8, device=dev)
            outs.append((y, ws))
            fns.append(lambda x=x, y=y, ws=ws: sa.sparse_attn_rope_wo_a(
                x["q"], x["kv"], x["sink"], x["idx"], wl.scale, rope, x["wo_a"], out=y,
                workspace=ws))
    else:
        odt = torch.float32 if wl.out_f32 else torch.bfloat16
        for x in sets:
            o = torch.empty((wl.B, wl.T, wl.H, wl.D), dtype=odt, device=dev)
            ws = torch.zeros(sa.workspace_size(wl.B, wl.T, wl.K), dtype=torch.uint8, device=dev)
            outs.append((o, ws))
            fns.append(lambda x=x, o=o, ws=ws: sa.sparse_attn(
                x["q"], x["kv"], x["sink"], x["idx"], wl.scale, out=o, workspace=ws))
    secs, (t0, t1) = time_graph_steps(fns, steps, warmup)
    for _, ws in outs:
        sa.check_errors(ws)
    work = [algorithmic(wl, x["idx"]) for x in sets]
    per_step_bytes = np.mean([w["bytes"] for w in work])
    per_step_flops = np.mean([w["flops"] for w in work])
    step_s = secs / steps
    res = {
        "workload": name, "B": wl.B, "T": wl.T, "K": wl.K, "N": wl.N,
        "input_sets": len(sets), "steps": steps, "ms_per_step": step_s * 1e3,
        "queries_per_s": wl.n_queries / step_s,
        "gbs": per_step_bytes / step_s / 1e9, "tflops": per_step_flops / step_s / 1e12,
        "bytes_per_step": int(per_step_bytes), "flops_per_step": int(per_step_flops),
        "valid_pairs_per_step": int(np.mean([w["pairs"] for w in work])),
        "window": (t0, t1),
        "gpu_launches": steps * launches_per_call(
            wl, torch.cuda.get_device_properties(dev).multi_processor_count),
    }
    if with_e2e:
        res["e2e"] = bench_e2e(wl, sets[0], steps, warmup, dev)
    if cpu_s > 0:
        res["cpu"] = cpu_rate(name, sets[0], cpu_s)
    del sets, outs, fns
    torch.cuda.empty_cache()
    return res


def bench_e2e(wl: I.Workload, x: dict, steps: int, warmup: int, dev) -> dict:
    """Same call end to end, every input starting in pinned host memory: each
    step copies q, sink and the index lists to the device, runs the C-ABI call
    with kv left in pinned host memory (the kernel gathers the rows the lists
    name straight from there over the CPU-GPU link) and copies the output
    back.  Steps are pipelined as a caller would run them: copies in on one
    stream, calls on another, results out on a third, with two sets of device
    buffers, so that step i+1's copies and step i-1's read-back overlap step
    i's call.  h2d bytes = the copies + the gathered kv rows."""
    import sparse_latent_attention_02_gb300 as sa
    keys = ["q", "sink", "idx"]
    host = {k: x[k].cpu().pin_memory() for k in keys + ["kv"]}
    devb = [{k: torch.empty_like(x[k], device=dev) for k in keys} for _ in range(2)]
    outs = [torch.empty((wl.B, wl.T, wl.H, wl.D), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    outs_h = [torch.empty(outs[0].shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    ws = torch.zeros(sa.workspace_size(wl.B, wl.T, wl.K), dtype=torch.uint8, device=dev)
    idx = x["idx"].cpu()
    kv_rows = int(((idx >= 0) & (idx < wl.N)).sum())
    copied = sum(host[k].numel() * host[k].element_size() for k in keys)
    h2d = copied + kv_rows * wl.D * 2
    d2h = outs[0].numel() * outs[0].element_size()
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    ev_in = [ev(), ev()]      # set b's inputs are on the device
    ev_ran = [ev(), ev()]     # the call on set b is done (inputs free, output ready)
    ev_out = [ev(), ev()]     # set b's output has been read back (output free)
    used = [False, False]

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_ran[b])
            for k in keys:
                devb[b][k].copy_(host[k], non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_in[b])
            if used[b]:
                s_run.wait_event(ev_out[b])
            sa.sparse_attn(devb[b]["q"], host["kv"], devb[b]["sink"], devb[b]["idx"], wl.scale,
                           out=outs[b], workspace=ws, stream=s_run)
            ev_ran[b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_ran[b])
            outs_h[b].copy_(outs[b], non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(max(warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        step(i)
    # the last read-back completes after every copy and call of the timed steps
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_run)
    e1.record(s_out)
    e1.synchronize()
    sa.check_errors(ws)
    secs = e0.elapsed_time(e1) / 1e3
    return {"value": wl.n_queries * steps / secs, "unit": "queries/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "note": f"per step: {copied} bytes copied (q, sink, idx) + {kv_rows * wl.D * 2} bytes of kv "
                    f"rows gathered by the kernel from pinned host memory ({kv_rows} rows); "
                    f"output copied back; copies, calls and read-backs pipelined on three streams"}


def bench_topk(steps: int, warmup: int, dev, pk: dict, cpu_s: float = 0.0) -> dict:
    """Top-k selection of 512 of 4096 compressed positions for the 8192 queries
    of the prefill workload (scores N(0,1), each query's visible prefix
    causal): one call per step, inputs rotating over sets larger than L2."""
    import sparse_latent_attention_02_gb300 as sa
    rows, L, k = 8192, 4096, 512
    n_sets = 3
    sets = []
    vis = (torch.arange(rows, device=dev) // 2 + 1).clamp(max=L)
    cols = torch.arange(L, device=dev)
    for i in range(n_sets):
        g = torch.Generator(device=dev).manual_seed(100 + i)
        sc = torch.randn((rows, L), generator=g, device=dev)
        sc[cols[None, :] >= vis[:, None]] = float("-inf")
        sets.append((sc, torch.empty((rows, k), dtype=torch.int32, device=dev)))
    fns = [lambda sc=sc, o=o: sa.topk_indices(sc, k, offset=128, out=o) for sc, o in sets]
    secs, _ = time_graph_steps(fns, steps, warmup)
    step_s = secs / steps
    nbytes = rows * L * 4 + rows * k * 4
    gbs = nbytes / step_s / 1e9
    res = {"ms_per_step": step_s * 1e3, "rows_per_s": rows / step_s, "bytes_per_step": nbytes,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / pk["hbm_gbs"], "traffic": measured_traffic("topk")}}
    if cpu_s > 0:
        import oracle
        n = 256
        sc = sets[0][0][:n].cpu().numpy()
        t0 = time.time()
        oracle.topk_indices(sc, k, offset=128)
        dt = time.time() - t0
        res["cpu"] = {"value": n / dt, "unit": "rows/s", "cores": 1, "kind": "oracle",
                      "sample": f"{n} rows, {dt:.1f} s"}
    return res


def bench_decode_fp4(steps: int, warmup: int, dev, pk: dict, cpu_s: float = 0.0) -> dict:
    """The decode workload with its compressed cache stored as fp4 (e2m1 codes
    and an E4M3 scale per 16 features, 288 bytes per row) next to the bf16
    window: the same lists, the two-source fp4 call, rotating input sets larger
    than L2."""
    import sparse_latent_attention_02_gb300 as sa
    wl = I.WORKLOADS["decode"]
    D = wl.D
    n_sets = 4
    sets = []
    for i in range(n_sets):
        x = I.make_inputs(wl, seed=200 + i, device=dev)
        g = torch.Generator(device=dev).manual_seed(300 + i)
        codes = torch.randint(0, 256, (wl.B, wl.C, D // 2), generator=g, device=dev,
                              dtype=torch.int32).to(torch.uint8)
        scales = (0x20 + torch.randint(0, 8, (wl.B, wl.C, D // 16), generator=g, device=dev,
                                       dtype=torch.int32)).to(torch.uint8)
        win = x["kv"][:, :wl.W].contiguous()
        out = torch.empty((wl.B, wl.T, wl.H, D), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(sa.workspace_size(wl.B, wl.T, wl.K), dtype=torch.uint8, device=dev)
        sets.append((x, win, codes, scales, out, ws))
        del x["kv"]
    fns = [lambda x=x, win=win, c=c, sc=sc, o=o, ws=ws: sa.sparse_attn_two_source_fp4(
        x["q"], win, c, sc, x["sink"], x["idx"], wl.scale, out=o, workspace=ws)
        for x, win, c, sc, o, ws in sets]
    secs, _ = time_graph_steps(fns, steps, warmup)
    for *_, ws in sets:
        sa.check_errors(ws)
    step_s = secs / steps
    idx = sets[0][0]["idx"]
    win_rows = int(((idx >= 0) & (idx < wl.W)).sum())
    fp4_rows = int((idx >= wl.W).sum())
    nbytes = (win_rows * D * 2 + fp4_rows * (D // 2 + D // 16) + wl.n_queries * wl.H * D * 4
              + idx.numel() * 4 + wl.H * 4)
    gbs = nbytes / step_s / 1e9
    res = {"ms_per_step": step_s * 1e3, "queries_per_s": wl.n_queries / step_s, "bytes_per_step": nbytes,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / pk["hbm_gbs"], "traffic": measured_traffic("decode_fp4")}}
    if cpu_s > 0:
        import oracle
        x, win, c, sc = sets[0][:4]
        args = (x["q"].cpu(), win.cpu(), wl.W, c.cpu().numpy(), sc.cpu().numpy(), wl.C, x["sink"].cpu(),
                x["idx"].cpu(), wl.scale)
        oracle.sparse_attn_two_source_fp4(*args)
        done, t0 = 0, time.time()
        while True:
            oracle.sparse_attn_two_source_fp4(*args)
            done += 1
            if time.time() - t0 >= cpu_s or done >= 1000:
                break
        dt = time.time() - t0
        res["cpu"] = {"value": wl.n_queries * done / dt, "unit": "queries/s", "cores": oracle.threads(0),
                      "kind": "oracle", "sample": f"{done} whole calls"}
    return res


def bench_fused_tail_fp8(steps: int, warmup: int, dev, pk: dict, cpu_s: float = 0.0) -> dict:
    """The fused-tail workload (attention, inverse RoPE, grouped wo_a) with wo_a
    kept as an fp8 checkpoint (E4M3 + an fp32 scale per 128 x 128 block,
    decoded by the call into a bf16 workspace copy): same inputs and flops as
    the bf16 line."""
    import sparse_latent_attention_02_gb300 as sa
    wl = I.WORKLOADS["fused_tail"]
    sets = sets_for(wl, dev)
    rope = sa.rope_table(wl.theta, 0, wl.T, wl.rope_dim).to(dev)
    fns, wss = [], []
    for x in sets:
        x["w8"], x["w8_scales"] = I.fp8_weight(x.pop("wo_a"))
        y = torch.empty((wl.B, wl.T, wl.G * wl.R), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(sa.fused_fp8_workspace_size(wl.B, wl.T, wl.K, wl.G, wl.R), dtype=torch.uint8,
                         device=dev)
        wss.append(ws)
        fns.append(lambda x=x, y=y, ws=ws: sa.sparse_attn_rope_wo_a_fp8(
            x["q"], x["kv"], x["sink"], x["idx"], wl.scale, rope, x["w8"], x["w8_scales"], out=y, workspace=ws))
    secs, _ = time_graph_steps(fns, steps, warmup)
    for ws in wss:
        sa.check_errors(ws)
    step_s = secs / steps
    flops = float(np.mean([algorithmic(wl, x["idx"])["flops"] for x in sets]))
    tflops = flops / step_s / 1e12
    peak, note = tensor_peak(pk, secs)
    res = {"ms_per_step": step_s * 1e3, "queries_per_s": wl.n_queries / step_s, "flops_per_step": int(flops),
           "gpu_launches": 3 * steps,
           "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                        "frac": tflops / peak, "traffic": measured_traffic("fused_tail_fp8"), "peak_note": note}}
    if cpu_s > 0:
        import oracle
        x = dict(sets[0])
        t0 = time.time()
        w8 = x["w8"].cpu().numpy()
        x["wo_a"] = torch.from_numpy(oracle.dequant_fp8_weight(w8.reshape(-1, w8.shape[-1]),
                                                                x["w8_scales"].cpu().numpy()).view(np.int16)
                                     ).view(torch.bfloat16).reshape(w8.shape)
        deq = time.time() - t0
        r = cpu_rate("fused_tail", x, cpu_s)
        call_s = wl.n_queries / r["value"] + deq
        res["cpu"] = {"value": wl.n_queries / call_s, "unit": "queries/s", "cores": r["cores"], "kind": "oracle",
                      "sample": r["sample"] + f", + weight decoding {deq:.1f} s"}
    del sets, fns
    torch.cuda.empty_cache()
    return res


# the additional lines that are not attention workloads, by name
def bench_fp4_quant(steps: int, warmup: int, dev, pk: dict, cpu_s: float = 0.0) -> dict:
    """fp4 quantization of the decode workload's compressed cache (64 batch
    rows x 4096 latent rows x 512 features, RMS-normalised N(0,1)) into codes
    and E4M3 group scales: one call per step, two input sets rotating (each
    larger than L2)."""
    import sparse_latent_attention_02_gb300 as sa
    wl = I.WORKLOADS["decode"]
    rows, D = wl.B * wl.C, wl.D
    sets = []
    for i in range(2):
        g = torch.Generator(device=dev).manual_seed(400 + i)
        lat = torch.empty((rows, D), dtype=torch.bfloat16, device=dev)
        for r0 in range(0, rows, 65536):
            r1 = min(rows, r0 + 65536)
            lat[r0:r1] = I.rms_rows(torch.randn((r1 - r0, D), generator=g, device=dev)).to(torch.bfloat16)
        sets.append((lat, torch.empty((rows, D // 2), dtype=torch.uint8, device=dev),
                     torch.empty((rows, D // 16), dtype=torch.uint8, device=dev)))
    fns = [lambda lat=lat, c=c, s=s: sa.fp4_quantize(lat, c, s) for lat, c, s in sets]
    secs, _ = time_graph_steps(fns, steps, warmup)
    step_s = secs / steps
    nbytes = rows * (2 * D + D // 2 + D // 16)
    gbs = nbytes / step_s / 1e9
    res = {"ms_per_step": step_s * 1e3, "rows_per_s": rows / step_s, "bytes_per_step": nbytes,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / pk["hbm_gbs"], "traffic": measured_traffic("fp4_quant")}}
    if cpu_s > 0:
        import oracle
        n = 16384
        bits = sets[0][0][:n].cpu().view(torch.int16).numpy().view(np.uint16)
        t0 = time.time()
        oracle.fp4_quantize(bits)
        dt = time.time() - t0
        res["cpu"] = {"value": n / dt, "unit": "rows/s", "cores": 1, "kind": "oracle",
                      "sample": f"{n} rows, {dt:.1f} s"}
    del sets, fns
    torch.cuda.empty_cache()
    return res


EXTRA_LINES = {
    "topk": bench_topk,
    "decode_fp4": bench_decode_fp4,
    "fused_tail_fp8": bench_fused_tail_fp8,
    "fp4_quant": bench_fp4_quant,
}


def _oracle_chain(wl: I.Workload, q, kv, sink, idx, wo_a=None, wo_b=None):
    """The oracle's steps for a block of queries (q [1, n, H, D] etc. on the
    host): attention, and for the tails inverse RoPE, wo_a and wo_b."""
    import oracle
    o, _ = oracle.sparse_attn(q, kv, sink, idx, wl.scale)
    if wl.tail:
        n = q.shape[1]
        pos = np.arange(n)   # positions only shift the angles; the work is the same
        o = oracle.inverse_rope(o.reshape(n, wl.H, wl.D), pos, wl.rope_dim, wl.theta)
        y = oracle.wo_a(o.reshape(n, wl.G, -1), wo_a)
        if wl.wo_b:
            oracle.wo_b(y.reshape(n, -1), wo_b)


def cpu_rate(name: str, x: dict, budget_s: float) -> dict:
    """The fp64 oracle, as it stands, on the host cores on one input set of a
    workload (x: its tensors, on any device): whole calls repeated for about
    `budget_s` when a call is short (the decode workloads), else one contiguous
    block of queries of the first batch element (attention and, for the tails,
    the projections), scaled to the whole call by algorithmic flops.  Returns
    queries/s, the threads used and what was timed."""
    import oracle
    wl = I.WORKLOADS[name]
    cores = oracle.threads(0)
    cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in x.items()
           if k in ("q", "kv", "sink", "idx", "wo_a", "wo_b")}
    if wl.T == 1:   # decode: whole calls
        oracle.sparse_attn(cpu["q"], cpu["kv"], cpu["sink"], cpu["idx"], wl.scale)
        done, t0 = 0, time.time()
        while True:
            oracle.sparse_attn(cpu["q"], cpu["kv"], cpu["sink"], cpu["idx"], wl.scale)
            done += 1
            if time.time() - t0 >= budget_s or done >= 1000:
                break
        secs = time.time() - t0
        return {"value": wl.n_queries * done / secs, "unit": "queries/s", "cores": cores, "kind": "oracle",
                "sample": f"{done} whole calls"}
    n = 512 if not wl.tail else (256 if not wl.wo_b else 128)
    t_a = wl.T // 2
    blk = dict(q=cpu["q"][:1, t_a:t_a + n], kv=cpu["kv"][:1], sink=cpu["sink"], idx=cpu["idx"][:1, t_a:t_a + n])
    t0 = time.time()
    _oracle_chain(wl, blk["q"], blk["kv"], blk["sink"], blk["idx"], cpu.get("wo_a"), cpu.get("wo_b"))
    secs = time.time() - t0
    full = algorithmic(wl, cpu["idx"])["flops"]
    part = algorithmic(I.scaled(wl, B=1, T=n), blk["idx"])["flops"]
    call_s = secs * full / part
    return {"value": wl.n_queries / call_s, "unit": "queries/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} queries (t {t_a}..{t_a + n - 1}), {secs:.1f} s, scaled by flops"}


def cpu_baseline(name: str, budget_s: float = 12.0) -> dict:
    """The headline's oracle baseline on a fresh host input set."""
    x = I.make_inputs(I.WORKLOADS[name], seed=0)
    return cpu_rate(name, x, budget_s)


def _entry(r: dict) -> dict:
    """A workload's compact entry in the printed line: milliseconds per call,
    throughput, the roofline (achieved in GB/s for "hbm", TFLOP/s for
    "tensor"; peak; fraction; measured DRAM bytes per launch of the dominant
    kernel or null) and the oracle's rate on the host cores."""
    rf = r["roofline"]
    e = {"ms": r["ms_per_step"]}
    if "queries_per_s" in r:
        e["qps"] = r["queries_per_s"]
    if "rows_per_s" in r:
        e["rows_per_s"] = r["rows_per_s"]
    e.update({"bound": rf["bound"], "ach": rf["achieved"], "peak": rf["peak"], "frac": rf["frac"],
              "traffic": rf.get("traffic")})
    if rf.get("peak_note", "").find("burst") >= 0:
        e["peak_kind"] = "burst"
    elif rf["bound"] == "tensor":
        e["peak_kind"] = "sustained"
    if r.get("cpu"):
        e["cpu"] = r["cpu"]["value"]
    return e


def run_ours(args):
    import sparse_latent_attention_02_gb300 as sa
    rank, world, local = dist_env()
    if rank == 0:
        sa.build()
    barrier()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk = peaks()
    cpu_s = args.cpu_seconds if world == 1 else 0.0
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    head_wl = I.WORKLOADS[args.workload]
    if args.kv_rows is not None:   # profiling aid: a smaller compressed cache, the same lists' shape
        head_wl = I.scaled(head_wl, C=args.kv_rows)
    head = bench_workload(args.workload, args.steps, args.warmup, dev,
                          with_e2e=not args.no_e2e and world == 1, n_sets=args.sets, cpu_s=cpu_s, wl=head_wl)
    secs, units = aggregate_over_ranks(head["ms_per_step"] * 1e-3 * args.steps,
                                       head["queries_per_s"] * head["ms_per_step"] * 1e-3 * args.steps)
    head["job_queries_per_s"] = units / secs
    head["job_ms_per_step"] = secs / args.steps * 1e3
    clocks = sampler.summary(*head.pop("window"))
    if rank != 0:
        sampler.stop()
        barrier()
        return
    extra = {}
    if not args.headline_only and world == 1:
        per_line_cpu = min(cpu_s, 3.0)
        for name in ("long_decode", "prefill", "fused_tail", "block_tail"):
            steps = max(3, min(args.steps, 20))
            r = bench_workload(name, steps, max(args.warmup, 3), dev, with_e2e=False, cpu_s=per_line_cpu)
            sampler.summary(*r.pop("window"))
            if name in ("prefill", "fused_tail", "block_tail"):
                peak, note = tensor_peak(pk, r["ms_per_step"] * 1e-3 * steps)
                r["roofline"] = {"bound": "tensor", "achieved": r["tflops"], "peak": peak, "unit": "TFLOP/s",
                                 "frac": r["tflops"] / peak, "traffic": measured_traffic(name), "peak_note": note}
            else:
                r["roofline"] = {"bound": "hbm", "achieved": r["gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                                 "frac": r["gbs"] / pk["hbm_gbs"], "traffic": measured_traffic(name)}
            extra[name] = _entry(r)
        extra["topk"] = _entry(bench_topk(max(3, min(args.steps, 50)), max(args.warmup, 3), dev, pk, per_line_cpu))
        extra["decode_fp4"] = _entry(bench_decode_fp4(max(3, min(args.steps, 200)), max(args.warmup, 3), dev, pk,
                                                      per_line_cpu))
        extra["fused_tail_fp8"] = _entry(bench_fused_tail_fp8(max(3, min(args.steps, 20)), max(args.warmup, 3), dev,
                                                              pk, per_line_cpu))
        extra["fp4_quant"] = _entry(bench_fp4_quant(max(3, min(args.steps, 50)), max(args.warmup, 3), dev, pk,
                                                    per_line_cpu))
    sampler.stop()
    e2e = head.pop("e2e", None)
    if e2e:
        e2e.pop("note", None)
    cpu = head.pop("cpu", None)
    line = {
        "metric": METRIC, "value": head["job_queries_per_s"], "unit": "queries/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["job_ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: B={head['B']} T={head['T']} H=64 D=512 "
                               f"N={head['N']} K={head['K']}",
                   "parallelism": f"replicas only ({world} GPU{'s' if world > 1 else ''}, no collective)",
                   "l2": f"{head['input_sets']} rotating input sets, > 2x L2"},
        "gbs": head["gbs"], "tflops": head["tflops"],
        "roofline": {"bound": "hbm", "achieved": head["gbs"], "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": head["gbs"] / pk["hbm_gbs"],
                     "traffic": measured_traffic(args.workload),
                     "bytes_per_call": head["bytes_per_step"]},
        "e2e": e2e,
        "gpu_launches": head["gpu_launches"] * world,
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons") if k in clocks},
        "cpu_baseline": cpu,
        "workloads": extra,
    }
    print(json.dumps(sig(line), separators=(",", ":")))
    barrier()


def run_reference(args):
    import oracle
    wl = I.WORKLOADS[HEADLINE]
    x = I.make_inputs(wl, seed=0)
    cores = oracle.threads(0)
    # each step: a bounded sample (a quarter of the decode batch) of the workload
    sample = np.arange(0, wl.n_queries, 4, dtype=np.int64)
    for _ in range(args.warmup):
        oracle.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, queries=sample)
    t0 = time.time()
    for _ in range(args.steps):
        oracle.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, queries=sample)
    secs = time.time() - t0
    v = sample.size * args.steps / secs
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "queries/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{HEADLINE}: B={wl.B} T={wl.T} H=64 D=512 N={wl.N} K={wl.K}"},
        "cpu_baseline": {"value": v, "unit": "queries/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample.size} of {wl.n_queries} decode queries per step"},
        "e2e": {"value": v, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=6.0,
                    help="CPU-baseline budget; 0 skips it (profiling runs)")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(I.WORKLOADS),
                    help="workload of the headline line (default: decode)")
    ap.add_argument("--sets", type=int, default=None,
                    help="number of rotating input sets (default: enough for > 2x L2)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--kv-rows", type=int, default=None,
                    help="profiling aid: compressed rows per batch row of the headline workload "
                         "(the lists keep their length; only with --headline-only)")
    ap.add_argument("--extra", choices=sorted(EXTRA_LINES),
                    help="time only this additional line (one GPU) and print it as JSON")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.kv_rows is not None and (not args.headline_only or args.kv_rows < 1):
        ap.error("--kv-rows takes a positive count and --headline-only")
    if args.extra:
        import sparse_latent_attention_02_gb300 as sa
        sa.build()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(sig({"extra": args.extra,
                              **EXTRA_LINES[args.extra](args.steps, args.warmup, dev, peaks(),
                                                        min(args.cpu_seconds, 3.0))})))
        return
    rank, world, local = dist_env()
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; other ranks exit at once
        if rank == 0:
            run_reference(args)
        return
    if world > 1:
        # replicas only: one independent replica per GPU; the process group
        # carries the timing barrier and the max-over-ranks reduction only
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        run_ours(args)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
