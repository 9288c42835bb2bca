#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300: chunked prefill tokens/s and decode state GB/s.

Default run (N=1): the headline is the prefill_1m workload -- one sequence of
T = 1,048,576 tokens, H=16, dk=dv=128, bf16 inputs, fp32 state carried over
the whole length and emitted -- through kda_chunk_fwd; one step is one full
chunked forward (gate, intra-chunk transform, state recurrence, output).  The
same line carries the other workloads measured the same way (prefill_8k: one
8192-token sequence with 32 heads; varlen_64: 64 packed sequences of 512-4096
tokens with initial states), the decode workload (256 sequences x 1 token,
H=32, 128 consecutive in-place steps on a 512 MiB fp32 state) through
kda_decode_step, the roofline of each workload's dominant kernel, the
end-to-end number with host buffers, the CPU oracle timed on the host cores,
and the SM clocks seen during the timed region.

With --impl reference the fp64 CPU oracle runs the headline workload (the
same seeded inputs, drawn by the same generator on the same device) on the
host cores, a bounded prefix of the tokens per step, and prints the same JSON
line.

Multi-GPU (torchrun, one rank per GPU): every rank runs its own replica of the
workload (the (sequence, head) units are independent; no collective is on the
data path), so `value` is weak-scaling aggregate throughput = N x per-replica
work / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s and decode state GB/s per GB300; % of roofline"
HEADLINE = "prefill_1m"
EXTRA_PREFILL = ("prefill_8k", "varlen_64")
DECODE = "decode_256"
L2_BYTES = 129 * 1024 * 1024
FLUSH_BYTES = 256 * 1024 * 1024


def profiled_traffic(md_name: str, units_per_launch: float | None = None):
    """DRAM bytes per launch from a committed ncu summary under profiles/, or None when the
    summary is absent or the kernel sources it names have changed since the capture.  A
    summary taken on a smaller case of the same kernel gives bytes per token-head
    (`traffic_bytes_per_token_head`), scaled here by the token-heads one launch processes."""
    import hashlib
    keys = ("traffic_bytes_per_launch", "traffic_bytes_per_token_head", "source_sha256_16",
            "sources")
    try:
        text = open(os.path.join(ROOT, "profiles", md_name)).read()
        fields = dict(line.strip().split(": ", 1) for line in text.splitlines()
                      if line.strip().split(": ", 1)[0] in keys)
        h = hashlib.sha256()
        for f in fields["sources"].split():
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        if h.hexdigest()[:16] != fields["source_sha256_16"]:
            return None
        if "traffic_bytes_per_launch" in fields:
            return int(fields["traffic_bytes_per_launch"])
        if units_per_launch is None:
            return None
        return int(float(fields["traffic_bytes_per_token_head"]) * units_per_launch)
    except (OSError, KeyError, ValueError):
        return None


# fallbacks only when the measured peaks file is absent
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK), "fallback"


def prefill_bytes(seqlens, H, dk, dv, elt, h0: bool, hT: bool) -> int:
    """Algorithmic HBM bytes of one chunked forward: q, k, z, v, beta read, o written once,
    states read/written once (intermediates are not algorithmic)."""
    T = sum(seqlens)
    per_tok = H * ((2 * dk + dk + dv) * elt + elt + dv * elt)
    st = len(seqlens) * H * dk * dv * 4
    return T * per_tok + (st if h0 else 0) + (st if hT else 0)


def prefill_flops(seqlens, H, dk, dv) -> int:
    """Fixed flop convention per token-head: 6 dk dv + 64 (3 dk + 2 dv)."""
    return sum(seqlens) * H * (6 * dk * dv + 64 * (3 * dk + 2 * dv))


def kernel_names(n_events: int, tc_path: bool) -> list[str]:
    """Names of the kernels one kda_chunk_fwd_profiled call launched, in order (each
    kernel is bracketed by a pair of events recorded on its own stream)."""
    k = n_events // 2
    if not tc_path:
        return ["chunk_fwd_simt_kernel"] * k
    names = ["plan_chunks_kernel"]
    while len(names) < k:
        names += ["prep_kernel", "chain_kernel"]
    return names[:k]


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=self.out,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows
                                    if r[3].replace(".", "").isdigit()), default=None)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units: float, elapsed_s: float, world: int) -> tuple[float, float]:
    """(whole-job throughput, max-over-ranks seconds) for weak scaling."""
    tmax = max_over_ranks(elapsed_s, world)
    return per_rank_units * world / tmax, tmax


# ----------------------------------------------------------------------------- GPU arm

def workload_config(name: str, world: int = 1) -> dict:
    """The `config` object of a prefill workload's line (identical in both arms)."""
    from gated_delta_rule_43_gb300 import inputs

    w = inputs.WORKLOADS[name]
    if w.seqlens and w.seqlens[0] == "uniform":
        _, cnt, lo, hi = w.seqlens
        shape = f"{cnt} packed sequences, lengths uniform in [{lo}, {hi}]"
    else:
        shape = f"B={len(w.seqlens)}, T={sum(w.seqlens)}"
    h0 = (f"initial state N(0, {w.h0_sigma ** 2:g}) fp32" if w.h0_sigma > 0
          else "zero initial state")
    return {"workload": f"{name}: {shape}, H={w.H}, dk={w.dk}, dv={w.dv}, {w.dtype} "
                        f"q/k/v/z/beta, {h0}, fp32 final state emitted",
            "heads": w.H, "dk": w.dk, "dv": w.dv, "seed": w.seed,
            "inputs": "seeded synthetic (gated_delta_rule_43_gb300/inputs.py), drawn on the GPU",
            "l2": "flushed between timed steps (256 MiB write outside the events); the "
                  "1M-token inputs (17 GB) are also far larger than L2",
            "parallelism": f"replicas x{world}"}


def prefill_leg(name, dev, stream, K, warmup, world, pk, pk_src, clock=False, keep=False):
    """One prefill workload through kda_chunk_fwd: K timed whole calls (L2 flushed between
    them), then K calls through kda_chunk_fwd_profiled for per-kernel times on the streams
    the kernels run on.  Returns (result dict, inputs or None)."""
    import torch

    from gated_delta_rule_43_gb300 import inputs, kda

    w = inputs.WORKLOADS[name]
    d = inputs.make_workload(w, device=dev)
    T = sum(d["seqlens"])
    N = len(d["seqlens"])
    H, dk, dv = w.H, w.dk, w.dv
    ws = kda.alloc_workspace(kda.chunk_fwd_workspace_size(T, N, H, dk, dv, d["q"].dtype), dev)
    o = torch.empty(T, H, dv, dtype=d["q"].dtype, device=dev)
    hT = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"], d["cu_seqlens"],
                      d["h0"], o=o, final_state=hT, workspace=ws, stream=stream)

    for _ in range(warmup):
        step()
    kda.query_status(ws, stream, raise_on_error=True)

    NEV = 1024
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(NEV)] for _ in range(K)]
    for row in kev:                 # torch creates each CUDA event on its first record:
        for e_ in row:              # do that here, outside the timed region
            e_.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    clk = ClockSampler(dev.index or 0) if clock else None
    if clk:
        clk.__enter__()
    # whole calls of the public entry, timed on the caller's stream
    for i in range(K):
        flush.zero_()                       # evict L2 between timed steps
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    if clk:
        clk.__exit__(None, None, None)
    barrier(world)
    kda.query_status(ws, stream, raise_on_error=True)
    step_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    value, tmax = aggregate(T * K, sum(step_ms) / 1e3, world)
    # per-kernel times: the same K calls through the profiled entry, which brackets
    # every kernel with two events on the stream that kernel runs on
    used = []
    for i in range(K):
        flush.zero_()
        used.append(kda.chunk_fwd_profiled(d["q"], d["k"], d["v"], d["z"], d["beta"],
                                           d["A_log"], d["cu_seqlens"], d["h0"], o, hT, ws,
                                           kev[i], stream=stream))
    torch.cuda.synchronize(dev)
    kda.query_status(ws, stream, raise_on_error=True)
    names = kernel_names(used[0], tc_path=(d["q"].dtype == torch.bfloat16 and dk == 128
                                            and dv == 128))
    per_kernel = {}
    for i in range(K):
        for j, nm in enumerate(names):
            per_kernel.setdefault(nm, []).append(kev[i][2 * j].elapsed_time(kev[i][2 * j + 1]))
    totals = {nm: sum(v_) / K for nm, v_ in per_kernel.items()}       # ms per step
    launches = {nm: names.count(nm) for nm in totals}
    dom = max(totals, key=totals.get)
    algo_bytes = prefill_bytes(d["seqlens"], H, dk, dv, 2, d["h0"] is not None, True)
    step_s = statistics.mean(step_ms) / 1e3
    dom_s = totals[dom] / 1e3
    achieved_gbs = algo_bytes / dom_s / 1e9           # per launch: bytes/launches / (time/launches)
    flops = prefill_flops(d["seqlens"], H, dk, dv)
    tflops = flops / step_s / 1e12
    hbm_peak = pk.get("hbm_gbs", FALLBACK["hbm_gbs"])
    tc_peak = pk.get("bf16_tflops", FALLBACK["bf16_tflops"])
    units_per_launch = T * H / launches[dom]
    res = {
        "value": value, "unit": "tokens/s", "ms_per_step": tmax * 1e3 / K,
        "ms_per_step_all": step_ms, "steps": K, "tokens_per_step": T,
        "config": workload_config(name, world),
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved_gbs / hbm_peak,
                     "traffic": profiled_traffic(f"{dom}_{name}.md", units_per_launch),
                     "kernel": dom, "peak_source": pk_src,
                     "algorithmic_bytes_per_launch": algo_bytes / launches[dom],
                     "token_heads_per_launch": units_per_launch,
                     "launches_per_step": launches[dom],
                     "avg_launch_us": dom_s / launches[dom] * 1e6,
                     "kernel_ms_per_step": totals,
                     "kernel_launches_per_step": launches,
                     "step": {"achieved_gbs": algo_bytes / step_s / 1e9,
                              "frac": algo_bytes / step_s / 1e9 / hbm_peak,
                              "algorithmic_bytes": algo_bytes},
                     "tensor": {"achieved_tflops": tflops, "peak_tflops": tc_peak,
                                "frac": tflops / tc_peak, "flops_per_step": flops,
                                "convention": "6 dk dv + 64 (3 dk + 2 dv) per token-head"}},
        "gpu_launches": len(names) * K,
    }
    if clk:
        res["clocks"] = clk.summary()
    del ws, o, hT, flush
    if not keep:
        del d
        torch.cuda.empty_cache()
        return res, None
    return res, d


def run_ours(args, rank, world, local):
    import torch

    from gated_delta_rule_43_gb300 import _build, kda

    _build.build()
    kda.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    pk, pk_src = peaks()
    head, d = prefill_leg(args.workload, dev, stream, args.steps, args.warmup, world, pk, pk_src,
                          clock=True, keep=True)
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": head["config"], "roofline": head["roofline"],
        "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
        "ms_per_step_all": head["ms_per_step_all"],
    }
    if not args.no_e2e:
        line["e2e"] = e2e_bench(args, d, dev, stream, world)
    sample = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == HEADLINE:
        sample = host_prefix(d, CPU_SAMPLE_MAX)
    del d
    torch.cuda.empty_cache()
    if not args.headline_only:
        line["workloads"] = {}
        for name in [w for w in EXTRA_PREFILL if w != args.workload]:
            res, _ = prefill_leg(name, dev, stream, args.steps, args.warmup, world, pk, pk_src)
            line["workloads"][name] = res
        if not args.no_decode:
            line["decode"] = decode_bench(args, dev, stream, world, pk, pk_src)
        if not args.no_segmented:
            line["segmented"] = segmented_bench(dev)
    if sample is not None:
        line["cpu_baseline"] = cpu_baseline(sample, args)
    return line


# the segment-parallel entry's workload: one long sequence with few heads, where the plain
# walk keeps only H x 4 SMs busy (name, lengths, heads, segments)
SEGMENTED = ("prefill_1m_h4", (1 << 20,), 4, 8)


def segmented_bench(dev):
    """kda_chunk_fwd_segmented against kda_chunk_fwd on the same inputs (a long sequence
    with few heads): CUDA events, L2 flushed between steps, the median of three steps
    after one untimed call each."""
    import torch

    from gated_delta_rule_43_gb300 import inputs, kda

    name, lens, H, segs = SEGMENTED
    d = inputs.make_prefill(list(lens), H=H, dk=128, dv=128, dtype="bf16", seed=6, device=dev)
    T, N = sum(lens), len(lens)
    o = torch.empty(T, H, 128, dtype=torch.bfloat16, device=dev)
    hT = torch.empty(N, H, 128, 128, dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def run(seg):
        nbytes = kda.load().kda_chunk_fwd_segmented_workspace_size(T, N, H, 128, 128,
                                                                   kda.KDA_BF16, seg)
        ws = kda.alloc_workspace(nbytes, dev)

        def call():
            kda.chunk_fwd_segmented(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                                    d["cu_seqlens"], None, segments=seg, o=o, final_state=hT,
                                    workspace=ws)
        call()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(3):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            call()
            e.record()
            torch.cuda.synchronize(dev)
            ts.append(s.elapsed_time(e))
        kda.query_status(ws, raise_on_error=True)
        return sorted(ts)[1]

    plain_ms, seg_ms = run(1), run(segs)
    return {"workload": f"{name}: B=1, H={H}, T={T}, dk=dv=128, bf16, zero initial state",
            "segments": segs, "plain_ms": plain_ms, "segmented_ms": seg_ms,
            "plain_tokens_per_s": T / plain_ms * 1e3, "segmented_tokens_per_s": T / seg_ms * 1e3,
            "speedup": plain_ms / seg_ms}


def decode_bench(args, dev, stream, world, pk, pk_src):
    import torch

    from gated_delta_rule_43_gb300 import inputs, kda

    w = inputs.WORKLOADS[DECODE]
    ds = inputs.decode_workload(w, device=dev)
    S = ds.state0
    steps = args.decode_steps
    xs = [ds.step() for _ in range(min(steps, 8))]  # fresh inputs cycle (inputs are 10 MB)
    o = torch.empty(w.N, w.H, w.dv, dtype=torch.bfloat16, device=dev)
    ws = kda.alloc_workspace(kda.load().kda_decode_workspace_size(), dev)

    def step(i):
        x = xs[i % len(xs)]
        kda.decode_step(x["q"], x["k"], x["v"], x["z"], x["beta"], ds.A_log, S, o=o,
                        workspace=ws, stream=stream)

    for i in range(3):
        step(i)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    barrier(world)
    torch.cuda.synchronize(dev)
    ev[0].record(stream)
    for i in range(steps):
        step(i)
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    med = statistics.median(per) / 1e3
    state_bytes = 2 * w.N * w.H * w.dk * w.dv * 4
    io_bytes = w.N * w.H * ((3 * w.dk + 2 * w.dv) * 2 + 2)
    gbs_state = state_bytes / med / 1e9
    agg, tmax = aggregate(state_bytes * steps / 1e9, sum(per) / 1e3, world)
    hbm = pk.get("hbm_gbs", FALLBACK["hbm_gbs"])
    achieved = (state_bytes + io_bytes) / med / 1e9
    return {"workload": f"{DECODE}: N=256 x 1 token, H=32, dk=dv=128, bf16 q/k/v/z/beta, "
                        "fp32 state [256,32,128,128] (512 MiB, larger than L2) in place, "
                        f"{steps} consecutive steps",
            "value": agg, "unit": "state GB/s", "median_step_us": med * 1e6,
            "state_gbs_median_step": gbs_state, "steps": steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm,
                         "traffic": profiled_traffic("decode_step_kernel_decode_256.md"),
                         "kernel": "decode_step_kernel", "peak_source": pk_src,
                         "algorithmic_bytes_per_launch": state_bytes + io_bytes},
            "gpu_launches": steps}


class HostBuffers:
    """Page-locked host tensors for the end-to-end leg, each in an anonymous mapping advised
    for transparent huge pages, touched, then registered with the CUDA driver; torch's
    pinned allocator where a step of that is unavailable.  The mappings stay referenced
    (and registered) until release().  Measured on one box right after the GPU test suite
    had run (host memory fragmented by its processes): the same pipeline moved its inputs
    at 86 GB/s from torch-pinned buffers and at 188 GB/s from these, of a 211 GB/s link."""

    HUGE = 2 << 20

    def __init__(self):
        self.maps = []
        self.registered = []
        self.kind = "huge-page registered"

    def new(self, shape, dtype):
        import mmap

        import torch

        nbytes = torch.empty(0, dtype=dtype).element_size() * int(torch.Size(shape).numel())
        size = max(self.HUGE, (nbytes + self.HUGE - 1) // self.HUGE * self.HUGE)
        try:
            m = mmap.mmap(-1, size, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
            if hasattr(m, "madvise") and hasattr(mmap, "MADV_HUGEPAGE"):
                m.madvise(mmap.MADV_HUGEPAGE)
            raw = torch.frombuffer(m, dtype=torch.uint8, count=size)
            raw.zero_()                                  # allocate (and back) every page now
            if int(torch.cuda.cudart().cudaHostRegister(raw.data_ptr(), size, 0)) != 0:
                raise OSError("cudaHostRegister failed")
        except (OSError, ValueError, AttributeError, RuntimeError):
            self.kind = "pinned"
            return torch.empty(shape, dtype=dtype, pin_memory=True)
        self.maps.append(m)
        self.registered.append(raw)
        return raw[:nbytes].view(dtype).view(shape)

    def release(self):
        import torch

        for raw in self.registered:
            torch.cuda.cudart().cudaHostUnregister(raw.data_ptr())
        self.registered.clear()
        self.maps.clear()


def e2e_bench(args, d, dev, stream, world):
    """Same prefill metric through the public call with pinned host buffers: H2D of every
    input and D2H of o and the final state inside the timed region, every step.  What a
    caller streaming batches does: the host-to-device copies run back to back on their
    own stream (the host link is the bound), compute and device-to-host copies on two
    more, with two sets of device buffers and events between the three."""
    import torch

    from gated_delta_rule_43_gb300 import kda

    names = ("q", "k", "v", "z", "beta", "A_log", "cu_seqlens")
    hb = HostBuffers()
    host = {}
    for n in names:
        host[n] = hb.new(d[n].shape, d[n].dtype)
        host[n].copy_(d[n])
    T, H, dv = d["v"].shape
    N = d["cu_seqlens"].numel() - 1
    dk = d["q"].shape[2]
    ws_bytes = kda.chunk_fwd_workspace_size(T, N, H, dk, dv, d["q"].dtype)
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()
    lanes = []
    for _ in range(2):
        lanes.append({
            "dev": {n: torch.empty_like(d[n]) for n in names},
            "o": torch.empty(T, H, dv, dtype=d["q"].dtype, device=dev),
            "hT": torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev),
            "o_h": hb.new((T, H, dv), d["q"].dtype),
            "s_h": hb.new((N, H, dk, dv), torch.float32),
            "ws": kda.alloc_workspace(ws_bytes, dev),
            "loaded": ev(), "computed": ev(), "copied_out": ev(),
        })
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = lanes[0]["o"].numel() * lanes[0]["o"].element_size() + lanes[0]["hT"].numel() * 4

    def step(i):
        L = lanes[i % 2]
        b = L["dev"]
        with torch.cuda.stream(s_in):
            s_in.wait_event(L["computed"])          # step i - 2 has read these inputs
            for n in names:
                b[n].copy_(host[n], non_blocking=True)
            L["loaded"].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(L["loaded"])
            s_comp.wait_event(L["copied_out"])      # step i - 2's outputs have left
            kda.chunk_fwd(b["q"], b["k"], b["v"], b["z"], b["beta"], b["A_log"], b["cu_seqlens"],
                          None, o=L["o"], final_state=L["hT"], workspace=L["ws"], stream=s_comp)
            L["computed"].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(L["computed"])
            L["o_h"].copy_(L["o"], non_blocking=True)
            L["s_h"].copy_(L["hT"], non_blocking=True)
            L["copied_out"].record(s_out)

    for i in range(2):
        step(i)
    torch.cuda.synchronize(dev)
    K = max(4, args.steps)
    barrier(world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for x in (s_in, s_comp, s_out):
        x.wait_stream(stream)
    for i in range(K):
        step(i)
    for x in (s_in, s_comp, s_out):
        stream.wait_stream(x)
    e.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    for L in lanes:
        kda.query_status(L["ws"], raise_on_error=True)
    elapsed = s.elapsed_time(e) / 1e3
    val, _ = aggregate(T * K, elapsed, world)

    # the host link on its own, for reading the number above: pinned copies of one tensor
    # each way, one untimed, then three timed back to back
    def link_gbs(dst, src, reps=3):
        dst.copy_(src, non_blocking=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(dev)
        return reps * dst.numel() * dst.element_size() / (a.elapsed_time(b) / 1e3) / 1e9
    h2d_link = link_gbs(lanes[0]["dev"]["q"], host["q"])
    d2h_link = link_gbs(lanes[0]["o_h"], lanes[0]["o"])
    torch.cuda.synchronize(dev)
    kind = hb.kind
    del host, lanes
    hb.release()
    return {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K,
            "h2d_gbs": h2d * K / elapsed / 1e9,
            "link_h2d_gbs": h2d_link, "link_d2h_gbs": d2h_link, "host_buffers": kind,
            "note": "H2D, compute and D2H on three streams with two sets of device buffers: "
                    "the next step's inputs stream in while this step computes and its "
                    "outputs stream out; h2d_gbs is the input rate this reached, link_*_gbs "
                    "pinned copies of a single tensor each way on their own (one untimed, "
                    "three timed)"}


# ----------------------------------------------------------------------------- CPU oracle

# tokens of the headline workload copied to the host for the oracle's timed sample
CPU_SAMPLE_MAX = 1 << 16


def host_prefix(d, tmax: int) -> dict:
    """Host arrays (exact storage precision) of the first tmax tokens of a one-sequence
    prefill input, all heads; the oracle's timed sample is a prefix of these."""
    import numpy as np

    from gated_delta_rule_43_gb300 import inputs

    T = sum(d["seqlens"])
    t = min(T, tmax)
    out = {n: inputs.host_array(d[n][:t]) for n in ("q", "k", "v", "z", "beta")}
    out["A_log"] = d["A_log"].cpu().numpy().astype(np.float64)
    out["T"] = T
    out["H"] = d["q"].shape[1]
    return out


def oracle_sample_rate(hp, target_s: float, nthreads: int = 0):
    """Time the fp64 oracle on a prefix of the headline workload sized to ~target_s of
    host work.  Returns (tokens/s, prefix length, threads)."""
    from oracle import oracle as orc

    avail = hp["q"].shape[0]

    def run(t):
        t0 = time.perf_counter()
        orc.forward(hp["q"][:t], hp["k"][:t], hp["v"][:t], hp["z"][:t], hp["beta"][:t],
                    hp["A_log"], [0, t], None, want_o=True, want_state=True, nthreads=nthreads)
        return time.perf_counter() - t0

    probe = min(avail, 128)
    dt = run(probe)
    t_s = int(min(avail, max(probe, probe * target_s / max(dt, 1e-6))))
    dt = run(t_s)
    return t_s / dt, t_s, orc.threads() if nthreads <= 0 else nthreads


def cpu_baseline(hp, args):
    rate, t_s, thr = oracle_sample_rate(hp, args.cpu_seconds)
    return {"value": rate, "unit": "tokens/s", "cores": thr, "kind": "oracle",
            "sample": f"first {t_s} of {hp['T']} tokens of {HEADLINE}, all {hp['H']} heads, "
                      "fp64 sequential recurrence (C, OpenMP over head x column-block units), "
                      "the same inputs the GPU arm ran"}


def run_reference(args, rank, world):
    """--impl reference: the fp64 oracle on the host cores, a bounded prefix of the headline
    workload per step.  The inputs are drawn exactly as the GPU arm draws them (the same
    seeded generator on the GPU, then copied to the host), so both arms see the same values;
    without a GPU they are drawn on the host (same distributions, other values)."""
    import torch

    from gated_delta_rule_43_gb300 import inputs

    if rank != 0:
        return None
    on_gpu = torch.cuda.is_available()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0"))) if on_gpu else "cpu"
    d = inputs.make_workload(inputs.WORKLOADS[HEADLINE], device=dev)
    hp = host_prefix(d, CPU_SAMPLE_MAX)
    del d
    if on_gpu:
        torch.cuda.empty_cache()
    per_step = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample_rate(hp, per_step)
    rates = []
    for _ in range(args.steps):
        r, t_s, thr = oracle_sample_rate(hp, per_step)
        rates.append(r)
    value = statistics.mean(rates)
    sample = (f"first {t_s} of {hp['T']} tokens of {HEADLINE} per step, all {hp['H']} heads, "
              "fp64 sequential recurrence on the host cores; inputs drawn "
              + ("on the GPU with the GPU arm's generator (identical values)" if on_gpu else
                 "on the host (same recipe and seed, host generator: other values)"))
    return {"metric": METRIC, "impl": "reference", "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_s / value * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(HEADLINE, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": thr,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-steps", type=int, default=128)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-segmented", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="time the headline workload (and e2e / CPU baseline) only")
    ap.add_argument("--workload", default=HEADLINE,
                    help="prefill workload of the line (default: the headline, prefill_1m); "
                         "another name from inputs.WORKLOADS is for inspection and profiles")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    rank, world, local = dist_setup()
    line = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
