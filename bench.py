"""Benchmark of the KDA recurrence hot path on one GB300 per rank.

Default workload (N=1): one decode step of one KDA layer for 64 sequences,
96 heads, d_k = d_v = 128: the short conv (3-token bf16 ring, SiLU) followed
by the decode step on a 384 MiB fp32 state. `value` is whole-job algorithmic
bytes per second (GB/s) over the step; `prefill` reports the chunked prefill
of a 4096-token sequence (96 heads, d=128, C=64) in tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs as one process per GPU under torchrun; every rank runs an
independent replica (the path needs no exchange), rank 0 prints the line.
`--impl reference` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_attention_recurrence_02_gb300 import synth  # noqa: E402

METRIC = "KDA decode state GB/s & prefill tokens/s (H=96,d=128) vs HBM/TC roofline"
DEC = synth.DECODE
PRE = synth.PREFILL
B, H, D = DEC["B"], DEC["H"], DEC["D"]
UNITS = B * H
# Algorithmic bytes of one decode step per (sequence, head), conv included:
# state read + write, q/k/v in (bf16), g (fp32), beta, o out (bf16), conv ring
# read of 3 tokens x 3 projections and write of the newest token.
STATE_RW = 2 * D * D * 4
DEC_UNIT_BYTES = STATE_RW + 3 * D * 2 + D * 4 + 4 + D * 2 + 3 * 3 * D * 2 + 3 * D * 2
CONV_W_BYTES = 3 * H * D * 4 * 4
STEP_BYTES = UNITS * DEC_UNIT_BYTES + CONV_W_BYTES
GRAPH_STEPS = 100  # decode steps per CUDA graph in the headline's timed region
# prefill per token-head: q,k,v bf16 in, g fp32, beta, o bf16 out
PREFILL_TOKEN_HEAD_BYTES = 3 * D * 2 + D * 4 + 4 + D * 2
PREFILL_TOKEN_HEAD_FLOPS = 6 * D * D + 5 * PRE["C"] * D


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def _src_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "linear_attention_recurrence_02_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


TRAFFIC_NOTE = ("DRAM bytes of one launch from the committed ncu counters, scaled to this launch by the units "
                "processed; dram_write is a lower bound: dirty lines still in L2 when the kernel ends are not "
                "counted (algorithmic_write_bytes is what the kernel stores)")


def _traffic(kernel, src_files, units_in_launch):
    """DRAM read and write bytes per launch from the committed ncu summary,
    if it was taken on the current source of the kernel; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("src_sha") != _src_sha(*src_files):
        return None
    scale = units_in_launch / rec["units"]
    return {"traffic": rec["dram_bytes"] * scale, "dram_read": rec["dram_read"] * scale,
            "dram_write": rec["dram_write"] * scale, "dram_write_is_lower_bound": True}


def _traffic_fields(tr, algo_write):
    if tr is None:
        return {"traffic": None}
    return dict(tr, algorithmic_write_bytes=algo_write, traffic_note=TRAFFIC_NOTE)


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            args = ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.uuid:
                args.insert(1, f"--id={self.uuid}")
            self.proc = subprocess.Popen(args, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 7:
                        rows.append(parts)
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[3 + i]
                          and "Not" not in r[3 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max([num(r[2]) for r in rows if num(r[2]) is not None] or [0])}


def max_over_ranks(value, device=None):
    """Largest value over the ranks of the default process group (the value
    itself when there is one rank): per-step times are reported as the
    slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------- oracle timing
def _oracle_decode_sample(d, n_seqs, nthreads):
    """Oracle conv + decode for the first n_seqs sequences; returns seconds."""
    import oracle
    t0 = time.perf_counter()
    ry, _ = oracle.shortconv_step(d["x"][:n_seqs], d["ring"][:n_seqs], d["w"])
    oracle.decode_step(ry[:, 0], ry[:, 1], ry[:, 2], d["g"][:n_seqs], d["beta"][:n_seqs], d["s0"][:n_seqs],
                       nthreads=nthreads)
    return time.perf_counter() - t0


def _oracle_prefill_sample(n_heads, nthreads):
    """Oracle token recurrence over the 4096-token prefill workload's first n_heads heads (the
    workload's own seeded inputs for those heads); returns seconds."""
    import oracle
    p = synth.prefill_inputs(PRE["seed"], PRE["T"], H, D, True, heads=list(range(n_heads)))
    t0 = time.perf_counter()
    oracle.recurrence(p["q"], p["k"], p["v"], p["g"], p["beta"], nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(d, budget_s=12.0):
    cores = len(os.sched_getaffinity(0))
    t1 = _oracle_decode_sample(d, 1, cores)  # calibration: 1 sequence x 96 heads
    n = int(max(1, min(B, budget_s / 3 / max(t1, 1e-4))))
    reps, elapsed = 0, 0.0
    while elapsed < budget_s / 2 or reps == 0:
        elapsed += _oracle_decode_sample(d, n, cores)
        reps += 1
    bytes_done = reps * (n * H * DEC_UNIT_BYTES + CONV_W_BYTES)
    # the same oracle on one thread, over a smaller sample (about 2 s)
    t_one = _oracle_decode_sample(d, 1, 1)
    n1 = int(max(1, min(B, 2.0 / max(t_one, 1e-4))))
    e1 = _oracle_decode_sample(d, n1, 1)
    return {"value": bytes_done / elapsed / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} x conv+decode step of {n} of {B} sequences x {H} heads (d={D}), fp64, "
                      f"{cores} threads over (sequence, head) units, {elapsed:.1f} s",
            "single_thread": {"value": (n1 * H * DEC_UNIT_BYTES + CONV_W_BYTES) / e1 / 1e9, "unit": "GB/s",
                              "sample": f"conv+decode step of {n1} of {B} sequences x {H} heads, 1 thread, "
                                        f"{e1:.1f} s"},
            "prefill": _prefill_cpu(cores)}


def _prefill_cpu(cores, budget_s=4.0):
    """The prefill metric on the host: the oracle over a head sample of the 4096-token workload, as
    tokens/s for all H heads (the heads are independent units)."""
    nh = min(H, max(1, cores))
    t = _oracle_prefill_sample(nh, cores)
    if t < budget_s / 4 and nh < H:  # enough time left for a larger sample
        nh = min(H, int(nh * budget_s / 2 / max(t, 1e-3)))
        t = _oracle_prefill_sample(nh, cores)
    T = PRE["T"]
    return {"value": T / (t * H / nh), "unit": "tokens/s", "cores": cores,
            "sample": f"fp64 token recurrence over {nh} of {H} heads x {T} tokens, {cores} threads, {t:.1f} s"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    d = synth.decode_inputs(DEC["seed"], B, H, D, True)
    cores = len(os.sched_getaffinity(0))
    t1 = _oracle_decode_sample(d, 1, cores)
    budget = 90.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(B, budget / max(t1, 1e-4))))
    for _ in range(args.warmup):
        _oracle_decode_sample(d, n, cores)
    times = [_oracle_decode_sample(d, n, cores) for _ in range(args.steps)]
    tot = sum(times)
    value = args.steps * (n * H * DEC_UNIT_BYTES + CONV_W_BYTES) / tot / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"KDA decode step with short conv, B={B} sequences (sample of {n} per step), "
                               f"H={H}, d_k=d_v={D}, bf16 q/k/v inputs, fp32 state"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"conv+decode step of {n} of {B} sequences x {H} heads per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    from linear_attention_recurrence_02_gb300 import build as kbuild
    from linear_attention_recurrence_02_gb300 import kda

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kbuild.build_library()
    hbm_peak, tc_peak, tc_sus, peak_src = _peaks()

    d = synth.decode_inputs(DEC["seed"] + 1000 * rank, B, H, D, True)
    bf = torch.bfloat16

    def up(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev, dt)

    x, ring, w = up(d["x"], bf), up(d["ring"], bf), up(d["w"], torch.float32)
    g, beta, state = up(d["g"], torch.float32), up(d["beta"], torch.float32), up(d["s0"], torch.float32)
    out = torch.empty((B, H, D), dtype=bf, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(st=None):
        # one launch: short conv + decode (kda_shortconv_decode_step)
        kda.kda_shortconv_decode_step(x, ring, w, g, beta, state, out, stream=stream if st is None else st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the same steps issued one by one from the host, reported beside the graph-timed value
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    one_by_one_ms = start.elapsed_time(end) / args.steps
    # The timed steps run from CUDA graphs of up to GRAPH_STEPS launches (a serving loop's decode
    # form): each launch is the same call on the same resident state, and the graph removes the
    # host's launch gap between steps (about 2 us on this part), not any work.
    G = min(GRAPH_STEPS, args.steps)
    graphs = []
    for n_g in sorted({G, args.steps % G} - {0}, reverse=True):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            cs = torch.cuda.current_stream(dev)
            for _ in range(n_g):
                step(cs)
        graphs.append((n_g, gr))
    for _, gr in graphs:
        gr.replay()  # warm-up of the graphs themselves
    torch.cuda.synchronize(dev)
    replays = [graphs[0][1]] * (args.steps // G) + ([graphs[1][1]] if len(graphs) > 1 else [])
    if ws > 1:
        dist.barrier()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    with ClockSampler(uuid) as clk:
        torch.cuda.synchronize(dev)
        start.record(stream)
        for gr in replays:
            gr.replay()
        end.record(stream)
        torch.cuda.synchronize(dev)
    clocks = clk.summary()
    ms = start.elapsed_time(end)
    # the timed region holds only this kernel's launches, one per step
    dec_ms = [ms / args.steps]
    ms = max_over_ranks(ms, dev)
    if ws > 1:
        dist.barrier()
    kda.kda_sync_status(stream)
    ms_per_step = ms / args.steps
    value = ws * STEP_BYTES / (ms_per_step * 1e-3) / 1e9

    dec_avg_ms = statistics.mean(dec_ms)
    dec_bytes = STEP_BYTES
    achieved = dec_bytes / (dec_avg_ms * 1e-3) / 1e9
    traffic = _traffic("fused_decode_bulk_kernel", ["kda_fused_decode.cu", "kda_common.cuh", "kda_tc.cuh"], UNITS)
    # state written back, o, the shifted 3-slot ring
    dec_write = UNITS * (D * D * 4 + D * 2 + 9 * D * 2)

    # End to end through the public API, the way a serving loop runs it: every
    # step's inputs (x, g, beta, packed in one pinned host buffer) go host ->
    # device and its output comes back device -> host inside the timed region.
    # The copies run on their own streams, double-buffered, so that step t+1's
    # input copy and step t-1's output copy overlap step t's launch.
    nx, ng, nb = x.numel() * 2, g.numel() * 4, beta.numel() * 4
    host_in = torch.empty(nx + ng + nb, dtype=torch.uint8).pin_memory()
    host_in[:nx].copy_(torch.from_numpy(np.ascontiguousarray(d["x"])).to(bf).view(-1).view(torch.uint8))
    host_in[nx:nx + ng].copy_(torch.from_numpy(np.ascontiguousarray(d["g"])).view(-1).view(torch.uint8))
    host_in[nx + ng:].copy_(torch.from_numpy(np.ascontiguousarray(d["beta"])).view(-1).view(torch.uint8))
    dev_in = [torch.empty(nx + ng + nb, dtype=torch.uint8, device=dev) for _ in range(2)]
    xs = [b_[:nx].view(bf).view(x.shape) for b_ in dev_in]
    gs = [b_[nx:nx + ng].view(torch.float32).view(g.shape) for b_ in dev_in]
    bs = [b_[nx + ng:].view(torch.float32).view(beta.shape) for b_ in dev_in]
    outs = [out, torch.empty_like(out)]
    host_out = [torch.empty((B, H, D), dtype=bf).pin_memory() for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    k_done = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]
    k_e2e = max(1, min(args.steps, 1000))

    def e2e_step(t):
        i = t % 2
        h2d_s.wait_event(k_done[i])          # launch t-2 has read this input buffer
        with torch.cuda.stream(h2d_s):
            dev_in[i].copy_(host_in, non_blocking=True)
        in_ready[i].record(h2d_s)
        stream.wait_event(in_ready[i])
        stream.wait_event(out_read[i])       # output t-2 has been read back
        kda.kda_shortconv_decode_step(xs[i], ring, w, gs[i], bs[i], state, outs[i], stream=stream)
        k_done[i].record(stream)
        d2h_s.wait_event(k_done[i])
        with torch.cuda.stream(d2h_s):
            host_out[i].copy_(outs[i], non_blocking=True)
        out_read[i].record(d2h_s)

    for t in range(min(args.warmup, 20)):
        e2e_step(t)
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    h2d_s.wait_event(s2)
    for t in range(k_e2e):
        e2e_step(t)
    e2.record(d2h_s)                          # after the last output copy
    torch.cuda.synchronize(dev)
    e2e_ms = s2.elapsed_time(e2) / k_e2e
    e2e_ms = max_over_ranks(e2e_ms, dev)
    h2d = nx + ng + nb
    d2h = out.numel() * 2

    dec_unfused = bench_decode_unfused(torch, kda, dev, stream, ws, hbm_peak, d)
    dec_epi = bench_decode_epi(torch, kda, dev, stream, ws, hbm_peak, d, ms_per_step)
    conv_step = bench_shortconv_step(torch, kda, dev, stream, ws, hbm_peak)

    prefill = None
    if not args.no_prefill:
        prefill = bench_prefill(args, torch, kda, dev, stream, ws, hbm_peak, tc_peak, peak_src)
    stack = None
    if not args.no_stack:
        stack = bench_stack(torch, kda, dev, ws, hbm_peak)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
            "data": "synthetic (seeded N(0,1) q/k/v, g=-softplus(N(0,1)), beta=sigmoid(N(0,1)), "
                    "state N(0,0.02^2))",
            "config": {"workload": f"KDA decode step with short conv (fused, one launch): B={B} sequences, "
                                   f"H={H}, d_k=d_v={D}, bf16 q/k/v, fp32 state (384 MiB), 1 layer",
                       "B": B, "H": H, "d": D, "l2": "state (384 MiB) larger than L2 (129 MB); no flush",
                       "launch": f"the K steps replayed from CUDA graphs of {min(GRAPH_STEPS, args.steps)} launches",
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
            "one_by_one": {"ms_per_step": one_by_one_ms,
                           "value": ws * STEP_BYTES / (one_by_one_ms * 1e-3) / 1e9, "unit": "GB/s",
                           "note": "the same K steps issued one by one from the host, before the graph-timed region"},
            "roofline": {"bound": "hbm", "kernel": "fused_decode_bulk_kernel", "achieved": achieved,
                         "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                         "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                         **_traffic_fields(traffic, dec_write), "algorithmic_bytes": dec_bytes,
                         "avg_launch_us": dec_avg_ms * 1e3},
            "e2e": {"value": ws * STEP_BYTES / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "copies": "one packed pinned H2D copy and one D2H copy per step on their own streams, "
                              "double-buffered, overlapping the neighbouring steps' launches"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "decode_unfused": dec_unfused,
            "decode_epilogue": dec_epi,
            "shortconv_step": conv_step,
        }
        if prefill is not None:
            line["prefill"] = prefill
        if stack is not None:
            line["stack"] = stack
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(d)
        print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()
    return 0


def bench_prefill(args, torch, kda, dev, stream, ws, hbm_peak, tc_peak, peak_src):
    """Chunked prefill of one 4096-token sequence, 96 heads, d=128, C=64."""
    T, C = PRE["T"], PRE["C"]
    p = synth.prefill_inputs(PRE["seed"], T, H, D, bf16=True)
    bf = torch.bfloat16

    def up(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev, dt)

    q, k, v = (up(p[n], bf) for n in ("q", "k", "v"))
    g, beta = up(p["g"], torch.float32), up(p["beta"], torch.float32)
    out = torch.empty_like(q)
    sf = torch.empty((1, H, D, D), dtype=torch.float32, device=dev)
    ws_bytes = kda.kda_chunk_prefill_workspace_bytes(T, 1, H, D, C)
    wsb = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    try:
        kda.kda_chunk_prefill(q, k, v, g, beta, out, final_state=sf, chunk_size=C, workspace=wsb, stream=stream)
    except kda.KdaError as e:
        return {"unavailable": str(e)}
    n = max(3, min(args.steps, 200))
    for _ in range(max(3, min(args.warmup, 10))):
        kda.kda_chunk_prefill(q, k, v, g, beta, out, final_state=sf, chunk_size=C, workspace=wsb, stream=stream)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        a.record(stream)
        kda.kda_chunk_prefill(q, k, v, g, beta, out, final_state=sf, chunk_size=C, workspace=wsb, stream=stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    kda.kda_sync_status(stream)
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evs), dev)
    toks = T * 1.0
    by = T * H * PREFILL_TOKEN_HEAD_BYTES + H * D * D * 4
    fl = T * H * PREFILL_TOKEN_HEAD_FLOPS
    varlen = bench_varlen(torch, kda, dev, stream, ws, hbm_peak)
    conv = bench_conv_prefill(torch, kda, dev, stream, ws, hbm_peak)
    epilogue = bench_epilogue(torch, kda, dev, stream, ws, hbm_peak)
    # the prefill and its output epilogue in one call (kda_chunk_prefill_epi)
    egen = torch.Generator(device=dev).manual_seed(PRE["seed"] + 13)
    egate = torch.randn((T, H, D), generator=egen, device=dev).to(bf)
    ew = torch.rand((D,), generator=egen, device=dev) + 0.5

    def ecall():
        kda.kda_chunk_prefill_epi(q, k, v, g, beta, out, egate, ew, final_state=sf, chunk_size=C, workspace=wsb,
                                  stream=stream)
    for _ in range(3):
        ecall()
    torch.cuda.synchronize(dev)
    ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a0, b0 in ee:
        a0.record(stream)
        ecall()
        b0.record(stream)
    torch.cuda.synchronize(dev)
    kda.kda_sync_status(stream)
    ems = max_over_ranks(statistics.mean(a0.elapsed_time(b0) for a0, b0 in ee), dev)
    epilogue["with_prefill"] = {
        "ms_per_call": ems, "unit": "ms", "prefill_alone_ms": ms,
        "workload": "kda_chunk_prefill_epi on the 4096-token prefill (sigmoid gate): the prefill, then the "
                    "epilogue pass in place"}
    del egate
    long_seq = bench_long_sequence(torch, kda, dev, stream, ws)
    # the same workload with a per-head gate (Gated DeltaNet) and with none (DeltaNet)
    gates = {}
    gh = g[..., 0].contiguous()
    for name, gg, gbytes in (("head", gh, 4), ("none", None, 0)):
        def gcall():
            kda.kda_chunk_prefill_gated(q, k, v, gg, beta, out, gate=name, final_state=sf, chunk_size=C,
                                        workspace=wsb, stream=stream)
        for _ in range(3):
            gcall()
        torch.cuda.synchronize(dev)
        ge = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a0, b0 in ge:
            a0.record(stream)
            gcall()
            b0.record(stream)
        torch.cuda.synchronize(dev)
        gms = max_over_ranks(statistics.mean(a0.elapsed_time(b0) for a0, b0 in ge), dev)
        gby = T * H * (PREFILL_TOKEN_HEAD_BYTES - 512 + gbytes) + H * D * D * 4
        gates[name] = {"value": ws * toks / (gms * 1e-3), "unit": "tokens/s", "ms_per_call": gms,
                       "roofline_hbm": {"achieved": gby / (gms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                                        "frac": gby / (gms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": gby}}
    # the same workload in fp32: the tensor-core kernel in tf32 with a 3-term hi/lo split per product
    simt = None
    try:
        q32, k32, v32 = (t_.float() for t_ in (q, k, v))
        o32 = torch.empty_like(q32)

        def scall():
            kda.kda_chunk_prefill(q32, k32, v32, g, beta, o32, final_state=sf, chunk_size=C, workspace=wsb,
                                  stream=stream)
        for _ in range(2):
            scall()
        torch.cuda.synchronize(dev)
        se = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
        for a0, b0 in se:
            a0.record(stream)
            scall()
            b0.record(stream)
        torch.cuda.synchronize(dev)
        sms = max_over_ranks(statistics.mean(a0.elapsed_time(b0) for a0, b0 in se), dev)
        sby = T * H * (3 * D * 4 + D * 4 + 4 + D * 4) + H * D * D * 4
        # tensor-pipe work as issued: per chunk-head the five products (G1 128x64x128, G0 128x128x128,
        # G2, G3 128x64x64, G4 128x128x64) at 2 flops per multiply-add, three tf32 MMAs each
        sfl = 3 * 2 * (128 * 64 * 128 + 128 * 128 * 128 + 2 * 128 * 64 * 64 + 128 * 128 * 64) * (T // C) * H
        tf32_peak = tc_peak / 2.0  # dense tf32 runs at half the bf16 rate (nominal 1.1 vs 2.25 PFLOP/s)
        simt = {"value": ws * toks / (sms * 1e-3), "unit": "tokens/s", "ms_per_call": sms,
                "kernel": "prefill_tf32_kernel (fp32 q/k/v/out; tcgen05 kind::tf32, 3xTF32 products)",
                "roofline_hbm": {"achieved": sby / (sms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                                 "frac": sby / (sms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": sby,
                                 **_traffic_fields(_traffic("prefill_tf32_kernel",
                                                            ["kda_prefill_tf32.cu", "kda_tc.cuh", "kda_prefill.cuh",
                                                             "kda_common.cuh"], T * H),
                                                   T * H * D * 4 + H * D * D * 4)},
                "roofline_tensor": {"achieved": sfl / (sms * 1e-3) / 1e12, "peak": tf32_peak, "unit": "TFLOP/s",
                                    "frac": sfl / (sms * 1e-3) / 1e12 / tf32_peak, "flops_issued": sfl,
                                    "peak_source": f"{peak_src} bf16_tflops (burst) x 1/2 (tf32 : bf16 nominal)"}}
        del q32, k32, v32, o32
    except kda.KdaError as e:
        simt = {"unavailable": str(e)}
    return {"value": ws * toks / (ms * 1e-3), "unit": "tokens/s", "ms_per_call": ms, "varlen": varlen,
            "conv": conv, "epilogue": epilogue, "long_sequence": long_seq, "gates": gates, "fp32": simt,
            "config": {"workload": f"chunked prefill T={T}, H={H}, d={D}, C={C}, bf16 q/k/v, zero S0, "
                                   "fp32 final state", "calls": n},
            "roofline_hbm": {"achieved": by / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                             "frac": by / (ms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": by,
                             **_traffic_fields(_traffic("prefill_tc_pipe_kernel",
                                                        ["kda_prefill_tc.cu", "kda_tc.cuh", "kda_prefill.cuh",
                                                         "kda_common.cuh"], T * H),
                                               T * H * D * 2 + H * D * D * 4)},
            "roofline_tensor": {"achieved": fl / (ms * 1e-3) / 1e12, "peak": tc_peak, "unit": "TFLOP/s",
                                "frac": fl / (ms * 1e-3) / 1e12 / tc_peak, "algorithmic_flops": fl,
                                "peak_source": f"{peak_src} bf16_tflops (burst)"}}


def bench_conv_prefill(torch, kda, dev, stream, ws, hbm_peak, n=30):
    """Short conv + SiLU over one 4096-token prompt (96 heads, d=128, bf16)
    with the ring handed in and out. Timing only; inputs drawn on the device
    by a seeded torch generator. Three input/output sets are rotated so that
    every call reads and writes 151 MB that the previous two calls did not
    touch (450 MB in all, above the 129 MB L2)."""
    T = PRE["T"]
    gen = torch.Generator(device=dev).manual_seed(PRE["seed"])
    bf = torch.bfloat16
    sets = []
    for _ in range(3):
        x = torch.randn((T, 3, H, D), generator=gen, device=dev).to(bf)
        y = torch.empty((3, T, H, D), dtype=bf, device=dev)
        sets.append((x, y))
    rin = torch.randn((1, 3, H, 3, D), generator=gen, device=dev).to(bf)
    rout = torch.empty_like(rin)
    w = torch.randn((3, H, D, 4), generator=gen, device=dev) * 0.5

    def call(st, i):
        x, y = sets[i % 3]
        kda.kda_shortconv_prefill(x, w, y, ring_in=rin, ring_out=rout, stream=st)
    try:
        call(stream, 0)
    except kda.KdaError as e:
        return {"unavailable": str(e)}
    for i in range(6):
        call(stream, i)
    torch.cuda.synchronize(dev)
    ms, loop_ms = _graph_and_loop_ms(torch, dev, stream, call, n, per_graph=n)
    kda.kda_sync_status(stream)
    ms = max_over_ranks(ms, dev)
    by = 2 * (T * 3 * H * D * 2) + 2 * (9 * H * D * 2) + 3 * H * D * 16
    return {"value": ws * T / (ms * 1e-3), "unit": "tokens/s", "ms_per_call": ms,
            "config": {"workload": f"short conv + SiLU prefill T={T}, H={H}, d={D}, bf16, ring in and out",
                       "calls": n, "l2": "3 rotating input/output sets (450 MB)", "launch": f"CUDA graph of {n} calls"},
            "one_by_one_ms_per_call": loop_ms,
            "roofline_hbm": {"achieved": by / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                             "frac": by / (ms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": by,
                             **_traffic_fields(_traffic("shortconv_prefill_kernel",
                                                        ["kda_shortconv.cu", "kda_common.cuh", "kda_tc.cuh"], T),
                                               T * 3 * H * D * 2 + 9 * H * D * 2)}}


def bench_shortconv_step(torch, kda, dev, stream, ws, hbm_peak, n=200, nsets=6, per_graph=60, replays=10):
    """The standalone short conv decode step (kda_shortconv_step) on the
    headline batch: B=64, H=96, d=128, bf16, writing y for callers that need
    the post-conv q, k, v. Timing only; inputs drawn on the device by a seeded
    torch generator. `nsets` sets of x, ring and y (38 MB each, 226 MB in all,
    above the 129 MB L2) rotate so that every call misses in L2.

    The value is timed on launches replayed from a CUDA graph (`per_graph`
    calls per graph): a 38 MB step lasts about as long as the gap between two
    launches issued one by one from the host, and a plain device copy of the
    same bytes measures 55 % of HBM that way against 74-78 % from a graph.
    The one-by-one figure is reported beside it."""
    gen = torch.Generator(device=dev).manual_seed(DEC["seed"] + 21)
    bf = torch.bfloat16
    sets = [(torch.randn((B, 3, H, D), generator=gen, device=dev).to(bf),
             torch.randn((B, 3, H, 3, D), generator=gen, device=dev).to(bf),
             torch.empty((3, B, H, D), dtype=bf, device=dev)) for _ in range(nsets)]
    w = torch.randn((3, H, D, 4), generator=gen, device=dev) * 0.5

    def call(i, st):
        x, ring, y = sets[i % nsets]
        kda.kda_shortconv_step(x, ring, w, y, stream=st)
    for i in range(2 * nsets):
        call(i, stream)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(n):
        call(i, stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    kda.kda_sync_status(stream)
    ms_loop = max_over_ranks(a.elapsed_time(b) / n, dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cs = torch.cuda.current_stream(dev)
        for i in range(per_graph):
            call(i, cs)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize(dev)
    a.record()
    for _ in range(replays):
        graph.replay()
    b.record()
    torch.cuda.synchronize(dev)
    kda.kda_sync_status()
    ms = max_over_ranks(a.elapsed_time(b) / (replays * per_graph), dev)
    # per (sequence, head): x read, the 3-slot ring read and rewritten (shifted), y written; plus the taps
    by = B * H * (3 * D * 2 + 2 * 9 * D * 2 + 3 * D * 2) + 3 * H * D * 16
    return {"value": ws * by / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "kernel": "shortconv_step_kernel",
            "config": {"workload": f"short conv decode step alone (kda_shortconv_step): B={B}, H={H}, d={D}, bf16, "
                                   "y written", "steps": replays * per_graph,
                       "launch": f"CUDA graph of {per_graph} calls, replayed {replays} times",
                       "l2": f"{nsets} rotating x/ring/y sets (226 MB)"},
            "one_by_one": {"ms_per_step": ms_loop, "steps": n,
                           "frac": by / (ms_loop * 1e-3) / 1e9 / hbm_peak},
            "roofline_hbm": {"achieved": by / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                             "frac": by / (ms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": by,
                             **_traffic_fields(_traffic("shortconv_step_kernel", ["kda_shortconv.cu",
                                                                                  "kda_common.cuh", "kda_tc.cuh"], B * H),
                                               B * H * 12 * D * 2)}}


def bench_epilogue(torch, kda, dev, stream, ws, hbm_peak, n=20):
    """Output epilogue (gated RMSNorm, sigmoid gate) over the 4096-token
    prefill output, 96 heads, d=128, bf16. Timing only; inputs drawn on the
    device by a seeded torch generator. Two sets of o, gate and y (604 MB in
    all, above the 129 MB L2) alternate."""
    T = PRE["T"]
    gen = torch.Generator(device=dev).manual_seed(PRE["seed"] + 7)
    bf = torch.bfloat16
    sets = [(torch.randn((T, H, D), generator=gen, device=dev).to(bf),
             torch.randn((T, H, D), generator=gen, device=dev).to(bf),
             torch.empty((T, H, D), dtype=bf, device=dev)) for _ in range(2)]
    w = torch.rand((D,), generator=gen, device=dev) + 0.5

    def call(st, i):
        o, gt, y = sets[i % 2]
        kda.kda_gated_rmsnorm(o, gt, w, y, stream=st)
    for i in range(4):
        call(stream, i)
    torch.cuda.synchronize(dev)
    ms, loop_ms = _graph_and_loop_ms(torch, dev, stream, call, n, per_graph=n)
    kda.kda_sync_status(stream)
    ms = max_over_ranks(ms, dev)
    by = 3 * T * H * D * 2 + D * 4
    return {"value": ws * T / (ms * 1e-3), "unit": "tokens/s", "ms_per_call": ms,
            "config": {"workload": f"gated RMSNorm output epilogue T={T}, H={H}, d={D}, bf16, sigmoid gate",
                       "calls": n, "l2": "2 alternating sets (604 MB)", "launch": f"CUDA graph of {n} calls"},
            "one_by_one_ms_per_call": loop_ms,
            "roofline_hbm": {"achieved": by / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                             "frac": by / (ms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": by,
                             **_traffic_fields(_traffic("gated_rmsnorm_kernel", ["kda_epilogue.cu", "kda_common.cuh"],
                                                        T * H), T * H * D * 2)}}


def bench_long_sequence(torch, kda, dev, stream, ws, T=65536, Hs=8, segments=0, n=3):
    """One 65,536-token sequence with 8 heads, d=128, C=64, bf16, per-channel
    gate: the serial prefill (one chain of 1024 chunks per head, 8 SMs busy)
    against kda_chunk_prefill_scan with the automatic segment count
    (floor(SMs / H): one pass over the segments fills the GPU once). Timing
    only; inputs drawn on the device by a seeded torch generator with the
    workloads' distributions."""
    gen = torch.Generator(device=dev).manual_seed(PRE["seed"] + 11)

    def rnd(shape):
        return torch.randn(shape, generator=gen, device=dev)
    q, k, v = (rnd((T, Hs, D)).to(torch.bfloat16) for _ in range(3))
    g = -torch.nn.functional.softplus(rnd((T, Hs, D)))
    beta = torch.sigmoid(rnd((T, Hs)))
    out = torch.empty_like(q)
    sf = torch.empty((Hs, D, D), device=dev)
    wsb = torch.empty(max(16, kda.kda_chunk_prefill_scan_workspace_bytes(T, Hs, D, 64, segments)),
                      dtype=torch.uint8, device=dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return max_over_ranks(a.elapsed_time(b) / n, dev)
    # an empty workspace keeps kda_chunk_prefill on the serial path (with the workspace it asks for, the
    # call would split this sequence itself)
    no_ws = torch.empty(0, dtype=torch.uint8, device=dev)
    ms_serial = timed(lambda: kda.kda_chunk_prefill(q, k, v, g, beta, out, final_state=sf[None], chunk_size=64,
                                                    workspace=no_ws, stream=stream))
    ms_scan = timed(lambda: kda.kda_chunk_prefill_scan(q, k, v, g, beta, out, segments, final_state=sf,
                                                       workspace=wsb, stream=stream))
    # the same rows as a packed batch of five sequences, one of them long: kda_chunk_prefill_split
    # (host-side lengths; it splits the long one and runs the rest in one launch) against one
    # kda_chunk_prefill_gated call over the batch
    lens = [59904, 512, 3000, 120, 2000]
    cu_h = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int64)
    cu_d = cu_h.to(dev)
    sfb = torch.empty((len(lens), Hs, D, D), device=dev)
    seg, _ = kda.kda_chunk_prefill_split_plan(cu_h, Hs, 64)
    ms_batch_whole = timed(lambda: kda.kda_chunk_prefill_gated(q, k, v, g, beta, out, final_state=sfb,
                                                               cu_seqlens=cu_d, chunk_size=64, stream=stream))
    ms_batch_split = timed(lambda: kda.kda_chunk_prefill_split(q, k, v, g, beta, out, cu_h, final_state=sfb,
                                                               chunk_size=64, stream=stream))
    kda.kda_sync_status(stream)
    mixed = {"ms_per_call": ms_batch_split, "whole_ms_per_call": ms_batch_whole,
             "speedup": ms_batch_whole / ms_batch_split, "segments": [int(x) for x in seg],
             "config": {"workload": f"packed batch of {len(lens)} sequences {lens} (65,536 tokens), H={Hs}, d={D}, "
                                    "C=64, bf16: kda_chunk_prefill_split vs kda_chunk_prefill_gated"}}
    return {"value": ws * T / (ms_scan * 1e-3), "unit": "tokens/s", "ms_per_call": ms_scan,
            "serial_ms_per_call": ms_serial, "speedup": ms_serial / ms_scan, "mixed_batch": mixed,
            "config": {"workload": f"one sequence of {T} tokens, H={Hs}, d={D}, C=64, bf16, per-channel gate: "
                                   "kda_chunk_prefill_scan vs kda_chunk_prefill",
                       "segments": segments if segments else max(2, torch.cuda.get_device_properties(dev)
                                                                 .multi_processor_count // Hs),
                       "calls": n}}


def bench_varlen(torch, kda, dev, stream, ws, hbm_peak):
    """Variable-length prefill with carry-in: 8 sequences of 512..65536 tokens
    (130,560 in all), H=96, d=128, C=64, bf16. Timing only; inputs drawn on
    the device by a seeded torch generator with the workload's distributions."""
    cu = synth.varlen_cu_seqlens()
    T, N = int(cu[-1]), len(cu) - 1
    gen = torch.Generator(device=dev).manual_seed(synth.VARLEN["seed"])

    def rnd(shape):
        return torch.randn(shape, generator=gen, device=dev)
    q, k, v = (rnd((T, H, D)).to(torch.bfloat16) for _ in range(3))
    g = -torch.nn.functional.softplus(rnd((T, H, D)))
    beta = torch.sigmoid(rnd((T, H)))
    s0 = rnd((N, H, D, D)) * 0.02
    sf = torch.empty_like(s0)
    out = torch.empty_like(q)
    tcu = torch.from_numpy(cu).to(dev)
    wsb = torch.empty(max(16, kda.kda_chunk_prefill_workspace_bytes(T, N, H, D, 64)), dtype=torch.uint8, device=dev)

    def call():
        kda.kda_chunk_prefill(q, k, v, g, beta, out, initial_state=s0, final_state=sf, cu_seqlens=tcu,
                              chunk_size=64, workspace=wsb, stream=stream)
    for _ in range(3):
        call()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 5
    a.record(stream)
    for _ in range(n):
        call()
    b.record(stream)
    torch.cuda.synchronize(dev)
    kda.kda_sync_status(stream)
    ms = max_over_ranks(a.elapsed_time(b) / n, dev)
    by = T * H * PREFILL_TOKEN_HEAD_BYTES + 2 * N * H * D * D * 4
    return {"value": ws * T / (ms * 1e-3), "unit": "tokens/s", "ms_per_call": ms,
            "config": {"workload": "varlen prefill, 8 sequences 512..65536 (130,560 tokens), H=96, d=128, C=64, "
                                   "bf16, S0 ~ N(0,0.02^2), final states", "calls": n},
            "roofline_hbm": {"achieved": by / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                             "frac": by / (ms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": by}}


def _graph_and_loop_ms(torch, dev, stream, call, steps, per_graph=GRAPH_STEPS):
    """ms per call of `call(st, i)` (the i-th call, on stream st) issued one by one on `stream`, then
    replayed from a CUDA graph of `per_graph` calls (steps // per_graph replays, at least one):
    (graph_ms, one_by_one_ms)."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        call(stream, i)
    b.record(stream)
    torch.cuda.synchronize(dev)
    loop_ms = a.elapsed_time(b) / steps
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        cs = torch.cuda.current_stream(dev)
        for i in range(per_graph):
            call(cs, i)
    gr.replay()
    torch.cuda.synchronize(dev)
    reps = max(1, steps // per_graph)
    a.record(stream)
    for _ in range(reps):
        gr.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / (reps * per_graph), loop_ms


def bench_decode_unfused(torch, kda, dev, stream, ws, hbm_peak, d, steps=200):
    """The decode step alone (kda_decode_step, post-conv q/k/v, no conv) on
    the headline workload: B=64, H=96, d=128, bf16 q/k/v, its own 384 MiB
    fp32 state (larger than L2, so no flush)."""
    bf = torch.bfloat16

    def up(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev, dt)
    q, k, v = up(d["q"], bf), up(d["k"], bf), up(d["v"], bf)
    g, beta, state = up(d["g"], torch.float32), up(d["beta"], torch.float32), up(d["s0"], torch.float32)
    out = torch.empty_like(q)

    def step(st, i=0):
        kda.kda_decode_step(q, k, v, g, beta, state, out, stream=st)
    for _ in range(5):
        step(stream)
    torch.cuda.synchronize(dev)
    ms, loop_ms = _graph_and_loop_ms(torch, dev, stream, step, steps)
    kda.kda_sync_status(stream)
    ms = max_over_ranks(ms, dev)
    by = B * H * (2 * D * D * 4 + 3 * D * 2 + D * 4 + 4 + D * 2)
    tr = _traffic("decode_step_kernel", ["kda_decode.cu", "kda_common.cuh"], B * H)
    return {"value": ws * by / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "kernel": "decode_step_kernel", "dram": _traffic_fields(tr, B * H * (D * D * 4 + D * 2)),
            "config": {"workload": f"decode step without conv (kda_decode_step): B={B}, H={H}, d={D}, bf16 q/k/v, "
                                   "fp32 state 384 MiB", "steps": steps,
                       "launch": f"CUDA graph of {GRAPH_STEPS} calls, as the headline"},
            "one_by_one_ms_per_step": loop_ms,
            "roofline_hbm": {"achieved": by / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                             "frac": by / (ms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": by}}


def bench_decode_epi(torch, kda, dev, stream, ws, hbm_peak, d, fused_ms, steps=200):
    """The fused conv + decode step with the gated RMSNorm output epilogue in
    the same launch (kda_shortconv_decode_step_epi) on the headline workload:
    the step's bytes plus the output gate read (bf16) and the norm weight;
    the output is the epilogue's y instead of o."""
    bf = torch.bfloat16

    def up(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev, dt)
    x, ring, w = up(d["x"], bf), up(d["ring"], bf), up(d["w"], torch.float32)
    g, beta, state = up(d["g"], torch.float32), up(d["beta"], torch.float32), up(d["s0"], torch.float32)
    e = synth.epilogue_inputs(DEC["seed"] + 50, B, H, D, True)
    og, nw = up(e["gate"], bf), up(e["weight"], torch.float32)
    y = torch.empty((B, H, D), dtype=bf, device=dev)

    def step(st, i=0):
        kda.kda_shortconv_decode_step_epi(x, ring, w, g, beta, state, og, nw, y, stream=st)
    for _ in range(5):
        step(stream)
    torch.cuda.synchronize(dev)
    ms, loop_ms = _graph_and_loop_ms(torch, dev, stream, step, steps)
    kda.kda_sync_status(stream)
    ms = max_over_ranks(ms, dev)
    by = STEP_BYTES + B * H * D * 2 + D * 4
    tr = _traffic("fused_decode_bulk_kernel_epilogue", ["kda_fused_decode.cu", "kda_common.cuh", "kda_tc.cuh"], B * H)
    return {"value": ws * by / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "dram": _traffic_fields(tr, B * H * (D * D * 4 + D * 2 + 9 * D * 2)),
            "fused_step_without_epilogue_ms": fused_ms, "kernel": "fused_decode_bulk_kernel (output epilogue)",
            "config": {"workload": f"fused conv + decode step with the gated RMSNorm epilogue (sigmoid gate) in "
                                   f"one launch: B={B}, H={H}, d={D}, bf16, fp32 state 384 MiB", "steps": steps,
                       "launch": f"CUDA graph of {GRAPH_STEPS} calls, as the headline"},
            "one_by_one_ms_per_step": loop_ms,
            "roofline_hbm": {"achieved": by / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                             "frac": by / (ms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": by}}


def bench_stack(torch, kda, dev, ws, hbm_peak, steps_per_graph=16, replays=8):
    """Full-stack decode: 69 independent layers x 8 sequences x 96 heads
    (414 MiB of fp32 state per sequence, 3.3 GB in all), one fused conv+decode
    launch per layer per step in model order, `steps_per_graph` steps captured
    in one CUDA graph with each step's own inputs. Inputs are drawn on the
    device by a seeded torch generator with the workload's distributions."""
    L, Bs = synth.STACK["layers"], synth.STACK["B"]
    gen = torch.Generator(device=dev).manual_seed(synth.STACK["seed"])

    def rnd(shape):
        return torch.randn(shape, generator=gen, device=dev)
    G = steps_per_graph
    x = [rnd((G, Bs, 3, H, D)).to(torch.bfloat16) for _ in range(L)]
    g = [-torch.nn.functional.softplus(rnd((G, Bs, H, D))) for _ in range(L)]
    beta = [torch.sigmoid(rnd((G, Bs, H))) for _ in range(L)]
    state = [rnd((Bs, H, D, D)) * 0.02 for _ in range(L)]
    ring = [rnd((Bs, 3, H, 3, D)).to(torch.bfloat16) for _ in range(L)]
    w = [rnd((3, H, D, 4)) * 0.5 for _ in range(L)]
    out = [torch.empty((G, Bs, H, D), dtype=torch.bfloat16, device=dev) for _ in range(L)]

    def run_steps():
        # each launch follows another layer's, which never writes this layer's
        # state: it may stream that state while the previous launch drains
        for t in range(G):
            for li in range(L):
                kda.kda_shortconv_decode_step_ex(x[li][t], ring[li], w[li], g[li][t], beta[li][t], state[li],
                                                 out[li][t], overlap_prev=True)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        run_steps()  # warm-up outside the graph
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_steps()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        graph.replay()
    b.record()
    torch.cuda.synchronize(dev)
    kda.kda_sync_status()
    ms_step = max_over_ranks(a.elapsed_time(b) / (replays * G), dev)
    by = L * (Bs * H * DEC_UNIT_BYTES + CONV_W_BYTES)
    del graph, x, g, beta, out

    # Upper bound: the same 69 x 8 sequences' states in one tensor, stepped by one fused launch (one set
    # of conv weights), so that no layer boundary stands between the heads
    Bu = L * Bs
    xu, ringu = rnd((Bu, 3, H, D)).to(torch.bfloat16), rnd((Bu, 3, H, 3, D)).to(torch.bfloat16)
    gu, betau = -torch.nn.functional.softplus(rnd((Bu, H, D))), torch.sigmoid(rnd((Bu, H)))
    stu, outu = rnd((Bu, H, D, D)) * 0.02, torch.empty((Bu, H, D), dtype=torch.bfloat16, device=dev)

    def one(st, i=0):
        kda.kda_shortconv_decode_step(xu, ringu, w[0], gu, betau, stu, outu, stream=st)
    cs = torch.cuda.current_stream(dev)
    for _ in range(3):
        one(cs)
    torch.cuda.synchronize(dev)
    ub_ms, _ = _graph_and_loop_ms(torch, dev, cs, one, 20, per_graph=10)
    kda.kda_sync_status()
    ub_ms = max_over_ranks(ub_ms, dev)
    by_ub = Bu * H * DEC_UNIT_BYTES + CONV_W_BYTES
    del xu, ringu, gu, betau, stu, outu
    return {"value": ws * by / (ms_step * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms_step,
            "upper_bound_single_launch": {
                "ms_per_step": ub_ms, "frac": by_ub / (ub_ms * 1e-3) / 1e9 / hbm_peak,
                "workload": f"the {Bu} sequences' states ({L} layers x {Bs}) in one [{Bu},{H},{D},{D}] tensor, one "
                            "fused launch per step with one layer's conv weights, CUDA graph of 10 steps"},
            "config": {"workload": f"full-stack decode: {L} layers x {Bs} sequences x {H} heads, d={D}, bf16 q/k/v, "
                                   f"fp32 state 3.3 GB, {L} fused launches per step in a CUDA graph of {G} steps, "
                                   f"each a programmatic dependent launch overlapping the previous layer's tail",
                       "steps_timed": replays * G},
            "roofline_hbm": {"achieved": by / (ms_step * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                             "frac": by / (ms_step * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": by}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stack", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
