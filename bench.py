#!/usr/bin/env python
"""Benchmark of the gated delta rule hot path on GB300.

One step = one chunked forward (gate cumsum and norms, UT transform,
inter-chunk recurrence, final-state write) over the headline workload
  B=4, H=16, L=2048, d_k=d_v=128, chunk 64, bf16 q/k/v, fp32 gates/state,
with inputs resident in HBM.  The decode half of the metric (64 successive
single-token steps on N=256, H=16, d=128, fp32 state) is measured in the same
run and reported under "decode".

Timing: W warm-up steps, then K timed steps, each bracketed by CUDA events on
the launching stream; the L2 cache is flushed (a 512 MiB buffer is written)
before every timed step, outside the events.  Under torchrun every rank runs
its own replica of the workload (independent sequences: weak scaling, no
collective on the data path); rank 0 prints the max over ranks.

--impl reference times the fp64 CPU oracle on the host cores instead, on the
same workload, and prints the same JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_delta_rule_12_gb300 import inputs  # noqa: E402

METRIC = "tokens/s chunked fwd (H=16,d=128,L=2048) + decode steps/s; % roofline"
PREFILL = "prefill_b4_h16_l2048_d128_bf16"
DECODE = "decode_n256_h16_d128_bf16"
MULTI_T = 4          # tokens per call of the multi-token decode line
PROLOGUE_K = 4       # short-convolution width of the prologue line
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["source"] = "measured"
        return d
    return dict(PEAKS_FALLBACK)


def prefill_algorithmic_bytes(w: inputs.Workload) -> int:
    """q, k, v, out once (element size s), g and beta fp32, states in/out once per sequence."""
    s = 2 if w.dtype == "bf16" else 4
    th = w.B * w.L * w.H
    per_th = (2 * w.dk + 2 * w.dv) * s + 8
    nseq = w.num_seqs if w.kind == "varlen" else w.B
    states = nseq * w.H * w.dv * w.dk * 4 * (2 if w.init_state else 1)
    return th * per_th + states


def prefill_algorithmic_flops(w: inputs.Workload) -> int:
    C = w.chunk_size
    return w.B * w.L * w.H * (2 * C * (3 * w.dk + 2 * w.dv) + 6 * w.dk * w.dv)


def decode_multi_algorithmic_bytes(w: inputs.Workload, T: int) -> int:
    """Per call of T tokens: the fp32 state read and written once, plus T tokens of q, k, v, out, g, beta."""
    s = 2 if w.dtype == "bf16" else 4
    nh = w.num_seqs * w.H
    return nh * (2 * w.dv * w.dk * 4 + T * ((2 * w.dk + 2 * w.dv) * s + 8))


def decode_algorithmic_bytes(w: inputs.Workload) -> int:
    """Per step: the fp32 state read and written once, plus q, k, v, out, g, beta."""
    s = 2 if w.dtype == "bf16" else 4
    nh = w.num_seqs * w.H
    return nh * (2 * w.dv * w.dk * 4 + (2 * w.dk + 2 * w.dv) * s + 8)


FP32_FMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12   # CUDA-core fp32 FMA rate at the maximum SM clock (nominal)


def prefill_roofline(w: inputs.Workload, ms: float, peaks, traffic=None, kernel: str = "") -> dict:
    """Roofline of one chunked-forward call: the time bound is the larger of the algorithmic bytes at
    the measured HBM bandwidth and the algorithmic FLOPs at the tensor (bf16 workloads) or fp32 FMA
    (fp32 workloads) peak; `frac` is that bound over the measured time."""
    nbytes = prefill_algorithmic_bytes(w)
    flops = prefill_algorithmic_flops(w)
    t_bytes = nbytes / (peaks["hbm_gbs"] * 1e9)
    fpeak = peaks["bf16_tflops"] if w.dtype == "bf16" else FP32_FMA_TFLOPS
    t_flops = flops / (fpeak * 1e12)
    t = ms * 1e-3
    if t_bytes >= t_flops:
        r = {"bound": "hbm", "achieved": nbytes / t / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        r = {"bound": "tensor" if w.dtype == "bf16" else "alu", "achieved": flops / t / 1e12, "peak": fpeak,
             "unit": "TFLOP/s"}
    r.update({"frac": max(t_bytes, t_flops) / t, "traffic": traffic, "algorithmic_bytes": nbytes,
              "algorithmic_flops": flops, "t_bytes_us": t_bytes * 1e6, "t_flops_us": t_flops * 1e6,
              "frac_bytes": t_bytes / t, "frac_flops": t_flops / t,
              "flop_peak_source": "measured bf16" if w.dtype == "bf16" else "nominal fp32 FMA (152 SMs x 128 lanes x 2 x 2.07 GHz)",
              "peak_source": peaks["source"]})
    if kernel:
        r["kernel"] = kernel
    return r


def bench_prefill_workload(name: str, dev, flush, stream, reps: int, peaks) -> dict:
    """One gdn_chunk_fwd call on another workload of the table (inputs resident in HBM, L2 flushed
    before each call, CUDA events on the launching stream, median of `reps`)."""
    import gated_delta_rule_12_gb300 as gdn
    w = inputs.WORKLOADS[name]
    host = inputs.make(w)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in host.items()}
    del host
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    B = w.B if w.kind != "varlen" else 1
    N = w.num_seqs if w.kind == "varlen" else w.B
    num_seqs = N if w.kind == "varlen" else 0
    out = torch.empty((B, w.L, w.H, w.dv), dtype=tdt, device=dev)
    sf = torch.empty((N, w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    work = torch.empty(gdn.chunk_fwd_workspace_size(B, w.L, w.H, w.dk, w.dv, num_seqs, tdt), dtype=torch.uint8,
                       device=dev)

    def call():
        gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], init_state=d["init_state"],
                      cu_seqlens=d["cu_seqlens"], scale=w.scale, use_qk_l2norm=True, out=out, final_state=sf,
                      workspace=work)

    for _ in range(3):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    t = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        torch.cuda.synchronize()
        t.append(a.elapsed_time(b))
    ms = statistics.median(t)
    launches = gdn.chunk_fwd_kernel_count(B, w.L, w.H, w.dk, w.dv, num_seqs, tdt)
    shape = {"B": B, "T": w.L, "H": w.H, "dk": w.dk, "dv": w.dv, "chunk": w.chunk_size, "dtype": w.dtype}
    if w.kind == "varlen":
        cu = d["cu_seqlens"].cpu().tolist()
        shape["lengths"] = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    del d, out, sf, work
    torch.cuda.empty_cache()
    return {"workload": name, "shape": shape, "unit": "tokens/s", "value": w.B * w.L / (ms * 1e-3) if w.kind != "varlen" else w.L / (ms * 1e-3),
            "ms_per_call": ms, "kernels_per_call": launches,
            "roofline": prefill_roofline(w, ms, peaks, kernel="one gdn_chunk_fwd call"),
            "timing": f"median of {reps} calls, L2 flushed (512 MiB write) before each"}


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons around the timed region.

    nvidia-smi polls every `interval_ms`; each line is stamped with the host
    clock.  The timed region of one step is far shorter than a poll, so the
    summary keeps the samples within `margin_s` of the region (the bench marks
    its start and end with `mark()`), and the sampler is started, and has
    produced its first line, before the warm-up steps run.
    """
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: int = 50, margin_s: float = 0.5):
        self.index = index
        self.interval_ms = interval_ms
        self.margin_s = margin_s
        self.proc = None
        self.lines = []
        self.marks = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            t0 = time.monotonic()
            while not self.lines and time.monotonic() - t0 < 5.0:
                time.sleep(0.01)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark(self):
        self.marks.append(time.monotonic())

    def __exit__(self, *exc):
        if self.proc is not None:
            # one more poll after the region ends
            t0 = time.monotonic()
            while time.monotonic() - t0 < 3 * self.interval_ms / 1e3:
                time.sleep(0.01)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo = (min(self.marks) - self.margin_s) if self.marks else float("-inf")
        hi = (max(self.marks) + self.margin_s) if self.marks else float("inf")
        for ts, ln in self.lines:
            if not (lo <= ts <= hi):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        window = (f"nvidia-smi every {self.interval_ms} ms, samples within {self.margin_s} s of the timed region"
                  if self.marks else f"nvidia-smi every {self.interval_ms} ms")
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "window": window}


def traffic_record(kernel: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel source is unchanged since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        rec = json.load(open(p)).get(kernel)
    except (ValueError, OSError):
        return None
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if h != rec.get("source_sha256_16"):
        return None
    return rec.get("dram_bytes_per_launch")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def make_group(ws):
    if ws <= 1:
        return None
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world_size: int, ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time (ms)."""
    return units_per_rank * world_size / (ms * 1e-3)


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def bench_ours(args):
    import gated_delta_rule_12_gb300 as gdn
    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = make_group(ws_n)
    gdn.load_library()
    dev = torch.device("cuda", local)
    peaks = load_peaks()

    w = inputs.WORKLOADS[PREFILL]
    host = inputs.make(w)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in host.items()}
    out = torch.empty((w.B, w.L, w.H, w.dv), dtype=torch.bfloat16, device=dev)
    sf = torch.empty((w.B, w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    wsz = gdn.chunk_fwd_workspace_size(w.B, w.L, w.H, w.dk, w.dv, 0, torch.bfloat16)
    work = torch.empty(wsz, dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], init_state=d["init_state"], scale=w.scale,
                      use_qk_l2norm=True, out=out, final_state=sf, workspace=work)

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            flush.zero_()
            step()
        torch.cuda.synchronize()
        barrier(dist)
        torch.cuda.synchronize()
        clk.mark()
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        clk.mark()
    barrier(dist)
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    ms = max_over_ranks(dist, ms)
    clocks = clk.summary()

    tokens = w.B * w.L
    value = job_throughput(tokens, ws_n, ms)
    algo_bytes = prefill_algorithmic_bytes(w)
    achieved = algo_bytes / (ms * 1e-3) / 1e9
    launches_per_step = gdn.chunk_fwd_kernel_count(w.B, w.L, w.H, w.dk, w.dv, 0, torch.bfloat16)

    # end to end through the C ABI with host buffers: pinned H2D of the inputs,
    # the call, D2H of the outputs, every step
    pin = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in host.items()}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    sf_h = torch.empty(sf.shape, dtype=sf.dtype).pin_memory()
    names = ["q", "k", "v", "g", "beta"]
    h2d = sum(pin[n].numel() * pin[n].element_size() for n in names)
    d2h = out_h.numel() * out_h.element_size() + sf_h.numel() * sf_h.element_size()

    def e2e_step():
        for n in names:
            d[n].copy_(pin[n], non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)
        sf_h.copy_(sf, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(dist, e0.elapsed_time(e1) / args.steps)

    # the same steps as a serving loop would run them: step i+1's inputs are copied in while step i
    # computes and step i-1's outputs are copied out (two device buffer sets, one stream per copy
    # direction, events between them); every step still moves its own inputs in and outputs out
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    bufs = [dict({n: torch.empty_like(d[n]) for n in names}, out=torch.empty_like(out), sf=torch.empty_like(sf))
            for _ in range(2)]
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def pipelined(nsteps: int):
        for i in range(nsteps):
            b, bf = i % 2, bufs[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[b])   # step i-2 has read this buffer set
                for n in names:
                    bf[n].copy_(pin[n], non_blocking=True)
                in_done[b].record(s_in)
            stream.wait_event(in_done[b])
            if i >= 2:
                stream.wait_event(out_done[b])      # step i-2's outputs have left this buffer set
            gdn.chunk_fwd(bf["q"], bf["k"], bf["v"], bf["g"], bf["beta"], init_state=d["init_state"],
                          scale=w.scale, use_qk_l2norm=True, out=bf["out"], final_state=bf["sf"], workspace=work)
            comp_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                out_h.copy_(bf["out"], non_blocking=True)
                sf_h.copy_(bf["sf"], non_blocking=True)
                out_done[b].record(s_out)
        stream.wait_stream(s_out)

    pipelined(max(args.warmup, 2))
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    pipelined(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1) / args.steps)

    # decode half of the metric
    wd = inputs.WORKLOADS[DECODE]
    dh = inputs.make(wd)
    dd = {k: v.to(dev) for k, v in dh.items()}
    state = dd["state0"].clone()
    dout = torch.empty((wd.num_seqs, wd.H, wd.dv), dtype=torch.bfloat16, device=dev)

    def decode_all():
        for t in range(wd.steps):
            gdn.decode_step(state, dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t],
                            scale=wd.scale, use_qk_l2norm=True, out=dout)

    for _ in range(max(1, args.warmup)):
        decode_all()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        decode_all()
    graph.replay()
    torch.cuda.synchronize()
    reps = max(3, args.steps // 4)
    t_ms = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        t_ms.append(a.elapsed_time(b) / wd.steps)
    dms = max_over_ranks(dist, statistics.median(t_ms))
    dbytes = decode_algorithmic_bytes(wd)
    d_ach = dbytes / (dms * 1e-3) / 1e9

    # The same steps over two state sets in turn (two batches of the workload served alternately):
    # a step never reads the state the step before it wrote, so none of it can still sit in the
    # 129 MB L2 and every state byte of the roofline comes from DRAM.
    state2 = [dd["state0"].clone(), dd["state0"].clone()]

    def decode_alt():
        for t in range(wd.steps):
            gdn.decode_step(state2[t % 2], dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t],
                            scale=wd.scale, use_qk_l2norm=True, out=dout)

    decode_alt()
    torch.cuda.synchronize()
    agraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(agraph):
        decode_alt()
    agraph.replay()
    torch.cuda.synchronize()
    a_ms = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        agraph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        a_ms.append(a.elapsed_time(b) / wd.steps)
    dms_cold = max_over_ranks(dist, statistics.median(a_ms))
    del state2, agraph

    # several tokens per call: the same 64 tokens as MULTI_T tokens x (64 / MULTI_T) calls,
    # the state read and written once per call
    tmaj = lambda x: x.transpose(0, 1).contiguous()          # [steps, N, ...] -> [N, steps, ...]
    dm = {k2: tmaj(dd[k2]) for k2 in ("q", "k", "v", "g", "beta")}
    calls = wd.steps // MULTI_T
    mstate = dd["state0"].clone()
    mout = torch.empty((wd.num_seqs, MULTI_T, wd.H, wd.dv), dtype=torch.bfloat16, device=dev)
    msl = [{k2: dm[k2][:, c * MULTI_T:(c + 1) * MULTI_T].contiguous() for k2 in dm} for c in range(calls)]

    def decode_multi_all():
        for c in range(calls):
            x = msl[c]
            gdn.decode_multi(mstate, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=wd.scale, out=mout)

    for _ in range(max(1, args.warmup)):
        decode_multi_all()
    torch.cuda.synchronize()
    mgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(mgraph):
        decode_multi_all()
    mgraph.replay()
    torch.cuda.synchronize()
    m_ms = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        mgraph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        m_ms.append(a.elapsed_time(b) / calls)
    mms = max_over_ranks(dist, statistics.median(m_ms))
    mbytes = decode_multi_algorithmic_bytes(wd, MULTI_T)
    m_ach = mbytes / (mms * 1e-3) / 1e9

    # the same calls over two state sets in turn (see decode_alt)
    mstate2 = [dd["state0"].clone(), dd["state0"].clone()]

    def decode_multi_alt():
        for c in range(calls):
            x = msl[c]
            gdn.decode_multi(mstate2[c % 2], x["q"], x["k"], x["v"], x["g"], x["beta"], scale=wd.scale, out=mout)

    decode_multi_alt()
    torch.cuda.synchronize()
    magraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(magraph):
        decode_multi_alt()
    magraph.replay()
    torch.cuda.synchronize()
    ma_ms = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        magraph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ma_ms.append(a.elapsed_time(b) / calls)
    mms_cold = max_over_ranks(dist, statistics.median(ma_ms))
    del mstate2, magraph

    # backward of the chunked forward on the bench shape
    bwd = bench_backward(w, d, dev, flush, stream, reps, peaks)
    bwd["value"] = job_throughput(w.B * w.L, ws_n, max_over_ranks(dist, bwd["ms_per_call"]))

    # block prologue (short conv + SiLU for q, k, v; gate activations) on the bench shape
    pro = bench_prologue(w, dev, flush, stream, reps, peaks)
    pro["value"] = job_throughput(w.B * w.L, ws_n, max_over_ranks(dist, pro["ms_per_call"]))

    # the block prologue fused into the chunked forward, against the two calls
    fused = bench_prologue_chunk(w, dev, flush, stream, reps, peaks)
    fused["value"] = job_throughput(w.B * w.L, ws_n, max_over_ranks(dist, fused["ms_per_call"]))

    # the other chunked-forward workloads of the table (parity cases, timed here too)
    others = {}
    for key, name in (("small_f32", "prefill_b1_h2_l256_d64_f32"), ("varlen", "varlen_t32768_h16_d128_bf16"),
                      ("large", "prefill_b8_h32_l8192_dk128_dv256_bf16")):
        others[key] = bench_prefill_workload(name, dev, flush, stream, max(5, reps), peaks)
        tokens_w = others[key]["value"] * others[key]["ms_per_call"] * 1e-3
        others[key]["value"] = job_throughput(tokens_w, ws_n, max_over_ranks(dist, others[key]["ms_per_call"]))

    if rank == 0:
        cpu = cpu_baseline(w) if ws_n == 1 else None
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws_n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": PREFILL, "B": w.B, "T": w.L, "H": w.H, "dk": w.dk, "dv": w.dv,
                       "chunk": w.chunk_size, "tokens_per_step": tokens, "l2": "flushed (512 MiB write) before each timed step",
                       "parallelism": f"replicas x{ws_n}"},
            "roofline": prefill_roofline(w, ms, peaks, traffic=traffic_record("chunk_fwd"),
                                         kernel="one gdn_chunk_fwd call (ut_tc_kernel + recur_tc_kernel)"),
            "e2e": {"value": job_throughput(tokens, ws_n, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "mode": "pipelined: step i+1's inputs in and step i-1's outputs out while step i computes",
                    "serial": {"value": job_throughput(tokens, ws_n, e2e_serial_ms), "unit": "tokens/s",
                               "ms_per_step": e2e_serial_ms,
                               "mode": "copy in, call, copy out, one stream, one step after another"}},
            "decode": {"workload": DECODE, "value": job_throughput(1, ws_n, dms), "unit": "steps/s",
                       "tokens_per_s": job_throughput(wd.num_seqs, ws_n, dms), "ms_per_step": dms,
                       "roofline": {"bound": "hbm", "achieved": d_ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": d_ach / peaks["hbm_gbs"], "traffic": traffic_record("decode"),
                                    "algorithmic_bytes": dbytes},
                       "timing": f"{wd.steps} steps in one CUDA graph, median of {reps}",
                       "l2_cold": {"ms_per_step": dms_cold, "frac": dbytes / (dms_cold * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                   "how": "the same steps over two state sets in turn, so no step reads a state "
                                          "still in L2 from the step before"}},
            "decode_multi": {"workload": DECODE, "tokens_per_call": MULTI_T,
                             "value": job_throughput(wd.num_seqs * MULTI_T, ws_n, mms), "unit": "tokens/s",
                             "ms_per_call": mms,
                             "roofline": {"bound": "hbm", "achieved": m_ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                          "frac": m_ach / peaks["hbm_gbs"], "algorithmic_bytes": mbytes},
                             "timing": f"{wd.steps} tokens as {calls} calls in one CUDA graph, median of {reps}",
                             "l2_cold": {"ms_per_call": mms_cold,
                                         "frac": mbytes / (mms_cold * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                         "how": "the same calls over two state sets in turn"}},
            "prologue": pro,
            "prologue_chunk_fwd": fused,
            "backward": bwd,
            **others,
            "gpu_launches": args.steps * launches_per_step,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def bench_backward(w: inputs.Workload, d, dev, flush, stream, reps: int, peaks):
    """One gdn_chunk_bwd call on the workload (inputs resident, L2 flushed before each call)."""
    import gated_delta_rule_12_gb300 as gdn
    gen = torch.Generator().manual_seed(w.seed + 200)
    dO = torch.randn((w.B, w.L, w.H, w.dv), generator=gen).to(torch.bfloat16).to(dev)
    dS = torch.randn((w.B, w.H, w.dv, w.dk), generator=gen).to(dev)
    need = gdn.load_library().gdn_chunk_bwd_workspace_size(w.B, w.L, w.H, w.dk, w.dv, 0, gdn.GDN_BF16)
    work = torch.empty(need, dtype=torch.uint8, device=dev)

    def call():
        gdn.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], dO, init_state=d["init_state"], dfinal_state=dS,
                      scale=w.scale, workspace=work)

    for _ in range(2):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    t = []
    for _ in range(max(3, reps)):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        torch.cuda.synchronize()
        t.append(a.elapsed_time(b))
    ms = statistics.median(t)
    s = 2
    per_th = (2 * w.dk + 2 * w.dv) * s + 8 + (2 * w.dk + w.dv) * s + 8   # q, k, v, dO, g, beta in; dq, dk, dv, dg, dbeta out
    nbytes = w.B * w.L * w.H * per_th + 2 * w.B * w.H * w.dv * w.dk * 4
    ach = nbytes / (ms * 1e-3) / 1e9
    # bf16 with dk = dv = 128: prep, the chunk-local and saving-recurrence pair of the forward scan,
    # the reverse scan and the local kernel
    return {"workload": PREFILL, "unit": "tokens/s", "ms_per_call": ms, "kernels": 5,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"], "algorithmic_bytes": nbytes},
            "timing": f"median of {max(3, reps)} calls, L2 flushed before each"}


def bench_prologue(w: inputs.Workload, dev, flush, stream, reps: int, peaks, K: int = PROLOGUE_K):
    """One gdn_prologue call on the workload's shape: raw projections in, q, k, v, g, beta out."""
    import gated_delta_rule_12_gb300 as gdn
    gen = torch.Generator().manual_seed(w.seed + 100)
    rn = lambda *shape: torch.randn(shape, generator=gen, dtype=torch.float32)
    B, T, H, dk, dv = w.B, w.L, w.H, w.dk, w.dv
    x = [rn(B, T, H, dk).to(torch.bfloat16).to(dev), rn(B, T, H, dk).to(torch.bfloat16).to(dev),
         rn(B, T, H, dv).to(torch.bfloat16).to(dev)]
    wts = [(0.5 * rn(H, dk, K)).to(dev), (0.5 * rn(H, dk, K)).to(dev), (0.5 * rn(H, dv, K)).to(dev)]
    ab = [rn(B, T, H).to(dev), rn(B, T, H).to(dev)]
    par = [(0.5 * rn(H)).to(dev), (0.5 * rn(H)).to(dev)]
    s_in = torch.zeros((B, K - 1, H, 2 * dk + dv), dtype=torch.bfloat16, device=dev)
    s_out = torch.empty_like(s_in)
    outs = (torch.empty_like(x[0]), torch.empty_like(x[1]), torch.empty_like(x[2]),
            torch.empty((B, T, H), dtype=torch.float32, device=dev),
            torch.empty((B, T, H), dtype=torch.float32, device=dev))

    def call():
        gdn.prologue(*x, *wts, *ab, *par, conv_state_in=s_in, conv_state_out=s_out, out=outs)

    for _ in range(3):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    t = []
    for _ in range(max(reps, 5)):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        torch.cuda.synchronize()
        t.append(a.elapsed_time(b))
    ms = statistics.median(t)
    nbytes = B * T * H * ((2 * dk + dv) * 2 * 2 + 16) + 2 * B * (K - 1) * H * (2 * dk + dv) * 2
    ach = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"{PREFILL} projections, conv width {K}", "unit": "tokens/s", "ms_per_call": ms,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"], "traffic": traffic_record("prologue"),
                         "algorithmic_bytes": nbytes},
            "timing": f"median of {max(reps, 5)} calls, L2 flushed before each"}


def bench_prologue_chunk(w: inputs.Workload, dev, flush, stream, reps: int, peaks, K: int = PROLOGUE_K):
    """gdn_prologue_chunk_fwd (the block prologue fused into the chunked forward) on the workload's shape,
    against gdn_prologue followed by gdn_chunk_fwd on the same projections."""
    import gated_delta_rule_12_gb300 as gdn
    gen = torch.Generator().manual_seed(w.seed + 300)
    rn = lambda *shape: torch.randn(shape, generator=gen, dtype=torch.float32)
    B, T, H, dk, dv = w.B, w.L, w.H, w.dk, w.dv
    x = [rn(B, T, H, dk).to(torch.bfloat16).to(dev), rn(B, T, H, dk).to(torch.bfloat16).to(dev),
         rn(B, T, H, dv).to(torch.bfloat16).to(dev)]
    wts = [(0.5 * rn(H, dk, K)).to(dev), (0.5 * rn(H, dk, K)).to(dev), (0.5 * rn(H, dv, K)).to(dev)]
    ab = [rn(B, T, H).to(dev), rn(B, T, H).to(dev)]
    par = [(0.5 * rn(H) - 1.0).to(dev), (0.5 * rn(H)).to(dev)]
    s_in = torch.zeros((B, K - 1, H, 2 * dk + dv), dtype=torch.bfloat16, device=dev)
    s_out = torch.empty_like(s_in)
    s0 = torch.zeros((B, H, dv, dk), dtype=torch.float32, device=dev)
    out = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device=dev)
    sf = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    ws_f = torch.empty(int(gdn.load_library().gdn_prologue_chunk_fwd_workspace_size(B, T, H, dk, dv, 0, gdn.GDN_BF16)),
                       dtype=torch.uint8, device=dev)
    ws_s = torch.empty(gdn.chunk_fwd_workspace_size(B, T, H, dk, dv, 0, torch.bfloat16), dtype=torch.uint8, device=dev)
    mid = (torch.empty_like(x[0]), torch.empty_like(x[1]), torch.empty_like(x[2]),
           torch.empty((B, T, H), dtype=torch.float32, device=dev), torch.empty((B, T, H), dtype=torch.float32, device=dev))

    def fused():
        gdn.prologue_chunk_fwd(*x, *wts, *ab, *par, conv_state_in=s_in, conv_state_out=s_out, init_state=s0,
                               scale=w.scale, out=out, final_state=sf, workspace=ws_f)

    def separate():
        q, k, v, g, beta = gdn.prologue(*x, *wts, *ab, *par, conv_state_in=s_in, conv_state_out=s_out, out=mid)
        gdn.chunk_fwd(q, k, v, g, beta, init_state=s0, scale=w.scale, out=out, final_state=sf, workspace=ws_s)

    def timed(fn):
        for _ in range(3):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        t = []
        for _ in range(max(reps, 5)):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            t.append(a.elapsed_time(b))
        return statistics.median(t)

    ms_f, ms_s = timed(fused), timed(separate)
    th = B * T * H
    # algorithmic bytes of the fused call: projections and gate projections in, out, the states once
    nbytes = th * ((2 * dk + dv) * 2 + 8 + dv * 2) + 2 * B * (K - 1) * H * (2 * dk + dv) * 2 + 2 * B * H * dv * dk * 4
    # the separate calls also write q, k, v, g, beta and read them back
    extra = 2 * th * ((2 * dk + dv) * 2 + 8)
    ach = nbytes / (ms_f * 1e-3) / 1e9
    return {"workload": f"{PREFILL} from projections, conv width {K}", "unit": "tokens/s",
            "value": B * T / (ms_f * 1e-3), "ms_per_call": ms_f, "separate_ms_per_call": ms_s,
            "separate_value": B * T / (ms_s * 1e-3),
            "algorithmic_bytes": nbytes, "bytes_not_moved_vs_separate": extra,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"], "algorithmic_bytes": nbytes},
            "timing": f"median of {max(reps, 5)} calls each, L2 flushed before each"}


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(w: inputs.Workload, host=None, seqs=1, heads=None):
    """A bounded sample of the workload: `seqs` sequences x `heads` heads, full length."""
    host = host if host is not None else inputs.make(w)
    hs = heads or w.H
    sel = lambda t: t[:seqs, :, :hs].contiguous()
    return {k: sel(host[k]) for k in ("q", "k", "v", "g", "beta")}, seqs * w.L * hs


def cpu_baseline(w: inputs.Workload, host=None, budget_s: float = 10.0):
    """The fp64 oracle on the host cores over the whole workload, repeated for about `budget_s`."""
    import oracle
    s, token_heads = oracle_sample(w, host, seqs=w.B)

    def one_pass() -> float:
        t0 = time.perf_counter()
        oracle.recurrent_fwd(s["q"], s["k"], s["v"], s["g"], s["beta"], scale=w.scale, use_qk_l2norm=True)
        return time.perf_counter() - t0

    dt = one_pass()
    reps = max(1, int(budget_s / dt))   # the first pass sizes the sample
    dt += sum(one_pass() for _ in range(reps - 1))
    cores = min(oracle.num_threads(), w.B * w.H)
    # one host core: one sequence of the workload (all heads), one pass
    s1, th1 = oracle_sample(w, host, seqs=1)
    t0 = time.perf_counter()
    oracle.recurrent_fwd(s1["q"], s1["k"], s1["v"], s1["g"], s1["beta"], scale=w.scale, use_qk_l2norm=True,
                         nthreads=1)
    dt1 = time.perf_counter() - t0
    return {"value": token_heads / w.H * reps / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"the whole workload ({w.B} x {w.L} tokens x {w.H} heads), fp64 recurrence, "
                      f"{reps} passes in {dt:.1f} s",
            "single_core": {"value": th1 / w.H / dt1, "unit": "tokens/s", "cores": 1,
                            "sample": f"one sequence ({w.L} tokens x {w.H} heads), one pass in {dt1:.2f} s"}}


def bench_reference(args):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = inputs.WORKLOADS[PREFILL]
    host = inputs.make(w)
    s, token_heads = oracle_sample(w, host, seqs=w.B)
    cores = min(oracle.num_threads(), w.B * w.H)

    def step():
        oracle.recurrent_fwd(s["q"], s["k"], s["v"], s["g"], s["beta"], scale=w.scale, use_qk_l2norm=True)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = token_heads / w.H / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": PREFILL, "B": w.B, "T": w.L, "H": w.H, "dk": w.dk, "dv": w.dv, "chunk": w.chunk_size},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: the whole workload ({w.B} x {w.L} tokens x {w.H} heads), fp64 recurrence"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
