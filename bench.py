#!/usr/bin/env python3
"""Benchmark of the GB300 4-bit MoE layer library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Default workload ``stack40-T16384+T1``: 40 independently seeded MoE layers of
Qwen3.6-35B-A3B's shape (18.2 GB of MLX affine 4-bit weights, residual add between
layers, no attention).  One step = one prefill pass of T=16384 tokens through the
40 layers plus one decode pass of T=1 token through the 40 layers, i.e. every step
of the layer's hot path (routing, permutation, grouped gate/up and down GEMMs,
combine, and the decode GEMVs).  Inputs are synthetic and seeded (``synth``).

``value`` is MoE-layer tokens/s: (16384 + 1) tokens x 40 layers / step time, timed
with CUDA events on the launching stream, inputs resident in HBM, max over ranks.
The weights read per step (18.2 GB) are far larger than L2, so no L2 flush is needed.
``e2e`` is the same metric through the C entry ``moe_stack_forward_host`` with the
input copied from pinned host memory and the output copied back inside the timed
region.  ``roofline`` is for the dominant kernel (the grouped gate/up GEMM; on the
decode-only workloads the fused decode kernel against HBM), timed live by the library's
event profiler during the timed steps.  ``cpu_baseline`` times the
CPU oracle on a bounded sample.  With N>1 (torchrun) every rank runs an independent
replica on its own GPU (weak scaling, no collective on the data path).

``--impl reference`` times the CPU oracle (the only reference that exists: the pages'
engine is Metal-only) on a bounded sample per step of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

METRIC = "MoE-layer tokens/s (prefill T=512..16K), decode µs/layer; % HBM/BF16 roofline"
UNIT = "layer-tokens/s"
FLOP_PER_TOKEN = 57_675_776          # per layer: 8 routed + 1 shared SwiGLU expert, router, shared gate
GATEUP_FLOP_PER_ROW = 2 * 2 * 512 * 2048
LAYER_BYTES = 455_806_976
EXPERT_BYTES = 1_769_472              # one expert: 3 packed 4-bit matrices + scales + biases
ROUTER_BYTES = 1_048_576 + 4_096      # router matrix + shared-expert gate vector

WORKLOADS = {
    "stack40-T16384+T1": dict(layers=40, T_prefill=16384, T_decode=1, skew=False),
    "layer-T4096-skew": dict(layers=1, T_prefill=4096, T_decode=0, skew=True),
    "layer-T4096": dict(layers=1, T_prefill=4096, T_decode=0, skew=False),
    "layer-T16384": dict(layers=1, T_prefill=16384, T_decode=0, skew=False),
    "layer-T8192": dict(layers=1, T_prefill=8192, T_decode=0, skew=False),
    "layer-T2048": dict(layers=1, T_prefill=2048, T_decode=0, skew=False),
    "layer-T1024": dict(layers=1, T_prefill=1024, T_decode=0, skew=False),
    "layer-decode-T1": dict(layers=1, T_prefill=0, T_decode=1, skew=False),
    "layer-decode-T8": dict(layers=1, T_prefill=0, T_decode=8, skew=False),
    "layer-T512": dict(layers=1, T_prefill=512, T_decode=0, skew=False),
    "layer-T32": dict(layers=1, T_prefill=32, T_decode=0, skew=False),
    "layer-T64": dict(layers=1, T_prefill=64, T_decode=0, skew=False),
    "layer-T256": dict(layers=1, T_prefill=256, T_decode=0, skew=False),
    "layer-T192": dict(layers=1, T_prefill=192, T_decode=0, skew=False),
    "layer-T128": dict(layers=1, T_prefill=128, T_decode=0, skew=False),
    "decode-T1": dict(layers=40, T_prefill=0, T_decode=1, skew=False),
    "decode-T8": dict(layers=40, T_prefill=0, T_decode=8, skew=False),
    # grouped-query decode attention alone (the full-attention layers' decode step)
    "gqa-decode-ctx4K-B8": dict(layers=0, T_prefill=0, T_decode=0, skew=False, gqa=(8, 4096)),
    "gqa-decode-ctx32K-B8": dict(layers=0, T_prefill=0, T_decode=0, skew=False, gqa=(8, 32768)),
}
DEFAULT_WORKLOAD = "stack40-T16384+T1"


def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time; every rank receives it."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank_step: int, steps: int, elapsed_ms: float) -> float:
    """Units all ranks processed (each rank its own replica's work) / the slowest rank's
    time: weak scaling, no data-path collective."""
    return world * units_per_rank_step * steps / (elapsed_ms / 1e3)


def make_hosts(wl):
    import synth
    n = wl["layers"]
    if n == 1:
        return [synth.make_layer(0, skew=wl["skew"])]
    with ThreadPoolExecutor(4) as ex:
        return list(ex.map(lambda l: synth.stack_layer(l, threads=2), range(n)))


def kernel_hash() -> str:
    """Hash of the gate/up kernel's source with comments and blank lines removed, so that a
    stored DRAM-traffic capture stays attached to the code it was taken on."""
    import re
    h = hashlib.sha256()
    for f in ("expert_gemm.cu", "common.cuh", "gemm_common.cuh"):
        src = open(os.path.join(ROOT, "bit_expert_layer_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in src.splitlines()]
        h.update("\n".join(ln for ln in lines if ln.strip()).encode())
    return h.hexdigest()[:16]


# The ncu DRAM-traffic record that holds a workload's gate/up launch: the stack's gate/up
# launch at T=16384 is the same kernel on the same token count as a single layer's, and
# the capture is taken on the single layer (a few GB on the device, not the 19 GB stack).
TRAFFIC_RECORD = {"stack40-T16384+T1": "layer-T16384", "layer-T16384": "layer-T16384"}


def load_traffic(workload: str):
    """DRAM bytes per gate/up launch from a committed ncu summary, if it was taken on the
    current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "gateup_traffic.json")
    try:
        d = json.load(open(p))
    except Exception:
        return None
    e = d.get(TRAFFIC_RECORD.get(workload, workload))
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("bytes_per_launch")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d["bf16_tflops_sustained"]), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "100", "-i", gpu_id], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return dict(sm_mhz=statistics.median(sm), sm_max_mhz=mx, reasons=sorted(reasons), samples=len(sm))


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), with the core count."""
    name = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                name = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not name:
        try:
            for ln in open("/proc/cpuinfo"):
                if ln.lower().startswith(("model name", "cpu part")):
                    name = ln.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return f"{name or 'unknown'} ({os.cpu_count()} logical CPUs)"


def oracle_sample(hosts, wl, n_prefill: int, n_decode: int, threads: int | None = None):
    """Time the CPU oracle on a bounded sample of the workload; returns (layer-tokens, s, threads)."""
    import synth
    from oracle import Oracle, default_threads
    o = Oracle()
    threads = threads or default_threads()
    n_layers = len(hosts)
    resid = n_layers > 1
    layer_tokens = 0
    t0 = time.perf_counter()
    for T, n in ((wl["T_prefill"], n_prefill), (wl["T_decode"], n_decode)):
        if T == 0 or n == 0:
            continue
        x = synth.make_x(0, T)[:n]
        for h in hosts:
            x = o.forward(h, x, residual=resid, nthreads=threads)["out"]
        layer_tokens += n * n_layers
    return layer_tokens, time.perf_counter() - t0, threads


def run_reference(args, wl):
    rank, world, _ = rank_info()
    if rank != 0:
        return 0
    from oracle import default_threads
    hosts = make_hosts(wl)
    n_pf = min(wl["T_prefill"], max(16, default_threads())) if wl["T_prefill"] else 0
    n_dc = 1 if wl["T_decode"] else 0
    for _ in range(args.warmup):
        oracle_sample(hosts[:1], wl, 1, 0 if n_pf else 1)
    tot_tokens, tot_s, threads = 0, 0.0, 1
    for _ in range(args.steps):
        n, s, threads = oracle_sample(hosts, wl, n_pf, n_dc)
        tot_tokens += n
        tot_s += s
    value = tot_tokens / tot_s
    sample = (f"per step: {n_pf} of the {wl['T_prefill']} prefill tokens and {n_dc} decode token(s) "
              f"through all {wl['layers']} layers on {threads} host threads; CPU: {cpu_model()}")
    line = dict(impl="reference", metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=1e3 * tot_s / args.steps, higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="f64", data="synthetic",
                config=dict(workload=args.workload, **wl),
                cpu_baseline=dict(value=value, unit=UNIT, cores=threads, kind="oracle", sample=sample),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)
    return 0


def use_burst_peak(clk) -> bool:
    """The burst bf16 peak applies when the sampled SM clock sat at its maximum with no
    power-cap sample (the conditions the burst figure was measured under); otherwise the
    sustained one does."""
    if not clk:
        return False
    return clk["sm_mhz"] >= 0.97 * clk["sm_max_mhz"] and "sw_power_cap" not in clk["reasons"]


def peak_reason(clk) -> str:
    if not clk:
        return "no clock samples"
    return (f"median SM clock {clk['sm_mhz']:.0f} of {clk['sm_max_mhz']:.0f} MHz, "
            f"{'power cap seen' if 'sw_power_cap' in clk['reasons'] else 'no power-cap sample'}")


def decode_bytes(layers, x0, resid: bool) -> int:
    """Algorithmic HBM bytes of one decode pass: per layer the touched experts (counted from
    the routing of that layer's actual input; the shared expert included), the router
    matrix and the shared gate."""
    import torch
    x = x0.clone()
    total = 0
    for L in layers:
        n_e = int(torch.unique(L.route(x)["idx"]).numel())
        total += (n_e + 1) * EXPERT_BYTES + ROUTER_BYTES
        if resid:
            x = L.forward(x, residual=True)
    torch.cuda.synchronize()
    return total


def time_configs(ml, dev, stream, stack, stack_layers, peaks, burst, steps: int = 10, warmup: int = 3):
    """Whole-layer time, tokens/s and roofline fraction of each single-layer configuration
    (CUDA events around the forward on the launching stream, a 256 MB L2 flush between
    steps, outside the events; median of `steps`), the 40-layer decode at T=8, and the
    grouped-query decode attention."""
    import torch
    import synth
    from bit_expert_layer_gb300 import _abi
    bf16 = peaks["bf16"] if burst else peaks["bf16_sustained"]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    host_u = synth.make_layer(0)
    host_s = synth.make_layer(0, skew=True)
    lay_u = ml.MoELayer(ml.DeviceWeights(host_u, dev), 4096)
    lay_s = ml.MoELayer(ml.DeviceWeights(host_s, dev), 4096)

    def timed(fn, pre=None):
        for _ in range(warmup):
            if pre:
                pre()
            fn()
            flush.zero_()
        ts = []
        for _ in range(steps):
            if pre:
                pre()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            flush.zero_()
            ts.append((a, b))
        torch.cuda.synchronize(dev)
        return statistics.median(a.elapsed_time(b) for a, b in ts)

    for name, layer, T in (("layer-T32", lay_u, 32), ("layer-T512", lay_u, 512), ("layer-T4096", lay_u, 4096),
                           ("layer-T4096-skew", lay_s, 4096)):
        x = torch.from_numpy(synth.make_x(0, T).view(np.int16)).to(dev).view(torch.bfloat16)
        y = torch.empty_like(x)
        ms = timed(lambda: layer.forward(x, out=y))
        assert layer.get_error() == 0
        n_e = int(torch.unique(layer.route(x)["idx"]).numel())
        hbm_bytes = (n_e + 1) * EXPERT_BYTES + ROUTER_BYTES + 2 * T * 2048 * 2
        tflops = FLOP_PER_TOKEN * T / (ms / 1e3) / 1e12
        gbs = hbm_bytes / (ms / 1e3) / 1e9
        out[name] = dict(us_per_layer=1e3 * ms, tokens_per_s=T / (ms / 1e3), tflops=tflops,
                         tensor_frac=tflops / bf16, hbm_bytes=hbm_bytes, hbm_gbs=gbs, hbm_frac=gbs / peaks["hbm"],
                         touched_experts=n_e,
                         bound="tensor" if FLOP_PER_TOKEN * T / (bf16 * 1e12) > hbm_bytes / (peaks["hbm"] * 1e9)
                         else "hbm")
    if stack is not None:
        T = 8
        xs = torch.from_numpy(synth.make_x(1, T).view(np.int16)).to(dev).view(torch.bfloat16)
        xw = torch.empty_like(xs)

        ms = timed(lambda: stack.forward_(xw), pre=lambda: xw.copy_(xs))
        assert stack_layers[0].get_error() == 0
        nb = decode_bytes(stack_layers, xs, True)
        gbs = nb / (ms / 1e3) / 1e9
        out["decode-T8"] = dict(us_per_layer=1e3 * ms / len(stack_layers), us_per_stack=1e3 * ms,
                                hbm_bytes_per_pass=nb, hbm_gbs=gbs, hbm_frac=gbs / peaks["hbm"], layers=len(stack_layers))
    # grouped-query decode attention (the full-attention layers' decode step): 8 sequences
    # of 4K and 32K cached positions, HBM-bound on the KV rows
    for name, S in (("gqa-decode-ctx4K-B8", 4096), ("gqa-decode-ctx32K-B8", 32768)):
        B = 8
        q, k, v, lens = synth.make_gqa(7, B, S)
        dv = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
        qd, kd, vd = dv(q), dv(k), dv(v)
        od = torch.empty_like(qd)
        nws = _abi.gqa_decode_workspace_bytes(B)
        gws = torch.zeros(nws, dtype=torch.uint8, device=dev)
        lens_l = [int(x) for x in lens]
        ms = timed(lambda: _abi.gqa_decode_attention(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), lens_l, B, S,
                                                     od.data_ptr(), gws.data_ptr(), nws, stream.cuda_stream))
        assert _abi.gqa_decode_get_error(gws.data_ptr()) == 0
        nb = B * 2 * S * 128 * 2 * 2 + 2 * B * 16 * 128 * 2
        gbs = nb / (ms / 1e3) / 1e9
        out[name] = dict(us=1e3 * ms, kv_bytes=nb, hbm_gbs=gbs, hbm_frac=gbs / peaks["hbm"], bound="hbm",
                         shape="16 query heads, 2 KV heads, head 128, bf16 KV cache")
        del kd, vd
    out["peak_bf16_tflops"] = bf16
    out["peak_hbm_gbs"] = peaks["hbm"]
    out["method"] = "median of 10 CUDA-event timings per configuration, 256 MB L2 flush between steps"
    del lay_u, lay_s
    return out


def cpu_baseline(hosts, wl, n_layers):
    """The oracle on the host cores: as many prefill tokens as host threads (and one
    decode token) through every layer on all threads, and one prefill token through every
    layer on one thread."""
    from oracle import default_threads
    threads = default_threads()
    n_pf = min(wl["T_prefill"], max(16, threads)) if wl["T_prefill"] else 0
    n_dc = 1 if wl["T_decode"] else 0
    n, s, threads = oracle_sample(hosts, wl, n_pf, n_dc, threads)
    n1, s1, _ = oracle_sample(hosts, wl, 1 if n_pf else 0, 0 if n_pf else 1, 1)
    return dict(value=n / s, unit=UNIT, cores=threads, kind="oracle",
                sample=f"{n_pf} prefill + {n_dc} decode tokens through all {n_layers} layers on {threads} threads "
                       f"({n} layer-tokens, {s:.1f} s)",
                one_thread=dict(value=n1 / s1, unit=UNIT,
                                sample=f"1 token through all {n_layers} layers on 1 thread ({s1:.1f} s)"),
                cpu=cpu_model())


def run_gqa(args, wl):
    """Grouped-query decode attention alone: one call per step over B sequences of S cached
    positions (16 query heads, 2 KV heads, head 128), CUDA events around each call on the
    launching stream, the KV cache (B * 2 * S * 512 bytes) read from HBM every step."""
    import torch

    import synth
    from bit_expert_layer_gb300 import _abi
    from bit_expert_layer_gb300.build import build
    rank, world, local = rank_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build()
    B, S = wl["gqa"]
    q, k, v, lens = synth.make_gqa(7, B, S)
    dv = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
    qd, kd, vd = dv(q), dv(k), dv(v)
    od = torch.empty_like(qd)
    nws = _abi.gqa_decode_workspace_bytes(B)
    ws = torch.zeros(nws, dtype=torch.uint8, device=dev)
    lens_l = [int(x) for x in lens]
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    call = lambda: _abi.gqa_decode_attention(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), lens_l, B, S, od.data_ptr(),
                                             ws.data_ptr(), nws, stream.cuda_stream)
    for _ in range(args.warmup):
        call()
        flush.zero_()
    torch.cuda.synchronize(dev)
    evs = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        flush.zero_()
        evs.append((a, b))
    torch.cuda.synchronize(dev)
    assert _abi.gqa_decode_get_error(ws.data_ptr()) == 0
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    peaks = load_peaks()
    nb = B * 2 * S * 128 * 2 * 2 + 2 * B * 16 * 128 * 2
    gbs = nb / (ms / 1e3) / 1e9
    line = dict(metric="GQA decode attention, µs per step", value=1e3 * ms, unit="us/step", n_gpus=1,
                steps=args.steps, warmup=args.warmup, ms_per_step=ms, higher_is_better=False, scaling="weak",
                vs_baseline=None, dtype="bf16", data="synthetic",
                config=dict(workload=args.workload, B=B, S=S, heads="16 query / 2 KV, head 128",
                            l2="256 MB L2 flush between steps (outside the events)"),
                roofline=dict(kernel="gqa_decode", bound="hbm", achieved=gbs, peak=peaks["hbm"], unit="GB/s",
                              frac=gbs / peaks["hbm"], traffic=None,
                              algorithmic=f"K and V rows read once: {nb} B per step"),
                gpu_launches=args.steps)
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    import synth
    from bit_expert_layer_gb300 import _abi
    from bit_expert_layer_gb300 import layer as ml
    from bit_expert_layer_gb300.build import build

    rank, world, local = rank_info()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build()
    if world > 1:
        dist.barrier()
    build()

    hosts = make_hosts(wl)
    Tp, Td, n_layers = wl["T_prefill"], wl["T_decode"], wl["layers"]
    Tmax = max(Tp, Td, 1)
    ws = ml.new_workspace(Tmax, dev)
    layers = [ml.MoELayer(ml.DeviceWeights(h, dev), Tmax, workspace=ws) for h in hosts]
    stack = ml.MoEStack(layers)
    resid = n_layers > 1
    stream = torch.cuda.current_stream(dev)

    def to_dev(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    xp_src = to_dev(synth.make_x(0, Tp)) if Tp else None
    xd_src = to_dev(synth.make_x(1, Td)) if Td else None
    xp = torch.empty_like(xp_src) if Tp else None
    xd = torch.empty_like(xd_src) if Td else None
    outp = torch.empty_like(xp_src) if (Tp and not resid) else None
    outd = torch.empty_like(xd_src) if (Td and not resid) else None
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if n_layers == 1 else None

    ev = lambda: torch.cuda.Event(enable_timing=True)
    part = {"prefill": [], "decode": []}

    def step(record: bool):
        if Tp:
            a, b = ev(), ev()
            xp.copy_(xp_src)
            a.record(stream)
            if resid:
                stack.forward_(xp)
            else:
                layers[0].forward(xp, out=outp)
            b.record(stream)
            if record:
                part["prefill"].append((a, b))
        if Td:
            a, b = ev(), ev()
            xd.copy_(xd_src)
            a.record(stream)
            if resid:
                stack.forward_(xd)
            else:
                layers[0].forward(xd, out=outd)
            b.record(stream)
            if record:
                part["decode"].append((a, b))
        if flush is not None:
            flush.zero_()      # single-layer workloads: evict the weights from L2 between steps

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize(dev)
    assert layers[0].get_error() == 0

    # ---------------- timed region (device)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    gpu_id = str(local)
    cvd = [c.strip() for c in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if c.strip()]
    if local < len(cvd):
        gpu_id = cvd[local]
    else:
        try:
            u = str(getattr(torch.cuda.get_device_properties(dev), "uuid", ""))
            if u:
                gpu_id = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
    clocks = ClockSampler(gpu_id)
    time.sleep(0.3)
    t0 = ev()
    t1 = ev()
    t0.record(stream)
    for _ in range(args.steps):
        step(True)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    # the same steps again with the library's per-launch events on (every launch bracketed
    # by two CUDA events on its stream): the per-kernel times and the roofline come from
    # this pass, the step time above from a pass without that instrumentation
    _abi.moe_profiler_read()
    _abi.moe_profiler_enable(True)
    for _ in range(args.steps):
        step(False)
    torch.cuda.synchronize(dev)
    _abi.moe_profiler_enable(False)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    if clk is not None:
        clk["gpu"] = gpu_id
    kern = _abi.moe_profiler_read()
    # with the single-layer flush the step total excludes the flush: sum the parts
    part_ms = {k: sum(a.elapsed_time(b) for a, b in v) for k, v in part.items()}
    elapsed_ms = t0.elapsed_time(t1) if flush is None else part_ms["prefill"] + part_ms["decode"]
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    status = layers[0].get_error()
    assert status == 0, f"device error word {status}"

    tokens_per_step = (Tp + Td) * n_layers
    value = job_throughput(world, tokens_per_step, args.steps, elapsed_ms)
    def call_launches(T):
        if not T:
            return 0
        if resid:
            return _abi.moe_stack_forward_launches([l.handle for l in layers], T)
        return _abi.moe_forward_launches(layers[0].handle, T)
    launches = args.steps * (call_launches(Tp) + call_launches(Td))

    # ---------------- e2e: host buffers through the C entry, copies inside the region
    e2e = None
    if resid:
        xh_p = torch.from_numpy(synth.make_x(0, Tp).view(np.int16)).pin_memory() if Tp else None
        oh_p = torch.empty_like(xh_p).pin_memory() if Tp else None
        xh_d = torch.from_numpy(synth.make_x(1, Td).view(np.int16)).pin_memory() if Td else None
        oh_d = torch.empty_like(xh_d).pin_memory() if Td else None

        def e2e_step():
            if Tp:
                stack.forward_host(xh_p, oh_p)
            if Td:
                stack.forward_host(xh_d, oh_d)

        e2e_step()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(args.steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(a.elapsed_time(b), world, dev)
        nbytes = (Tp + Td) * 2048 * 2
        e2e = dict(value=job_throughput(world, tokens_per_step, args.steps, e_ms), unit=UNIT,
                   h2d_bytes_per_step=nbytes, d2h_bytes_per_step=nbytes, ms_per_step=e_ms / args.steps)

    # ---------------- roofline of the dominant kernel
    peaks = load_peaks()
    burst = use_burst_peak(clk)
    bf16_peak = peaks["bf16"] if burst else peaks["bf16_sustained"]
    bf16_src = f"{peaks['src']} bf16 {'burst' if burst else 'sustained'} ({peak_reason(clk)})"
    roof = None
    gu_ms, gu_n = kern.get("gateup", (0.0, 0))
    if Tp and gu_n:
        flop = GATEUP_FLOP_PER_ROW * 9 * Tp
        achieved = flop / (gu_ms / gu_n / 1e3) / 1e12
        tb = load_traffic(args.workload)
        roof = dict(kernel="gateup", bound="tensor", achieved=achieved, peak=bf16_peak, unit="TFLOP/s",
                    frac=achieved / bf16_peak, traffic=tb,
                    algorithmic=f"{GATEUP_FLOP_PER_ROW} FLOP x 9T rows per launch (T={Tp})",
                    peak_source=bf16_src,
                    launch_time=f"{1e3 * gu_ms / gu_n:.1f} us: mean of {gu_n} gate/up launches, each between two "
                                f"CUDA events on its stream, in a second pass of the timed steps")
    dec = None
    dec_roof = None
    if Td:
        dms = part_ms["decode"] / args.steps
        dbytes = decode_bytes(layers, xd_src, resid)
        gbs = dbytes / (dms / 1e3) / 1e9
        dec = dict(us_per_layer=1e3 * dms / n_layers, us_per_stack=1e3 * dms,
                   hbm_bytes_per_pass=dbytes, hbm_gbs=gbs, hbm_frac=gbs / peaks["hbm"])
        dec_roof = dict(kernel="decode_layers", bound="hbm", achieved=gbs, peak=peaks["hbm"], unit="GB/s",
                        frac=gbs / peaks["hbm"], T=Td, us_per_layer=1e3 * dms / n_layers,
                        algorithmic=f"touched experts x {EXPERT_BYTES} B + {ROUTER_BYTES} B per layer, "
                                    f"{dbytes} B per pass of {n_layers} layer(s), T={Td}",
                        peak_source=f"{peaks['src']} HBM copy")
        if roof is None:
            roof = dict(dec_roof, traffic=None)

    # ---------------- the other configurations, timed in the same run (single layers with
    # an L2 flush between steps; decode at T=8 through the same 40-layer stack)
    cfg_block = None
    if rank == 0 and not args.no_configs and args.workload == DEFAULT_WORKLOAD:
        cfg_block = time_configs(ml, dev, stream, stack if resid else None, layers, peaks, burst)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(hosts, wl, n_layers)

    per_kernel = {k: dict(ms_avg=(v[0] / v[1]) if v[1] else None, launches=v[1], ms_total=v[0])
                  for k, v in kern.items() if v[1]}
    line = dict(
        metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps, warmup=args.warmup,
        ms_per_step=elapsed_ms / args.steps, higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="bf16", data="synthetic",
        config=dict(workload=args.workload, layers=n_layers, T_prefill=Tp, T_decode=Td, skew=wl["skew"],
                    weights="MLX affine 4-bit g64 (u4 codes, bf16 scale/bias); bf16 MMA, fp32 accumulate",
                    l2=("weights read per step larger than L2" if n_layers > 1 else
                        "256 MB L2 flush between steps (outside the events)"),
                    parallelism=f"replicas x{world}"),
        prefill_layer_tokens_per_s=(Tp * n_layers * args.steps / (part_ms["prefill"] / 1e3)) if Tp else None,
        prefill_tflops=(FLOP_PER_TOKEN * Tp * n_layers * args.steps / (part_ms["prefill"] / 1e3) / 1e12)
        if Tp else None,
        decode=dec, roofline=roof, decode_roofline=dec_roof, configs=cfg_block, cpu_baseline=cpu, e2e=e2e,
        gpu_launches=launches, clocks=clk, kernels=per_kernel,
    )
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def spawn_ranks(n: int, argv) -> int:
    """Run this script as n ranks of one node under torch.distributed.run (one rank per
    GPU, rendezvous on 127.0.0.1); returns the launcher's exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration block")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)      # at least 3 untimed warm-up steps
    wl = WORKLOADS[args.workload]
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return spawn_ranks(args.gpus, sys.argv[1:] if argv is None else list(argv))
    if "gqa" in wl:
        if args.impl == "reference":
            print(json.dumps(dict(impl="reference", unavailable="the attention workloads have no CPU-timed arm; "
                                                                "the default workload carries it")))
            return 0
        return run_gqa(args, wl)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
