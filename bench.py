#!/usr/bin/env python3
"""MoE-layer forward benchmark on B300.

One step = one pass of the whole layer (route -> capacity dispatch -> grouped
SwiGLU experts (up, down) -> combine) over one batch of synthetic tokens: one
moe_forward call through the C ABI.  The headline value times K such steps; a
second loop runs the same layer as separate stage calls with CUDA events
between them for the per-kernel breakdown and roofline; a third runs
moe_forward end to end from pinned host buffers.
Default workload: the Mixtral-shaped layer at prefill size, bf16, T=16384,
d=4096, E=8, d_ff=14336, top-2 softmax renormalised, per-expert logit offsets
(the largest configuration, where the grouped expert GEMM is bound by the tensor
cores; its 2.8 GB of expert weights and 0.4 GB of tokens exceed the 126 MB L2).
After the headline, every other workload is measured once the same way and
reported under "per_config" (tokens/s, layer-roofline fraction, grouped-GEMM
TFLOP/s, per-stage device time and GB/s, SM clock).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--T T]
    python bench.py --impl reference ...     # the CPU oracle on the same workload
    python bench.py --stage S --workload W   # one stage alone (route | dispatch |
                                             # ffn | combine), e.g. under ncu

Prints one JSON line (rank 0).  With N > 1 (torchrun), every rank runs its own
replica on its own batch (no data exchange; the layer is replicated, tokens are
independent), timing is the max over ranks, value = all ranks' tokens / time.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "MoE-layer fwd tokens/s; grouped-GEMM TFLOP/s as % of B300 bf16 peak"
DEFAULT_WORKLOAD = "mixtral_T16384"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
STAGES = ("route", "dispatch", "ffn", "combine")
# workloads of the per_config table (the headline's own is skipped there)
PER_CONFIG = ("tiny_top2_fp32", "switch_top1_cap1.25", "mixtral_T16", "mixtral_T256", "mixtral_T4096",
              "mixtral_T16384", "deepseek_v3", "expert_choice_zipf")
# the same layers with the up projection on E4M3 operands (MOE_BF16_FP8UP), beside them
PER_CONFIG_FP8UP = ("switch_top1_cap1.25", "mixtral_T4096", "mixtral_T16384", "deepseek_v3")
KERNEL_SOURCES = {   # files whose content defines each stage's kernels (for the ncu traffic record)
    # moe_api.cu holds the default tile-group shares that set the FFN's tile order
    "ffn": ["csrc/ffn_tcgen05.cu", "csrc/tc_gemm.cuh", "csrc/tc_common.cuh", "csrc/moe_internal.cuh",
            "csrc/moe_api.cu"],
    "route": ["csrc/route.cu", "csrc/route_tcgen05.cu", "csrc/tc_gemm.cuh", "csrc/tc_common.cuh"],
    "dispatch": ["csrc/dispatch.cu"],
    "combine": ["csrc/combine.cu"],
}


# ------------------------------------------------------------------------------------ helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def layer_config(wl, ws_n):
    """The layer both arms run (the `config` of the JSON line, before measured keys)."""
    return {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "d_ff": wl.f, "k": wl.k, "gate": wl.gate,
            "mode": wl.mode, "capacity_factor": wl.capacity_factor, "ec_capacity": wl.ec_capacity,
            "n_shared": wl.n_shared, "f_shared": wl.f_shared,
            "expert_weights": {"fp8w": "e4m3 + fp32 scale per output channel",
                               "fp8up": "W1|W3 e4m3 + scale per channel, x e4m3 + scale per token, W2 bf16"}.get(
                                   wl.dtype, wl.dtype),
            "drop_policy": wl.drop_policy,
            "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "single GPU"}


def kernel_hash(stage):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[stage]:
        with open(os.path.join(ROOT, "mixture_experts_sparse_gemm_b300", rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(stage, workload):
    """DRAM bytes per launch from the committed ncu record, if the kernel source
    still matches the one that was profiled; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_hash(stage)
    with open(path) as fh:
        for line in fh:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == stage and parts[1] == workload:
                if parts[3] == want:
                    return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background;
    window(t_lo, t_hi) summarises the samples inside one timed region."""
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, bus_id=None):
        self.bus_id = bus_id
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu=timestamp,{self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def _rows(self):
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                c = [x.strip() for x in line.split(",")]
                if len(c) < 11:
                    continue
                if self.bus_id and self.bus_id.lower() not in c[2].lower():
                    continue
                try:
                    ts = datetime.datetime.strptime(c[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                rows.append((ts, c))
        return rows

    def window(self, t_lo, t_hi):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = self._rows()
        win = [c for ts, c in rows if t_lo - 0.25 <= ts <= t_hi + 0.25]
        if not win:   # a region shorter than the sampling period: the nearest sample
            near = sorted(rows, key=lambda r: abs(r[0] - 0.5 * (t_lo + t_hi)))[:1]
            win = [c for _, c in near]
        sm = [float(r[3]) for r in win if r[3].replace(".", "").isdigit()]
        mx = [float(r[4]) for r in win if r[4].replace(".", "").isdigit()]
        pw = [float(r[5]) for r in win if r[5].replace(".", "").isdigit()]
        reasons = sorted({self.REASONS[i] for r in win for i in range(4) if r[7 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(win)}

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()

    def close(self):
        self.stop()
        try:
            os.unlink(self.f.name)
        except OSError:
            pass


def pci_bus(dev):
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
        return f"{bus:02x}:" if isinstance(bus, int) else None
    except Exception:
        return None


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(v, device=None):
    """Largest value over the ranks of the default process group (v itself alone)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, tokens_per_rank, steps, max_ms):
    """Whole-job tokens/s of `world` replicas that each ran `steps` steps of
    `tokens_per_rank` tokens, the slowest rank taking `max_ms`."""
    return world * tokens_per_rank * steps / (max_ms * 1e-3)


# ------------------------------------------------------------------------------------ work model
def work_model(wl, off, E_used):
    """Algorithmic bytes and FLOPs per stage launch (bf16 b = 2 or fp32 b = 4).
    A = assignments computed; touched = experts with at least one row."""
    b = 4 if wl.dtype == "f32" else 2
    bw = 1 if wl.dtype == "fp8w" else b   # bytes per stored expert weight (E4M3 codes)
    up8 = wl.dtype == "fp8up"             # E4M3 up projection: W1|W3 one byte, W2 bf16
    T, d, E, f = wl.T, wl.d, wl.E, wl.f
    A = int(off[-1])
    touched = int(E_used)
    kslots = wl.k if wl.mode == "tc" else E
    fs = wl.n_shared * wl.f_shared
    Ts = T if wl.n_shared else 0
    m = {}
    m["route"] = {"bytes": T * d * b + d * E * b + (T * wl.k * 8 if wl.mode == "tc" else 3 * T * E * 4 + E * wl.ec_capacity * 8),
                  "flops": 2 * T * d * E}
    m["dispatch"] = {"bytes": (T * wl.k * 4 * 3 if wl.mode == "tc" else E * wl.ec_capacity * 4 + T * E * 4) + 2 * A * d * b,
                     "flops": 0}
    # grouped experts (up + down): touched weights, x_perm read, H written and read, Y written
    # (FP8 weights: one byte per weight plus one fp32 scale per output channel)
    sc = 4 * (2 * f + d) if wl.dtype == "fp8w" else 0
    scs = 4 * (2 * fs + d) if (wl.dtype == "fp8w" and fs) else 0
    m["ffn"] = {"bytes": touched * (3 * d * f * bw + sc) + 2 * A * d * b + 2 * A * f * b
                         + (3 * d * fs * bw + scs + 2 * Ts * d * b + 2 * Ts * fs * b),
                "flops": 6 * A * d * f + 6 * Ts * d * fs}
    if up8:
        # weights: E4M3 W1|W3 + one scale per column, bf16 W2; rows: the stage quantises
        # x_perm (and x) to E4M3 (read bf16, write codes), the up tiles read the codes
        m["ffn"]["bytes"] = (touched * (2 * d * f + 4 * 2 * f + d * f * 2) + A * d * (2 + 1 + 1) + 2 * A * f * 2
                             + A * d * 2 + (2 * d * fs + 4 * 2 * fs + d * fs * 2 + Ts * d * (2 + 1 + 1)
                                            + 2 * Ts * fs * 2 + Ts * d * 2))
        # the up FLOPs run at twice the bf16 rate: their bf16-equivalent count is half
        m["ffn"]["flops_bf16_equiv"] = 4 * A * d * f + 4 * Ts * d * fs
    m["combine"] = {"bytes": A * d * b + T * kslots * 8 + T * d * b + Ts * d * b, "flops": 2 * A * d}
    return m, A, touched


# ------------------------------------------------------------------------------------ our arm
_WEIGHT_KEYS = ("W1", "W3", "W2", "W1s", "W3s", "W2s")


class LayerRun:
    """One layer on the device: seeded inputs, packed expert weights, the stage
    buffers, and the C-ABI calls of one step.  keep_weights=False frees the
    unpacked expert weights once they are packed (the layer only reads the packed
    copy)."""

    def __init__(self, wl, dev, keep_weights=False):
        from mixture_experts_sparse_gemm_b300 import binding as B
        from mixture_experts_sparse_gemm_b300.layer import MoELayer
        self.B = B
        self.wl = wl
        self.dev = dev
        self.stream = torch.cuda.current_stream()
        self.inp = make_inputs(wl, dev)
        i = self.inp
        self.cfg = B.config_from_workload(wl)
        self.layer = MoELayer(self.cfg, i["W1"], i["W3"], i["W2"], i.get("W1s"), i.get("W3s"), i.get("W2s"))
        if not keep_weights:
            for k in _WEIGHT_KEYS:
                i.pop(k, None)
        T, d = wl.T, wl.d
        dt = self.layer.dtype
        ec = wl.mode == "ec"
        sel = (wl.E, wl.ec_capacity) if ec else (T, wl.k)
        slots = (T, wl.E) if ec else (T, wl.k)
        self.idx = torch.empty(sel, dtype=torch.int32, device=dev)
        self.gw = torch.empty(sel, dtype=torch.float32, device=dev)
        self.off = torch.empty(wl.E + 1, dtype=torch.int32, device=dev)
        self.cnt = torch.empty(wl.E, dtype=torch.int32, device=dev)
        self.slot_of = torch.empty(slots, dtype=torch.int32, device=dev)
        self.x_perm = torch.empty(self.layer.rows_routed, d, dtype=dt, device=dev)
        self.Y = torch.empty(self.layer.rows_total, d, dtype=dt, device=dev)
        self.y = torch.empty(T, d, dtype=dt, device=dev)
        self.ws = {s: self.layer.workspace(s) for s in (B.MOE_STAGE_ROUTE, B.MOE_STAGE_DISPATCH,
                                                      B.MOE_STAGE_GROUPED_FFN, B.MOE_STAGE_FORWARD)}

    @property
    def x(self):
        return self.inp["x"]

    def forward(self, s=None, x=None, y=None):
        i, B = self.inp, self.B
        B.moe_forward(self.cfg, self.x if x is None else x, i["W_r"], i["logit_offset"], i["sel_bias"],
                      self.layer.packed, self.y if y is None else y, self.ws[B.MOE_STAGE_FORWARD],
                      self.stream if s is None else s)

    def stage_calls(self):
        """The four stage calls of one step, each taking the stream to enqueue on."""
        i, B, c = self.inp, self.B, self.cfg
        return {
            "route": lambda s: B.moe_route(c, self.x, i["W_r"], i["logit_offset"], i["sel_bias"], self.idx, self.gw,
                                           self.ws[B.MOE_STAGE_ROUTE], s),
            "dispatch": lambda s: B.moe_dispatch(c, self.idx, self.x, self.off, self.cnt, self.slot_of, self.x_perm,
                                                 self.ws[B.MOE_STAGE_DISPATCH], s, self.gw),
            "ffn": lambda s: B.moe_grouped_ffn(c, self.x_perm, self.off, self.layer.packed, self.x, self.Y,
                                               self.ws[B.MOE_STAGE_GROUPED_FFN], s),
            "combine": lambda s: B.moe_combine(c, self.Y, self.slot_of, self.gw, self.y, None, s),
        }

    def staged_step(self, ev=None):
        """One step as the four stage calls, an event before and after each when given."""
        calls = self.stage_calls()
        for j, name in enumerate(STAGES):
            if ev is not None:
                ev[j].record(self.stream)
            calls[name](self.stream)
        if ev is not None:
            ev[len(STAGES)].record(self.stream)

    def work(self):
        """Work model of the step the stage buffers hold (after a staged step)."""
        offs = self.off.cpu().numpy()
        return work_model(self.wl, offs, int((np.diff(offs) > 0).sum()))


def time_calls(fn, n, stream):
    """Device milliseconds of n calls of fn() on `stream` (CUDA events, synchronised)."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def graph_call_us(fn_s, stream, n_cap=10, budget_s=0.2, max_reps=50):
    """Device microseconds per call of fn_s(stream): n_cap back-to-back calls
    captured in a CUDA graph on a side stream and replayed (no host launch gaps;
    the inputs of a stage stay where the previous call left them, in L2 when they
    fit)."""
    cs = torch.cuda.Stream()
    cs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        for _ in range(n_cap):
            fn_s(cs)
    with torch.cuda.stream(cs):
        g.replay()
        one = time_calls(g.replay, 1, cs)
        reps = int(max(1, min(max_reps, budget_s * 1e3 / max(one, 1e-3))))
        ms = time_calls(g.replay, reps, cs)
    del g
    return ms / (reps * n_cap) * 1e3


def stage_table(stage_s, model, peaks):
    """Per-stage achieved GB/s and TFLOP/s and the fraction of the stage's bound
    (HBM copy bandwidth, or for a compute-bound expert stage the bf16 peak)."""
    bw = peaks["hbm_gbs"]
    out = {}
    for s in STAGES:
        t = stage_s[s]
        gbs = model[s]["bytes"] / t / 1e9
        tfl = model[s]["flops"] / t / 1e12
        t_mem = model[s]["bytes"] / (bw * 1e9)
        t_cmp = model[s]["flops"] / (peaks["bf16_tflops"] * 1e12)
        bound = "tensor" if (s == "ffn" and t_cmp > t_mem) else "hbm"
        out[s] = {"us": round(t * 1e6, 2), "GB/s": round(gbs, 1), "TFLOP/s": round(tfl, 2), "bound": bound,
                  "frac": round(gbs / bw if bound == "hbm" else tfl / peaks["bf16_tflops"], 4)}
    return out


def layer_roofline_ms(model, peaks):
    layer_bytes = sum(model[s]["bytes"] for s in STAGES)
    flops = model["ffn"].get("flops_bf16_equiv", model["ffn"]["flops"])
    return max(flops / (peaks["bf16_tflops"] * 1e12), layer_bytes / (peaks["hbm_gbs"] * 1e9)) * 1e3, layer_bytes


def measure_config(wl, dev, peaks, clocks):
    """One workload measured on its own: moe_forward timed over ~0.4 s of steps,
    then each stage replayed from a CUDA graph.  Returns the per_config entry."""
    run = LayerRun(wl, dev)
    B, st = run.B, run.stream
    for _ in range(3):
        run.forward()
    run.staged_step()
    est = time_calls(run.forward, 3, st) / 3
    K = int(min(2000, max(10, 400.0 / max(est, 1e-3))))
    t_lo = time.time()
    ms = time_calls(run.forward, K, st)
    t_hi = time.time()
    clk = clocks.window(t_lo, t_hi)
    B.moe_check_device_error(st)
    calls = run.stage_calls()
    stage_us = {s: graph_call_us(calls[s], st) for s in STAGES}
    B.moe_check_device_error(st)
    model, A, touched = run.work()
    step_ms = ms / K
    roof_ms, layer_bytes = layer_roofline_ms(model, peaks)
    ffn_s = stage_us["ffn"] * 1e-6
    gemm_tf = model["ffn"]["flops"] / ffn_s / 1e12
    entry = {
        "T": wl.T, "steps": K, "ms_per_step": round(step_ms, 5), "tokens_per_s": round(wl.T / (step_ms * 1e-3), 1),
        "assignments_computed": A, "experts_touched": touched,
        "layer_roofline": {"ms": round(roof_ms, 5), "frac": round(roof_ms / step_ms, 4)},
        "grouped_gemm": {"tflops": round(gemm_tf, 2), "pct_bf16_peak": round(100 * gemm_tf / peaks["bf16_tflops"], 2)},
        "stage_device": stage_table({s: stage_us[s] * 1e-6 for s in STAGES}, model, peaks),
        "sm_mhz": clk["sm_mhz"], "clock_reasons": clk["reasons"],
        "ms_x_mhz": round(step_ms * clk["sm_mhz"], 1) if clk["sm_mhz"] else None,
        "launches_per_step": B.moe_launch_count(run.cfg, B.MOE_STAGE_FORWARD),
    }
    del run, calls
    torch.cuda.empty_cache()
    return entry


def run_gpu(args):
    from mixture_experts_sparse_gemm_b300 import binding as B
    from mixture_experts_sparse_gemm_b300 import build as build_mod

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        build_mod.build()
    if ws_n > 1:
        dist.barrier()
    B.lib()

    wl = WORKLOADS[args.workload]
    if args.T:
        wl = wl.with_(T=args.T)
    if args.fp8_weights:
        wl = wl.with_(dtype="fp8w")
    if args.fp8_up:
        wl = wl.with_(dtype="fp8up")
    if args.affinity_drop:
        wl = wl.with_(drop_policy="affinity")
    if ws_n > 1:   # each replica gets its own batch of tokens
        wl = wl.with_(index=wl.index + 1000 * rank) if rank else wl
    want_cpu = rank == 0 and ws_n == 1 and not args.no_cpu_baseline
    run = LayerRun(wl, dev, keep_weights=want_cpu)
    stream = run.stream
    T, d = wl.T, wl.d
    peaks, peak_src = load_peaks()
    clocks = ClockSampler(pci_bus(dev))

    def barrier():
        if ws_n > 1:
            dist.barrier()

    def slowest(v):
        return max_over_ranks(v, dev)

    # ---- headline timed region: K layer forwards through moe_forward, inputs resident
    K = args.steps
    for _ in range(args.warmup):
        run.forward()
        run.staged_step()
    torch.cuda.synchronize()
    B.moe_check_device_error(stream)
    barrier()
    t_lo = time.time()
    total_ms = slowest(time_calls(run.forward, K, stream))
    t_hi = time.time()
    barrier()
    clk = clocks.window(t_lo, t_hi)
    B.moe_check_device_error(stream)

    # ---- the same forward captured once in a CUDA graph and replayed K times (the
    # library never synchronises the host, so a serving loop can capture it): the
    # kernels are the same, only the launch overhead between them differs
    try:
        cap_s = torch.cuda.Stream()
        cap_s.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap_s):
            run.forward(cap_s)
        torch.cuda.synchronize()
        with torch.cuda.stream(cap_s):
            for _ in range(max(3, args.warmup)):
                g.replay()
            g_ms = slowest(time_calls(g.replay, K, cap_s))
        B.moe_check_device_error(stream)
        graph = {"ms_per_step": round(g_ms / K, 5), "value": round(replica_throughput(ws_n, T, K, g_ms), 1),
                 "unit": "tokens/s"}
        del g
    except Exception as ex:   # capture unsupported here: report why
        graph = {"unavailable": str(ex).splitlines()[0][:200]}

    # ---- stage breakdown: the same layer as separate C-ABI stage calls, CUDA events
    # between them on the launching stream (the roofline of each kernel comes from here)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        run.staged_step(evs[i])
    torch.cuda.synchronize()
    staged_ms = evs[0][0].elapsed_time(evs[K - 1][len(STAGES)]) / K
    stage_ms = {s: float(np.mean([evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)]))
                for j, s in enumerate(STAGES)}
    B.moe_check_device_error(stream)
    model, A, touched = run.work()

    # ---- per-stage device time without host launch gaps (graph replay of each stage)
    try:
        calls = run.stage_calls()
        stage_dev_us = {s: graph_call_us(calls[s], stream) for s in STAGES}
        B.moe_check_device_error(stream)
        stage_device = stage_table({s: stage_dev_us[s] * 1e-6 for s in STAGES}, model, peaks)
        stage_device["method"] = ("10 back-to-back calls of the stage replayed from a CUDA graph; "
                                  "route/dispatch/combine inputs L2-warm between calls")
    except Exception as ex:   # capture unsupported here: report why
        stage_device = {"unavailable": str(ex).splitlines()[0][:200]}

    # ---- load statistics (outside the timed regions): the router with its score sums,
    # and the statistics kernel, each averaged over a short loop of its own
    E = wl.E
    psum = torch.empty(E, dtype=torch.float32, device=dev)
    frac = torch.empty(E, dtype=torch.float32, device=dev)
    pmean = torch.empty(E, dtype=torch.float32, device=dev)
    summary = torch.empty(5, dtype=torch.float64, device=dev)
    i_, ws_r = run.inp, run.ws[B.MOE_STAGE_ROUTE]

    def route(prob_sum=None):
        B.moe_route(run.cfg, run.x, i_["W_r"], i_["logit_offset"], i_["sel_bias"], run.idx, run.gw, ws_r, stream,
                    prob_sum)

    for _ in range(3):
        route(psum)
    route_plain_ms = time_calls(route, 20, stream) / 20
    route_probs_ms = time_calls(lambda: route(psum), 20, stream) / 20
    run.stage_calls()["dispatch"](stream)
    stats_ms = time_calls(lambda: B.moe_load_stats(run.cfg, run.idx, run.cnt, psum, frac, pmean, summary, stream),
                          20, stream) / 20
    B.moe_check_device_error(stream)
    load_stats = {"route_ms": round(route_plain_ms, 5), "route_with_prob_sum_ms": round(route_probs_ms, 5),
                  "stats_kernel_ms": round(stats_ms, 5),
                  "lif": round(float(summary[0]), 4), "cv": round(float(summary[1]), 4),
                  "router_entropy": round(float(summary[2]), 4), "switch_aux": round(float(summary[3]), 4),
                  "expert_balance": round(float(summary[4]), 4)}

    # ---- end to end through the C ABI with host buffers (pinned): every step copies its
    # tokens host -> device, runs moe_forward and copies its output device -> host.  The
    # copies of neighbouring steps overlap the compute on their own streams (double
    # buffers), as a serving loop would run it.
    dt = run.layer.dtype
    x_host = [run.x.cpu().pin_memory(), run.x.cpu().pin_memory()]
    y_host = [torch.empty(T, d, dtype=dt).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(run.x) for _ in range(2)]
    y_dev = [torch.empty_like(run.y) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n):
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[b])          # step i-2 finished reading x_dev[b]
                x_dev[b].copy_(x_host[b], non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])             # step i-2's output has left y_dev[b]
            run.forward(x=x_dev[b], y=y_dev[b])
            ev_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                y_host[b].copy_(y_dev[b], non_blocking=True)
                ev_out[b].record(s_out)

    e2e_steps(args.warmup)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    e2e_steps(K)
    e1.record(s_out)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = slowest(e0.elapsed_time(e1))
    B.moe_check_device_error(stream)
    del x_host, y_host, x_dev, y_dev

    # ---- work model and roofline of the dominant kernel
    stage_info = stage_table({s: stage_ms[s] * 1e-3 for s in STAGES}, model, peaks)
    for s in STAGES:
        stage_info[s]["ms"] = round(stage_ms[s], 5)
    dom = max(STAGES, key=lambda s: stage_ms[s])
    di = stage_info[dom]
    if di["bound"] == "hbm":
        bw = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": di["GB/s"], "peak": bw, "unit": "GB/s", "frac": round(di["GB/s"] / bw, 4)}
        peak_kind = "copy bandwidth"
    else:
        # the denominator matching the clock the kernel ran at: the burst bf16 figure
        # when the timed region held the maximum SM clock, the power-capped sustained
        # figure when the clock sat lower
        capped = clk.get("sm_mhz") and clk.get("sm_max_mhz") and clk["sm_mhz"] < 0.95 * clk["sm_max_mhz"]
        key = "bf16_tflops_sustained" if capped else "bf16_tflops"
        p = peaks[key]
        roof = {"bound": "tensor", "achieved": di["TFLOP/s"], "peak": p, "unit": "TFLOP/s",
                "frac": round(di["TFLOP/s"] / p, 4)}
        peak_kind = ("sustained bf16 (timed region under the power cap)" if capped
                     else "burst bf16 (timed region at the maximum SM clock)")
    roof["kernel"] = dom
    roof["peak_source"] = (f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'}), "
                           f"{peak_kind}")
    roof["traffic"] = recorded_traffic(dom, wl.name + {"fp8up": "+fp8up", "fp8w": "+fp8w"}.get(wl.dtype, ""))
    roof["algorithmic_bytes_per_launch"] = model[dom]["bytes"]
    roof["algorithmic_flops_per_launch"] = model[dom]["flops"]

    step_ms = total_ms / K
    gemm_flops = model["ffn"]["flops"]
    gemm_tflops = gemm_flops / (stage_ms["ffn"] * 1e-3) / 1e12
    roof_ms, layer_bytes = layer_roofline_ms(model, peaks)
    value = replica_throughput(ws_n, T, K, total_ms)
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": ws_n,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"bf16": "bf16", "f32": "f32", "fp8w": "bf16 (E4M3 expert weights)",
                  "fp8up": "bf16 (E4M3 up projection)"}[wl.dtype],
        "data": "synthetic (seeded; random-init expert weights)",
        "config": {**layer_config(wl, ws_n),
                   "assignments_computed": A, "experts_touched": touched,
                   "l2": "inputs larger than L2: the expert weights read per step exceed 126 MB"
                         if touched * 3 * d * wl.f * run.x.element_size() > 126e6 else "working set fits L2"},
        "grouped_gemm": {"tflops": round(gemm_tflops, 2),
                         "pct_bf16_peak": round(100 * gemm_tflops / peaks["bf16_tflops"], 2),
                         "bf16_peak_tflops": peaks["bf16_tflops"], "flops_per_step": gemm_flops},
        "layer_roofline": {"ms": round(roof_ms, 5), "frac": round(roof_ms / step_ms, 4),
                           "bytes_per_step": layer_bytes, "flops_per_step": gemm_flops},
        "stages": stage_info,
        "staged_ms_per_step": round(staged_ms, 5),
        "stage_device": stage_device,
        "graph_replay": graph,
        "load_stats": load_stats,
        "roofline": roof,
        "e2e": {"value": round(replica_throughput(ws_n, T, K, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": T * d * run.x.element_size(),
                "d2h_bytes_per_step": T * d * run.y.element_size(),
                "ms_per_step": round(e2e_ms / K, 5)},
        "gpu_launches": K * B.moe_launch_count(run.cfg, B.MOE_STAGE_FORWARD),
        "clocks": {**clk, "ms_x_mhz": round(step_ms * clk["sm_mhz"], 1) if clk.get("sm_mhz") else None},
    }
    inp = run.inp
    del run
    torch.cuda.empty_cache()
    if want_cpu:
        out["cpu_baseline"] = cpu_baseline(wl, inp, args.cpu_tokens, args.cpu_budget)
    del inp
    torch.cuda.empty_cache()

    # ---- every other workload, measured once the same way (single GPU only)
    if ws_n == 1 and not args.no_per_config:
        per = {}
        for name in PER_CONFIG:
            if name == wl.name:
                continue
            try:
                per[name] = measure_config(WORKLOADS[name], dev, peaks, clocks)
            except Exception as ex:   # report, keep the headline
                per[name] = {"error": str(ex).splitlines()[0][:200]}
                torch.cuda.empty_cache()
        for name in PER_CONFIG_FP8UP:
            key = name + "+fp8up"
            try:
                per[key] = measure_config(WORKLOADS[name].with_(dtype="fp8up"), dev, peaks, clocks)
            except Exception as ex:   # report, keep the headline
                per[key] = {"error": str(ex).splitlines()[0][:200]}
                torch.cuda.empty_cache()
        out["per_config"] = {"method": "moe_forward timed over about 0.4 s of steps (CUDA events); stages from "
                                       "CUDA-graph replays of 10 calls; fractions of MEASURED_PEAKS.json "
                                       "(burst bf16, copy bandwidth); sm_mhz = median nvidia-smi SM clock "
                                       "during the forward loop; '+fp8up' = the same layer with the up "
                                       "projection on E4M3 operands (MOE_BF16_FP8UP)", **per}
    clocks.close()
    if ws_n > 1:
        dist.destroy_process_group()
    return out if rank == 0 else None


# ------------------------------------------------------------------------------------ one stage alone
def run_stage(args):
    """One stage of the layer called --steps times after --warmup calls, with only
    the buffers it needs on the device (the small captures of ncu).  Prints the
    stage's device time per call and its achieved bandwidth against the work model."""
    from mixture_experts_sparse_gemm_b300 import binding as B
    from mixture_experts_sparse_gemm_b300 import build as build_mod
    from mixture_experts_sparse_gemm_b300.layer import MoELayer
    build_mod.build()
    B.lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = WORKLOADS[args.workload]
    if args.T:
        wl = wl.with_(T=args.T)
    if args.fp8_weights:
        wl = wl.with_(dtype="fp8w")
    if args.fp8_up:
        wl = wl.with_(dtype="fp8up")
    S = args.stage
    st = torch.cuda.current_stream()
    cfg = B.config_from_workload(wl)
    need_w = S == "ffn"
    inp = make_inputs(wl, dev, weights=need_w)
    layer = None
    if need_w:
        layer = MoELayer(cfg, inp["W1"], inp["W3"], inp["W2"], inp.get("W1s"), inp.get("W3s"), inp.get("W2s"))
        for k in _WEIGHT_KEYS:
            inp.pop(k, None)
        torch.cuda.empty_cache()

    def ws(stage):
        n = B.moe_workspace_size(cfg, stage)
        return torch.empty(max(n, 1), dtype=torch.uint8, device=dev)

    ec = wl.mode == "ec"
    sel = (wl.E, wl.ec_capacity) if ec else (wl.T, wl.k)
    idx = torch.empty(sel, dtype=torch.int32, device=dev)
    gw = torch.empty(sel, dtype=torch.float32, device=dev)
    ws_r = ws(B.MOE_STAGE_ROUTE)
    x, Wr, lo, sb = inp["x"], inp["W_r"], inp["logit_offset"], inp["sel_bias"]
    B.moe_route(cfg, x, Wr, lo, sb, idx, gw, ws_r, st)
    rows_routed, rows_total = B.moe_buffer_rows(cfg)
    off = torch.zeros(wl.E + 1, dtype=torch.int32, device=dev)
    fn = lambda: B.moe_route(cfg, x, Wr, lo, sb, idx, gw, ws_r, st)   # noqa: E731
    if S != "route":
        cnt = torch.empty(wl.E, dtype=torch.int32, device=dev)
        slot_of = torch.empty((wl.T, wl.E) if ec else (wl.T, wl.k), dtype=torch.int32, device=dev)
        x_perm = torch.empty(rows_routed, wl.d, dtype=x.dtype, device=dev)
        ws_d = ws(B.MOE_STAGE_DISPATCH)
        B.moe_dispatch(cfg, idx, x, off, cnt, slot_of, x_perm, ws_d, st, gw)
        fn = lambda: B.moe_dispatch(cfg, idx, x, off, cnt, slot_of, x_perm, ws_d, st, gw)   # noqa: E731
        if S == "ffn":
            Y = torch.empty(rows_total, wl.d, dtype=x.dtype, device=dev)
            ws_f = ws(B.MOE_STAGE_GROUPED_FFN)
            fn = lambda: B.moe_grouped_ffn(cfg, x_perm, off, layer.packed, x, Y, ws_f, st)   # noqa: E731
        elif S == "combine":
            # the combine's input rows: seeded values in the expert outputs' place
            # (the stage's traffic and time do not depend on them)
            Y = torch.empty(rows_total, wl.d, dtype=x.dtype, device=dev).normal_()
            y = torch.empty(wl.T, wl.d, dtype=x.dtype, device=dev)
            fn = lambda: B.moe_combine(cfg, Y, slot_of, gw, y, None, st)   # noqa: E731
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    B.moe_check_device_error(st)
    ms = time_calls(fn, args.steps, st)
    B.moe_check_device_error(st)
    offs = off.cpu().numpy()
    model, A, touched = work_model(wl, offs, int((np.diff(offs) > 0).sum()))
    peaks, peak_src = load_peaks()
    t = ms * 1e-3 / args.steps
    m = model[S]
    return {"stage": S, "workload": wl.name, "calls": args.steps, "us_per_call": round(t * 1e6, 3),
            "launches_per_call": B.moe_launch_count(cfg, {"route": B.MOE_STAGE_ROUTE, "dispatch": B.MOE_STAGE_DISPATCH,
                                                          "ffn": B.MOE_STAGE_GROUPED_FFN,
                                                          "combine": B.MOE_STAGE_COMBINE}[S]),
            "algorithmic_bytes": m["bytes"], "algorithmic_flops": m["flops"],
            "GB/s": round(m["bytes"] / t / 1e9, 1), "frac_hbm": round(m["bytes"] / t / 1e9 / peaks["hbm_gbs"], 4),
            "TFLOP/s": round(m["flops"] / t / 1e12, 2),
            "frac_bf16_burst": round(m["flops"] / t / 1e12 / peaks["bf16_tflops"], 4),
            "peaks": f"{peak_src}", "note": "back-to-back calls on one stream; inputs stay in L2 when they fit"}


# ------------------------------------------------------------------------------------ oracle arms
def _oracle_host_inputs(wl, inp):
    """Host fp32 copies of the workload (exact run-dtype values) for the oracle."""
    h = {}
    for k, v in inp.items():
        h[k] = None if v is None else np.ascontiguousarray(v.detach().float().cpu().numpy())
    return h


def _oracle_setup(oracle, wl, h):
    """Routing and capacity dispatch of the whole batch, once: which slots are
    dropped depends on the global token order, so the sampled steps reuse it."""
    if wl.mode == "ec":
        tok, w, _ = oracle.route_ec(h["x"], h["W_r"], wl.ec_capacity, h["logit_offset"])
        return {"ec_tok": tok, "ec_w": w}
    idx, w, _ = oracle.route_tc(h["x"], h["W_r"], wl.k, wl.gate, h["logit_offset"], h["sel_bias"], wl.renorm)
    cap = oracle.capacity(wl.capacity_factor, wl.T, wl.k, wl.E)
    _, _, slot, _ = oracle.dispatch_tc(idx, wl.E, cap)
    return {"idx": idx, "w": w, "slot": slot, "cap": cap}


def _oracle_step(oracle, wl, h, st, tokens):
    """One oracle step over a token sample, one thread: the sample's routing
    (scores and top-k, or the Expert Choice affinities and a proportional
    column top-cap), the capacity dispatch of the batch, then experts + combine
    for the sample.  Returns seconds."""
    t0 = time.perf_counter()
    xs = h["x"][tokens]
    if wl.mode == "ec":
        cap = max(1, wl.ec_capacity * len(tokens) // wl.T)
        oracle.route_ec(xs, h["W_r"], cap, h["logit_offset"])
        oracle.forward_ec_streamed(h["x"], st["ec_tok"], st["ec_w"], h["W1"], h["W3"], h["W2"], tokens,
                                   h.get("W1s"), h.get("W3s"), h.get("W2s"))
    else:
        oracle.route_tc(xs, h["W_r"], wl.k, wl.gate, h["logit_offset"], h["sel_bias"], wl.renorm)
        oracle.dispatch_tc(st["idx"], wl.E, st["cap"])
        oracle.forward_tc_streamed(h["x"], st["idx"], st["w"], st["slot"], h["W1"], h["W3"], h["W2"], tokens,
                                   h.get("W1s"), h.get("W3s"), h.get("W2s"))
    return time.perf_counter() - t0


def _sample_tokens(wl, n, seed=20261202):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(wl.T, size=min(max(1, n), wl.T), replace=False)).astype(np.int64)


def _sample_text(wl, n):
    return (f"fp64 C oracle, 1 thread; per step a seeded sample of {n} of the {wl.T} tokens: their routing, "
            f"the capacity dispatch of the batch, their experts + combine; tokens/s = sample tokens / step time")


def cpu_baseline(wl, inp, max_tokens, budget_s):
    """The oracle, as it stands, on 1 host thread, on a seeded token sample of the
    same batch sized to about budget_s seconds (at most max_tokens tokens)."""
    import oracle
    oracle.build()
    h = _oracle_host_inputs(wl, inp)
    st = _oracle_setup(oracle, wl, h)
    probe = _sample_tokens(wl, 2, seed=1)
    per_tok = _oracle_step(oracle, wl, h, st, probe) / len(probe)
    n = int(max(4, min(max_tokens, budget_s / max(per_tok, 1e-9))))
    toks = _sample_tokens(wl, n)
    dt = _oracle_step(oracle, wl, h, st, toks)
    return {"value": round(len(toks) / dt, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": _sample_text(wl, len(toks)) + f" ({dt:.1f} s)", "host_cpus": os.cpu_count()}


def run_reference(args):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    wl = WORKLOADS[args.workload]
    if args.T:
        wl = wl.with_(T=args.T)
    inp = make_inputs(wl, "cpu")
    h = _oracle_host_inputs(wl, inp)
    del inp
    st = _oracle_setup(oracle, wl, h)
    # size the per-step sample so that warm-up + timed steps take about args.ref_budget seconds
    probe = _sample_tokens(wl, 4, seed=1)
    per_tok = _oracle_step(oracle, wl, h, st, probe) / len(probe)
    n = int(max(1, min(args.ref_tokens, args.ref_budget / max(1, args.steps + args.warmup) / per_tok)))
    for i in range(args.warmup):
        _oracle_step(oracle, wl, h, st, _sample_tokens(wl, n, seed=100 + i))
    wall = []
    for i in range(args.steps):
        wall.append(_oracle_step(oracle, wl, h, st, _sample_tokens(wl, n, seed=1000 + i)))
    value = n * len(wall) / sum(wall)
    sample = _sample_text(wl, n)
    return {"metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws_n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * float(np.mean(wall)), 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": layer_config(wl, ws_n),
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--T", type=int, default=0, help="override the token count")
    ap.add_argument("--cpu-tokens", type=int, default=768, help="largest oracle sample for cpu_baseline")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds the cpu_baseline sample aims to take")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per_config table of the other workloads")
    ap.add_argument("--stage", choices=list(STAGES), default=None,
                    help="time one stage alone (only its buffers on the device) and print its line")
    ap.add_argument("--ref-tokens", type=int, default=256, help="largest oracle sample per reference step")
    ap.add_argument("--ref-budget", type=float, default=120.0, help="seconds the reference arm aims to take")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--affinity-drop", action="store_true",
                    help="capacity drop by descending gate weight (DeepSeek-V2) instead of token order")
    ap.add_argument("--fp8-weights", action="store_true",
                    help="store the expert weights as FP8 E4M3 with per-channel scales (MOE_BF16_FP8W)")
    ap.add_argument("--fp8-up", action="store_true",
                    help="run the up projection on E4M3 activations and weights (MOE_BF16_FP8UP)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.stage:
        out = run_stage(args)
    else:
        out = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
