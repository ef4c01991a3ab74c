#!/usr/bin/env python3
"""MoE-layer throughput on one GB300 (and N independent replicas under torchrun).

Headline workload ("decode"): the decode MoE layer -- hidden 2048, 128 routed
experts, top-8 softmax gates renormalised, expert intermediate 768, SwiGLU,
Q4_K gate/up/down, fp32 router, bf16 activations -- at T = 1 token.  One step
is one pass of the whole hot path (router GEMV + top-k, permute, gate/up +
SwiGLU, down, combine) over L = 16 such layers with distinct weights, replayed
as one captured CUDA graph.  The L layers touch ~360 MB of distinct weights per
step, well above the 129 MB L2, so no layer's bytes are still cached when it
runs again.  value = layer-token applications per second = T * L * steps / time.

Other workloads (--workload): decode2 (T = 2), prefill (T = 4096, Zipf(1)
popularity), deepseek (hidden 7168, 256 experts, sigmoid + bias group routing,
shared Q8_0 expert, T = 2).

--impl reference times the fp64 CPU oracle (the baseline the library is
checked against) on the same workload, on the host cores.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

WORKLOADS = {
    # name: (shape, T, layers in the chain, seed, description)
    "decode": (synth.DECODE, 1, 16, 2,
               "decode MoE layer T=1: H=2048 E=128 top-8 softmax I=768 Q4_K, bf16 x, 16 distinct layers per step"),
    "decode2": (synth.DECODE, 2, 16, 2,
                "decode MoE layer T=2: H=2048 E=128 top-8 softmax I=768 Q4_K, bf16 x, 16 distinct layers per step"),
    "prefill": (synth.DECODE, 4096, 2, 3,
                "prefill MoE layer T=4096: H=2048 E=128 top-8 softmax I=768 Q4_K, Zipf(1) popularity, 2 layers per step"),
    "deepseek512": (synth.DEEPSEEK, 512, 2, 4,
                    "MoE layer T=512 (verification batch): H=7168 E=256 sigmoid+bias 8 groups/4 kept top-8 scale 2.5 "
                    "I=2048 Q4_K, shared I=2048 Q8_0, 2 layers per step"),
    "stack": (synth.DECODE, 1, 48, 5,
              "48-layer stack captured as one CUDA graph: per layer RMSNorm (eps 1e-6) -> decode MoE layer "
              "(H=2048 E=128 top-8 I=768 Q4_K) -> residual add, fp32 residual, bf16 layer input"),
    "deepseek": (synth.DEEPSEEK, 2, 4, 4,
                 "MoE layer T=2: H=7168 E=256 sigmoid+bias 8 groups/4 kept top-8 scale 2.5 I=2048 Q4_K, shared I=2048 Q8_0"),
}

CLOCK_QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


def sources_digest(files):
    """sha1 over the given library sources (paths relative to the package's csrc/)."""
    h = hashlib.sha1()
    for f in files:
        with open(os.path.join(ROOT, "quantized_routed_expert_sigmoid_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(kernel, args):
    """DRAM bytes per launch of `kernel` on this workload from the committed ncu summary
    (profiles/traffic.json), or None when there is none or the kernel's sources changed
    since the counters were taken."""
    try:
        key = f"{kernel} {args.workload}" + (f" T={args.tokens}" if args.tokens else "")
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            entry = json.load(f).get(key)
        if entry and sources_digest(entry["sources"]) == entry["sources_sha1"]:
            return entry["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        pass
    return None


# ------------------------------------------------------------------ clocks

class NvmlClocks:
    """Read-only NVML queries (SM clock, max SM clock, clock-event reasons, power) through
    ctypes on libnvidia-ml; None when the library or the device is not available."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        ct = self.ct
        mhz, mx, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz))          # NVML_CLOCK_SM
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
        self.reasons_fn(self.h, ct.byref(rs))
        return time.time(), float(mhz.value), float(mx.value), mw.value / 1000.0, int(rs.value)


class ClockSampler:
    """Samples the SM clock every `period_s` on a thread (NVML), or through nvidia-smi every
    200 ms when NVML is not available; summary() keeps the samples of the timed region."""

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.dev = device_index
        self.period = period_s
        self.rows = []
        self.proc = None
        self.path = None
        self.thread = None
        self.stop = False
        self.source = "nvml"

    def _loop(self, nv):
        while not self.stop:
            try:
                t, mhz, mx, w, bits = nv.sample()
                self.rows.append((t, mhz, mx, [n for b, n in NvmlClocks.REASONS.items() if bits & b]))
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        import threading
        try:
            nv = NvmlClocks(self.dev)
            nv.sample()
            self.thread = threading.Thread(target=self._loop, args=(nv,), daemon=True)
            self.thread.start()
            time.sleep(3 * self.period)
            return self
        except Exception:
            self.thread = None
        self.source = "nvidia-smi"
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={CLOCK_QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.thread is not None:
            time.sleep(2 * self.period)
            self.stop = True
            self.thread.join(timeout=2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t_begin=None, t_end=None):
        """Median SM clock, max clock and active throttle reasons over the samples taken in
        [t_begin, t_end] (host epoch seconds: the timed region); all samples when none fell in it."""
        if self.thread is not None:
            rows = [(t, mhz, mx, ["active"] + [("Active" if n in rs else "Not Active") for n in
                                                ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                                 "sw_power_cap")])
                    for t, mhz, mx, rs in self.rows]
            out = summarize_clocks(rows, t_begin, t_end)
        else:
            if self.proc is None or not self.path or not os.path.exists(self.path):
                return None
            rows = parse_clock_samples(open(self.path).read().splitlines())
            os.unlink(self.path)
            out = summarize_clocks(rows, t_begin, t_end)
        if out is not None:
            out["source"] = self.source
        return out


def parse_clock_samples(lines):
    """(epoch seconds or None, sm MHz, max sm MHz, [reason flags]) per nvidia-smi CSV line of
    CLOCK_QUERY (noheader, nounits)."""
    import datetime
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            ts = None
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                pass
            rows.append((ts, float(parts[2]), float(parts[3]), parts[5:10]))
        except ValueError:
            continue
    return rows


def summarize_clocks(rows, t_begin=None, t_end=None):
    if not rows:
        return None
    window = "timed region"
    if t_begin is not None and t_end is not None:
        inside = [r for r in rows if r[0] is not None and t_begin <= r[0] <= t_end]
        if inside:
            rows = inside
        else:
            window = "whole run (no sample fell in the timed region)"
    names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = set()
    for r in rows:
        for n, v in zip(names[1:], r[3][1:]):
            if v.lower().startswith("active"):
                reasons.add(n)
    return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": max(r[2] for r in rows),
            "samples": len(rows), "reasons": sorted(reasons), "window": window}


# ------------------------------------------------------------------ replicas (one process per GPU)

def ranks_max(v, world, device):
    """The largest of the ranks' values of v; v itself for one process.  Every rank calls it."""
    if world <= 1:
        return v
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.item()


def agree_steps(seconds_per_step, world, device, target_s=1.2, lo=200, hi=20000):
    """Timed steps for about target_s seconds of work, the same count on every rank (the
    slowest rank's probe sets it, so no rank's timed region is shorter than target_s)."""
    k = min(hi, max(lo, int(target_s / max(seconds_per_step, 1e-6)) + 1))
    return int(ranks_max(k, world, device))


def job_tokens_per_s(world, T, L, steps, t_ms):
    """Whole-job throughput of N replicas: each rank applies L layers to its own T tokens per
    step, and t_ms, the slowest rank's time for all steps, bounds the job."""
    return world * T * L * steps / (t_ms / 1e3)


# ------------------------------------------------------------------ workload construction

def build_layers(shape, T, L, seed, device, shared_router=False, decode_chain=True, tc_min_tokens=0):
    """L layers with distinct expert weights.  Router weights and biases are drawn on the
    CPU (small) so that a workload built around them (the Zipf prefill) sees the same values;
    shared_router gives every layer layer 0's router.  tc_min_tokens (0: the library's
    default) is the smallest T that takes the tensor-core path."""
    from quantized_routed_expert_sigmoid_gb300 import MoeLayer
    layers = []
    for l in range(L):
        gate = synth.expert_stack(shape, seed, l, "gate", device)
        up = synth.expert_stack(shape, seed, l, "up", device)
        down = synth.expert_stack(shape, seed, l, "down", device)
        lr = 0 if shared_router else l
        Wr = synth.router_weight(shape, seed, lr).to(device)
        b = synth.bias(shape, seed, lr)
        b = None if b is None else b.to(device)
        sh, sh_run, sq = None, None, shape.shared_qtype
        if shape.I_s > 0:
            sh = [synth.expert_matrix(shape, seed, l, n, 0, device) for n in ("s_gate", "s_up", "s_down")]
            sh_run = sh
            if shape.shared_qtype == synth.Q8_0:
                # a Q8_0 shared expert is prepared once (moe_weights_prepare), as a user would
                from quantized_routed_expert_sigmoid_gb300.layer import prepare_q8_0
                sh_run = [prepare_q8_0(sh[0], shape.I_s, shape.H), prepare_q8_0(sh[1], shape.I_s, shape.H),
                          prepare_q8_0(sh[2], shape.H, shape.I_s)]
                sq = "q8_0_r"
        lay = MoeLayer(mode=shape.mode, E=shape.E, k=shape.k, H=shape.H, I=shape.I, qtype=shape.qtype,
                       gate=gate, up=up, down=down, W_router=Wr, bias=b, n_groups=shape.n_groups,
                       topk_groups=shape.topk_groups, scale=shape.scale, renormalize=shape.renormalize,
                       x_dtype=shape.x_dtype, I_s=shape.I_s, shared_qtype=sq,
                       s_gate=sh_run[0] if sh else None, s_up=sh_run[1] if sh else None,
                       s_down=sh_run[2] if sh else None, decode_chain=decode_chain, tc_min_tokens=tc_min_tokens)
        lay.stored_shared = sh                   # the GGUF bytes, for the oracle
        layers.append(lay)
    return layers


def resolve_workload(args):
    """(shape, T, layers per step, seed, description) of args.workload with --tokens / --layers."""
    shape, T, L, seed, desc = WORKLOADS[args.workload]
    if args.tokens:
        T = args.tokens
        desc = desc.replace("T=1:", f"T={T}:").replace("T=2:", f"T={T}:")
    if args.layers:
        L = args.layers
        desc = desc.replace("16 distinct layers", f"{L} distinct layers")
    return shape, T, L, seed, desc


def workload_config(args, shape, T, L, desc, world):
    """The `config` of a bench line: the workload and its sizes (the same on both arms)."""
    return {"workload": desc, "T": T, "layers_per_step": L, "H": shape.H, "E": shape.E, "k": shape.k,
            "I": shape.I, "qtype": shape.qtype, "l2": "inputs larger than L2 (distinct weights per layer)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            **({"tc_min_tokens": args.tc_min_tokens} if args.tc_min_tokens else {})}


def make_x(shape, T, seed, device, workload):
    if workload == "prefill":
        Wr = synth.router_weight(shape, seed, 0).numpy()
        L = synth.zipf_target_logits(T, shape.E, shape.k, seed)
        return synth.activations_for_logits(L, Wr, seed).to(device)
    return synth.activations(T, shape.H, seed, shape.x_dtype, device="cpu").to(device)


def algorithmic_bytes(shape, T, offsets_host):
    """Distinct chosen experts' blocks + router weight + x in + out (one layer)."""
    u = int(np.count_nonzero(np.diff(offsets_host)))
    xb = T * shape.H * (2 if shape.x_dtype == "bf16" else 4)
    b = u * synth.bytes_per_expert(shape) + shape.E * shape.H * 4 + xb + T * shape.H * 4
    b += synth.shared_bytes(shape)
    gu = u * 2 * shape.I * synth.row_bytes(shape.qtype, shape.H) + xb + T * shape.k * shape.I * 4
    return b, gu, u


def launches_per_layer(shape, T, stack=False, path=None):
    """Kernel launches of one moe_layer call on the given path (the library's own launch order)."""
    P = T * shape.k
    if path == "decode_chain":
        return 3                                     # logits (+ RMSNorm), routing + gate/up, down + combine
    n = 2 + (1 if P <= 1024 else 2) + 2 + 1          # logits, top-k, permute, gate/up, down, combine
    if path == "tensor":
        n += 2                                       # fp16 copy of x, token-block list
        if shape.x_dtype == "bf16" and T > 32 and shape.H % 64 == 0 and shape.E % 4 == 0 and shape.E <= 1024:
            n += 1                                   # router logits on tcgen05: W_r split into bf16 parts first
    if shape.I_s > 0:
        n += 2                                       # the shared expert's gate/up and down
    return n + (1 if stack else 0)                   # the layer's own RMSNorm launch in the stack


# ------------------------------------------------------------------ our arm

SUB_WORKLOADS = ("decode2", "prefill")       # the metric's other two points, measured beside the headline


def run_ours(args, rank, world):
    """The headline line (decode T=1) with the metric's other points (decode T=2, prefill
    T=4096) as sub-records measured in the same run, each with its own timing, roofline and
    end-to-end figure."""
    import copy
    steps_given = args.steps
    head = measure(args, rank, world)
    if args.workload == "decode" and not (args.tokens or args.layers or args.no_sub):
        subs = {}
        for name in SUB_WORKLOADS:
            torch.cuda.empty_cache()
            a = copy.copy(args)
            a.workload, a.steps, a.no_cpu_baseline = name, steps_given, True
            r = measure(a, rank, world)
            subs[name] = {k: r[k] for k in ("value", "unit", "steps", "ms_per_step", "config", "layer", "roofline",
                                            "e2e", "gpu_launches", "clocks") if k in r}
        head["workloads"] = subs
    return head


def measure(args, rank, world):
    """One workload: build its layers, capture one step as a CUDA graph, time K steps."""
    import quantized_routed_expert_sigmoid_gb300 as moe
    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(device)
    shape, T, L, seed, desc = resolve_workload(args)
    stack = args.workload == "stack"
    layers = build_layers(shape, T, L, seed + 1000 * rank, device, shared_router=(args.workload == "prefill"),
                          decode_chain=not args.separate_decode, tc_min_tokens=args.tc_min_tokens)
    x = make_x(shape, T, seed + 1000 * rank, device, args.workload)
    outs = [torch.empty(T, shape.H, dtype=torch.float32, device=device) for _ in range(L)]
    for lay in layers:
        lay.ensure_workspace(T, device)
    if stack:
        import quantized_routed_expert_sigmoid_gb300._native as N
        gammas = [synth.gamma(shape.H, seed, l).to(device) for l in range(L)]
        for lay, gm in zip(layers, gammas):
            # one call per layer is a residual block: resid += layer(bf16(RMSNorm(resid) * gamma))
            lay.desc.accumulate = 1
            lay.desc.x_type = N.MOE_F32
            lay.desc.norm_gamma = gm.data_ptr()
            lay.desc.norm_eps = 1e-6
            lay._keep.append(gm)
            lay.rebuild_plan()
            lay.ensure_workspace(T, device)
        resid = x.float().clone()
        u = torch.empty(T, shape.H, dtype=torch.bfloat16, device=device)

    def chain(stream=None):
        if stack:
            for lay in layers:
                lay(resid, out=resid, stream=stream)
            return
        for lay, o in zip(layers, outs):
            lay(x, out=o, stream=stream)

    chain()
    torch.cuda.synchronize()
    # one captured graph per step
    s = torch.cuda.Stream(device=device)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        chain(stream=s)
    torch.cuda.synchronize()

    # per-layer routing facts (for algorithmic bytes)
    per_layer = []
    for lay in layers:
        _, _, offs = lay.debug_views(T)
        per_layer.append(algorithmic_bytes(shape, T, offs.numpy()))
    layer_bytes = float(np.mean([p[0] for p in per_layer]))
    gu_bytes = float(np.mean([p[1] for p in per_layer]))
    u_mean = float(np.mean([p[2] for p in per_layer]))

    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream(device)          # CUDAGraph.replay() launches on the current stream
    if args.steps is None:
        # no --steps given: about a second of timed work, so the clock samples fall inside it
        t_probe = time.perf_counter()
        for _ in range(10):
            graph.replay()
        torch.cuda.synchronize()
        args.steps = agree_steps((time.perf_counter() - t_probe) / 10, world, device)
    with ClockSampler(device.index) as clk:
        torch.cuda.synchronize()
        t_begin = time.time()
        ev0.record(cur)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(cur)
        torch.cuda.synchronize()
        t_end = time.time()
    t_ms = ranks_max(ev0.elapsed_time(ev1), world, device)
    ms_per_step = t_ms / args.steps
    value = job_tokens_per_s(world, T, L, args.steps, t_ms)

    # ---- the dominant kernel alone (the routed gate/up + SwiGLU launch)
    path = layers[0].path(T)           # which kernels the library runs for this T
    tc_path = path == "tensor"
    chain_path = path == "decode_chain"
    gu_ms = None
    if stack:
        # the gate/up kernel's input: the residual stream for the chain (which normalizes it
        # itself), the bf16 normalized stream for the other paths
        if chain_path or tc_path:
            x = resid.clone()
        else:
            moe.moe_rmsnorm_bf16(resid, gammas[0], T, shape.H, 1e-6, u)
            x = u
    try:
        if tc_path or chain_path:
            gu_ms = time_gateup_events(moe, layers, x, outs, T, args)
        else:
            gu_ms = time_gateup(moe, layers, x, shape, T, device, args)
    except Exception as exc:  # keep the headline even if this sub-measurement fails
        print(f"gate/up timing skipped: {exc}", file=sys.stderr)

    # ---- end to end through the public call, host buffers, copies inside the timed region
    x_host = x.cpu().pin_memory()
    out_host = torch.empty(L, T, shape.H, dtype=torch.float32).pin_memory()
    x_dev = torch.empty_like(x)
    out_stack = torch.empty(L, T, shape.H, dtype=torch.float32, device=device)
    e2e_steps = max(3, min(args.steps, 50))

    def e2e_step():
        x_dev.copy_(x_host, non_blocking=True)
        if stack:
            resid.copy_(x_dev)
            for lay in layers:
                lay(resid, out=resid)
            out_stack[0].copy_(resid)
        else:
            for i, lay in enumerate(layers):
                lay(x_dev, out=out_stack[i])
        out_host.copy_(out_stack, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(2):
        e2e_step()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_ms = ranks_max((time.perf_counter() - t0) * 1e3, world, device)
    e2e = {"value": job_tokens_per_s(world, T, L, e2e_steps, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": x.numel() * x.element_size(),
           "d2h_bytes_per_step": out_stack.numel() * 4, "calls": "moe_layer x %d per step" % L}

    hbm_peak, tc_peak, peak_kind = measured_peaks()
    roof = None
    if gu_ms is not None and chain_path:
        # routing + gate/up (+ the shared expert's gate/up rows) of the chain
        cb = gu_bytes + (2 * shape.I_s * synth.row_bytes(shape.shared_qtype, shape.H) if shape.I_s > 0 else 0)
        achieved = cb / (gu_ms * 1e-3) / 1e9
        roof = {"kernel": "chain_gateup_kernel (routing + gate/up + SwiGLU)", "bound": "hbm",
                "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": profiled_traffic("chain_gateup_kernel", args),
                "peak_source": peak_kind, "bytes_per_launch": round(cb), "us_per_launch": round(gu_ms * 1e3, 3),
                "timing": "CUDA events recorded around the gate/up launch, eager calls"}
    elif gu_ms is not None and not tc_path:
        achieved = gu_bytes / (gu_ms * 1e-3) / 1e9
        # Q4_K experts (up to 256 of them) take the persistent segmented kernel, others qgemv
        kern = ("seg_gateup_kernel (persistent segmented gate/up + SwiGLU)" if shape.qtype == "q4_k" and shape.E <= 256
                else "qgemv_kernel (gate/up + SwiGLU)")
        roof = {"kernel": kern, "bound": "hbm", "achieved": round(achieved, 1),
                "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                "traffic": profiled_traffic(kern.split(" ")[0], args),
                "peak_source": peak_kind, "bytes_per_launch": round(gu_bytes), "us_per_launch": round(gu_ms * 1e3, 3)}
    elif gu_ms is not None:
        # the tensor-core gate/up: report the binding roofline (tensor pipe or HBM, whichever
        # fraction is higher) and the other one beside it
        flops = 2.0 * T * shape.k * 2 * shape.H * shape.I
        tflops = flops / (gu_ms * 1e-3) / 1e12
        gbs = gu_bytes / (gu_ms * 1e-3) / 1e9
        tc_frac, hbm_frac = tflops / tc_peak, gbs / hbm_peak
        kern = "tc_gemm_kernel (tcgen05 gate/up + SwiGLU, fp16 operands, fp32 accumulate)"
        if tc_frac >= hbm_frac:
            roof = {"kernel": kern, "bound": "tensor", "achieved": round(tflops, 1), "peak": tc_peak,
                    "unit": "TFLOP/s", "frac": round(tc_frac, 4), "traffic": profiled_traffic("tc_gemm_kernel", args),
                    "peak_source": peak_kind + " (bf16 burst; fp16 runs at the bf16 rate)",
                    "flops_per_launch": flops, "us_per_launch": round(gu_ms * 1e3, 3),
                    "other": {"bound": "hbm", "achieved": round(gbs, 1), "unit": "GB/s", "frac": round(hbm_frac, 4)}}
        else:
            roof = {"kernel": kern, "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(hbm_frac, 4), "traffic": profiled_traffic("tc_gemm_kernel", args), "peak_source": peak_kind,
                    "bytes_per_launch": round(gu_bytes), "us_per_launch": round(gu_ms * 1e3, 3),
                    "other": {"bound": "tensor", "achieved": round(tflops, 1), "unit": "TFLOP/s",
                              "frac": round(tc_frac, 4)}}
    layer_us = ms_per_step * 1e3 / L
    extra = {}
    if stack:
        extra["stack_tokens_per_s"] = round(job_tokens_per_s(world, T, 1, args.steps, t_ms), 1)
    result = {
        "metric": "MoE-layer tokens/s (decode T=1,2 / prefill T=4096); % of HBM roofline",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(args, shape, T, L, desc, world), "path": path,
        "layer": {"us_per_layer": round(layer_us, 3), "algorithmic_bytes": round(layer_bytes),
                  "GBps": round(layer_bytes / (layer_us * 1e-6) / 1e9, 1),
                  "frac_hbm": round(layer_bytes / (layer_us * 1e-6) / 1e9 / hbm_peak, 4),
                  "distinct_experts_mean": u_mean},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": launches_per_layer(shape, T, stack, path) * L * args.steps,
        "clocks": clk.summary(t_begin, t_end),
    }
    result.update(extra)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.workload, layers[0], x, shape, T, budget_s=args.cpu_seconds)
    return result


def time_gateup_events(moe, layers, x, outs, T, args):
    """Average duration of the routed gate/up launch measured with CUDA events recorded
    around it by moe_layer_timed (eager calls queued behind a short sleep so the host
    is never the bottleneck)."""
    import quantized_routed_expert_sigmoid_gb300._native as N
    durations = []
    rounds = max(5, min(args.steps, 20))
    for _ in range(rounds):
        evs = []
        torch.cuda._sleep(20_000_000)
        for lay, o in zip(layers, outs):
            eb, ea = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            eb.record()                  # torch creates the CUDA event on first record;
            ea.record()                  # the library records both again around the kernel
            N.moe_layer_timed(lay.plan, x, T, o, lay.ws, lay.ws.numel(), None, eb, ea)
            evs.append((eb, ea))
        torch.cuda.synchronize()
        durations += [eb.elapsed_time(ea) for eb, ea in evs]
    # the events tick in steps of about 1 us: the mean over many launches (whose start times
    # fall anywhere within a tick) estimates the duration without the rounding of a median
    return statistics.fmean(durations)


def time_gateup(moe, layers, x, shape, T, device, args):
    """Average duration of the gate/up kernel: one graph of L launches, replayed."""
    k, E, H, I = shape.k, shape.E, shape.H, shape.I
    P = T * k
    import quantized_routed_expert_sigmoid_gb300._native as N
    xt = N.MOE_BF16 if x.dtype == torch.bfloat16 else N.MOE_F32   # the kernels read x as it is
    routed = []
    for lay in layers:
        ids = torch.empty(T, k, dtype=torch.int32, device=device)
        w = torch.empty(T, k, device=device)
        lg = torch.empty(T, E, device=device)
        moe.moe_route(lay.desc.route, x, xt, T, H, lay.desc.W_router, lay.desc.bias, None, lg, ids, w)
        sp = torch.empty(P, dtype=torch.int32, device=device)
        pp = torch.empty(P, dtype=torch.int32, device=device)
        off = torch.empty(E + 1, dtype=torch.int32, device=device)
        nb = moe.moe_permute_workspace_size(T, k, E)
        ws = torch.empty(nb, dtype=torch.uint8, device=device)
        moe.moe_permute(ids, T, k, E, sp, off, pp, ws, nb)
        h = torch.empty(P, I, device=device)
        routed.append((lay, sp, off, h))
    torch.cuda.synchronize()

    def run(stream=None):
        for lay, sp, off, h in routed:
            moe.moe_expert_gateup(lay.desc.gate, lay.desc.up, E, x, xt, T, H, I, sp, off, k, h,
                                  stream)

    s = torch.cuda.Stream(device=device)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(stream=s)
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(10, args.steps)
    cur = torch.cuda.current_stream(device)
    e0.record(cur)
    for _ in range(reps):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * len(routed))


# ------------------------------------------------------------------ oracle (CPU baseline / reference arm)

def oracle_layer_spec(shape, layer_tensors):
    import oracle
    gate, up, down, Wr, bias = layer_tensors
    return oracle.LayerSpec(mode=oracle.ROUTE_SIGMOID_GROUP if shape.mode == "sigmoid_group" else oracle.ROUTE_SOFTMAX,
                            E=shape.E, k=shape.k, H=shape.H, I=shape.I,
                            qtype=oracle.Q4_K if shape.qtype == synth.Q4_K else oracle.Q8_0,
                            gate=gate, up=up, down=down, Wr=Wr, bias=bias, n_groups=shape.n_groups,
                            topk_groups=shape.topk_groups, renormalize=shape.renormalize, scale=shape.scale)


def oracle_threads(workload):
    return 1 if workload in ("decode", "decode2") else (os.cpu_count() or 1)


def cpu_baseline(workload, layer, x, shape, T, budget_s=10.0):
    """The oracle, as it stands, on a bounded sample of the same workload (host cores)."""
    import oracle
    gate, up, down = layer._keep[0], layer._keep[1], layer._keep[2]
    Wr, b = layer._keep[3], layer._keep[4]
    spec = oracle_layer_spec(shape, (gate.cpu().numpy(), up.cpu().numpy(), down.cpu().numpy(), Wr.cpu().numpy(),
                                     None if b is None else b.cpu().numpy()))
    if shape.I_s > 0:
        sg, su, sd = layer.stored_shared
        spec.shared_qtype, spec.I_s = oracle.Q8_0, shape.I_s
        spec.s_gate, spec.s_up, spec.s_down = sg.cpu().numpy(), su.cpu().numpy(), sd.cpu().numpy()
    xs = x.float().cpu().double().numpy()
    n_sample = T if T <= 8 else 8                 # tokens per oracle call
    threads = oracle_threads(workload)
    times = []
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < budget_s and len(times) < 200:
        t0 = time.perf_counter()
        oracle.moe_layer(spec, xs[:n_sample], n_threads=threads)
        times.append(time.perf_counter() - t0)
    per_call = statistics.median(times)
    return {"value": round(n_sample / per_call, 3), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(times)} oracle calls of {n_sample} token(s) of one layer of the same workload, "
                      f"median {per_call * 1e3:.1f} ms per call"}


def run_reference(args):
    """The fp64 oracle timed on the host cores on this workload (no GPU)."""
    import oracle
    shape, T, L, seed, desc = resolve_workload(args)
    tensors = (synth.expert_stack(shape, seed, 0, "gate").numpy(), synth.expert_stack(shape, seed, 0, "up").numpy(),
               synth.expert_stack(shape, seed, 0, "down").numpy(), synth.router_weight(shape, seed, 0).numpy(),
               None if shape.bias_std <= 0 else synth.bias(shape, seed, 0).numpy())
    spec = oracle_layer_spec(shape, tensors)
    if shape.I_s > 0:
        spec.shared_qtype, spec.I_s = oracle.Q8_0, shape.I_s
        spec.s_gate, spec.s_up, spec.s_down = [synth.expert_matrix(shape, seed, 0, n, 0).numpy()
                                               for n in ("s_gate", "s_up", "s_down")]
    x = make_x(shape, T, seed, "cpu", args.workload).float().double().numpy()
    n_sample = T if T <= 8 else 8
    threads = oracle_threads(args.workload)
    for _ in range(args.warmup):
        oracle.moe_layer(spec, x[:n_sample], n_threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.moe_layer(spec, x[:n_sample], n_threads=threads)
    dt = (time.perf_counter() - t0) / args.steps
    value = n_sample / dt
    return {"impl": "reference", "metric": "MoE-layer tokens/s (decode T=1,2 / prefill T=4096); % of HBM roofline",
            "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": workload_config(args, shape, T, L, desc, 1),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step: one oracle call on {n_sample} token(s) of one layer"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about a second of work; the reference arm: 200)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="override the layers per step (default per workload)")
    ap.add_argument("--tokens", type=int, default=0, help="override T (tokens per layer call)")
    ap.add_argument("--tc-min-tokens", type=int, default=0,
                    help="smallest T that takes the tensor-core path (default: the library's, 65)")
    ap.add_argument("--no-sub", action="store_true",
                    help="decode: skip the sub-records of decode T=2 and prefill T=4096")
    ap.add_argument("--separate-decode", action="store_true",
                    help="decode sizes: run the separate route/permute/GEMV/combine kernels, not the single-launch layer")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if args.steps is None:
            args.steps = 200
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    try:
        result = run_ours(args, rank, world)
        if rank == 0:
            print(json.dumps(result), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
