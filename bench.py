"""Throughput of the fused trellis-MoE layer on synthetic inputs.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload decode|prefill|odd|large-decode|large-prefill|linear] [--tokens T]

One step is one pass of the whole hot path over one token batch: router on the
logits, route map, fused rotate+quantize, FC1 with its activation epilogue,
FC2 with the unrotation epilogue, and the top-k combine -- all in the
library's CUDA kernels, replayed from CUDA graphs captured per batch.

The default workload is the decode layer (H=1024, I=512, E=128, top-k 8,
W4A8, K=4 trellis) at T=8 tokens per step. Its touched weights (~41 MB per
step) would sit in the 129 MB L2, so the step cycles through several copies of
the layer living at different addresses (touched bytes between two uses of one
copy exceed 2x L2) and through as many token batches.

Output: one JSON line on rank 0. ``roofline`` is for the dominant kernel
(FC1; on the tensor-core path the one launch that runs FC1 and FC2 where the
library fuses them): algorithmic bytes (or FLOPs) per launch divided by its
CUDA-event duration, timed inside the captured graphs of the timed region. The default
run also measures the metric's other configurations -- decode at T = 1, 2
and 4 and the T=2048 W4A16 prefill -- each with the same keys, under
``sub`` (``--no-sub`` skips them). ``cpu_baseline`` times the float64 CPU
oracle on a bounded sample. ``--impl reference`` runs only that oracle (the
CPU reference arm).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from trellis_quantized_moe_route_gb300 import synth  # noqa: E402

METRIC = "fused trellis-MoE layer tokens/s (decode T=1-8, prefill T=2048); % of roofline"
L2_BYTES = 129e6

WORKLOADS = {
    # name: (config, T, mode)
    "decode": ("decode", 8, "w4a8"),
    "prefill": ("prefill", 2048, "w4a16"),
    "odd": ("odd", 512, "w4a16"),
    "large-decode": ("large", 1, "w4a8"),
    "large-prefill": ("large", 4096, "w4a16"),
}


def job_time_ms(local_ms: float, world: int) -> float:
    """The job's timed region: the slowest rank's (every rank calls this)."""
    if world <= 1:
        return local_ms
    import torch
    t = torch.tensor([local_ms], dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(steps: int, tokens_per_step: int, world: int, total_ms: float) -> float:
    """Whole-job tokens/s: every rank runs its own replica (weak scaling)."""
    return round(steps * tokens_per_step * world / (total_ms / 1e3), 2)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu = gpu_index
        self.period = period_ms
        self.samples = []
        self._stop = threading.Event()
        self._t = None

    def _query(self):
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=5)
            if r.returncode == 0 and r.stdout.strip():
                self.samples.append([v.strip() for v in r.stdout.strip().split(",")])
        except Exception:
            pass

    def _run(self):
        while not self._stop.is_set():
            self._query()
            self._stop.wait(self.period / 1000.0)

    def start(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def stop(self):
        self._stop.set()
        if self._t:
            self._t.join()
        self._query()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in self.samples:
            for n, v in zip(names, s[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.samples)}


# ------------------------------------------------------------------- ours ---
def touched_bytes_fc1(cfg, ids, T, mode):
    """Algorithmic DRAM bytes of one FC1 launch: trellis payload, per-channel
    scales and rotation rows of every touched expert, the quantised input rows
    read, and the FC1 epilogue's output rows written."""
    E, H, I = cfg.E, cfg.H, cfg.I
    K = max(cfg.bits)
    d = len(np.unique(ids))
    R = ids.size
    act_b = 1 if mode == "w4a8" else 2
    weights = d * (2 * I * H * K // 8 + 2 * I * 2 + 3 * I * 2)
    acts = T * H * act_b + (T * H // 32 if act_b == 1 else 0)
    outs = R * I * act_b + (R * I // 32 if act_b == 1 else 0)
    return weights + acts + outs, d



def sleep_ahead(stream, steps: int):
    """A device-side spin on `stream` ahead of the timed region, long enough
    for the host to queue the timed steps (~150 us of host time per graph
    replay, plus 2 ms), so that the region measures the device's throughput
    on resident inputs rather than the host's launch rate. The end-to-end
    host-buffer figure (`e2e`) is the number with the host in the loop."""
    import torch
    us = min(200000.0, 2000.0 + 150.0 * steps)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2.0e3))   # ~us at 2 GHz


def sampler_started(dev):
    """A clock sampler whose first sample is taken before the timed region."""
    smp = ClockSampler(dev)
    smp.start()
    t_end = time.time() + 5.0
    while not smp.samples and time.time() < t_end:
        time.sleep(0.01)
    return smp


def roofline_record(cfg, T, mode, stages_us, fc1_bytes, pk, ncu):
    """The roofline object of one layer workload, from its stage times (us),
    the FC1 launch's algorithmic bytes and the peaks. Returns (roofline,
    decode_path, fused): the decode rows are bound by HBM bytes, the tensor-core
    path by FLOPs. Where FC1 and FC2 both take 256-row units the library runs
    them as one tensor-core launch (FC2 units fill FC1's last wave); the stage
    after its event is then empty and that launch's work is both GEMMs."""
    K = max(cfg.bits)
    R = T * cfg.topk
    decode_path = R <= 1024 and (mode == "w4a8" or R < 4 * cfg.E)   # the library's decode-rows regime
    fused = not decode_path and stages_us["fc2"] < 0.1 * stages_us["fc1"]
    if decode_path:
        achieved = fc1_bytes / (stages_us["fc1"] * 1e-6) / 1e9
        roof = {"bound": "hbm", "kernel": "k_dec_warp<%s,FC1,K=%d> (decode rows, persistent warp items)" % (
                    mode.upper(), K),
                "achieved": round(achieved, 1),
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                "traffic": ncu[0] if ncu else None, "traffic_source": ncu[1] if ncu else None,
                "peak_source": pk["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst)",
                "bytes_per_launch": int(fc1_bytes)}
    else:
        flops = 2 * R * 2 * cfg.I * cfg.H + (2 * R * cfg.H * cfg.I if fused else 0)
        achieved = flops / (stages_us["fc1"] * 1e-6) / 1e12
        kern = "k_tc_fc<FC1+FC2,K=%d> (tcgen05, W4A16, one launch)" if fused else "k_tc_fc<FC1,K=%d> (tcgen05, W4A16)"
        roof = {"bound": "tensor", "kernel": kern % K, "achieved": round(achieved, 2),
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / pk["bf16_tflops"], 4),
                "traffic": ncu[0] if ncu else None, "traffic_source": ncu[1] if ncu else None,
                "peak_source": pk["source"] + " (bf16 dense burst; fp16 runs at the bf16 rate)",
                "flops_per_launch": flops}
    return roof, decode_path, fused


def launches_per_layer_step(R, decode_path, fused):
    """Our kernels per layer step: decode rows: prologue, FC1, FC1 epilogue,
    FC2, FC2 epilogue; otherwise router, route map (1 kernel, 3 above 1024
    routes), rotate, FC1 and FC2 (one launch when fused), combine."""
    if decode_path:
        return 5
    return 6 + (2 if R > 1024 else 0) - (1 if fused else 0)


def measure_layer(name, T, mode, steps, warmup, rank, world, dev, e2e_steps):
    """One workload of the layer: graphs per (layer copy, token batch), K timed
    steps between CUDA events on the launching stream, stage durations from
    events recorded inside the last few timed steps, and the host-buffer call
    end to end. Returns the record (metric keys, roofline, stages, e2e)."""
    import torch
    from trellis_quantized_moe_route_gb300 import binding

    cfg = synth.CONFIGS[name]
    K = max(cfg.bits)
    R = T * cfg.topk
    # layer copies at distinct addresses so that the bytes touched between two
    # uses of one copy exceed twice the L2
    layer = synth.make_layer(cfg)
    per_expert = 3 * cfg.H * cfg.I * K // 8
    touched_est = min(cfg.E, R) * per_expert
    copies = int(min(16, max(1, np.ceil(2 * L2_BYTES / max(touched_est, 1)) + 1)))
    moes = [binding.TrellisMoE(layer, max_tokens=T) for _ in range(copies)]
    batches = []
    for b in range(copies):
        x_bits, logits = synth.make_tokens(cfg, T=T, seed=1000 + 17 * rank + b)
        x = torch.from_numpy(np.ascontiguousarray(x_bits.view(np.int16))).cuda()
        lg = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
        out = torch.empty((T, cfg.H), dtype=torch.float32, device="cuda")
        batches.append((x, lg, out, x_bits, logits))
    stream = torch.cuda.Stream()

    # warm-up (eager; also fixes kernel attributes before capture)
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 1)):
            b = i % copies
            moes[b].forward_logits(batches[b][0], batches[b][1], mode=mode, out=batches[b][2])
    torch.cuda.synchronize()

    # per (copy, batch): one plain graph and one that also records the
    # library's stage-boundary events (used for the last few timed steps, so
    # that the per-kernel durations come from inside the timed region)
    graphs, graphs_ev, evsets = [], [], []
    for b in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            moes[b].forward_logits(batches[b][0], batches[b][1], mode=mode, out=batches[b][2])
        graphs.append(g)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
        for ev in evs:
            ev.record(stream)
        torch.cuda.synchronize()
        moes[b].set_stage_events(evs)
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge, stream=stream):
            moes[b].forward_logits(batches[b][0], batches[b][1], mode=mode, out=batches[b][2])
        moes[b].set_stage_events(None)
        graphs_ev.append(ge)
        evsets.append(evs)
    for i in range(max(warmup, 3)):
        graphs[i % copies].replay()
        graphs_ev[i % copies].replay()
    torch.cuda.synchronize()

    sampler = sampler_started(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sleep_ahead(stream, steps)
    t0.record(stream)
    # the last three timed steps (or fewer) use the event-recording graphs: the
    # stage statistics need only a few samples, and every recorded event adds
    # its own overhead to the timed region
    n_ev = min(copies, steps, 3)
    with torch.cuda.stream(stream):
        for i in range(steps):
            (graphs_ev if i >= steps - n_ev else graphs)[i % copies].replay()
    t1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = job_time_ms(t0.elapsed_time(t1), world)

    # stage times of the event graphs replayed at the end of the timed region
    stage = {k: [] for k in ("router", "route_map", "rotate", "fc1", "fc2", "combine", "step")}
    used = sorted(set(i % copies for i in range(steps - n_ev, steps)))
    for evs in [evsets[i] for i in used]:
        e = [evs[i] for i in range(7)]
        stage["router"].append(e[0].elapsed_time(e[1]) * 1e3)
        stage["route_map"].append(e[1].elapsed_time(e[2]) * 1e3)
        stage["rotate"].append(e[2].elapsed_time(e[3]) * 1e3)
        stage["fc1"].append(e[3].elapsed_time(e[4]) * 1e3)
        stage["fc2"].append(e[4].elapsed_time(e[5]) * 1e3)
        stage["combine"].append(e[5].elapsed_time(e[6]) * 1e3)
        stage["step"].append(e[0].elapsed_time(e[6]) * 1e3)
    stages_us = {k: round(statistics.mean(v), 3) for k, v in stage.items()}
    for m in moes:
        assert m.poll_error() == 0

    # algorithmic work per FC1 launch, from each batch's routes
    fc1_bytes, distinct = [], []
    for b in used:
        ids, _ = binding.route(batches[b][1], cfg.topk)
        nb, d = touched_bytes_fc1(cfg, ids.cpu().numpy(), T, mode)
        fc1_bytes.append(nb)
        distinct.append(d)
    pk = peaks()
    roof, decode_path, fused = roofline_record(cfg, T, mode, stages_us, statistics.mean(fc1_bytes), pk,
                                               NCU_TRAFFIC.get((name, T, mode)))

    # end to end through the host-buffer C-ABI call
    xh = [torch.from_numpy(np.ascontiguousarray(b[3].view(np.int16))).pin_memory() for b in batches]
    lh = [torch.from_numpy(np.ascontiguousarray(b[4])).pin_memory() for b in batches]
    oh = [torch.empty((T, cfg.H), dtype=torch.float32).pin_memory() for _ in batches]
    # warm-up: every buffer set the timed calls use, twice (the first call on
    # a buffer set captures the CUDA graph the later calls replay)
    with torch.cuda.stream(stream):
        for i in range(copies * 2):
            moes[i % copies].forward_host(xh[i % copies], lh[i % copies], oh[i % copies], mode=mode)
    torch.cuda.synchronize()
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    h0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            b = i % copies
            moes[b].forward_host(xh[b], lh[b], oh[b], mode=mode)
    h1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = job_time_ms(h0.elapsed_time(h1), world)
    e2e = {"value": round(e2e_steps * T * world / (e2e_ms / 1e3), 2), "unit": "tokens/s",
           "h2d_bytes_per_step": T * cfg.H * 2 + T * cfg.E * 4, "d2h_bytes_per_step": T * cfg.H * 4,
           "steps": e2e_steps, "api": "trellis_moe_forward_host",
           "transfer": "pinned host buffers mapped into the device address space: the kernels read x and the "
                       "logits and write the fp32 result over NVLink-C2C each call (no staging copies); the call "
                       "replays a graph cached for the buffer set and synchronises the stream"}

    launches_per_step = launches_per_layer_step(R, decode_path, fused)
    for m in moes:
        m.close()
    return {
        "value": job_value(steps, T, world, total_ms), "unit": "tokens/s",
        "ms_per_step": round(total_ms / steps, 5), "steps": steps,
        "dtype": "e4m3" if mode == "w4a8" else "f16",
        "config": {"workload": workload_string(name, cfg, K, mode, T), "tokens_per_step": T,
                   "layer_copies": copies,
                   "l2": "inputs larger than L2: %d layer copies and token batches cycled" % copies,
                   "distinct_experts_per_step": round(statistics.mean(distinct), 2),
                   "graphs": "one CUDA graph per (layer copy, batch), replayed; the last %d timed steps use "
                             "graphs that also record stage events; a device-side spin precedes the "
                             "timed region so that the host has queued the steps" % n_ev},
        "roofline": roof, "stages_us": stages_us, "e2e": e2e,
        "gpu_launches": launches_per_step * steps, "clocks": sampler.summary(),
    }


def workload_string(name, cfg, K, mode, T):
    """The workload named identically by both arms."""
    return "%s: H=%d I=%d E=%d top-k=%d K=%d %s T=%d" % (name, cfg.H, cfg.I, cfg.E, cfg.topk, K, mode.upper(), T)


# DRAM bytes per launch of the dominant kernel from one ncu capture of this
# program (profiles/); workloads without a capture of the current kernel get
# None
NCU_TRAFFIC = {
    ("decode", 8, "w4a8"): (28.400e6, "profiles/k_dec_warp_fc1_decode_w4a8_T8.md"),
    ("prefill", 2048, "w4a16"): (212.30e6, "profiles/k_tc_fc_fused_prefill_w4a16_T2048.md"),
}

# The metric's other configurations, measured in the same run as the headline
# (decode T=8): decode at T = 1, 2 and 4 and the T=2048 prefill.
SUB_RUNS = [("decode", 1, "w4a8"), ("decode", 2, "w4a8"), ("decode", 4, "w4a8"), ("prefill", 2048, "w4a16")]


def run_ours(args, rank, world):
    import torch
    from trellis_quantized_moe_route_gb300 import binding, build

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    build.build()
    binding.load_library()
    name, T_default, mode = WORKLOADS[args.workload]
    cfg = synth.CONFIGS[name]
    T = args.tokens or T_default
    e2e_steps = min(args.steps, 200)
    head = measure_layer(name, T, mode, args.steps, args.warmup, rank, world, dev, e2e_steps)
    res = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic", "config": head["config"],
           "roofline": head["roofline"], "stages_us": head["stages_us"], "e2e": head["e2e"],
           "gpu_launches": head["gpu_launches"], "clocks": head["clocks"]}
    if args.workload == "decode" and not args.tokens and not args.no_sub:
        subs = []
        for (n2, t2, m2) in SUB_RUNS:
            r = measure_layer(n2, t2, m2, args.steps, args.warmup, rank, world, dev, e2e_steps)
            r["metric"] = METRIC
            r["higher_is_better"] = True
            subs.append(r)
        res["sub"] = subs
        res["gpu_launches"] += sum(r["gpu_launches"] for r in subs)
    return res, (cfg, T, mode, None)


# -------------------------------------------------------------- reference ---
def oracle_sample(cfg, T, mode, budget_s, seed=1000):
    """Time the float64 CPU oracle on whole batches of the workload (or on a
    prefix of one batch) for about ``budget_s`` seconds. Returns (tokens/s,
    description)."""
    from oracle import layer as olayer, route as oroute
    L = synth.make_layer(cfg)
    x_bits, logits = synth.make_tokens(cfg, T=T, seed=seed)
    done, t_start = 0, time.perf_counter()
    n = min(T, 8)
    while True:
        toks = np.arange(done % T, done % T + n) % T
        ids, w = oroute.route_topk_softmax(logits[toks], cfg.topk)
        olayer.layer_forward(L, x_bits[toks], ids, w, mode=mode)
        done += n
        el = time.perf_counter() - t_start
        if el > budget_s:
            break
    return done / el, "%d tokens of the %s workload in %.1f s (oracle: router, per-expert decode, float64 GEMMs)" % (
        done, cfg.name, el)


def cpu_baseline(cfg, T, mode, budget_s=12.0):
    v, desc = oracle_sample(cfg, T, mode, budget_s)
    return {"value": round(v, 3), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle", "sample": desc}


def run_reference(args, rank, world):
    if args.workload == "linear":
        c = LINEAR
        T = args.tokens or c["T"]
        lin = synth.make_linear(c["N"], c["K"], c["bits"], c["rot_in"], c["rot_out"], seed=40)
        cb = linear_cpu_baseline(lin, T, budget_s=min(60.0, 5.0 * max(args.steps, 1)))
        return {
            "impl": "reference", "metric": LINEAR_METRIC, "value": cb["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * 64 / cb["value"], 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "linear: N=%d K=%d W4A16 T=%d" % (c["N"], c["K"], T)}, "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
    cfg_name, T_default, mode = WORKLOADS[args.workload]
    cfg = synth.CONFIGS[cfg_name]
    T = args.tokens or T_default
    budget = max(1.0, min(8.0, 150.0 / max(args.steps + args.warmup, 1)))
    for _ in range(min(args.warmup, 2)):
        oracle_sample(cfg, T, mode, 0.0)
    vals = []
    t0 = time.perf_counter()
    for i in range(args.steps):
        v, desc = oracle_sample(cfg, T, mode, budget, seed=2000 + i)
        vals.append(v)
        if time.perf_counter() - t0 > 170.0:
            break
    value = statistics.mean(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * min(T, 8) / value, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_string(cfg_name, cfg, max(cfg.bits), mode, T)},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "%d steps of about %.1f s each, up to 8 tokens per oracle call (%s)" % (
                             len(vals), budget, desc)},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------- dense linear ---
LINEAR = dict(N=4096, K=4096, bits=4, rot_in=128, rot_out=128, T=2048)
LINEAR_METRIC = "dense trellis linear tokens/s (N=K=4096, K=4 trellis, W4A16, T=2048); % of tensor roofline"


def run_linear(args, rank, world):
    """The dense trellis linear layer (no routing): rotate + tensor-core
    projection per step, replayed from one graph per weight copy."""
    import torch
    from trellis_quantized_moe_route_gb300 import binding, build

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    build.build()
    binding.load_library()
    c = LINEAR
    T = args.tokens or c["T"]
    N, K = c["N"], c["K"]
    # weights + x + out per copy ~ N*K/2 + 2TK + 4TN bytes; copies until two
    # uses of one copy are more than 2x L2 apart
    per_copy = N * K * c["bits"] // 8 + 2 * T * K + 4 * T * N
    copies = int(min(16, max(2, np.ceil(2 * L2_BYTES / per_copy) + 1)))
    lins = [synth.make_linear(N, K, c["bits"], c["rot_in"], c["rot_out"], seed=40 + i) for i in range(copies)]
    mods = [binding.TrellisLinear(l, max_tokens=T) for l in lins]
    xs = [torch.from_numpy(np.ascontiguousarray(synth.make_linear_tokens(l, T, seed=1000 + 17 * rank + i).view(np.int16))).cuda()
          for i, l in enumerate(lins)]
    outs = [torch.empty((T, N), dtype=torch.float32, device="cuda") for _ in range(copies)]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            mods[i % copies].forward(xs[i % copies], out=outs[i % copies])
    torch.cuda.synchronize()
    graphs = []
    for i in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            mods[i].forward(xs[i], out=outs[i])
        graphs.append(g)
    for i in range(max(args.warmup, 3)):
        graphs[i % copies].replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            graphs[i % copies].replay()
    t1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = job_time_ms(t0.elapsed_time(t1), world)
    step_us = total_ms * 1e3 / args.steps
    for i in range(copies):
        assert mods[i].poll_error() == 0
    pk = peaks()
    flops = 2 * T * N * K
    achieved = flops / (step_us * 1e-6) / 1e12
    res = {
        "metric": LINEAR_METRIC, "value": round(job_value(args.steps, T, world, total_ms), 2), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": "linear: N=%d K=%d K_trellis=%d W4A16 rot %d/%d T=%d" % (N, K, c["bits"], c["rot_in"],
                                                                                      c["rot_out"], T),
                   "tokens_per_step": T, "weight_copies": copies,
                   "l2": "inputs larger than L2: %d weight copies with their token batches cycled" % copies,
                   "graphs": "one CUDA graph per copy (route map, rotate, projection), replayed"},
        "roofline": {"bound": "tensor", "kernel": "whole call: k_linear_map + k_rotate_quant + k_tc_fc<FC2> (tcgen05)",
                     "achieved": round(achieved, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / pk["bf16_tflops"], 4),
                     # DRAM bytes of the projection launch from one ncu capture of this workload
                     "traffic": 26.36e6 if (N, K, T) == (4096, 4096, 2048) else None,
                     "traffic_source": "profiles/k_tc_fc_fc2_linear_w4a16_N4096_T2048.md (k_tc_fc<FC2> launch)",
                     "peak_source": pk["source"] + " (bf16 dense burst; fp16 runs at the bf16 rate)",
                     "flops_per_launch": flops},
        "e2e": None, "gpu_launches": 3 * args.steps, "clocks": sampler.summary(),
    }
    return res, (lins[0], T)


def linear_cpu_baseline(lin, T, budget_s=10.0):
    """The float64 oracle on a bounded sample of the linear workload's tokens
    (weights decoded once, counted in the time)."""
    from oracle import linear as olinear
    x = synth.make_linear_tokens(lin, T, seed=1000)
    t0 = time.perf_counter()
    w = olinear.linear_weights(lin)
    done, n = 0, 64
    while True:
        olinear.linear_apply(lin, synth.bf16_to_f64(x[done % T:done % T + n]), True, w)
        done += n
        el = time.perf_counter() - t0
        if el > budget_s:
            break
    return {"value": round(done / el, 3), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": "%d tokens of the linear workload in %.1f s (oracle: decode W once, float64 rotations and GEMM)"
                      % (done, el)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS) + ["linear"])
    ap.add_argument("--tokens", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="headline workload only (no decode T=1/2/4 and prefill lines)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("gloo")
    if args.workload == "linear":
        res, (lin, T) = run_linear(args, rank, world)
        if rank == 0:
            if not args.no_cpu_baseline:
                res["cpu_baseline"] = linear_cpu_baseline(lin, T)
            print(json.dumps(res), flush=True)
        if world > 1:
            import torch
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return
    res, (cfg, T, mode, _) = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(cfg, T, mode)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
