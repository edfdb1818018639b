"""Benchmark of the single-GPU MoE layer forward pass (one JSON line on rank 0).

Default workload: the DeepSeek-V3-shaped prefill layer (T=8192 tokens, d=7168, 256 routed
experts of inner width 2048 plus one shared expert, top-8, sigmoid scores with a selection
bias), bf16 with fp32 accumulation, on synthetic seeded inputs resident in HBM.  A step is one
full forward pass (router GEMM, top-k, dispatch, gather, gate/up GEMM + SwiGLU, down GEMM,
combine).  The decode-shaped layer (T=128, same shapes) is measured the same way and
reported under "decode".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config C]

Under torchrun each rank runs an independent replica on its own tokens (data parallel, no
collective on the data path); the time is the max over ranks and the value counts the tokens
of all ranks.  ``--impl reference`` times the fp64 CPU oracle (the reference arm) on a
bounded sample of the same workload, on rank 0 only.
"""
import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_inputs import configs  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
# oracle sample sizes (tokens) giving roughly 10-30 s of single-core fp64 work
CPU_SAMPLE = {0: 64, 1: 8, 2: 12, 3: 12, 4: 16}
# the one metric string both arms print (the reference arm is the fp64 oracle on host cores)
METRIC = ("MoE-layer tokens/s, DeepSeek-V3 shape (T=8192 prefill; T=128 decode under "
          "'decode')")
REF_SAMPLE = {0: 64, 1: 4, 2: 3, 3: 3, 4: 8}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def layer_flops(c):
    """Active-parameter FLOPs of one pass: router + k routed experts + shared expert."""
    T, d, E, k, F, Fs = c["T"], c["d"], c["E"], c["k"], c["F"], c["Fs"]
    return T * (2 * d * E + 6 * d * F * k + 6 * d * Fs)


def layer_bytes(c, counts):
    """Bytes the method must move: x, router weights, touched experts, shared expert, out."""
    s = 2 if c["dtype"] == "bf16" else 4
    T, d, E, F, Fs = c["T"], c["d"], c["E"], c["F"], c["Fs"]
    touched = int((np.asarray(counts) > 0).sum())
    return T * d * s + E * d * s + touched * 3 * d * F * s + 3 * d * Fs * s + T * d * s


def gateup_flops(c):
    T, d, k, F, Fs = c["T"], c["d"], c["k"], c["F"], c["Fs"]
    return 2 * d * (T * k * 2 * F + T * 2 * Fs)


def gateup_weight_bytes(c, counts):
    touched = int((np.asarray(counts) > 0).sum())
    return 2 * (touched * 2 * c["F"] * c["d"] + 2 * c["Fs"] * c["d"])


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, kept for the timed region."""

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(1.0)

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t0, t1):
        rows = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
                rows.append((ts, float(f[2]), float(f[3]), f[6:10], float(f[4])))
            except (ValueError, IndexError):
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        note = None
        if not inside:
            inside = sorted(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))[:3]
            note = "timed region shorter than the sampling period: nearest samples used"
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        out = {"sm_mhz": float(np.median([r[1] for r in inside])),
               "sm_max_mhz": float(max(r[2] for r in inside)), "reasons": reasons,
               "samples": len(inside),
               "power_w_median": float(np.median([r[4] for r in inside])),
               "power_w_max": float(max(r[4] for r in inside)),
               "sw_power_cap_samples": sum(1 for r in inside if r[3][3] == "Active")}
        if note:
            out["note"] = note
        return out


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value, world):
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def rank_inputs(c, rank):
    """Model weights are shared by all replicas; each rank draws its own tokens."""
    import moe_inputs
    dev = moe_inputs.device_inputs(c)
    if rank > 0:
        dev["x"] = moe_inputs.device_tensor(dict(c, seed=c["seed"] + 7919 * rank), "x")
    return dev


class Runner:
    """Device buffers and one-step closures for a config."""

    def __init__(self, c, dev):
        import torch
        import mixture_experts_layer_83_b300 as moe
        self.moe, self.torch, self.c, self.dev = moe, torch, c, dev
        T, d, E, k = c["T"], c["d"], c["E"], c["k"]
        dt = moe.MOE_DTYPE_BF16 if c["dtype"] == "bf16" else moe.MOE_DTYPE_F32
        self.shape = moe.make_shape(T, d, E, k, c["F"], c["Fs"], dt)
        self.ws_bytes = moe.moe_layer_workspace_size(self.shape)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        self.out = torch.empty_like(dev["x"])
        self.counts = torch.empty(E, dtype=torch.int32, device="cuda")
        self.shared = (dev["sh_gate_up"], dev["sh_down"]) if c["Fs"] > 0 else None
        self.stream = torch.cuda.current_stream()
        self.launches = moe.moe_layer_num_launches(self.shape)
        self.options = {}   # routing options of moe_layer_forward (group limits, capacity)

    def step(self, x=None, events=None):
        d = self.dev
        self.moe.moe_layer_forward(self.shape, d["x"] if x is None else x, d["w_router"],
                                   d["w_gate_up"], d["w_down"], self.c["score"], d.get("bias"),
                                   self.shared, self.out, self.counts, self.ws, self.ws_bytes,
                                   self.stream, stage_events=events, **self.options)

    def timed(self, steps, warmup, world, with_stages=True):
        torch = self.torch
        nst = self.moe.MOE_NUM_STAGE_EVENTS
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(steps)]
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        start.record(self.stream)
        for i in range(steps):
            self.step(events=evs[i] if with_stages else None)
        stop.record(self.stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
        ms = start.elapsed_time(stop) / steps
        stages = None
        if with_stages:
            per = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(nst - 1)]
                            for i in range(steps)])
            stages = per.mean(0)
        return ms, stages, (t0, t1)

    def timed_e2e(self, steps, warmup, world):
        """End to end through the public entry point, every step: pinned host x -> device,
        forward, device out + expert counts -> pinned host.  Copies run on their own streams,
        double-buffered, so step i+1's upload and step i-1's read-back overlap step i; the timed
        region spans the first upload to the last read-back."""
        torch = self.torch
        x_host = self.dev["x"].cpu().pin_memory()
        nbuf = 2
        x_dev = [torch.empty_like(self.dev["x"]) for _ in range(nbuf)]
        out_dev = [torch.empty_like(self.out) for _ in range(nbuf)]
        cnt_dev = [torch.empty_like(self.counts) for _ in range(nbuf)]
        out_host = [torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory() for _ in range(nbuf)]
        cnt_host = [torch.empty(self.counts.shape, dtype=torch.int32).pin_memory() for _ in range(nbuf)]
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        comp = self.stream
        uploaded = [torch.cuda.Event() for _ in range(nbuf)]
        computed = [torch.cuda.Event() for _ in range(nbuf)]
        consumed = [torch.cuda.Event() for _ in range(nbuf)]   # x buffer free again
        read_back = [torch.cuda.Event() for _ in range(nbuf)]  # out buffer free again
        for e in consumed + read_back:
            e.record(comp)

        def run(n):
            for i in range(n):
                b = i % nbuf
                with torch.cuda.stream(up):
                    up.wait_event(consumed[b])
                    x_dev[b].copy_(x_host, non_blocking=True)
                    uploaded[b].record(up)
                comp.wait_event(uploaded[b])
                comp.wait_event(read_back[b])
                self.moe.moe_layer_forward(self.shape, x_dev[b], self.dev["w_router"],
                                           self.dev["w_gate_up"], self.dev["w_down"],
                                           self.c["score"], self.dev.get("bias"), self.shared,
                                           out_dev[b], cnt_dev[b], self.ws, self.ws_bytes, comp)
                consumed[b].record(comp)
                computed[b].record(comp)
                with torch.cuda.stream(down):
                    down.wait_event(computed[b])
                    out_host[b].copy_(out_dev[b], non_blocking=True)
                    cnt_host[b].copy_(cnt_dev[b], non_blocking=True)
                    read_back[b].record(down)

        run(warmup)
        torch.cuda.synchronize()
        barrier(world)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(up)
        run(steps)
        down.wait_stream(up)
        down.wait_stream(comp)
        stop.record(down)
        torch.cuda.synchronize()
        barrier(world)
        ms = start.elapsed_time(stop) / steps
        h2d = x_host.numel() * x_host.element_size()
        d2h = out_host[0].numel() * out_host[0].element_size() + cnt_host[0].numel() * 4
        return ms, h2d, d2h


def code_digest(files):
    """sha256 of C/C++/CUDA sources with comments and blank lines removed: a change to the code
    changes it, an edit of comments alone does not."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in files:
        text = open(os.path.join(ROOT, f), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()


def traffic_record(kernel):
    """Per-launch DRAM bytes from a committed ncu summary, if the kernel code is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    return rec["bytes_per_launch"] if code_digest(rec.get("sources", [])) == rec.get("sha256") else None


def cpu_oracle_sample(c, dev, ntok, rank_seed_note=""):
    """Time the oracle (single thread, as it stands) on the first ``ntok`` tokens of the
    workload: router scores, top-k, routed experts, shared expert, combine."""
    import torch
    import oracle
    oracle.build()
    bf = c["dtype"] == "bf16"

    def host(t):
        t = t.contiguous()
        return t.view(torch.int16).cpu().numpy().view(np.uint16) if bf else t.cpu().numpy()

    x = host(dev["x"][:ntok])
    wr = host(dev["w_router"])
    bias = dev["bias"].cpu().numpy() if "bias" in dev else None
    # experts the sample needs (input plumbing, outside the timed region)
    _, sc, key = oracle.router_scores(x, wr, c["score"], bias)
    idx, _, _ = oracle.topk(key, sc, c["k"])
    experts = sorted(set(idx.ravel().tolist()))
    gu = {e: host(dev["w_gate_up"][e]) for e in experts}
    dn = {e: host(dev["w_down"][e]) for e in experts}
    shg = host(dev["sh_gate_up"]) if c["Fs"] > 0 else None
    shd = host(dev["sh_down"]) if c["Fs"] > 0 else None
    t0 = time.perf_counter()
    _, sc, key = oracle.router_scores(x, wr, c["score"], bias)
    idx, w, _ = oracle.topk(key, sc, c["k"])
    oracle.layer_rows(x, idx, w, gu, dn, shg, shd)
    dt = time.perf_counter() - t0
    return ntok / dt, dt


def cpu_baseline_entry(args, world, rank, c, dev):
    """The oracle timed on a bounded sample of config ``c`` (rank 0 of a one-GPU run only)."""
    if args.no_cpu_baseline or world != 1 or rank != 0:
        return None
    n = next(CPU_SAMPLE[i] for i, x in configs.CONFIGS.items() if x["name"] == c["name"])
    v, dt = cpu_oracle_sample(c, dev, n)
    return {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", **host_cores(),
            "sample": f"first {n} tokens of the {c['name']} batch: router, top-k, routed "
                      f"experts{', shared expert' if c['Fs'] > 0 else ''}, combine in fp64 "
                      f"({dt:.1f} s)"}


def run_reference(args, c):
    world, rank, local = dist_info()
    if rank != 0:
        return 0
    import torch
    torch.cuda.set_device(local)
    import moe_inputs
    dev = moe_inputs.device_inputs(c)
    torch.cuda.synchronize()
    n = REF_SAMPLE[args.config]
    for _ in range(args.warmup):
        cpu_oracle_sample(c, dev, n)
    times = [cpu_oracle_sample(c, dev, n)[1] for _ in range(args.steps)]
    t = float(np.sum(times))
    value = n * args.steps / t
    line = {"impl": "reference", "metric": METRIC, "value": value,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(c),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             **host_cores(),
                             "sample": f"{n} tokens per step (first {n} of the batch), router + "
                                       f"top-k + routed and shared experts + combine"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def host_cores():
    """The host's core counts, stated beside the single-threaded oracle's figure."""
    try:
        usable = len(os.sched_getaffinity(0))
    except AttributeError:
        usable = os.cpu_count()
    return {"host_nproc": os.cpu_count(), "host_cores_usable": usable}


def workload_config(c):
    return {"workload": f"{c['name']}: T={c['T']} d={c['d']} E={c['E']} top-{c['k']} "
                        f"F={c['F']} shared Fs={c['Fs']} "
                        f"{'sigmoid+bias' if c['score'] == configs.SIGMOID else 'softmax'} "
                        f"{c['dtype']} seed={c['seed']}",
            "T": c["T"], "d": c["d"], "E": c["E"], "k": c["k"], "F": c["F"], "Fs": c["Fs"],
            "l2": "inputs larger than L2 (every step streams the touched expert weights, "
                  "GBs per step, through a 126 MB L2)",
            "parallelism": "replicas (data parallel, no collective on the data path)"}


def measure(c, args, world, rank, peaks, sampler, kind):
    import torch
    dev = rank_inputs(c, rank)
    torch.cuda.synchronize()
    r = Runner(c, dev)
    ms, stages, (t0, t1) = r.timed(args.steps, args.warmup, world)
    ms_max = max_over_ranks(ms, world)
    counts = r.counts.cpu().numpy()
    res = {"ms": ms_max, "ms_local": ms, "stages": stages, "t0": t0, "t1": t1, "counts": counts,
           "runner": r, "dev": dev, "kernel_clocks": kernel_clocks(r)}
    res["layer"] = layer_roofline(c, counts, ms_max, peaks)
    return res


# Nominal dense bf16 rate of one SM per clock (2.25 PFLOP/s over 148 SMs at 1.86 GHz).
NOMINAL_BF16_FLOP_PER_CLK_SM = 8192
B300_SMS = 148


def kernel_clocks(r):
    """SM clock (MHz) and duration (ms) of the last timed pass's tensor-core kernels, as CTA 0
    of each recorded them (bf16 layers only): the clock the kernels really ran at."""
    if r.c["dtype"] != "bf16":
        return None
    kc = r.moe.moe_workspace_kernel_clocks(r.ws)
    return {k: {"sm_mhz": round(v[0], 1), "ms": round(v[1], 4)} for k, v in kc.items() if v[0] > 0}


def layer_roofline(c, counts, ms, peaks):
    """Layer roofline: t_roof = max(FLOPs / bf16 peak, bytes / HBM peak) over the step time.
    The timed region is a fraction of a second of back-to-back passes, which runs at the
    maximum SM clock (the clock record of the run shows it), so the peak is the measured
    burst bf16 figure; the fraction against the sustained (seconds-long, power-capped) figure
    is given beside it as context only."""
    fl = layer_flops(c)
    by = layer_bytes(c, counts)
    t_mem = by / (peaks["hbm_gbs"] * 1e9)
    t_tc = fl / (peaks["bf16_tflops"] * 1e12)
    t_roof = max(t_tc, t_mem)
    t_roof_sus = max(fl / (peaks["bf16_tflops_sustained"] * 1e12), t_mem)
    return {"tflops": fl / (ms * 1e-3) / 1e12, "gbs": by / (ms * 1e-3) / 1e9,
            "flop": fl, "bytes": by, "roofline_ms": t_roof * 1e3,
            "roofline_frac": t_roof * 1e3 / ms,
            "roofline_peaks": "bf16 burst and HBM copy, measured",
            "bound": "tensor" if t_tc >= t_mem else "hbm",
            "context_roofline_frac_at_sustained_bf16": t_roof_sus * 1e3 / ms}


def other_configs(args, world, rank, peaks):
    """The tiny fp32 and the Mixtral-8x7B-shaped layers: time per pass and roofline fraction."""
    import torch
    out = {}
    for cid in (0, 1):
        c = configs.CONFIGS[cid]
        res = measure(c, args, world, rank, peaks, None, c["name"])
        out[c["name"]] = {"workload": workload_config(c)["workload"], "ms_per_step": res["ms"],
                          "tokens_per_s": c["T"] * world / (res["ms"] * 1e-3),
                          "layer": res["layer"], "kernel_clocks": res["kernel_clocks"],
                          "stages_ms": {n: float(v) for n, v in
                                        zip(res["runner"].moe.STAGE_NAMES, res["stages"])}}
        if c["dtype"] != "bf16":
            out[c["name"]]["note"] = ("true-fp32 CUDA-core path, launch-bound at this size: the "
                                      "bf16 tensor roofline does not bound it")
        out[c["name"]]["cpu_baseline"] = cpu_baseline_entry(args, world, rank, c, res["dev"])
        del res
        torch.cuda.empty_cache()
    return out


def eplb_report(counts, n_gpus):
    """The library's replica plan on this pass's expert counts: per-GPU expected load, max over
    mean, for the contiguous placement and for plans with 0, 1 and 4 redundant slots per GPU."""
    import mixture_experts_layer_83_b300 as moe
    contiguous = counts.reshape(n_gpus, -1).sum(1)
    out = {"gpus": n_gpus, "contiguous_max_over_mean": float(contiguous.max() / contiguous.mean())}
    for per_gpu in (0, 1, 4):
        t0 = time.perf_counter()
        _, _, gl = moe.moe_eplb_plan(counts, n_gpus, per_gpu * n_gpus)
        out[f"plan_redundant_{per_gpu * n_gpus}"] = {
            "gpu_max_over_mean": float(gl.max() / gl.mean()),
            "plan_us": (time.perf_counter() - t0) * 1e6}
    return out


def skew_report(args, world, rank):
    """The Zipf-skewed layer: time per pass and the expert / group load (max over mean of the
    dispatched assignments; the 8 contiguous groups of 16 experts stand for an expert-parallel
    placement over 8 GPUs), dropless and under the two routing options that act on skew."""
    import torch
    c = configs.CONFIGS[4]
    dev = rank_inputs(c, rank)
    torch.cuda.synchronize()
    r = Runner(c, dev)
    dropped = torch.zeros(4, dtype=torch.int32, device="cuda")
    groups = c["groups"]
    res = {"workload": workload_config(c)["workload"],
           "groups": f"{groups} contiguous groups of {c['E'] // groups} experts"}
    variants = (("dropless", {}),
                ("group_limited_4_of_8", dict(n_groups=groups, topk_groups=4)),
                ("capacity_1.25", dict(capacity_factor=1.25, dropped=dropped)),
                ("capacity_1.25_reroute_4", dict(capacity_factor=1.25, dropped=dropped, reroute=4)))
    for name, opts in variants:
        r.options = opts
        ms, _, _ = r.timed(args.steps, args.warmup, world, with_stages=False)
        counts = r.counts.cpu().numpy()
        load = r.moe.moe_load_report(counts, groups)
        entry = {"ms_per_step": ms, "tokens_per_s": c["T"] / (ms * 1e-3),
                 "expert_max_over_mean": load["expert_max_over_mean"],
                 "group_max_over_mean": load["group_max_over_mean"],
                 "experts_touched": load["experts_touched"]}
        if "capacity_factor" in opts:
            entry["dropped_assignments"] = int(dropped[0].item())
            entry["dropped_fraction"] = int(dropped[0].item()) / (c["T"] * c["k"])
        if name == "dropless":
            entry["eplb"] = eplb_report(counts.astype(np.int32), groups)
        res[name] = entry
    res["cpu_baseline"] = cpu_baseline_entry(args, world, rank, c, dev)
    del r, dev
    torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--decode-config", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--T", type=int, default=None, help="override tokens (profiling cases)")
    ap.add_argument("--E", type=int, default=None, help="override routed experts (profiling)")
    ap.add_argument("--F", type=int, default=None,
                    help="override the expert inner width (profiling: smaller weights)")
    ap.add_argument("--profile", action="store_true",
                    help="only warm-up + timed steps of the main workload (for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    c = dict(configs.CONFIGS[args.config])
    if args.T is not None or args.E is not None or args.F is not None:
        c["T"] = args.T or c["T"]
        c["E"] = args.E or c["E"]
        c["F"] = args.F or c["F"]
        c["Fs"] = min(c["Fs"], c["F"])
        c["name"] = f"{c['name']} (T={c['T']}, E={c['E']}, F={c['F']} profiling case)"
    if args.profile:
        return run_profile(args, c)
    if args.impl == "reference":
        return run_reference(args, c)

    world, rank, local = dist_info()
    import torch
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import mixture_experts_layer_83_b300 as moe
    moe.lib()
    peaks, peak_src = load_peaks()

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    main_res = measure(c, args, world, rank, peaks, sampler, "prefill")
    r = main_res["runner"]
    e2e_ms, h2d, d2h = r.timed_e2e(args.steps, args.warmup, world)
    e2e_ms = max_over_ranks(e2e_ms, world)
    dc = configs.CONFIGS[args.decode_config]
    del main_res["runner"], r
    torch.cuda.empty_cache()
    dec = measure(dc, args, world, rank, peaks, sampler, "decode")
    del dec["runner"]
    torch.cuda.empty_cache()
    skew = skew_report(args, world, rank)
    others = other_configs(args, world, rank, peaks)
    if rank == 0:
        sampler.stop()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    ms = main_res["ms"]
    T = c["T"]
    value = T * world / (ms * 1e-3)
    st = main_res["stages"]
    names = moe.STAGE_NAMES
    gu_ms = float(st[names.index("gateup_gemm")])
    gu_fl = gateup_flops(c)
    achieved = gu_fl / (gu_ms * 1e-3) / 1e12
    traffic = traffic_record("gemm_gateup_prefill")
    # samples taken inside each workload's own timed region
    clocks = sampler.summary(main_res["t0"], main_res["t1"])
    dec_clocks = sampler.summary(dec["t0"], dec["t1"])
    # The timed region is a fraction of a second of back-to-back passes: the gate/up GEMM's
    # peak is the measured burst bf16 figure (the burst rate of a kernel timed alone), although
    # the board reaches its power limit within it and the GEMMs run below the maximum SM clock
    # (their own clock records: "sm_mhz_in_kernel").  The fraction of the sustained
    # (seconds-long, power-capped) figure is context only.
    roof = {"kernel": "gemm_tc_kernel<1,2,1> gate/up + SwiGLU (tcgen05, wide CTA pairs)",
            "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
            "traffic": traffic,
            "peak_source": f"{peak_src} bf16 burst (timed region {ms * args.steps:.0f} ms of "
                           f"{args.steps} back-to-back passes)",
            "algorithmic_flop_per_launch": gu_fl, "ms_per_launch": gu_ms,
            "sm_mhz_median": clocks.get("sm_mhz"),
            "ms_x_ghz": gu_ms * clocks["sm_mhz"] / 1e3 if clocks.get("sm_mhz") else None,
            "context_frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
    kc = main_res["kernel_clocks"] or {}
    if "gateup_gemm" in kc:
        # the clock the GEMM ran at (its CTA 0's SM clock counter over the global timer, last
        # timed pass), and its tensor-pipe use per clock against the nominal per-SM rate
        mhz = kc["gateup_gemm"]["sm_mhz"]
        roof["sm_mhz_in_kernel"] = mhz
        roof["tensor_util_at_kernel_clock"] = achieved * 1e12 / (
            B300_SMS * NOMINAL_BF16_FLOP_PER_CLK_SM * mhz * 1e6)

    dms = dec["ms"]
    dst = dec["stages"]
    d_gu_ms = float(dst[names.index("gateup_gemm")])
    d_dn_ms = float(dst[names.index("down_gemm")])
    d_gu_bytes = gateup_weight_bytes(dc, dec["counts"])
    d_dn_bytes = d_gu_bytes // 2   # down weights: d x F per touched expert (+ the shared one)
    # summary keys last, so that they survive in the end of the printed line
    decode = {"workload": workload_config(dc)["workload"],
              "stages_ms": {n: float(v) for n, v in zip(names, dst)},
              "kernel_clocks": dec["kernel_clocks"],
              "clocks": dec_clocks,
              "cpu_baseline": cpu_baseline_entry(args, world, rank, dc, dec["dev"]),
              "experts_touched": int((dec["counts"] > 0).sum()),
              "down_gemm_hbm_frac": d_dn_bytes / (d_dn_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
              "layer": dec["layer"],
              "roofline": {"kernel": "gemm_tc_kernel<1,2,0> gate/up + SwiGLU (tcgen05, narrow CTA "
                                     "pairs)", "bound": "hbm",
                           "achieved": d_gu_bytes / (d_gu_ms * 1e-3) / 1e9,
                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": d_gu_bytes / (d_gu_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                           "traffic": traffic_record("gemm_gateup_decode"),
                           "peak_source": f"{peak_src} HBM copy"},
              "unit": "tokens/s", "value": dc["T"] * world / (dms * 1e-3), "ms_per_step": dms,
              "layer_roofline_frac": dec["layer"]["roofline_frac"]}

    cpu = cpu_baseline_entry(args, world, rank, c, main_res["dev"])
    line = {
        "metric": METRIC,
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(c),
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": T * world / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copies": "pinned host buffers, every step; uploads and read-backs on their own "
                          "streams, double-buffered, overlapping the neighbouring steps' compute"},
        "gpu_launches": int(r_launches(c) * args.steps),
        "clocks": clocks,
        "kernel_clocks": main_res["kernel_clocks"],
        "layer": main_res["layer"],
        "stages_ms": {n: float(v) for n, v in zip(names, st)},
        "other_configs": others,
        # kept last: a reader that keeps only the end of the line still sees these two
        "skewed": skew,
        "decode": decode,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_profile(args, c):
    """Warm-up + timed steps of one workload, nothing else (keeps ncu captures small)."""
    import torch
    import mixture_experts_layer_83_b300 as moe
    moe.lib()
    dev = rank_inputs(c, 0)
    torch.cuda.synchronize()
    r = Runner(c, dev)
    ms, stages, _ = r.timed(args.steps, args.warmup, 1)
    print(json.dumps({"profile": c["name"], "ms_per_step": ms,
                      "stages_ms": {n: float(v) for n, v in zip(moe.STAGE_NAMES, stages)}}))
    return 0


def r_launches(c):
    import mixture_experts_layer_83_b300 as moe
    dt = moe.MOE_DTYPE_BF16 if c["dtype"] == "bf16" else moe.MOE_DTYPE_F32
    return moe.moe_layer_num_launches(moe.make_shape(c["T"], c["d"], c["E"], c["k"], c["F"],
                                                     c["Fs"], dt))


if __name__ == "__main__":
    sys.exit(main())
