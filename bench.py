#!/usr/bin/env python3
"""Benchmark: INT4 block-quantized MoE FFN layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config decode|tiny|verify|prefill|stack|e128_decode|e128_prefill|e256_decode|e256_prefill]

A step is one pass of the whole layer (router, expert FFNs, weighted
combine) over one batch of T tokens.  The default workload is the
Qwen1.5-MoE-A2.7B-shaped decode layer (T=1, H=2048, I=1408, E=60, top-4,
uint4 block 32 with zero points, fp16).  Weights rotate over a pool of
independent layers far larger than L2, so every step streams its experts
from HBM.  Prints one JSON line (rank 0).  The default decode run also
measures, in the same run and line ("configs"), the T=16 verify-sized decode
layer, the T=512 prefill layer and the 24-layer T=2048 stack.  Every timed
region is K steps bracketed by a barrier and a synchronize, repeated at
least ten times (and for at least 0.3 s while the SM clock is sampled); the
reported time is the median region, with p10 and p90.

--impl reference times the fp64 CPU oracle (the correctness reference) on
the same workload instead: a deliberately slow baseline, not a target.
N > 1 (torchrun): independent replicas, one per GPU, no collective on the
data path; value = tokens of all ranks / the slowest rank's time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "QMoE layer tokens/s; decode HBM GB/s and prefill TFLOPS as % of GB300 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant
# kernel from an ncu capture of the current build (profiles/; None: not
# captured since the kernel last changed)
NCU_TRAFFIC = {("decode", "layer"): 20924672.0, ("prefill", "gateup"): 132435456.0,
               ("verify", "gateup"): 133735424.0}
POOL = {"tiny": 4, "decode": 24, "verify": 24, "prefill": 8, "stack": 24,
        "e128_decode": 24, "e128_prefill": 8, "e256_decode": 24, "e256_prefill": 8}
DEFAULT_STEPS = {"tiny": 2400, "decode": 24000, "verify": 4800, "prefill": 480, "stack": 60,
                 "e128_decode": 24000, "e128_prefill": 480, "e256_decode": 24000, "e256_prefill": 480}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="decode", choices=list(POOL) + ["gptq_repack"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="decode headline only (no verify / prefill / stack measurements in the same line)")
    ap.add_argument("--pool", type=int, default=None,
                    help="resident weight sets (default: enough that a revisit misses L2); "
                         "smaller pools only for profiler captures, which flush caches themselves")
    a = ap.parse_args()
    if a.steps is None:
        a.steps = DEFAULT_STEPS.get(a.config, 50)
    if a.warmup is None:
        a.warmup = max(3, min(240, a.steps // 10))
    a.warmup = max(3, a.warmup)
    return a


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None

    def start(self):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def dist_init():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def is_decode(wl):
    from int4_block_quantized_gb300 import binding
    return wl.T <= binding.AUTO_DECODE_MAX_TOKENS  # the path QMOE_PATH_AUTO takes


def workload_bytes(wl, D):
    """Algorithmic bytes and FLOPs of one layer: weights of the D distinct
    selected experts, router, x in, out; per kernel the same for its share."""
    from int4_block_quantized_gb300 import synthetic as S
    A = wl.T * wl.k
    nbh, nbi = wl.H // wl.block_size, wl.I // wl.block_size
    zp = 1 if wl.has_zp else 0
    gu = 2 * wl.I * (wl.H // 2 + nbh * 2 + nbh * zp)          # gate + up of one expert
    dn = wl.H * (wl.I // 2 + nbi * 2 + nbi * zp)               # down of one expert
    assert gu + dn == S.expert_bytes(wl)
    router = wl.H * wl.E * 2 + (wl.E * 4 if wl.zipf_s else 0)
    xio = 2 * wl.T * wl.H * 2
    layer = D * (gu + dn) + router + xio
    if is_decode(wl):
        gateup_kernel = D * gu + wl.T * wl.H * 2 + A * wl.I * 4    # x in, fp32 act out
        down_kernel = D * dn + A * wl.I * 4 + wl.T * wl.H * 2      # act in, out
    else:
        gateup_kernel = D * gu + A * wl.H * 2 + A * wl.I * 2       # gathered x in, act out
        down_kernel = D * dn + A * wl.I * 2 + wl.T * wl.H * 4      # act in, fp32 sum out
    flops = 2 * A * 3 * wl.H * wl.I + 2 * wl.T * wl.H * wl.E
    return dict(layer=layer, gateup=gateup_kernel, down=down_kernel, flops=flops,
                gateup_flops=2 * A * 2 * wl.H * wl.I, down_flops=2 * A * wl.H * wl.I)


def cpu_baseline(wl, layer_cpu, xs_cpu, budget_s=12.0):
    """The oracle as it stands, single-threaded, on a bounded sample of tokens
    through one layer; for the stack the rate is divided by its layer count
    (every layer has the same shape and cost)."""
    import oracle
    t0 = time.perf_counter()
    tokens = 0
    i = 0
    while True:
        L = dict(layer_cpu, x=xs_cpu[i % len(xs_cpu)], T=xs_cpu[i % len(xs_cpu)].shape[0])
        oracle.qmoe_forward(L)
        tokens += L["T"]
        i += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return tokens / el / wl.layers, tokens, el


def run_reference(a, wl):
    """--impl reference: the fp64 oracle on the host cores, same workload.
    A step pushes a bounded sample of the batch's tokens through the whole
    path (for the stack: RMSNorm + layer, 24 times, alternating between two
    generated weight sets of the stack's shape)."""
    import numpy as np
    import torch
    from int4_block_quantized_gb300 import synthetic as S
    import oracle
    oracle._load()
    nw = 2 if wl.layers > 1 else 1
    layers = [S.make_weights(wl, seed=0, device="cpu", layer=l) for l in range(nw)]
    T1 = min(wl.T, 1 if wl.T <= 16 else 2)  # one step = a bounded sample of the batch
    xs = [S.make_x(wl, seed=0, device="cpu", layer=l)[:T1].contiguous() for l in range(4)]
    tdt = torch.bfloat16 if wl.act_dtype else torch.float16

    def one_step(i):
        x = xs[i % 4]
        if wl.layers == 1:
            oracle.qmoe_forward(dict(layers[0], x=x, T=T1))
            return
        xd = x.to(torch.float64)
        for l in range(wl.layers):
            xn = oracle.rmsnorm(torch.from_numpy(xd.numpy()).to(tdt), wl.act_dtype, T1, wl.H, 1e-6)
            xn16 = torch.from_numpy(xn).to(tdt)
            y, _, _, _ = oracle.qmoe_forward(dict(layers[l % nw], x=xn16, T=T1))
            xd = torch.from_numpy(xd.numpy() + y)

    budget = 150.0
    tw0 = time.perf_counter()
    for i in range(a.warmup):
        one_step(i)
        if time.perf_counter() - tw0 > 20.0:
            break
    t0 = time.perf_counter()
    steps = 0
    while steps < a.steps:
        one_step(steps)
        steps += 1
        if time.perf_counter() - t0 > budget:
            break
    el = time.perf_counter() - t0
    v = steps * T1 / el
    sample = "%d step(s) of %d token(s) of the %s workload through %s (all %d experts resident), fp64, one thread" % (
        steps, T1, wl.name, "one layer" if wl.layers == 1 else
        "%d layers of RMSNorm + layer (two weight sets alternating)" % wl.layers, wl.E)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": a.gpus,
        "steps": steps, "warmup": a.warmup, "ms_per_step": 1000.0 * el / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(wl, a),
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def config_dict(wl, a):
    return {"workload": "%s: T=%d H=%d I=%d E=%d k=%d block=%d %s act, %s scales, %s" % (
        wl.name, wl.T, wl.H, wl.I, wl.E, wl.k, wl.block_size, "bf16" if wl.act_dtype else "fp16",
        "bf16" if wl.scale_dtype else "fp16", "uint4 zero points" if wl.has_zp else "no zero points"),
        "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k, "block_size": wl.block_size,
        "pool_layers": a.pool or POOL[wl.name],
        "l2": "weights rotate over %d independent layers (> L2 per revisit); no flush" % (a.pool or POOL[wl.name]),
        "parallelism": "replicas x%d" % a.gpus}


KERNELS = {True: ["route", "gateup", "down"],
           False: ["route", "permute", "gateup", "down", "convert"]}
# the configurations the default decode run adds to its line (name: steps per
# timed region, about 60-80 ms each; the region is repeated at least 10 times)
EXTRA = {"verify": 400, "prefill": 200, "stack": 4}


def host_info():
    """Core count and CPU model of the host the CPU baselines run on."""
    import platform
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            fields = {}
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
        model = fields.get("model name") or fields.get("Model") or (
            "CPU implementer %s part %s" % (fields.get("CPU implementer"), fields.get("CPU part"))
            if "CPU part" in fields else None)
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.processor() or platform.machine(),
            "machine": platform.machine()}


def near_tie_count(wl, layers, xs, ntok_max=512):
    """Tokens (over the pool, at most ntok_max per layer) whose oracle k-th
    and (k+1)-th router probabilities differ by less than 1e-4: their expert
    choice is not fixed by fp32 arithmetic, so the parity tests compare them
    by the near-tie rule instead of id for id."""
    import numpy as np
    import oracle
    n = 0
    tot = 0
    for l, L in enumerate(layers):
        x = xs[l % len(xs)][:ntok_max].cpu()
        T = x.shape[0]
        rb = L.get("router_bias")
        p = oracle.router_probs(x, wl.act_dtype, L["router_w"].cpu(), None if rb is None else rb.cpu(),
                                T, wl.H, wl.E)
        srt = -np.sort(-p, axis=1)
        if wl.E > wl.k:
            n += int(((srt[:, wl.k - 1] - srt[:, wl.k]) < 1e-4).sum())
        tot += T
    return n, tot


def measure(a, wl, steps, warmup, dev, rank, world, headline, cpu_budget):
    """Time one workload: K steps per timed region (barrier + synchronize on
    both sides, CUDA events on the launching stream), the region repeated at
    least 10 times and for at least 0.3 s while the SM clock is sampled;
    the reported time is the median region.  Returns the summary dict."""
    import torch
    from int4_block_quantized_gb300 import binding as B
    from int4_block_quantized_gb300 import synthetic as S
    dec = is_decode(wl)
    stack = wl.layers > 1
    names = KERNELS[dec]
    P = a.pool or POOL[wl.name]
    if stack:
        P = min(P, wl.layers)  # every step runs all the stack's layers
    layers = [S.make_weights(wl, seed=0, device=dev, layer=l) for l in range(P)]
    if stack:
        xs = [S.make_x(wl, seed=0, device=dev, layer=0)]
        xbuf = torch.empty_like(xs[0])
        xn = torch.empty_like(xs[0])
    else:
        xs = [S.make_x(wl, seed=0, device=dev, layer=l) for l in range(P)]
    outs = [torch.empty_like(x) for x in xs]
    ws = B.Workspace(wl.T, wl.H, wl.I, wl.E, wl.k, device=dev)
    Ds = []
    for l in range(P):
        _, ti, _, _ = B.qmoe_route(xs[l % len(xs)], layers[l]["router_w"], wl.k, layers[l]["router_bias"], ws=ws)
        Ds.append(int(torch.unique(ti).numel()))
    D_mean = sum(Ds) / len(Ds)
    wb = workload_bytes(wl, D_mean)
    nkern = B.qmoe_forward_kernels(layers[0], wl.T)
    fused = nkern == 1
    if fused:
        names = ["layer"]
    assert nkern == len(names), (nkern, names)
    launches_per_step = wl.layers * (nkern + (1 if stack else 0))

    def run_stack(x_in, x_out):
        x_out.copy_(x_in)
        for l in range(wl.layers):
            B.qmoe_rmsnorm(x_out, out=xn)
            B.qmoe_forward(layers[l % P], x=xn, out=x_out, ws=ws, accumulate=True)

    def step(i):
        if stack:
            run_stack(xs[0], xbuf)
            return
        j = i % P
        B.qmoe_forward(layers[j], x=xs[j], out=outs[j], ws=ws)

    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for i in range(3):
            step(i)
    torch.cuda.synchronize(dev)

    def capture(n, start):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(n):
                step(start + i)
        return g

    G = min(steps, 24 * P if dec else (4 if stack else 2 * P))
    g_warm = capture(warmup, 0)
    g_main = capture(G, warmup)
    rem = steps % G
    g_rem = capture(rem, warmup) if rem else None
    reps_in_region = steps // G
    g_warm.replay()
    torch.cuda.synchronize(dev)

    def region():
        barrier(world)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(reps_in_region):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
            e1.record(s)
        e1.synchronize()
        torch.cuda.synchronize(dev)
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1), world)

    clocks = Clocks(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    t_start = time.perf_counter()
    region_ms = []
    while len(region_ms) < 10 or (time.perf_counter() - t_start < 0.3 and len(region_ms) < 2000):
        region_ms.append(region())
    ck = clocks.stop()
    qs = sorted(region_ms)
    ms = statistics.median(qs)
    p10, p90 = qs[int(0.1 * (len(qs) - 1))], qs[int(0.9 * (len(qs) - 1))]
    value = wl.T * steps * world / (ms / 1000.0)
    ms_layer = ms / steps / wl.layers

    # per-kernel durations: the fused decode layer is one kernel, timed above
    # back to back; the multi-kernel paths are bracketed by events between
    # their kernels (run without programmatic overlap), replayed from a graph
    nrep = 3 if dec else 2
    xprof = [xn.copy_(B.qmoe_rmsnorm(xs[0])) if stack else None]

    def kernel_ms(knames, path):
        nk = len(knames)
        evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(nrep * P)]
        with torch.cuda.stream(s):
            for evs in evsets:
                for ev in evs:
                    ev.record(s)
        torch.cuda.synchronize(dev)
        g_prof = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_prof, stream=s):
            for i, evs in enumerate(evsets):
                j = i % P
                if stack:
                    B.qmoe_forward_profiled(layers[j], evs, x=xprof[0], out=outs[0], ws=ws, path=path)
                else:
                    B.qmoe_forward_profiled(layers[j], evs, x=xs[j], out=outs[j], ws=ws, path=path)
        g_prof.replay()
        torch.cuda.synchronize(dev)
        g_prof.replay()
        torch.cuda.synchronize(dev)
        return dict(zip(knames, [statistics.mean(evs[kk].elapsed_time(evs[kk + 1]) for evs in evsets[P:])
                                 for kk in range(nk)]))

    if fused:
        kdict = {"layer": ms_layer}
        split_kdict = kernel_ms(KERNELS[True], B.PATH_DECODE_SPLIT)
    else:
        kdict = kernel_ms(names, B.PATH_AUTO)
        split_kdict = None
    pk = peaks()
    if fused:
        kname, kb, kf = "layer", wb["layer"], wb["flops"]
        k_ms = ms_layer
    else:
        kname, kb, kf = "gateup", wb["gateup"], wb["gateup_flops"]
        k_ms = kdict["gateup"]
    k_gbs = kb / (k_ms * 1e-3) / 1e9
    k_tfs = kf / (k_ms * 1e-3) / 1e12
    if dec or kb / pk["hbm_gbs"] / 1e9 >= kf / pk["bf16_tflops"] / 1e12:
        roof = {"bound": "hbm", "achieved": k_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": k_gbs / pk["hbm_gbs"], "other": {"tflops": k_tfs, "tensor_frac": k_tfs / pk["bf16_tflops"]}}
    else:
        roof = {"bound": "tensor", "achieved": k_tfs, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": k_tfs / pk["bf16_tflops"], "other": {"gbs": k_gbs, "hbm_frac": k_gbs / pk["hbm_gbs"]}}
    kdesc = ("fused decode layer (router + gate-up + SwiGLU + down + weighted sum), timed back to back"
             if fused else "decode gate-up (+SwiGLU)" if dec else
             "grouped GEMM gate-up (+SwiGLU), exact hi+lo operands")
    roof.update({"traffic": NCU_TRAFFIC.get((wl.name, kname)),
                 "peak_source": pk["source"] + (" (copy GB/s)" if roof["bound"] == "hbm" else " (bf16 burst)"),
                 "kernel": kdesc, "bytes_per_launch": kb, "flops_per_launch": kf, "launch_ms": k_ms})

    res = {"workload": config_dict(wl, a)["workload"], "value": value, "unit": "tokens/s", "steps": steps,
           "warmup": warmup, "ms_per_step": ms / steps,
           "region_ms": {"median": ms, "p10": p10, "p90": p90, "repeats": len(qs)},
           "roofline": roof,
           "layer": {"path": ("decode, one fused kernel" if fused else "decode") if dec else
                     "prefill (exact hi+lo operands)",
                     "bytes": wb["layer"], "distinct_experts": D_mean, "ms": ms_layer,
                     "hbm_gbs": wb["layer"] / (ms_layer * 1e-3) / 1e9,
                     "hbm_frac": wb["layer"] / (ms_layer * 1e-3) / 1e9 / pk["hbm_gbs"],
                     "tflops": wb["flops"] / (ms_layer * 1e-3) / 1e12,
                     "tensor_frac": wb["flops"] / (ms_layer * 1e-3) / 1e12 / pk["bf16_tflops_sustained"],
                     "kernel_ms": kdict, **({"split_path_kernel_ms": split_kdict} if fused else {})},
           "gpu_launches": launches_per_step * steps,
           "clocks": {"sm_mhz": ck["sm_mhz"], "sm_max_mhz": ck["sm_max_mhz"], "reasons": ck["reasons"],
                      "samples": ck["samples"]}}
    if stack:
        res["layers"] = wl.layers
        res["tokens_per_s_per_layer"] = value * wl.layers

    if headline:
        # end to end through the public API: pinned H2D of x, forward, D2H of out
        xh = [x.cpu().pin_memory() for x in xs]
        oh = [torch.empty_like(x, device="cpu").pin_memory() for x in xs]
        xd = torch.empty_like(xs[0])
        od = torch.empty_like(xs[0])
        n_e2e = min(steps, 4000)

        def e2e_step(i):
            j = i % len(xs)
            xd.copy_(xh[j], non_blocking=True)
            if stack:
                run_stack(xd, od)
            else:
                B.qmoe_forward(layers[i % P], x=xd, out=od, ws=ws)
            oh[j].copy_(od, non_blocking=True)

        with torch.cuda.stream(s):
            for i in range(3):
                e2e_step(i)
            torch.cuda.synchronize(dev)
            barrier(world)
            f0 = torch.cuda.Event(enable_timing=True)
            f1 = torch.cuda.Event(enable_timing=True)
            f0.record(s)
            for i in range(n_e2e):
                e2e_step(i)
            f1.record(s)
        f1.synchronize()
        e2e_ms = max_over_ranks(f0.elapsed_time(f1), world)
        res["e2e"] = {"value": wl.T * n_e2e * world / (e2e_ms / 1000.0), "unit": "tokens/s",
                      "h2d_bytes_per_step": wl.T * wl.H * 2, "d2h_bytes_per_step": wl.T * wl.H * 2,
                      "steps": n_e2e}

    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        nt, tot = near_tie_count(wl, layers, xs if not stack else
                                 [B.qmoe_rmsnorm(xs[0])], ntok_max=512 if not stack else 256)
        res["near_ties"] = {"count": nt, "tokens_checked": tot, "gap": 1e-4,
                            "over": "the pool's layers" if not stack else "the first 256 tokens of layer 0's input against every layer's router"}
        lc = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in layers[0].items()}
        nt_cpu = wl.T if dec else 2  # tokens per oracle call: a bounded sample of the batch
        xc = [x.cpu()[:nt_cpu].contiguous() for x in xs[:4]]
        if stack:
            xc = [B.qmoe_rmsnorm(xs[0][i * nt_cpu:(i + 1) * nt_cpu].contiguous()).cpu() for i in range(4)]
        v, toks, el = cpu_baseline(wl, lc, xc, budget_s=cpu_budget)
        res["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                               "sample": "%d token(s) of the %s workload through one layer in %.1f s, fp64, one "
                                         "thread%s" % (toks, wl.name, el, "; rate divided by the %d layers"
                                                       % wl.layers if stack else ""),
                               **host_info()}
    del layers, xs, outs, ws
    torch.cuda.empty_cache()
    return res


def run_ours(a, wl):
    import torch
    from int4_block_quantized_gb300 import binding as B
    from int4_block_quantized_gb300 import synthetic as S
    rank, world, local = dist_init()
    dev = torch.device("cuda", local)
    B.lib()
    head = measure(a, wl, a.steps, a.warmup, dev, rank, world, True, 12.0)
    extra = {}
    if wl.name == "decode" and not a.no_extra and world == 1:
        # the rest of the metric: verify-sized decode, the prefill layer and the
        # 24-layer stack, each its own measurement in this same run
        for name, steps in EXTRA.items():
            extra[name] = measure(a, S.WORKLOADS[name], steps, max(3, min(a.warmup, 10)), dev, rank, world,
                                  False, 4.0)
    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp16" if wl.act_dtype == 0 else "bf16",
            "data": "synthetic", "config": config_dict(wl, a),
            "roofline": head["roofline"], "layer": head["layer"], "region_ms": head["region_ms"],
            "cpu_baseline": head.get("cpu_baseline"), "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
            **({"near_ties": head["near_ties"]} if "near_ties" in head else {}),
            **({"configs": extra} if extra else {}),
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_gptq_repack(a):
    """One Qwen1.5-MoE-A2.7B layer's GPTQ tensors (gate, up, down of 60
    experts, bs 32, fp16 scales, qzeros) converted to the canonical layout:
    bytes read + written per conversion over the CUDA-event time."""
    import torch
    from int4_block_quantized_gb300 import binding as B
    B.lib()
    E, H, I, bs = 60, 2048, 1408, 32
    g = torch.Generator(device="cuda").manual_seed(0)
    mats = []
    nbytes = 0
    for K, N in ((H, I), (H, I), (I, H)):
        qw = torch.randint(0, 2 ** 31 - 1, (E, K // 8, N), generator=g, device="cuda", dtype=torch.int32)
        qz = torch.randint(0, 2 ** 31 - 1, (E, K // bs, N // 8), generator=g, device="cuda", dtype=torch.int32) & 0x77777777
        sc = torch.rand((E, K // bs, N), generator=g, device="cuda").to(torch.float16)
        mats.append((qw, qz, sc))
        nbytes += 2 * (qw.numel() * 4 + sc.numel() * 2) + qz.numel() * 4 + E * N * (K // bs)
    steps = a.steps or 50
    warm = a.warmup if a.warmup is not None else 3

    def step():
        for qw, qz, sc in mats:
            B.qmoe_repack_gptq(qw, qz, sc, bs, zero_offset=1, check=False)
    for _ in range(warm):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    gbs = nbytes / (ms * 1e-3) / 1e9
    pk = peaks()
    print(json.dumps({"metric": "GPTQ -> canonical weight repack, GB/s (read + write)", "value": gbs, "unit": "GB/s",
                      "n_gpus": 1, "steps": steps, "warmup": warm, "ms_per_step": ms, "higher_is_better": True,
                      "dtype": "u32/u16/u8", "data": "synthetic",
                      "config": {"workload": "GPTQ gate+up+down of one layer: E=60 H=2048 I=1408 bs=32, qzeros, fp16 scales",
                                 "bytes_per_step": nbytes},
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                                   "frac": gbs / pk["hbm_gbs"], "traffic": None},
                      "gpu_launches": 9 * steps}))


def run_gptq_repack_reference(a):
    """--impl reference --config gptq_repack: the plain CPU definition
    (oracle/formats.py) converting a bounded sample of one layer's GPTQ
    tensors (row slices of the gate projection), in the same unit."""
    import numpy as np
    from oracle import formats as F
    K, N, bs = 2048, 1408, 32
    rng = np.random.default_rng(0)
    ncols = 16  # a sample: 16 output columns of one expert's gate projection
    qw = rng.integers(0, 2 ** 32, size=(K // 8, ncols), dtype=np.uint64).astype(np.uint32)
    qz = (rng.integers(0, 2 ** 32, size=(K // bs, ncols // 8), dtype=np.uint64).astype(np.uint32)
          & np.uint32(0x77777777))
    sc = rng.integers(0, 2 ** 16, size=(K // bs, ncols), dtype=np.uint64).astype(np.uint16)
    nbytes = 2 * (qw.nbytes + sc.nbytes) + qz.nbytes + ncols * (K // bs)
    for _ in range(min(a.warmup, 1)):
        F.gptq_to_canonical(qw, qz, sc, K, ncols, bs, 1)
    t0 = time.perf_counter()
    steps = 0
    while steps < a.steps and (steps == 0 or time.perf_counter() - t0 < 60.0):
        F.gptq_to_canonical(qw, qz, sc, K, ncols, bs, 1)
        steps += 1
    el = time.perf_counter() - t0
    gbs = steps * nbytes / el / 1e9
    sample = "%d conversion(s) of %d output columns of one GPTQ projection (K=%d, bs=%d), python, one thread" % (
        steps, ncols, K, bs)
    print(json.dumps({"impl": "reference", "metric": "GPTQ -> canonical weight repack, GB/s (read + write)",
                      "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": a.warmup,
                      "ms_per_step": el / steps * 1e3, "higher_is_better": True, "dtype": "u32/u16/u8",
                      "data": "synthetic", "config": {"workload": "GPTQ repack, bounded CPU sample"},
                      "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
                      "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


def main():
    a = parse()
    if a.config == "gptq_repack":
        if a.impl == "reference":
            if int(os.environ.get("RANK", "0")) == 0:
                run_gptq_repack_reference(a)
            return
        run_gptq_repack(a)
        return
    from int4_block_quantized_gb300 import synthetic as S
    wl = S.WORKLOADS[a.config]
    if a.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if world > 1 and rank != 0:
            return
        run_reference(a, wl)
        return
    run_ours(a, wl)


if __name__ == "__main__":
    main()
