"""Benchmark of the MoE expert layer on GB300 through libmoe's C-ABI.

One step = one moe_forward (plan -> quant/scatter -> GEMM1+act -> GEMM2 ->
combine) over one batch of synthetic tokens already resident in HBM.  Default
workload: the FP8 block-quantised compact-layout prefill (T=8192, K=7168,
I=2048, 256 experts, top-8, Zipf(1.2) expert popularity; e4m3 weights with
128x128 UE8M0 scales, 1x128 UE8M0 activation scales).  Prints one JSON line
(rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 (launched by torch.distributed.run, one rank per GPU) runs N
independent replicas: the layer has no cross-GPU step on one node's expert
set, so every rank processes its own batch; timing is the max over ranks.
"--impl reference" times the CPU oracle (fp64, numpy) on the host cores on a
bounded sample of the same workload.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s, grouped-GEMM TFLOPS & % of roofline on 1xGB300"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="fp8_prefill_zipf", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--T", type=int, default=None, help="override the token count")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="layer", choices=["layer", "requant", "router", "crossover"],
                    help="layer: the MoE layer step (default); requant: load-time UE8M0 weight requantisation; "
                         "router: the fp32 router (logits + top-k + softmax) on the workload's tokens; "
                         "crossover: masked vs compact layout across E_local and T")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms, world, device):
    """The slowest rank's time: every replica's batch counts toward `value`,
    so the job takes as long as its slowest rank."""
    if world <= 1:
        return ms
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_value(tokens_per_rank, world, steps, ms):
    """Whole-job throughput: the tokens all ranks processed / the max time."""
    return world * tokens_per_rank * steps / (ms / 1000.0)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [s for s in sm if mx and s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_source_digest():
    """Digest of the GEMM kernel sources with // comments and blank lines
    removed, so that a comment-only edit keeps a capture valid."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "moe_expert_layer_ep_gb300", "csrc")
    parts = []
    for f in ("gemm.cu", "common.cuh"):
        code = re.sub(r"//[^\n]*", "", open(os.path.join(csrc, f)).read())
        code = "\n".join(l.rstrip() for l in code.splitlines() if l.strip())
        parts.append(hashlib.sha256(code.encode()).hexdigest()[:16])
    return "-".join(parts)


def measured_traffic(workload_name, T_override=None, key="dram_bytes_per_launch"):
    """DRAM bytes per launch of a GEMM kernel (the dominant one, or GEMM2 with
    key="gemm2_dram_bytes_per_launch") from the committed ncu summary of this
    workload (and token count, when overridden), or None when there is no
    capture or the kernel code changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    name = workload_name if T_override is None else f"{workload_name}@T{T_override}"
    rec = json.load(open(path)).get(name)
    if not rec or key not in rec:
        return None
    return rec[key] if kernel_source_digest() == rec["code_digest"] else None


def workload(args):
    w = dict(synth.WORKLOADS[args.workload])
    if args.T:
        w["T"] = args.T
    return w


def routing_seed(w):
    """Routing seed of a workload: seed + 1, except that a workload holding
    only some of the experts (a masked, expert-parallel slice) takes the
    first of seed + 1, seed + 2, ... whose first token routes to at least one
    local expert, so that every batch size, T = 1 included, runs the expert
    GEMMs.  Token 0's logits do not depend on T, so neither does the seed."""
    seed = w["seed"] + 1
    if w["E_local"] == w["E_global"]:
        return seed
    es, El = w["expert_start"], w["E_local"]
    while True:
        ids, _ = synth.routing(1, w["E_global"], w["topk"], seed, w["zipf_s"])
        if ((ids >= es) & (ids < es + El)).any():
            return seed
        seed += 1


def build_inputs(w, device):
    T, K, I = w["T"], w["K"], w["I"]
    x = synth.activations(T, K, w["seed"], device)
    ids, wts = synth.routing(T, w["E_global"], w["topk"], routing_seed(w), w["zipf_s"])
    es = w["expert_start"]
    if w["dtype"] == "fp8":
        w13, w13s = synth.fp8_expert_weights(w["E_local"], 2 * I, K, w["seed"] + 2, device, es)
        w2, w2s = synth.fp8_expert_weights(w["E_local"], K, I, w["seed"] + 3, device, es)
    elif w["dtype"] in ("mxfp8", "mxfp4"):   # natural [E, N, C/32] scales (packed for the device by run_ours)
        gen = synth.mxfp8_expert_weights if w["dtype"] == "mxfp8" else synth.mxfp4_expert_weights
        w13, w13s = gen(w["E_local"], 2 * I, K, w["seed"] + 2, device, es)
        w2, w2s = gen(w["E_local"], K, I, w["seed"] + 3, device, es)
    else:
        w13 = synth.bf16_expert_weights(w["E_local"], 2 * I, K, w["seed"] + 2, device, es)
        w2 = synth.bf16_expert_weights(w["E_local"], K, I, w["seed"] + 3, device, es)
        w13s = w2s = None
    return x, ids, wts, (w13, w13s, w2, w2s)


def work_model(w, ids):
    """Algorithmic work of one step (valid rows only).  Bytes count what the
    method as described must move: the weights (and their scales) of the
    non-empty experts once, the valid a / h / y rows written and read, x and
    out; fused_bytes is the minimal fused bound (weights + x + out + routing)."""
    T, K, I, E_l, es, k = w["T"], w["K"], w["I"], w["E_local"], w["expert_start"], w["topk"]
    ids = ids.numpy()
    loc = (ids >= es) & (ids < es + E_l)
    A = int(loc.sum())
    nonempty = len(np.unique(ids[loc]))
    esz = 1 if w["dtype"] in ("fp8", "mxfp8", "mxfp4") else 2    # activations and h
    wsz = 0.5 if w["dtype"] == "mxfp4" else esz                   # weights
    # UE8M0 bytes per element: 1x128 activations / 128x128 weights, or 1x32 (MX)
    asf = {"fp8": 1 / 128, "mxfp8": 1 / 32, "mxfp4": 1 / 32}.get(w["dtype"], 0.0)
    wsf = {"fp8": 1 / 16384, "mxfp8": 1 / 32, "mxfp4": 1 / 32}.get(w["dtype"], 0.0)
    flops1 = 2.0 * A * K * 2 * I
    flops2 = 2.0 * A * I * K
    w13_bytes = nonempty * 2 * I * K * (wsz + wsf)
    w2_bytes = nonempty * K * I * (wsz + wsf)
    a_bytes = A * K * (esz + asf)
    h_bytes = A * I * (esz + asf)
    y_bytes = A * K * 2
    # GEMM1 reads its weights and the valid a rows and writes h; GEMM2 reads
    # its weights and h and writes y.
    g1_bytes = w13_bytes + a_bytes + h_bytes
    g2_bytes = w2_bytes + h_bytes + y_bytes
    route = T * k * 8
    # the memory-bound passes: quant-scatter reads x and the routing and
    # writes the a rows; combine reads the y rows and the routing and writes out
    quant = (T * K * 2 + T * k * 4, a_bytes)
    combine = (y_bytes + route, T * K * 2)
    return {"A": A, "nonempty": nonempty, "flops1": flops1, "flops2": flops2, "g1_bytes": g1_bytes,
            "g2_bytes": g2_bytes, "weights_bytes": w13_bytes + w2_bytes, "quant_rw": quant, "combine_rw": combine,
            "fused_bytes": w13_bytes + w2_bytes + 2 * T * K * 2 + route,
            "layer_bytes": w13_bytes + w2_bytes + 2 * T * K * 2 + route + 2 * (a_bytes + h_bytes + y_bytes)}


class OracleSample:
    """The fp64 oracle, as it stands, timed on a bounded sample of a workload.

    Sample: the first ``n_tok`` tokens, and of their assignments those routed
    to the ``n_exp`` local experts they use most (ties to the lower id); the
    other assignments are dropped, as a rank holding only those experts drops
    them.  One step is one ``oracle.forward_layout`` over that sample.  The
    expert work is what dominates the layer, so the rate is reported per
    assignment and scaled to tokens: tokens/s = assignments/s / topk.  Expert
    weights are fetched and dequantised once, before any timed call.
    """

    def __init__(self, w, x, ids, wts, expert_fn, n_tok=256, n_exp=8):
        import oracle
        self.oracle, self.w = oracle, w
        T, k, es, El = w["T"], w["topk"], w["expert_start"], w["E_local"]
        n_tok = min(T, n_tok)
        ids = ids[:n_tok].cpu().numpy().astype(np.int64)
        loc = ids - es
        is_loc = (ids >= 0) & (loc >= 0) & (loc < El)
        counts = np.bincount(loc[is_loc], minlength=El)
        order = sorted(range(El), key=lambda e: (-counts[e], e))
        chosen = sorted(e for e in order[:min(n_exp, El)] if counts[e] > 0)
        remap = np.full(El, -1, dtype=np.int64)
        remap[chosen] = np.arange(len(chosen))
        self.ids = np.where(is_loc, remap[np.where(is_loc, loc, 0)], -1).astype(np.int32)
        self.assignments = int((self.ids >= 0).sum())
        self.x64 = x[:n_tok].float().cpu().numpy().astype(np.float64)
        self.wts = wts[:n_tok].cpu().numpy()
        self.n_tok, self.experts = n_tok, chosen
        deq = []
        for e in chosen:
            w13, w13s, w2, w2s = expert_fn(e)
            if w["dtype"] in ("fp8", "mxfp8", "mxfp4"):
                f = {"fp8": oracle.dequant_fp8_weights, "mxfp8": oracle.dequant_mx_weights,
                     "mxfp4": oracle.dequant_mxfp4_weights}[w["dtype"]]
                deq.append((f(w13.numpy(), w13s.numpy().astype(np.int64) - 127)[0],
                            f(w2.numpy(), w2s.numpy().astype(np.int64) - 127)[0]))
            else:
                deq.append((w13[0].float().numpy().astype(np.float64), w2[0].float().numpy().astype(np.float64)))
        self.w13 = np.stack([d[0] for d in deq]) if deq else np.zeros((0, 2 * w["I"], w["K"]))
        self.w2 = np.stack([d[1] for d in deq]) if deq else np.zeros((0, w["K"], w["I"]))

    def describe(self):
        w = self.w
        return (f"first {self.n_tok} of {w['T']} tokens of workload {w['name']}, their {self.assignments} "
                f"assignments to their {len(self.experts)} most-used local experts (the rest dropped); fp64 numpy "
                f"oracle, layout path; tokens/s = assignments/s / topk")

    def step(self):
        t0 = time.perf_counter()
        self.oracle.forward_layout(self.x64, self.w13, self.w2, self.ids, self.wts, self.w["dtype"],
                                   E_global=max(1, len(self.experts)), layout="compact")
        return time.perf_counter() - t0

    def run(self, seconds_target):
        """Repeat the sample for about seconds_target of timed oracle work."""
        elapsed, reps = 0.0, 0
        while reps == 0 or elapsed < seconds_target:
            elapsed += self.step()
            reps += 1
        value = reps * self.assignments / self.w["topk"] / elapsed
        return {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                "sample": f"{self.describe()}; {reps} repetition(s), {elapsed:.1f} s"}


def expert_source(w, weights=None):
    """expert_fn(e) -> (w13, w13_sf, w2, w2_sf) CPU tensors of local expert e:
    sliced from the device weights when given, else generated on the host
    from the expert's own seed (synthetic weights are seeded per expert)."""
    I, K, es = w["I"], w["K"], w["expert_start"]

    def from_device(e):
        return tuple(t[e:e + 1].cpu() if t is not None else None for t in weights)

    def generated(e):
        if w["dtype"] == "fp8":
            gen = synth.fp8_expert_weights
        elif w["dtype"] in ("mxfp8", "mxfp4"):
            gen = synth.mxfp8_expert_weights if w["dtype"] == "mxfp8" else synth.mxfp4_expert_weights
        else:
            a = synth.bf16_expert_weights(1, 2 * I, K, w["seed"] + 2, "cpu", es + e)
            b = synth.bf16_expert_weights(1, K, I, w["seed"] + 3, "cpu", es + e)
            return a, None, b, None
        a, sa = gen(1, 2 * I, K, w["seed"] + 2, "cpu", es + e)
        b, sb = gen(1, K, I, w["seed"] + 3, "cpu", es + e)
        return a, sa, b, sb

    return from_device if weights is not None else generated


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    T, K = w["T"], w["K"]
    x = synth.activations(T, K, w["seed"], "cpu")
    ids, wts = synth.routing(T, w["E_global"], w["topk"], routing_seed(w), w["zipf_s"])
    sample = OracleSample(w, x, ids, wts, expert_source(w))
    per_step = []
    for s in range(args.warmup + args.steps):
        dt = sample.step()
        if s >= args.warmup:
            per_step.append(dt)
    elapsed = float(sum(per_step))
    value = len(per_step) * sample.assignments / w["topk"] / elapsed
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * elapsed / len(per_step),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w["name"], "T": w["T"], "K": w["K"], "I": w["I"],
                                            "E": w["E_local"], "topk": w["topk"]},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample.describe() + "; one sample per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def capture_graph(body, dev):
    """A CUDA graph of body() (one side-stream pass first, as capture needs
    the work to have run once outside it)."""
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        body(warm=True)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        body(warm=False)
    return graph


def tensor_peak_of(peaks, fp8):
    """Dense tensor peak for a GEMM timed inside the long power-capped step
    loop: the measured sustained bf16 figure (x 2, the nominal ratio, for the
    FP8 kinds).  The burst figure is the denominator only for a kernel timed
    alone."""
    return peaks["bf16_tflops_sustained"] * (2.0 if fp8 else 1.0)


def gemm_roofline(name, flops, nbytes, ms, peaks, fp8):
    """Roofline of one GEMM launch: the bound is whichever of the tensor time
    (algorithmic FLOPs at the dtype's sustained peak) and the HBM time
    (algorithmic bytes at the measured copy bandwidth) is larger."""
    tensor_peak = tensor_peak_of(peaks, fp8)
    sec = ms / 1000.0
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (tensor_peak * 1e12)
    gbs, tf = nbytes / sec / 1e9, flops / sec / 1e12
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": tensor_peak, "unit": "TFLOP/s",
                "frac": round(tf / tensor_peak, 4)}
    burst = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
    roof.update({"kernel": name, "ms": round(ms, 4), "algorithmic_bytes": int(nbytes),
                 "algorithmic_tflop": round(flops / 1e12, 4), "tflops": round(tf, 1),
                 "tensor_frac": round(tf / tensor_peak, 4), "hbm_gbs": round(gbs, 1),
                 "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                 # the same TFLOP/s against the measured burst peak (a GEMM timed alone)
                 "tensor_frac_of_burst": round(tf / burst, 4),
                 "peak_source": peaks["source"] + (" sustained bf16 x 2 for fp8" if fp8 else " sustained bf16")
                 + " (tensor); copy bandwidth (hbm)"})
    return roof


def measure_write_peak(dev):
    """Write-only HBM bandwidth of this GPU: torch's fill of a 512 MB buffer,
    CUDA events over 10 fills after 3 untimed ones.  A stream of writes
    alone runs well below the copy bandwidth (a read and a write per byte)
    the roofline peaks are measured with."""
    buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        buf.fill_(1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(10):
        buf.fill_(i)
    e1.record()
    torch.cuda.synchronize()
    gbs = 10 * buf.numel() / (e0.elapsed_time(e1) / 1e3) / 1e9
    del buf
    return gbs


def memory_pass(ms, rw, peaks, write_gbs):
    """An HBM-bound pass: achieved GB/s against the copy bandwidth, and its
    time against the time its writes alone take at the write-only bandwidth."""
    rd, wr = rw
    sec = ms / 1000.0
    gbs = (rd + wr) / sec / 1e9
    write_ms = wr / (write_gbs * 1e9) * 1000.0
    return {"ms": round(ms, 4), "read_bytes": int(rd), "write_bytes": int(wr), "achieved_gbs": round(gbs, 1),
            "frac_of_copy_peak": round(gbs / peaks["hbm_gbs"], 4), "writes_alone_ms": round(write_ms, 4),
            "frac_of_write_bound": round(write_ms / ms, 4)}


def pct(a, q):
    return round(float(np.percentile(np.asarray(a), q)), 4)


def run_ours(args, w, world, rank, local):
    import moe_expert_layer_ep_gb300 as M
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x, ids_host, w_host, weights = build_inputs(w, dev)
    ids, wts = ids_host.to(dev), w_host.to(dev)
    max_m = w.get("max_m", 0) or (w["T"] if w["layout"] == "masked" else 0)
    shape = M.make_shape(w["T"], w["K"], w["I"], w["E_global"], w["E_local"], w["topk"], w["dtype"], w["layout"],
                         w["expert_start"], max_m)
    ctx_weights = weights
    if w["dtype"] in ("mxfp8", "mxfp4"):   # the context takes packed MX scales; the oracle reads the natural ones
        ctx_weights = (weights[0], M.moe_pack_mx_scales(weights[1]), weights[2], M.moe_pack_mx_scales(weights[3]))
    ctx = M.moe_ctx_create(shape, *ctx_weights)
    ws = M.alloc_workspace(ctx, dev)
    out = torch.empty((w["T"], w["K"]), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    M.moe_clear_device_status(ws)

    stages = [lambda: M.moe_plan_layout(ctx, ids, ws),
              lambda: M.moe_quant_scatter(ctx, x, ws),
              lambda: M.moe_grouped_gemm_w13_act(ctx, ws),
              lambda: M.moe_grouped_gemm_w2(ctx, ws),
              lambda: M.moe_combine(ctx, wts, ws, out)]
    names = ["plan", "quant_scatter", "gemm_w13_act", "gemm_w2", "combine"]
    nst = len(stages)
    for _ in range(args.warmup):
        M.moe_forward(ctx, x, ids, wts, ws, out)
    torch.cuda.synchronize()
    status = M.moe_read_device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {M.STATUS_NAMES.get(status, status)} after warm-up")

    # The timed region replays graph A: args.steps forwards (moe_forward, the
    # layer is static-shape, so this is how it runs in production) with no
    # event between them, so consecutive kernels keep their programmatic
    # dependent launch across step boundaries too.  Three more graphs stay
    # out of the timed region, as their events cost time of their own:
    #   S: the same forwards with an event at each step boundary (per-step
    #      p10 / p50 / p90);
    #   B: the stage calls with an event between every stage (the stage
    #      breakdown and the GEMM rooflines; each stage time then includes its
    #      own launch latency);
    #   G1, G2: each GEMM stage alone, args.steps launches back to back (its
    #      throughput when launches overlap, as inside moe_forward).
    # Without graph-capturable events everything is launched eagerly.
    timing = "cuda-graph replay"
    step_ev = stage_ev = None

    def body_a(warm):
        for _ in range(args.steps):
            M.moe_forward(ctx, x, ids, wts, ws, out)

    def body_s(warm):
        for s in range(args.steps):
            if not warm:
                step_ev[s].record()
            M.moe_forward(ctx, x, ids, wts, ws, out)
        if not warm:
            step_ev[args.steps].record()

    def body_b(warm):
        for s in range(args.steps):
            if not warm:
                stage_ev[s][0].record()
            for i, fn in enumerate(stages):
                fn()
                if not warm:
                    stage_ev[s][i + 1].record()

    def body_gemm(fn):
        def body(warm):
            for _ in range(args.steps):
                fn()
        return body

    try:
        step_ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(args.steps + 1)]
        stage_ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(nst + 1)]
                    for _ in range(args.steps)]
        graphs = [capture_graph(b, dev) for b in (body_a, body_s, body_b, body_gemm(stages[2]), body_gemm(stages[3]))]
        run_a, run_s, run_b, run_g1, run_g2 = (g.replay for g in graphs)
    except Exception:                        # events in graphs unsupported: eager launches
        timing = "eager launches"
        step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(args.steps)]
        run_a, run_s, run_b = (lambda: body_a(False)), (lambda: body_s(False)), (lambda: body_b(False))
        run_g1, run_g2 = (lambda: body_gemm(stages[2])(False)), (lambda: body_gemm(stages[3])(False))
    for run in (run_a, run_s, run_b, run_g1, run_g2):
        run()
    torch.cuda.synchronize()

    def keep_busy(seconds):
        """Untimed replays around the timed one, so that the clock samples
        see the GPU under the same load."""
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            run_a()
            torch.cuda.synchronize()

    def timed(run):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # the untimed graphs run right after the timed one, under the same load
    # and inside the same clock record
    with ClockSampler(local) as clk:
        keep_busy(0.4)
        total_ms = timed(run_a)
        run_s()
        run_b()
        g1_steady_ms = timed(run_g1) / args.steps
        g2_steady_ms = timed(run_g2) / args.steps
        keep_busy(0.2)
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(total_ms, world, dev)
    step_ms = [step_ev[s].elapsed_time(step_ev[s + 1]) for s in range(args.steps)]
    stage_ms = np.array([[stage_ev[s][i].elapsed_time(stage_ev[s][i + 1]) for i in range(nst)]
                         for s in range(args.steps)])
    write_gbs = measure_write_peak(dev)

    # end to end through the C-ABI with host buffers, as a serving loop runs
    # it: every step copies its x / ids / weights from pinned host memory and
    # reads its output back, on copy streams that overlap the neighbouring
    # steps' forwards (two device buffer sets; events order every reuse).
    x_h = x.cpu().pin_memory()
    ids_h = ids.cpu().pin_memory()
    w_h = wts.cpu().pin_memory()
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    bufs = [(x, ids, wts, out), (torch.empty_like(x), torch.empty_like(ids), torch.empty_like(wts),
                                 torch.empty_like(out))]
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    s_fwd = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()                       # noqa: E731
    in_ready, fwd_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_steps(n, start_event=None):
        for i in range(n):
            b = i & 1
            xb, ib, wb, ob = bufs[b]
            with torch.cuda.stream(s_in):
                if start_event is not None and i == 0:
                    s_in.wait_event(start_event)
                if i >= 2:
                    s_in.wait_event(fwd_done[b])           # the forward two steps back read this buffer
                xb.copy_(x_h, non_blocking=True)
                ib.copy_(ids_h, non_blocking=True)
                wb.copy_(w_h, non_blocking=True)
                in_ready[b].record(s_in)
            s_fwd.wait_event(in_ready[b])
            if i >= 2:
                s_fwd.wait_event(out_done[b])              # its output was read back
            with torch.cuda.stream(s_fwd):
                M.moe_forward(ctx, xb, ib, wb, ws, ob)
                fwd_done[b].record(s_fwd)
            with torch.cuda.stream(s_out):
                s_out.wait_event(fwd_done[b])
                out_h[b].copy_(ob, non_blocking=True)
                out_done[b].record(s_out)
        s_fwd.wait_event(out_done[(n - 1) & 1])
        if n > 1:
            s_fwd.wait_event(out_done[(n - 2) & 1])

    torch.cuda.synchronize()
    e2e_steps(4)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_fwd)
    e2e_steps(args.steps, start_event=e0)
    e1.record(s_fwd)
    torch.cuda.synchronize()
    assert torch.equal(out_h[(args.steps - 1) & 1].view(torch.int16), out.cpu().view(torch.int16))
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    assert M.moe_read_device_status(ws) == 0

    if rank != 0:
        return
    peaks = load_peaks()
    wm = work_model(w, ids_host)
    T = w["T"]
    ms_per_step = total_ms / args.steps
    value = replica_value(T, world, args.steps, total_ms)
    med = np.median(stage_ms, axis=0)
    g1_ms, g2_ms = float(med[2]), float(med[3])
    fp8 = w["dtype"] in ("fp8", "mxfp8", "mxfp4")
    tensor_peak = tensor_peak_of(peaks, fp8)
    gemm_tflops = (wm["flops1"] + wm["flops2"]) / ((g1_ms + g2_ms) / 1000.0) / 1e12
    # dominant kernel: GEMM1; GEMM2 beside it
    roof = gemm_roofline("grouped_gemm_kernel<stage 1> (moe_grouped_gemm_w13_act)", wm["flops1"], wm["g1_bytes"],
                         g1_ms, peaks, fp8)
    roof2 = gemm_roofline("grouped_gemm_kernel<stage 2> (moe_grouped_gemm_w2)", wm["flops2"], wm["g2_bytes"],
                          g2_ms, peaks, fp8)
    # executed work: every row of the padded 128-row blocks goes through the MMAs
    padded_rows = int(M.ws_view(ctx, ws, "meta")[0].item())
    exec1 = 2.0 * padded_rows * w["K"] * 2 * w["I"] / (g1_ms / 1000.0) / 1e12
    exec2 = 2.0 * padded_rows * w["I"] * w["K"] / (g2_ms / 1000.0) / 1e12
    roof.update({"executed_tflops": round(exec1, 1), "executed_tensor_frac": round(exec1 / tensor_peak, 4),
                 "traffic": measured_traffic(w["name"], args.T)})
    roof2.update({"executed_tflops": round(exec2, 1), "executed_tensor_frac": round(exec2 / tensor_peak, 4),
                  "traffic": measured_traffic(w["name"], args.T, "gemm2_dram_bytes_per_launch")})
    # each GEMM stage launched back to back (programmatic dependent launch,
    # no events between launches): its time per launch when launches overlap
    for r, ms, fl, by in ((roof, g1_steady_ms, wm["flops1"], wm["g1_bytes"]),
                          (roof2, g2_steady_ms, wm["flops2"], wm["g2_bytes"])):
        r["back_to_back"] = {"ms": round(ms, 4), "tensor_frac": round(fl / (ms / 1000.0) / 1e12 / tensor_peak, 4),
                             "hbm_frac": round(by / (ms / 1000.0) / 1e9 / peaks["hbm_gbs"], 4)}
    layer_roof_ms = 1000.0 * max(wm["layer_bytes"] / (peaks["hbm_gbs"] * 1e9),
                                 (wm["flops1"] + wm["flops2"]) / (tensor_peak * 1e12))
    fused_ms = 1000.0 * max(wm["fused_bytes"] / (peaks["hbm_gbs"] * 1e9),
                            (wm["flops1"] + wm["flops2"]) / (tensor_peak * 1e12))
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": {"fp8": "fp8-e4m3/ue8m0", "mxfp8": "mxfp8-e4m3/ue8m0-1x32",
                  "mxfp4": "mxfp4-e2m1-weights/mxfp8-activations"}.get(w["dtype"], "bf16"),
        "data": "synthetic (seeded; random-init weights)",
        "config": {"workload": w["name"], "T": T, "K": w["K"], "I": w["I"], "E": w["E_local"],
                   "E_global": w["E_global"], "topk": w["topk"], "layout": w["layout"],
                   **({"max_m": max_m} if w["layout"] == "masked" else {}),
                   **({"zipf_s": w["zipf_s"]} if w["zipf_s"] else {}),
                   "l2": "weights larger than L2 (no flush needed)" if wm["weights_bytes"] > 2 * 129e6
                   else "L2 not flushed: weights fit in L2",
                   "parallelism": f"replicas x{world}", "timing": timing},
        "step_ms_p10_p50_p90": [pct(step_ms, 10), pct(step_ms, 50), pct(step_ms, 90)],
        "gemm_tflops": round(gemm_tflops, 1),
        "layer_roofline_frac": round(layer_roof_ms / ms_per_step, 4),
        "minimal_fused_bound": {"bytes": int(wm["fused_bytes"]), "ms": round(fused_ms, 4),
                                "frac": round(fused_ms / ms_per_step, 4),
                                "what": "weights of non-empty experts + x + out (+ routing) at the measured "
                                        "HBM bandwidth, or the tensor time if larger"},
        "memory_passes": {"write_peak_gbs": round(write_gbs, 1),
                          "write_peak_how": "torch fill of 512 MB, measured in this run",
                          "quant_scatter": memory_pass(float(med[1]), wm["quant_rw"], peaks, write_gbs),
                          "combine": memory_pass(float(med[4]), wm["combine_rw"], peaks, write_gbs)},
        "stage_ms": {n: round(float(v), 4) for n, v in zip(names, med)},
        "stage_ms_p10": {n: pct(stage_ms[:, i], 10) for i, n in enumerate(names)},
        "stage_ms_p90": {n: pct(stage_ms[:, i], 90) for i, n in enumerate(names)},
        "roofline": roof,
        "roofline_gemm2": roof2,
        "clocks": clk.summary(),
        "e2e": {"value": round(replica_value(T, world, args.steps, e2e_ms), 1), "unit": "tokens/s",
                "pipelining": "h2d / d2h on copy streams overlapping the neighbouring steps' forwards",
                "h2d_bytes_per_step": x.numel() * 2 + ids.numel() * 4 + wts.numel() * 4,
                "d2h_bytes_per_step": out.numel() * 2},
        "gpu_launches": M.moe_forward_launches(ctx) * args.steps,
        "work": {"assignments": wm["A"], "nonempty_experts": wm["nonempty"], "padded_rows": padded_rows},
    }
    if not args.no_cpu_baseline and world == 1:       # timed beside the N=1 line only
        sample = OracleSample(w, x, ids_host, w_host, expert_source(w, weights))
        line["cpu_baseline"] = sample.run(seconds_target=12.0)
    print(json.dumps(line), flush=True)


def run_requant(args, w, local):
    """Time moe_requant_weights_ue8m0 on the workload's w13 shape (load-time
    weight preparation; HBM-bound: reads and writes each weight byte once)."""
    import moe_expert_layer_ep_gb300 as M
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    E, N, C = w["E_local"], 2 * w["I"], w["K"]
    g = torch.Generator(device=dev).manual_seed(w["seed"])
    win = torch.randint(0, 126, (E, N, C), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    sin = torch.rand((E, N // 128, C // 128), generator=g, device=dev) * 2.0 ** -12 + 2.0 ** -13
    wout = torch.empty_like(win)
    sout = torch.empty((E, N // 128, C // 128), dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        M.moe_requant_weights_ue8m0(win, sin, wout, sout)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t0.record()
        for _ in range(args.steps):
            M.moe_requant_weights_ue8m0(win, sin, wout, sout)
        t1.record()
        torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    nbytes = 2 * win.numel() + sin.numel() * 4 + sout.numel()
    peaks = load_peaks()
    gbs = nbytes / (ms / 1000.0) / 1e9
    print(json.dumps({"metric": "load-time UE8M0 weight requantisation bandwidth", "value": round(gbs, 1),
                      "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "e4m3+fp32->e4m3+ue8m0",
                      "data": "synthetic", "config": {"workload": w["name"] + ":w13", "shape": [E, N, C]},
                      "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                                   "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                                   "kernel": "requant_kernel", "traffic": None},
                      "clocks": clk.summary(), "gpu_launches": args.steps}), flush=True)


def run_router(args, w, local):
    """Time moe_route (fp32 router logits + top-k + softmax) on the workload's
    tokens.  The fp32 GEMM runs on the tensor cores as three exact bf16 planes
    of the weights (prepared once, outside the timed region).  Each timed call
    is preceded by a 256 MB write that evicts L2, and the calls are replayed
    from one CUDA graph with events around each call only.  The bound is the
    larger of the executed bf16 tensor work (3 x 2TKE) over the measured bf16
    peak and the call's HBM bytes over the measured copy bandwidth."""
    import moe_expert_layer_ep_gb300 as M
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    T, K, E, k = w["T"], w["K"], w["E_global"], w["topk"]
    x = synth.activations(T, K, w["seed"], dev)
    g = torch.Generator(device=dev).manual_seed(w["seed"] + 5)
    wr = torch.randn((E, K), generator=g, device=dev) * 0.02
    planes = M.moe_router_prepare(wr)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    wts = torch.empty((T, k), dtype=torch.float32, device=dev)
    rws = torch.empty(M.moe_route_workspace_size(T, K, E), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call():
        M.moe_route(x, planes, k, logits, ids, wts, ws=rws)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    if M.moe_read_device_status(rws) != 0:
        raise RuntimeError("router device status after warm-up")
    timing = "cuda-graph replay"
    try:
        ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)] for _ in range(args.steps)]
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            call()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for s in range(args.steps):
                flush.fill_(s & 0xFF)
                ev[s][0].record()
                call()
                ev[s][1].record()
        graph.replay()
        torch.cuda.synchronize()
        run_timed = graph.replay
    except Exception:
        timing = "eager launches"
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        stream = torch.cuda.current_stream()

        def run_timed():
            for s in range(args.steps):
                flush.fill_(s & 0xFF)
                ev[s][0].record(stream)
                call()
                ev[s][1].record(stream)
    with ClockSampler(local) as clk:
        run_timed()
        torch.cuda.synchronize()
    per = np.array([e0.elapsed_time(e1) for e0, e1 in ev])
    ms = float(per.mean())
    sec = ms / 1000.0
    flops = 2.0 * T * K * E
    segs = (K + 1023) // 1024
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fold = ((T + 127) // 128) * ((E + 127) // 128) * 4 >= sms * 3
    # segment sums written and read back (small batches), or the logits
    # written, read and rewritten by the top-k kernel (folded tiles)
    nbytes = 6.0 * E * K + 2.0 * T * K + 4.0 * T * E * (3 if fold else 2 * segs + 1) + 8.0 * T * k
    peaks = load_peaks()
    t_tc = 3.0 * flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    if t_tc >= t_hbm:
        tf = 3.0 * flops / sec / 1e12
        roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(tf / peaks["bf16_tflops"], 4), "peak_source": peaks["source"] + " bf16",
                "work": "executed bf16 flops = 3 planes x 2TKE"}
    else:
        gbs = nbytes / sec / 1e9
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": peaks["source"]}
    roof.update({"kernel": "moe_route (router_logits_tc + topk_softmax)", "traffic": None,
                 "algorithmic_bytes": int(nbytes), "algorithmic_flops": flops})
    print(json.dumps({"metric": "fp32 router (logits + top-k + softmax) throughput", "value": round(T / sec, 1),
                      "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": round(ms, 4),
                      "ms_p10_p90": [round(float(np.percentile(per, q)), 4) for q in (10, 90)],
                      "higher_is_better": True, "dtype": "f32 (bf16x3 tensor-core planes, fp32 accumulate)",
                      "data": "synthetic", "fp32_equivalent_tflops": round(flops / sec / 1e12, 2),
                      "config": {"workload": w["name"], "T": T, "K": K, "E": E, "topk": k,
                                 "l2": "flushed before each call (256 MB write)", "timing": timing},
                      "roofline": roof, "clocks": clk.summary(), "gpu_launches": 2 * args.steps}), flush=True)


CROSSOVER_E_LOCAL = (8, 16, 32, 64, 128, 256)
CROSSOVER_T = (1, 16, 64, 256, 1024, 4096)


def run_crossover(args, w, local):
    """Masked vs compact layout: the whole layer, one graph of --steps
    forwards per point with events between the stages, for every E_local in
    CROSSOVER_E_LOCAL and T in CROSSOVER_T.  FP8, the workload's K and I,
    E_global 256 with the rank's experts first (ids outside them are dropped),
    uniform N(0, 1) router logits, top-8; masked max_m = T rounded up to 16.
    One JSON line per (E_local, T) with both layouts' stage times."""
    import moe_expert_layer_ep_gb300 as M
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    K, I, topk, E_g = w["K"], w["I"], 8, 256
    names = ["plan", "quant_scatter", "gemm_w13_act", "gemm_w2", "combine"]
    for E_l in CROSSOVER_E_LOCAL:
        w13, w13s = synth.fp8_expert_weights(E_l, 2 * I, K, w["seed"] + 2, dev)
        w2, w2s = synth.fp8_expert_weights(E_l, K, I, w["seed"] + 3, dev)
        for T in CROSSOVER_T:
            x = synth.activations(T, K, w["seed"], dev)
            ids_h, wts_h = synth.routing(T, E_g, topk, w["seed"] + 1)
            ids, wts = ids_h.to(dev), wts_h.to(dev)
            local_rows = int(((ids_h >= 0) & (ids_h < E_l)).sum())
            active = int(torch.unique(ids_h[(ids_h >= 0) & (ids_h < E_l)]).numel())
            res = {}
            for layout in ("compact", "masked"):
                max_m = (T + 15) // 16 * 16 if layout == "masked" else 0
                shape = M.make_shape(T, K, I, E_g, E_l, topk, "fp8", layout, 0, max_m)
                ctx = M.moe_ctx_create(shape, w13, w13s, w2, w2s)
                ws = M.alloc_workspace(ctx, dev)
                out = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
                stages = [lambda: M.moe_plan_layout(ctx, ids, ws), lambda: M.moe_quant_scatter(ctx, x, ws),
                          lambda: M.moe_grouped_gemm_w13_act(ctx, ws), lambda: M.moe_grouped_gemm_w2(ctx, ws),
                          lambda: M.moe_combine(ctx, wts, ws, out)]
                M.moe_clear_device_status(ws)
                for _ in range(max(args.warmup, 3)):
                    M.moe_forward(ctx, x, ids, wts, ws, out)
                torch.cuda.synchronize()
                ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(6)]
                      for _ in range(args.steps)]
                side = torch.cuda.Stream(device=dev)
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    M.moe_forward(ctx, x, ids, wts, ws, out)
                torch.cuda.current_stream().wait_stream(side)
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    for st in range(args.steps):
                        ev[st][0].record()
                        for i, fn in enumerate(stages):
                            fn()
                            ev[st][i + 1].record()
                graph.replay()
                torch.cuda.synchronize()
                graph.replay()
                torch.cuda.synchronize()
                status = M.moe_read_device_status(ws)
                if status != 0:
                    raise RuntimeError(f"device status {status} (E_local {E_l}, T {T}, {layout})")
                st_ms = np.median(np.array([[ev[s][i].elapsed_time(ev[s][i + 1]) for i in range(5)]
                                            for s in range(args.steps)]), axis=0)
                res[layout] = {"ms": round(float(st_ms.sum()), 4),
                               "stage_ms": {n: round(float(v), 4) for n, v in zip(names, st_ms)},
                               "ws_mb": round(M.moe_workspace_size(ctx) / 2 ** 20, 1)}
                del graph, ws, ctx          # the context is destroyed with its last reference
            print(json.dumps({"op": "crossover", "E_local": E_l, "T": T, "local_rows": local_rows,
                              "active_experts": active, "auto": "masked" if M.moe_choose_layout(E_g, E_l) == 2
                              else "compact", "masked_over_compact": round(res["masked"]["ms"] / res["compact"]["ms"], 3),
                              **res}), flush=True)
        del w13, w13s, w2, w2s
        torch.cuda.empty_cache()


def main():
    args = parse()
    world, rank, local = dist_env()
    w = workload(args)
    w["name"] = args.workload
    if world > 1:
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        torch.distributed.init_process_group(backend=backend)
    try:
        if args.op in ("requant", "router", "crossover"):
            if rank == 0:
                {"requant": run_requant, "router": run_router, "crossover": run_crossover}[args.op](args, w, local)
            return
        if args.impl == "reference":
            run_reference(args, w, world, rank)
        else:
            run_ours(args, w, world, rank, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
