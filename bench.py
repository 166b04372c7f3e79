"""Benchmark of the W4A8 block-32 linear on GB300.

Headline workload: decode FFN up-projection, M=1, K=2048, N=8192, with 16
distinct weight sets (151 MB of packed weights and scales, more than the
129 MB L2) used in rotation, so every call streams its weights from HBM.
A step is one CUDA-graph replay of `--calls-per-step` consecutive decode
calls cycling through the 16 sets.  The metric is effective HBM bandwidth:
algorithmic bytes (int4 weights + fp16 block scales + fp16 x + fp16 y) per
second.  Secondary records in the same JSON line (`--secondary`): the
prefill GEMM (M=512, K=2048, N=8192) in int8-equivalent TOPS (2*M*N*K per
call), one decode step over 26 decoder layers (7 linears per layer, and the
fused layer: q/k/v as one projection, gated gate/up, down), a shape sweep,
the decode linear on producer-quantised activations, and decode attention.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica (the linear has no
exchange step on one GPU); rank 0 prints one JSON line.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "decode_ffn_up_m1_k2048_n8192"
METRIC = "W4A8 linear: decode eff. HBM GB/s & prefill int8 TOPS, % of GB300 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--calls-per-step", type=int, default=512)
    ap.add_argument("--sets", type=int, default=16)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only-secondary", action="store_true",
                    help="time only the secondary workloads and print their records")
    ap.add_argument("--secondary", default="prefill,layers,sweep,q8,attention,sets32,ceiling",
                    help="comma list of secondary workloads to run: prefill, layers (both layer "
                         "workloads), layers_fused, sweep, q8 (decode on producer-quantised activations), "
                         "attention (decode attention over an fp16 KV cache), sets32 (the headline with 32 "
                         "rotating weight sets), ceiling (read-only HBM ceilings of the library's two load "
                         "mechanisms)")
    ap.add_argument("--layer-oracle-seconds", type=float, default=8.0,
                    help="CPU budget for timing the oracle on one decoder layer (0 skips it)")
    return ap.parse_args()


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            hbm = d.get("hbm_gbs")
            bf16 = d.get("bf16_tflops")
            if hbm and bf16:
                return float(hbm), float(bf16), float(d.get("bf16_tflops_sustained") or bf16), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel, files):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(kernel)
    except Exception:
        return None
    if not d or d.get("source_hash") != kernel_hash(files):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(ms, ws, device):
    """Slowest rank's time (ms); every rank returns the same value."""
    if ws <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_throughput(bytes_per_rank, ms, ws):
    """Whole-job GB/s: every rank moved bytes_per_rank in the slowest rank's time (weak scaling)."""
    return ws * bytes_per_rank / (ms * 1e-3) / 1e9


def oracle_inputs(lin, seed):
    from int4_weight_quantized_gb300 import workloads as wl
    x, codes, scales = wl.make_linear_inputs(lin, seed, 0)
    return x.numpy(), codes.numpy(), scales.numpy()


def time_oracle(inputs, seconds, max_calls=None):
    """The CPU oracle on this host, as it stands, on whole calls until `seconds` pass."""
    import oracle
    xn, cn, sn = inputs
    oracle.get()
    calls = 0
    t0 = time.perf_counter()
    while True:
        oracle.linear(xn, cn, sn)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_calls and calls >= max_calls):
            break
    return calls, el


def reference_arm(args):
    """The oracle timed on host cores: same metric, unit and workload as our arm.
    A step is one whole decode call (M=1, K=2048, N=8192) of the oracle."""
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    from int4_weight_quantized_gb300 import workloads as wl
    W = [w for w in wl.workloads() if w.name == HEADLINE][0]
    lin = W.linears[0]
    inputs = oracle_inputs(lin, W.seed)
    time_oracle(inputs, 0.0, max_calls=max(1, args.warmup))
    calls, secs = time_oracle(inputs, 1e9, max_calls=args.steps)
    gbs = lin.bytes * calls / secs / 1e9
    sample = f"{calls} whole M=1 K=2048 N=8192 calls of the plain C oracle, single thread"
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": calls, "warmup": args.warmup, "ms_per_step": 1e3 * secs / calls,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int4xint8",
            "data": "synthetic", "config": {"workload": HEADLINE, "calls_per_step": 1},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
        return
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import int4_weight_quantized_gb300 as w4
    from int4_weight_quantized_gb300 import workloads as wl
    from int4_weight_quantized_gb300.build import build
    if rank == 0:
        build()
    if ws > 1:
        dist.barrier()
    build()

    dev = torch.device("cuda", local)
    if args.only_secondary:
        hbm, bf16, _, peak_src = peaks()
        stream = torch.cuda.Stream(device=dev)
        print(json.dumps(run_secondary(w4, wl, dev, stream, hbm, bf16, peak_src, args.secondary)), flush=True)
        return
    W = [w for w in wl.workloads() if w.name == HEADLINE][0]
    lin = W.linears[0]
    S = args.sets
    xs = wl.make_x(lin.M, lin.K, W.seed, lin.outlier_frac).to(dev)
    sets = []
    for i in range(S):
        codes, scales = wl.make_weights(lin.N, lin.K, W.seed + 1 + i, lin.s_lo, lin.s_hi)
        sets.append((w4.pack(codes.to(dev)), scales.to(dev)))
    outs = [torch.empty((lin.M, lin.N), dtype=torch.float16, device=dev) for _ in range(S)]
    cps = args.calls_per_step

    def step_calls():
        for c in range(cps):
            i = c % S
            w4.linear(xs, sets[i][0], sets[i][1], out=outs[i], path=w4.PATH_DECODE)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        step_calls()                                  # first call sets kernel attributes
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step_calls()
        for _ in range(args.warmup):
            g.replay()
        stream.synchronize()
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk:
            e0.record(stream)
            for _ in range(args.steps):
                g.replay()
            e1.record(stream)
            e1.synchronize()
        torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    ms_step = ms / args.steps
    bytes_step = lin.bytes * cps
    value = job_throughput(bytes_step * args.steps, ms, ws)
    per_launch_s = ms * 1e-3 / (args.steps * cps)
    hbm, bf16, bf16_sus, peak_src = peaks()
    gemv_files = ["int4_weight_quantized_gb300/csrc/gemv_stream.cu", "int4_weight_quantized_gb300/csrc/common.cuh",
                  "int4_weight_quantized_gb300/csrc/sync.cuh"]
    achieved = lin.bytes / per_launch_s / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": traffic_for("gemv_stream_decode_ffn_up", gemv_files), "peak_source": peak_src,
            "kernel": "gemv_stream_kernel<1,2,1,false,false,false>", "algorithmic_bytes_per_launch": lin.bytes,
            "launch_time_us": per_launch_s * 1e6,
            "note": "launch time = timed region / launches (every launch in the step is this kernel)"}

    # ---- end to end through the C entry point with pinned host buffers
    # Every step copies the step's inputs from pinned host memory, runs the
    # cps calls of w4a8_linear (the plain C entry point) and reads all outputs
    # back, inside the timed region.  "graph": the step (input copy, the
    # calls, output copy) is captured once into a CUDA graph and replayed, as
    # a decode loop runs it; "eager": the copies and one Python call per
    # linear (host-bound: ctypes and launch overhead per call).
    e2e_steps = max(3, min(args.steps, 50))
    xh = torch.empty((cps, lin.M, lin.K), dtype=torch.float16).pin_memory()
    xh.copy_(xs.cpu().expand(cps, lin.M, lin.K))
    yh = torch.empty((cps, lin.M, lin.N), dtype=torch.float16).pin_memory()
    xd = torch.empty((cps, lin.M, lin.K), dtype=torch.float16, device=dev)
    yd = torch.empty((cps, lin.M, lin.N), dtype=torch.float16, device=dev)
    with torch.cuda.stream(stream):
        def e2e_calls():
            for c in range(cps):
                i = c % S
                w4.linear_c(xd[c], sets[i][0], sets[i][1], yd[c])

        def e2e_step(run):
            xd.copy_(xh, non_blocking=True)
            run()
            yh.copy_(yd, non_blocking=True)
            stream.synchronize()
        e2e_step(e2e_calls)
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge, stream=stream):
            xd.copy_(xh, non_blocking=True)
            e2e_calls()
            yh.copy_(yd, non_blocking=True)

        def graph_step():
            ge.replay()
            stream.synchronize()
        graph_step()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            graph_step()
        e2e_graph_s = time.perf_counter() - t0
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step(e2e_calls)
        e2e_eager_s = time.perf_counter() - t0
    e2e = {"value": ws * bytes_step * e2e_steps / e2e_graph_s / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": xh.numel() * 2, "d2h_bytes_per_step": yh.numel() * 2, "steps": e2e_steps,
           "note": "host wall clock per step: one CUDA graph of the step (pinned x -> device copy, the step's "
                   "w4a8_linear calls, all y -> pinned host copy), synchronize",
           "eager_value": ws * bytes_step * e2e_steps / e2e_eager_s / 1e9,
           "eager_note": "same step with one Python/ctypes w4a8_linear call per linear (host-bound)"}

    secondary = []
    if not args.no_secondary:
        secondary = run_secondary(w4, wl, dev, stream, hbm, bf16, peak_src, args.secondary, headline_gbs=value)

    layer_oracle = None
    if rank == 0 and args.layer_oracle_seconds > 0 and not args.no_secondary:
        layer_oracle = time_layer_oracle(wl, args.layer_oracle_seconds)

    cpu = None
    if rank == 0:
        calls, secs = time_oracle(oracle_inputs(lin, W.seed), args.cpu_seconds)
        cpu = {"value": lin.bytes * calls / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{calls} whole M=1 K=2048 N=8192 calls of the plain C oracle in {secs:.1f} s, single thread"}

    if rank == 0:
        summary = make_summary(value, roof, secondary, layer_oracle)
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "int4xint8", "data": "synthetic", "summary": summary,
                "config": {"workload": HEADLINE, "M": lin.M, "N": lin.N, "K": lin.K, "weight_sets": S,
                           "calls_per_step": cps, "l2": f"inputs larger than L2: {S} rotating weight sets = "
                           f"{S * lin.weight_bytes / 1e6:.1f} MB > 129 MB",
                           "launch": "CUDA graph of calls_per_step decode launches", "parallelism": f"replicas{ws}"},
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps * cps, "clocks": clk.summary(), "layer_oracle": layer_oracle,
                "secondary": secondary}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def make_summary(value, roof, secondary, layer_oracle):
    """One short record per workload (value, us, fraction of its roofline), placed
    early in the JSON line so that a truncated copy of the line still shows it."""
    out = {"decode_ffn_up_m1": {"GB_s": round(value, 1), "us_per_launch": round(roof["launch_time_us"], 3),
                                "frac_hbm": round(roof["frac"], 4)}}
    for r in secondary:
        name = r.get("workload", "")
        if "rows" in r:
            for row in r["rows"]:
                key = f"sweep_m{row['M']}_k{row['K']}_n{row['N']}"
                out[key] = {"path": row["path"], "us": round(row["us_per_call"], 2),
                            "frac": round(row["frac_fp16_tensor"] if row["path"] == "prefill" else row["frac_hbm"], 4)}
            continue
        rec = {"value": round(r["value"], 1), "unit": r["unit"].split(" ")[0]}
        for k in ("us_per_call", "us_per_decode_step"):
            if k in r:
                rec["us"] = round(r[k], 2)
        if "roofline" in r:
            rec["frac"] = round(r["roofline"]["frac"], 4)
        for k in ("epilogue_fp32_frac", "frac_of_bulk_read_ceiling"):
            if k in r:
                rec[k] = round(r[k], 4)
        out[name] = rec
    if layer_oracle:
        out["decoder_layers_oracle_cpu"] = {"s_per_step_extrapolated": round(layer_oracle["s_per_step_extrapolated"], 2),
                                            "cores": layer_oracle["cores"]}
    return out


def time_layer_oracle(wl, seconds):
    """The CPU oracle on one decoder layer (7 linears, M=1) of the 26-layer
    workload, repeated for about `seconds`; a decode step is 26 such layers and
    the workload has 128 steps, so those totals are extrapolated (x26, x128)."""
    import oracle
    W = [w for w in wl.workloads() if w.name == "decoder_layers_m1_26x7"][0]
    ins = []
    for li, lin in enumerate(W.linears):
        x, codes, scales = wl.make_linear_inputs(lin, W.seed + li)
        ins.append((x.numpy(), codes.numpy(), scales.numpy()))
    oracle.get()
    layers, t0 = 0, time.perf_counter()
    while True:
        for xn, cn, sn in ins:
            oracle.linear(xn, cn, sn)
        layers += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    per_layer = el / layers
    n_layers = W.extra["layers"]
    return {"kind": "oracle", "cores": 1, "s_per_layer": per_layer, "layers_timed": layers,
            "s_per_step_extrapolated": per_layer * n_layers,
            "s_per_128_steps_extrapolated": per_layer * n_layers * W.extra["decode_steps"],
            "GB_s": sum(l.bytes for l in W.linears) / per_layer / 1e9,
            "note": "measured on one layer of the 26 (7 linears at M=1, single thread); the step (x26) and the "
                    "128-step workload (x26x128) are extrapolations"}


def run_sets32(w4, wl, dev, stream, hbm, peak_src, cps=512, steps=20):
    """The headline decode shape with 32 rotating weight sets (302 MB, 2.3x the
    L2) instead of 16, to show that the 16-set figure is not helped by L2."""
    import torch
    W = [w for w in wl.workloads() if w.name == HEADLINE][0]
    lin = W.linears[0]
    S = 32
    xs = wl.make_x(lin.M, lin.K, W.seed, lin.outlier_frac).to(dev)
    sets = []
    for i in range(S):
        c, sc = wl.make_weights_on(dev, lin.N, lin.K, W.seed + 100 + i, lin.s_lo, lin.s_hi)
        sets.append((w4.pack(c), sc))
        del c
    outs = [torch.empty((lin.M, lin.N), dtype=torch.float16, device=dev) for _ in range(S)]
    with torch.cuda.stream(stream):
        def calls():
            for c in range(cps):
                i = c % S
                w4.linear(xs, sets[i][0], sets[i][1], out=outs[i], path=w4.PATH_DECODE)
        calls()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            calls()
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
        e1.synchronize()
    per = e0.elapsed_time(e1) * 1e-3 / (steps * cps)
    gbs = lin.bytes / per / 1e9
    return {"workload": HEADLINE + "_32sets", "value": gbs, "unit": "GB/s", "us_per_call": per * 1e6,
            "weight_set_bytes": S * lin.weight_bytes,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "peak_source": peak_src}}


def run_ceiling(w4, dev, stream, hbm, headline_gbs=None, nbytes=2 << 30, reps=10):
    """Read-only HBM ceilings of the library's two load mechanisms (bulk
    asynchronous copies, as the decode kernel streams its weights; 128-bit
    loads from every thread), each reading a 2 GiB buffer once per call."""
    import torch
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    buf.fill_(1)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    res = {"workload": "hbm_read_ceiling", "bytes_per_call": nbytes}
    with torch.cuda.stream(stream):
        for mode, name in ((0, "bulk_copy"), (1, "ld_128")):
            sink = torch.zeros(152, dtype=torch.int32, device=dev)
            w4.debug_stream_read(buf, mode, sink)
            best = None
            for _ in range(reps):
                flush.fill_(0)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                w4.debug_stream_read(buf, mode, sink)
                e1.record(stream)
                e1.synchronize()
                ms = e0.elapsed_time(e1)
                best = ms if best is None or ms < best else best
            res[name + "_GB_s"] = nbytes / (best * 1e-3) / 1e9
    res["value"] = res["bulk_copy_GB_s"]
    res["unit"] = "GB/s"
    res["copy_peak_GB_s"] = hbm
    if headline_gbs:
        res["frac_of_bulk_read_ceiling"] = headline_gbs / res["bulk_copy_GB_s"]
    res["note"] = "best of 10 calls; the copy peak (read + write bytes) is the roofline denominator, these are context"
    return res


def run_secondary(w4, wl, dev, stream, hbm, bf16, peak_src, which="prefill,layers,sweep,q8,attention",
                  headline_gbs=None):
    """Secondary workloads: prefill GEMM (M=512) in TOPS, the 26-layer decode
    step and the shape sweep, each timed with CUDA events on its stream."""
    import torch
    which = {s.strip() for s in which.split(",") if s.strip()}
    res = []
    if "prefill" in which:
        res.append(run_prefill(w4, wl, dev, stream, bf16, peak_src))
    if "layers" in which:
        res.append(run_decoder_layers(w4, wl, dev, stream, hbm, peak_src))
    if "layers_fused" in which or "layers" in which:
        res.append(run_decoder_layers(w4, wl, dev, stream, hbm, peak_src, name="decoder_layers_m1_26x4_fused"))
    if "sweep" in which:
        res.append(run_sweep(w4, wl, dev, stream, hbm, bf16, peak_src))
    if "q8" in which:
        res.append(run_decode_q8(w4, wl, dev, stream, hbm, peak_src))
    if "attention" in which:
        res.append(run_attention(w4, dev, stream, hbm, peak_src))
    if "sets32" in which:
        res.append(run_sets32(w4, wl, dev, stream, hbm, peak_src))
    if "ceiling" in which:
        res.append(run_ceiling(w4, dev, stream, hbm, headline_gbs))
    return res


def run_attention(w4, dev, stream, hbm, peak_src, B=32, Hq=8, Hkv=1, D=256, L=640, sets=8, cps=64, steps=20):
    """Decode attention for B sequences of L = 640 cached tokens (prefill 512 +
    128 decode steps) with the decoder layer's 8 query heads over one KV head of
    256; 8 rotating caches (168 MB > L2); GB/s of K + V + q + out."""
    import torch
    g = torch.Generator(device=dev).manual_seed(6000)
    caches = [(torch.randn((B, Hkv, L, D), generator=g, device=dev, dtype=torch.float32).half(),
               torch.randn((B, Hkv, L, D), generator=g, device=dev, dtype=torch.float32).half()) for _ in range(sets)]
    q = torch.randn((B, Hq, D), generator=g, device=dev, dtype=torch.float32).half()
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.float16, device=dev)
    ws = torch.empty(max(1, w4.lib().w4a8_decode_attention_workspace_bytes(B, Hq, Hkv, D, L)), dtype=torch.uint8,
                     device=dev)
    with torch.cuda.stream(stream):
        def calls():
            for c in range(cps):
                k, v = caches[c % sets]
                w4.decode_attention(q, k, v, lens, out=out, workspace=ws)
        calls()
        stream.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            calls()
        for _ in range(3):
            gr.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            gr.replay()
        e1.record(stream)
        e1.synchronize()
    per = e0.elapsed_time(e1) * 1e-3 / (steps * cps)
    byt = 2 * B * Hkv * L * D * 2 + 2 * 2 * B * Hq * D
    return {"workload": f"decode_attention_b{B}_hq{Hq}_hkv{Hkv}_d{D}_l{L}", "value": byt / per / 1e9, "unit": "GB/s",
            "us_per_call": per * 1e6,
            "roofline": {"bound": "hbm", "achieved": byt / per / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": byt / per / 1e9 / hbm, "peak_source": peak_src}}


def run_decode_q8(w4, wl, dev, stream, hbm, peak_src, cps=512, sets=16, steps=20):
    """The headline decode shape (M=1, K=2048, N=8192, 16 rotating weight sets)
    on activations quantised by their producer (w4a8_linear_q8: int8 codes and
    fp32 block scales in, no in-kernel quantisation), beside the fp16-input
    linear timed the same way; plus the producer itself (w4a8_rmsnorm_quant)
    followed by the linear.  CUDA graphs of cps calls."""
    import torch
    W = [w for w in wl.workloads() if w.name == HEADLINE][0]
    lin = W.linears[0]
    xs = wl.make_x(lin.M, lin.K, W.seed, lin.outlier_frac).to(dev)
    gamma = torch.ones(lin.K, dtype=torch.float16, device=dev)
    wsets = []
    for i in range(sets):
        c, s = wl.make_weights(lin.N, lin.K, W.seed + 1 + i, lin.s_lo, lin.s_hi)
        wsets.append((w4.pack(c.to(dev)), s.to(dev)))
    out = torch.empty((lin.M, lin.N), dtype=torch.float16, device=dev)
    with torch.cuda.stream(stream):
        q, sx = w4.rmsnorm_quant(xs, gamma, 1e-6)

        def timed(body):
            body()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                body()
            for _ in range(3):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                g.replay()
            e1.record(stream)
            e1.synchronize()
            return e0.elapsed_time(e1) * 1e-3 / (steps * cps)

        t_q8 = timed(lambda: [w4.linear_q8(q, sx, *wsets[c % sets], out=out) for c in range(cps)])
        t_fp16 = timed(lambda: [w4.linear(xs, *wsets[c % sets], out=out, path=w4.PATH_DECODE) for c in range(cps)])
        t_norm = timed(lambda: [(w4.rmsnorm_quant(xs, gamma, 1e-6, codes=q, sx=sx),
                                 w4.linear_q8(q, sx, *wsets[c % sets], out=out)) for c in range(cps)])
    byt = lin.weight_bytes + lin.M * lin.K + lin.M * (lin.K // 32) * 4 + 2 * lin.M * lin.N
    return {"workload": "decode_ffn_up_q8_m1_k2048_n8192", "value": byt / t_q8 / 1e9, "unit": "GB/s",
            "us_per_call": t_q8 * 1e6, "fp16_input_us_per_call": t_fp16 * 1e6,
            "rmsnorm_quant_plus_linear_us": t_norm * 1e6,
            "roofline": {"bound": "hbm", "achieved": byt / t_q8 / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": byt / t_q8 / 1e9 / hbm, "peak_source": peak_src},
            "note": "bytes = int4 weights + fp16 scales + int8 codes + fp32 block scales + fp16 y"}


def run_prefill(w4, wl, dev, stream, bf16, peak_src):
    """Prefill GEMM (M=512) in TOPS: a CUDA graph of 8 calls over 4 weight sets."""
    import torch
    W = [w for w in wl.workloads() if w.name == "prefill_ffn_up_m512_k2048_n8192"][0]
    lin = W.linears[0]
    x, codes, scales = wl.make_linear_inputs(lin, W.seed, 0)
    xd = x.to(dev)
    sets = []
    for i in range(4):
        c, s = wl.make_weights(lin.N, lin.K, W.seed + 1 + i, lin.s_lo, lin.s_hi)
        sets.append((w4.pack(c.to(dev)), s.to(dev)))
    out = torch.empty((lin.M, lin.N), dtype=torch.float16, device=dev)
    ws = w4.make_workspace(lin.M, lin.N, lin.K, w4.PATH_PREFILL, dev)
    reps = 8
    with torch.cuda.stream(stream):
        def calls():
            for r in range(reps):
                p, s = sets[r % len(sets)]
                w4.linear(xd, p, s, out=out, path=w4.PATH_PREFILL, workspace=ws)
        calls()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            calls()
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = 20
        e0.record(stream)
        for _ in range(n):
            g.replay()
        e1.record(stream)
        e1.synchronize()
    per_call = e0.elapsed_time(e1) * 1e-3 / (n * reps)
    tops = lin.ops / per_call / 1e12
    # the per-block scaling: one multiply (s_w * s_x) and one multiply-add per
    # output, token and 32-block, on 128 fp32 lanes per SM per clock
    fp32_ops = 2 * lin.M * lin.N * (lin.K // 32)
    sm_mhz = 2070.0                      # maximum SM clock of the part
    floor_us = fp32_ops / (152 * 128 * sm_mhz * 1e6) * 1e6
    return {"workload": W.name, "value": tops, "unit": "TOPS (2*M*N*K int8-equivalent)",
                "us_per_call": per_call * 1e6,
                "epilogue_fp32_ops": fp32_ops, "epilogue_fp32_floor_us": floor_us,
                "epilogue_fp32_frac": floor_us / (per_call * 1e6),
                "epilogue_note": "floor = 2*M*N*K/32 fp32 ops at 128 lanes/clock/SM on 152 SMs at the max SM clock; "
                                 "frac = floor / measured time",
                "roofline": {"bound": "tensor", "achieved": tops, "peak": bf16, "unit": "TFLOP/s",
                             "frac": tops / bf16, "peak_source": peak_src,
                             "note": "contraction runs on fp16 tensor cores (exact for int4 x int8 codes); "
                                     "peak is the dense fp16/bf16 tensor rate"}}


def run_sweep(w4, wl, dev, stream, hbm, bf16, peak_src, sets=5, reps=20):
    """The K/N shape sweep under the automatic stage-aware dispatch: per shape,
    a CUDA graph of calls over `sets` rotating weight sets (> L2 in total)."""
    import torch
    W = [w for w in wl.workloads() if w.name == "shape_sweep"][0]
    rows = []
    with torch.cuda.stream(stream):
        for li, lin in enumerate(W.linears):
            ws = []
            for i in range(sets):
                c, s = wl.make_weights_on(dev, lin.N, lin.K, W.seed + 10 * li + i, lin.s_lo, lin.s_hi)
                ws.append((w4.pack(c), s))
                del c
            x = wl.make_x(lin.M, lin.K, W.seed + li, lin.outlier_frac).to(dev)
            out = torch.empty((lin.M, lin.N), dtype=torch.float16, device=dev)
            path = w4.select_path(lin.M, lin.N, lin.K)
            wsp = w4.make_workspace(lin.M, lin.N, lin.K, path, dev)

            def calls():
                for p, s in ws:
                    w4.linear(x, p, s, out=out, path=path, workspace=wsp)
            calls()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                calls()
            for _ in range(3):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            e1.synchronize()
            per_call = e0.elapsed_time(e1) * 1e-3 / (reps * sets)
            gbs = lin.bytes / per_call / 1e9
            tops = lin.ops / per_call / 1e12
            rows.append({"M": lin.M, "K": lin.K, "N": lin.N,
                         "path": {w4.PATH_DECODE: "decode", w4.PATH_MID: "mid"}.get(path, "prefill"),
                         "us_per_call": per_call * 1e6, "GB_s": gbs, "TOPS": tops,
                         "frac_hbm": gbs / hbm, "frac_fp16_tensor": tops / bf16})
            del ws
    return {"workload": W.name, "rows": rows, "peak_source": peak_src,
            "note": "decode rows are measured in GB/s against HBM, prefill rows in TOPS against the fp16 tensor peak"}


def run_decoder_layers(w4, wl, dev, stream, hbm, peak_src, steps=20, name="decoder_layers_m1_26x7"):
    """One decode step over 26 decoder layers (M=1), captured as a CUDA graph:
    7 linears per layer (182 launches), or with name
    decoder_layers_m1_26x4_fused the fused layer (qkv, o, gated gate/up,
    down: 104 launches); effective HBM GB/s over the step."""
    import torch
    W = [w for w in wl.workloads() if w.name == name][0]
    layers = W.extra["layers"]
    linears = []
    with torch.cuda.stream(stream):
        for layer in range(layers):
            for li, lin in enumerate(W.linears):
                seed = W.seed + 100 * layer + li
                c, s = wl.make_weights_on(dev, lin.rows, lin.K, seed, lin.s_lo, lin.s_hi)
                x = wl.make_x(lin.M, lin.K, seed, lin.outlier_frac).to(dev)
                linears.append((x, w4.pack(c), s, torch.empty((lin.M, lin.N), dtype=torch.float16, device=dev),
                                lin.gated))
                del c
        step_bytes = layers * sum(l.bytes for l in W.linears)

        def step():
            for x, p, s, o, act in linears:
                if act:
                    w4.linear_gated(x, p, s, act=act, out=o)
                else:
                    w4.linear(x, p, s, out=o, path=w4.PATH_DECODE)
        step()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
        e1.synchronize()
    per_step = e0.elapsed_time(e1) * 1e-3 / steps
    gbs = step_bytes / per_step / 1e9
    return {"workload": W.name, "value": gbs, "unit": "GB/s", "us_per_decode_step": per_step * 1e6,
            "launches_per_step": len(linears), "bytes_per_step": step_bytes,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "peak_source": peak_src}}


if __name__ == "__main__":
    main()
