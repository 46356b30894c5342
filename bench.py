#!/usr/bin/env python
"""TTT-MLP layer benchmark: tokens/s at the Qwen3-4B MLP layer shape.

Workload (default): one SwiGLU MLP layer with an In-Place TTT fast W_down,
d=2560, f=9728, one document of T=32768 tokens per step, chunk C=256, Conv1D
k=5, eta=1e-3, bf16 activations/weights with an fp32 fast weight; synthetic
seeded inputs (X ~ N(0,1) rows RMS-normalised, weights ~ N(0, 0.02^2)).
A step is one forward call over the document: Conv1D target source, SwiGLU
producer, target projection, intra-group Gram blocks and the fused
apply+update group kernels (the fast weight is reset to W_0 at the document
start, so every step does identical work).

Prints one JSON line.  `value` is device-timed throughput with inputs resident
in HBM; `e2e` is the same metric through the host-buffer C-ABI call with the
host<->device copies inside the timed region; `roofline` is the dominant
kernel (the fused apply+update group kernel) timed live with CUDA events;
`cpu_baseline` is the CPU fp64 oracle timed on a bounded sample.

Multi-GPU (torchrun): every rank runs its own documents (the method's
documents are independent); no collective touches the data path, only the
barrier and the max-over-ranks of the timed interval.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TTT-MLP tokens/s at Qwen3-4B layer shape, C=256; % of TC/HBM roofline"
UNIT = "tokens/s"
KERNEL_SRC = os.path.join(ROOT, "chunk_wise_weight_ttt_b300", "csrc", "tc_gemm.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "group_kernel_traffic.json")
REF_CHUNKS = 2  # chunks of the document per reference-arm step (a bounded sample)
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--chunk", type=int, default=256)
    p.add_argument("--tokens", type=int, default=32768)
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--workload", choices=["layer", "long", "sweep", "stack"], default="layer",
                   help="layer: the headline workload (default, one JSON line with the full "
                        "contract); long / sweep / stack: the other measured configurations, "
                        "one JSON line per case (device-timed, inputs drawn on the GPU)")
    return p.parse_args(argv)


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, seconds: float, world: int, device=None):
    """Whole-job throughput: units summed over ranks / max-over-ranks time."""
    t = max_over_ranks(seconds, world, device)
    total = units_per_rank * world
    return total / t, t


# ---------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def group_tokens() -> int:
    """Target tokens per group of the fused apply+update kernel (the library's
    default, or the TTT_GROUP_TOKENS override it honours)."""
    v = os.environ.get("TTT_GROUP_TOKENS")
    n = int(v) if v and v.isdigit() else 2048
    return n if 256 <= n <= 4096 else 2048


def kernel_hash() -> str:
    """sha256 prefix of the kernel source's code: comments and blank space
    are dropped first, so that a comment edit keeps the stored counters."""
    import re
    with open(KERNEL_SRC) as fh:
        src = fh.read()
    src = re.sub(r"//[^\n]*", "", src)
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    code = "\n".join(line.strip() for line in src.splitlines() if line.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def stored_traffic(groups_per_launch: float, chunk: int, d: int, f: int):
    """DRAM bytes per group-kernel launch: the committed ncu figure per group
    times the groups one launch chains.  None when the kernel source has
    changed since the counters were taken, or for a shape or grouping other
    than the captured one."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as fh:
        rec = json.load(fh)
    if (rec.get("kernel_sha256_16") != kernel_hash() or "dram_bytes_per_group" not in rec
            or rec.get("captured_chunk") != chunk or rec.get("captured_group_tokens") != group_tokens()
            or rec.get("captured_shape") != {"d": d, "f": f}):
        return None
    return rec["dram_bytes_per_group"] * groups_per_launch


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        busy = [s for s, p in zip(sm, power) if p > 0.5 * max(power)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power)}


def pick_peak(peaks, clocks):
    """(bf16 peak TFLOP/s, name) that a kernel timed under `clocks` is held to.

    The burst figure was measured over a short region near the maximum SM
    clock; the sustained one over seconds under the power cap, at a lower
    clock.  A region whose sampled median SM clock is within 10% of the
    maximum is held to the burst figure, any other to the sustained one."""
    burst = float(peaks.get("bf16_tflops"))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    med = (clocks or {}).get("sm_mhz")
    mx = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz")
    if med is None or mx is None or med >= 0.9 * float(mx):
        return burst, "bf16_tflops"
    return sustained, "bf16_tflops_sustained"


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        info = [i for i in threadpool_info() if i.get("internal_api") in ("openblas", "mkl")]
        if info:
            return int(info[0]["num_threads"])
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample(cfg, seconds: float, min_chunks: int = 2):
    """Time the CPU oracle on the first chunks of the workload, chunk by chunk,
    until `seconds` of CPU work (or the whole document).  Returns (tokens/s,
    tokens, seconds)."""
    import numpy as np
    import oracle.ttt_oracle as orc
    C = cfg["chunk"]
    W = np.float64(cfg["w_down0"]).copy()
    done = 0
    t0 = time.perf_counter()
    while done < cfg["T"]:
        e = min(done + C, cfg["T"])
        o, W = orc.ttt_layer(cfg["x"][done:e], cfg["x0"][done:e], cfg["w_gate"], cfg["w_up"],
                             cfg["w_down0"], cfg["conv_w"], cfg["w_target"], cfg["eta"], C,
                             doc_starts=(0,) if done == 0 else (), w_init=W)
        done = e
        if done // C >= min_chunks and time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return done / dt, done, dt


def oracle_core_sample(cfg, seconds: float, min_chunks: int = 2):
    """Time the CPU oracle's apply+update recursion alone (ttt_core) on the
    first chunks of the workload, given their Z and V (computed by the oracle
    beforehand, outside the timed part).  Returns (tokens/s, tokens, seconds)."""
    import numpy as np
    import oracle.ttt_oracle as orc
    C, T = cfg["chunk"], cfg["T"]
    # size the sample from one timed chunk
    z1 = orc.swiglu_intermediate(cfg["x"][:C], cfg["w_gate"], cfg["w_up"])
    v1 = orc.chunk_target(cfg["x0"][:C], cfg["conv_w"], cfg["w_target"])
    t0 = time.perf_counter()
    orc.ttt_core(z1, v1, cfg["w_down0"], cfg["eta"], C, (0,))
    per_chunk = max(time.perf_counter() - t0, 1e-6)
    n = min(T, C * max(min_chunks, int(seconds / per_chunk)))
    z = orc.swiglu_intermediate(cfg["x"][:n], cfg["w_gate"], cfg["w_up"])
    v = np.zeros((n, cfg["d"]))
    for s0 in range(0, n, C):
        v[s0:s0 + C] = orc.chunk_target(cfg["x0"][s0:min(s0 + C, n)], cfg["conv_w"], cfg["w_target"])
    t0 = time.perf_counter()
    orc.ttt_core(z, v, cfg["w_down0"], cfg["eta"], C, (0,))
    dt = time.perf_counter() - t0
    return n / dt, n, dt


# ---------------------------------------------------------------- arms

def workload_x_seed(rank: int, world: int):
    """Seed of a rank's document X: the single-GPU workload uses the qwen
    recipe (X drawn first from seed 0); with several ranks every rank draws its
    own document from 1000 + rank after the shared weights (seed 0)."""
    return None if world == 1 else 1000 + rank


def make_workload(args, rank: int, world: int = 1):
    from ttt_inputs import CONFIGS, make_layer
    c = dict(CONFIGS["qwen"])
    return make_layer(c["d"], c["f"], args.tokens, args.chunk, c["k"], c["eta"], dtype="bf16",
                      seed=0, init="qwen", x_seed=workload_x_seed(rank, world))


def workload_config(args, extra=None):
    d = {"workload": f"qwen3-4b-shaped TTT-MLP layer, d=2560 f=9728 T={args.tokens} "
                     f"C={args.chunk} k=5 eta=1e-3, one document per step per GPU",
         "d": 2560, "f": 9728, "tokens_per_step_per_gpu": args.tokens, "chunk": args.chunk,
         "conv_k": 5, "eta": 1e-3,
         "l2": "inputs larger than L2 (X 168 MB, Z 637 MB per step at T=32768)",
         "parallelism": f"replicas{args.gpus} (independent documents per GPU)"}
    if extra:
        d.update(extra)
    return d


def run_reference(args):
    """CPU oracle arm: rank 0 only; each step is a bounded sample of the workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    cfg = make_workload(args, 0)
    for _ in range(args.warmup):
        oracle_sample(cfg, 0.0, min_chunks=REF_CHUNKS)
    tok, t = 0, 0.0
    for _ in range(args.steps):
        v, n, dt = oracle_sample(cfg, 0.0, min_chunks=REF_CHUNKS)
        tok += n
        t += dt
    value = tok / t
    cores = cpu_threads()
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"fp64 numpy/OpenBLAS oracle on the first {REF_CHUNKS} chunks "
                                       f"({tok // args.steps} tokens) of the document per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch
    rank, world = dist_init("nccl" if torch.cuda.is_available() else "gloo")
    _, _, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device for the kernel arm")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from chunk_wise_weight_ttt_b300 import TTTMLP
    from chunk_wise_weight_ttt_b300.build import build
    if rank == 0:
        build()
    barrier(world, dev)

    cfg = make_workload(args, rank, world)
    T, d, f = cfg["T"], cfg["d"], cfg["f"]

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev, torch.bfloat16)

    layer = TTTMLP(*[t(cfg[k]) for k in ("w_gate", "w_up", "w_down0", "conv_w", "w_target")],
                   chunk=cfg["chunk"], eta=cfg["eta"], max_tokens=T)
    x = t(cfg["x"])
    o = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(3, args.warmup)):
        layer.forward(x, doc_starts=(0,), out=o)
    layer.check()

    # ---- device-timed region: inputs resident in HBM, nothing but the steps
    # on the stream (no per-phase events between the kernels)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            layer.forward(x, doc_starts=(0,), out=o)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world, dev)
    layer.check()
    secs = e0.elapsed_time(e1) / 1e3
    value, tmax = aggregate_throughput(args.steps * T, secs, world, dev)

    # ---- per-phase events (the roofline's kernel time), on a separate pass
    prof_steps = max(3, min(args.steps, 50))
    layer.profile(True)
    with ClockSampler(local) as clk_prof:
        for _ in range(prof_steps):
            layer.forward(x, doc_starts=(0,), out=o)
        torch.cuda.synchronize(dev)
    prof = layer.profile_read()
    layer.profile(False)
    layer.check()

    # ---- end to end through the host-buffer C-ABI call (pinned host memory)
    e2e = None
    if not args.no_e2e:
        xh = x.cpu().pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        for _ in range(2):
            layer.forward_host(xh, out_host=oh, doc_starts=(0,))
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        h0 = torch.cuda.Event(enable_timing=True)
        h1 = torch.cuda.Event(enable_timing=True)
        k_e2e = max(3, min(args.steps, 50))
        h0.record(stream)
        for _ in range(k_e2e):
            layer.forward_host(xh, out_host=oh, doc_starts=(0,))
        h1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        ev, _ = aggregate_throughput(k_e2e * T, h0.elapsed_time(h1) / 1e3, world, dev)
        nbytes = T * d * 2
        e2e = {"value": ev, "unit": UNIT, "h2d_bytes_per_step": nbytes,
               "d2h_bytes_per_step": nbytes, "steps": k_e2e}
        layer.check()

    # ---- roofline of the dominant kernel (fused apply+update), live events
    peaks, peak_src = load_peaks()
    prof_clocks = clk_prof.summary()
    peak, peak_name = pick_peak(peaks, prof_clocks)
    burst = float(peaks.get("bf16_tflops"))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    ms = prof["ms"]
    group_s = ms["group"] / 1e3
    core_s = (ms["group"] + ms["gram"]) / 1e3
    n_launch = max(1, prof["group_launches"])
    flops = 4.0 * prof_steps * T * d * f          # algorithmic apply + update FLOPs
    achieved = flops / group_s / 1e12 if group_s > 0 else None
    core_achieved = flops / core_s / 1e12 if core_s > 0 else None
    group_len = max(1, group_tokens() // args.chunk) * args.chunk
    groups_per_step = -(-T // group_len)
    traffic = stored_traffic(groups_per_step * prof_steps / n_launch, args.chunk, d, f)
    frac = lambda a, p: (a / p) if a else None
    roofline = {"bound": "tensor", "kernel": "tc_gemm_kernel<kGroup> (apply+update)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": frac(achieved, peak),
                "peak_source": f"{peak_src} {peak_name}: median SM clock of the timed kernels "
                               f"{prof_clocks.get('sm_mhz')} MHz of {prof_clocks.get('sm_max_mhz')} "
                               f"(burst within 10% of the maximum clock, else sustained)",
                "frac_of_burst_peak": frac(achieved, burst),
                "frac_of_sustained_peak": frac(achieved, sustained),
                "traffic": traffic,
                "flops_per_launch": flops / n_launch,
                "ms_per_launch": 1e3 * group_s / n_launch,
                # the fused apply+update of this design: the group kernel plus
                # the Gram blocks that give the apply its intra-group correction
                "core_kernels": "tc_gemm_kernel<kSGram> + tc_gemm_kernel<kGroup>",
                "core_achieved": core_achieved,
                "core_frac": frac(core_achieved, peak),
                "core_frac_of_burst_peak": frac(core_achieved, burst),
                "core_tokens_per_s": (prof_steps * T / core_s) if core_s > 0 else None,
                "clocks": prof_clocks,
                "phase_ms_per_step": {k: v / prof_steps for k, v in ms.items()},
                "phase_steps": prof_steps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, ntok, dt = oracle_sample(cfg, args.cpu_seconds)
        vc, ntc, dtc = oracle_core_sample(cfg, args.cpu_seconds / 2)
        cpu = {"value": v, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
               "cpu_model": cpu_model(),
               "sample": f"fp64 numpy/OpenBLAS oracle, whole layer, on the first {ntok} tokens "
                         f"({ntok // cfg['chunk']} chunks) of the step's document, {dt:.1f} s",
               "core": {"value": vc, "unit": UNIT,
                        "sample": f"the oracle's apply+update recursion alone (ttt_core) on the "
                                  f"first {ntc} tokens, given their Z and V, {dtc:.1f} s"}}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": max(3, args.warmup),
                "ms_per_step": 1e3 * tmax / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": workload_config(args, {"group_tokens": group_tokens(),
                                                  "group_chunks": max(1, group_tokens() // args.chunk)}),
                "e2e": e2e, "gpu_launches": prof["launches"] // prof_steps * args.steps,
                "roofline": roofline,
                "cpu_baseline": cpu, "clocks": clk.summary(), "path": layer.path}
        print(json.dumps(line), flush=True)
    layer.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_extra(args):
    """The other configurations of the layer, timed on one GPU with inputs
    resident in HBM (drawn with torch's device generator: weights N(0, 0.02^2),
    X rows RMS-normalised; timing only, no oracle).  One JSON line per case."""
    import torch
    from chunk_wise_weight_ttt_b300 import TTTMLP, TTTStack
    from chunk_wise_weight_ttt_b300.build import build
    from ttt_inputs import CONFIGS, make_stack_device
    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)

    def weights(d, f, k, seed):
        g = torch.Generator(device=dev).manual_seed(seed)
        nrm = lambda *sh: (torch.randn(*sh, generator=g, device=dev) * 0.02).to(torch.bfloat16)
        return [nrm(f, d), nrm(f, d), nrm(d, f), nrm(k, d), nrm(d, d)]

    def tokens(T, d, seed):
        g = torch.Generator(device=dev).manual_seed(seed)
        x = torch.randn(T, d, generator=g, device=dev)
        return (x / torch.sqrt(x.pow(2).mean(1, keepdim=True) + 1e-6)).to(torch.bfloat16)

    def timed(fn, steps, warmup):
        for _ in range(max(3, warmup)):
            fn()
        torch.cuda.synchronize(dev)
        with ClockSampler(0) as clk:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                fn()
            e1.record()
            torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / 1e3 / steps, clk.summary()

    def emit(name, tok, sec, clocks, config):
        print(json.dumps({"metric": f"TTT-MLP tokens/s, {name}", "value": tok / sec,
                          "unit": UNIT, "ms_per_step": 1e3 * sec, "higher_is_better": True,
                          "dtype": "bf16", "data": "synthetic", "n_gpus": 1,
                          "config": config, "clocks": clocks}), flush=True)

    steps = max(3, min(args.steps, 20))
    if args.workload == "long":
        c = CONFIGS["long"]
        layer = TTTMLP(*weights(c["d"], c["f"], c["k"], 0), chunk=c["chunk"], eta=c["eta"],
                       max_tokens=c["T"])
        x = tokens(c["T"], c["d"], 1)
        o = torch.empty_like(x)
        sec, clk = timed(lambda: layer.forward(x, doc_starts=c["doc_starts"], out=o), steps,
                         args.warmup)
        layer.check()
        emit("131072-token call with a document every 32768 tokens", c["T"], sec, clk,
             {"workload": "long", "d": c["d"], "f": c["f"], "T": c["T"], "chunk": c["chunk"],
              "doc_starts": list(c["doc_starts"])})
    elif args.workload == "sweep":
        c = CONFIGS["sweep"]
        xs = [tokens(c["T"], c["d"], 1000 + b) for b in range(8)]
        outs = [torch.empty_like(x) for x in xs]
        w = weights(c["d"], c["f"], c["k"], 0)
        for C in (64, 128, 256, 512, 1024):
            layer = TTTMLP(*w, chunk=C, eta=c["eta"], n_docs=8, max_tokens=c["T"])
            for B in (1, 4, 8):
                def step():
                    for b in range(B):
                        layer.forward(xs[b], doc=b, doc_starts=(0,), out=outs[b])
                sec, clk = timed(step, steps, args.warmup)
                layer.check()
                emit(f"C={C}, batch {B} documents of {c['T']} tokens", B * c["T"], sec, clk,
                     {"workload": "sweep", "d": c["d"], "f": c["f"], "T_per_doc": c["T"],
                      "chunk": C, "batch": B})
            layer.close()
    else:
        c = CONFIGS["stack"]
        h0, layers = make_stack_device(c["n_layers"], c["d"], c["f"], c["T"], c["k"], seed=0)
        for every in (1, 6):
            stack = TTTStack(layers, chunk=c["chunk"], eta=c["eta"], max_tokens=c["T"],
                             ttt_every=every)
            sec, clk = timed(lambda: stack(h0), max(3, min(steps, 5)), 1)
            stack.check()
            n_ttt = sum(1 for li in range(c["n_layers"]) if (li + 1) % every == 0)
            emit(f"{c['n_layers']}-layer stack, TTT in every {every} block(s) "
                 f"(tokens through all layers)", c["T"], sec, clk,
                 {"workload": "stack", "n_layers": c["n_layers"], "ttt_every": every,
                  "ttt_layers": n_ttt, "d": c["d"], "f": c["f"], "T": c["T"], "chunk": c["chunk"],
                  "layer_tokens_per_s": c["n_layers"] * c["T"] / sec})
            stack.close()
            del stack
        # the single TTT layer on the same shape, for the per-layer comparison:
        # a step is as many calls as the stack has layers, so that both run
        # for as long and under the same power-cap clock
        w = layers[0]
        single = TTTMLP(w["w_gate"], w["w_up"], w["w_down0"], w["conv_w"], w["w_target"],
                        chunk=c["chunk"], eta=c["eta"], max_tokens=c["T"])
        x = h0.to(torch.bfloat16)
        o = torch.empty_like(x)

        def layer_calls():
            for _ in range(c["n_layers"]):
                single.forward(x, doc_starts=(0,), out=o)
        sec, clk = timed(layer_calls, max(3, min(steps, 5)), 1)
        single.check()
        emit(f"single TTT layer of the stack's shape, {c['n_layers']} calls per step "
             f"(layer-tokens)", c["n_layers"] * c["T"], sec, clk,
             {"workload": "stack-single-layer", "d": c["d"], "f": c["f"], "T": c["T"],
              "chunk": c["chunk"], "calls_per_step": c["n_layers"]})
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "layer":
        return run_extra(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
