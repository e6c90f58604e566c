#!/usr/bin/env python3
"""Benchmark of the GB300 4-bit quantized MoE layer forward (prefill and batch-1 decode).

A step is one pass of the layer-stack workload: 40 independent MoE layers (d=2048, 256 experts,
top-8, I=512, one shared expert, Q4 group-64 weights; seeds 0..39) each run on a 4096-token
prefill chunk, then 256 batch-1 decode steps through the 40 layers with fixed random inputs per
step. All layer weights (18.2 GB packed) stay resident in HBM and together exceed the 129 MB
L2 many times over, so no L2 flush is needed between steps.

Output: one JSON line (rank 0). `value` is MoE-layer prefill throughput in tok/s (tokens of
one layer per second, summed over ranks); `decode_us_per_layer` is the decode time per layer.
`--impl reference` times the CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "moe_layer_prefill_tok_per_s"
UNIT = "tok/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--layers", type=int, default=40)
    ap.add_argument("--prefill-tokens", type=int, default=4096)
    ap.add_argument("--decode-steps", type=int, default=256)
    ap.add_argument("--router-bias", choices=("none", "zipf"), default="none")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of replaying CUDA graphs")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-check", action="store_true",
                    help="accepted for older command lines; the sampled oracle check of this launch "
                         "configuration is tests/test_gpu_bench_config.py")
    ap.add_argument("--skip-diag", action="store_true", help="skip the diagnostics that run after the timed region (decode split, small batches, chunked prefill)")
    ap.add_argument("--skip-configs", action="store_true",
                    help="skip the per-workload sub-results after the timed region (single-layer cold "
                         "decode, 512-token prefill, skewed 2048-token prefill)")
    ap.add_argument("--rank-check", action="store_true",
                    help="only start the ranks, all-reduce one value and print the world size (rank 0)")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the nvidia-smi clock samples of the timed region in this file ({rank} is "
                         "replaced by the rank; default: a temporary file)")
    ap.add_argument("--oracle-child", default=None, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ------------------------------------------------------------------------------------------
# Peaks, algorithmic work per launch
# ------------------------------------------------------------------------------------------
def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


def expert_bytes(d: int, inter: int) -> dict:
    """Packed bytes of one expert: 4-bit codes plus one bf16 scale and bias per 64 weights."""
    per_w = 0.5 + 4.0 / 64
    return {"gate_up": int(2 * inter * d * per_w), "down": int(d * inter * per_w)}


def algorithmic_work(d: int, E: int, k: int, inter: int, T: int) -> dict:
    """Algorithmic FLOPs (real rows only) and bytes per launch of each kernel."""
    A = T * k
    eb = expert_bytes(d, inter)
    return {
        "prefill_router_gemm": {"flop": 2.0 * T * E * d},
        "prefill_gate_up_gemm": {"flop": 2.0 * (A + T) * 2 * inter * d},
        "prefill_down_gemm": {"flop": 2.0 * (A + T) * d * inter},
        # decode, per layer: router weights, the k+1 active experts' packed weights, x and y
        "decode_layer": {"bytes": E * d * 2 + (k + 1) * (eb["gate_up"] + eb["down"]) + 2 * d * 2},
    }


# ------------------------------------------------------------------------------------------
# Clock sampling during the timed region
# ------------------------------------------------------------------------------------------
_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
          "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
          "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_uuid: str | None):
        self.uuid, self.proc, self.path = gpu_uuid, None, None

    def start(self, path: str):
        self.path = path
        cmd = ["nvidia-smi", f"--query-gpu={_QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd[1:1] = ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(_REASONS, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------
# Ranks (one process per GPU; replicas of the whole workload, no data-path collective)
# ------------------------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_over_ranks(values: dict, op: str = "max") -> dict:
    """Max (timings) or sum (work) of scalar values over all ranks; identity without a group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return dict(values)
    keys = sorted(values)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(values[k]) for k in keys], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return {k: float(v) for k, v in zip(keys, t.tolist())}


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def src_sha(*rel_paths) -> str:
    h = hashlib.sha256()
    for rp in rel_paths:
        with open(os.path.join(ROOT, rp), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


_CSRC = "quantized_grouped_gemm_router_gb300/csrc/"
# the kernels' own device sources (the DRAM traffic of a capture holds while these are unchanged)
KERNEL_SOURCES = {
    "prefill_gate_up_gemm": (_CSRC + "gemm.cu", _CSRC + "ptx.cuh"),
    "prefill_down_gemm": (_CSRC + "gemm.cu", _CSRC + "ptx.cuh"),
    "prefill_router_gemm": (_CSRC + "gemm.cu", _CSRC + "ptx.cuh"),
    "decode_layer": (_CSRC + "decode.cu", _CSRC + "decode_common.cuh", _CSRC + "topk.cuh", _CSRC + "ptx.cuh"),
}


def device_info(device) -> dict:
    """The GPU the numbers were taken on (name, SM count, compute capability, memory)."""
    try:
        import torch
        p = torch.cuda.get_device_properties(device)
        return {"name": p.name, "sms": p.multi_processor_count, "cc": f"{p.major}.{p.minor}",
                "hbm_gib": round(p.total_memory / 2**30, 1)}
    except Exception as e:  # informational only: never fail the run for it
        return {"error": str(e)[:120]}


def measured_traffic(prefill_tokens: int, router_bias: str, path: str | None = None) -> dict:
    """DRAM bytes per launch from the committed ncu summary (profiles/dram_traffic.md), kept only
    for kernels whose sources still hash to the value recorded at capture time and whose captured
    workload is this run's: prefill rows name their tokens per layer and router bias
    (`T=4096 bias=none`), decode rows (`decode`) hold for any prefill setting."""
    out = {}
    try:
        lines = open(path or os.path.join(ROOT, "profiles", "dram_traffic.md")).read().splitlines()
    except OSError:
        return out
    here = f"T={prefill_tokens} bias={router_bias}"
    for ln in lines:
        m = re.match(r"\| `(\w+)` \| ([^|]+?) \| [^|]+ \| (\d+) \| (\w+) \|", ln)
        if not m or m.group(1) not in KERNEL_SOURCES or m.group(2) not in ("decode", here):
            continue
        if src_sha(*KERNEL_SOURCES[m.group(1)]) == m.group(4):
            out[m.group(1)] = int(m.group(3))
    return out


# ------------------------------------------------------------------------------------------
# CPU oracle: bounded samples of the same workload (baseline only, never the optimisation target)
# ------------------------------------------------------------------------------------------
def _oracle_child(spec: str) -> None:
    """Runs inside a child process (no CUDA): times the oracle on the sample in `spec` and
    prints one JSON object."""
    import numpy as np  # noqa: F401
    import oracle as O
    from synthetic import FULL, make_layer, make_tokens
    cfg = json.loads(spec)
    out = {"prefill_s": [], "decode_s": []}
    layers = {}
    for i in range(cfg["repeats"]):
        li = cfg["layer_ids"][i % len(cfg["layer_ids"])]
        if li not in layers:
            layers[li] = make_layer(FULL, seed=li, router_bias=cfg["router_bias"])
        L = layers[li]
        x = make_tokens(cfg["tokens"], FULL.d, seed=li, stream=1000 + i)
        t0 = time.perf_counter()
        O.moe_forward(x, L, tile_rows=256)
        out["prefill_s"].append(time.perf_counter() - t0)
        for j in range(cfg["decode_tokens"]):
            x1 = make_tokens(1, FULL.d, seed=li, stream=2000 + 16 * i + j)
            t0 = time.perf_counter()
            O.moe_forward(x1, L, tile_rows=256)
            out["decode_s"].append(time.perf_counter() - t0)
    print(json.dumps(out))


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def host_info() -> dict:
    """nproc, CPU model and machine of the host the oracle runs on."""
    import platform
    model = ""
    try:
        for ln in open("/proc/cpuinfo"):
            key = ln.split(":")[0].strip().lower()
            if key in ("model name", "cpu model", "hardware") and ":" in ln:
                model = ln.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for ln in out.splitlines():
                if ln.lower().startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or "unknown", "machine": platform.machine()}


def run_oracle_sample(tokens: int, decode_tokens: int, repeats: int, layer_ids, router_bias, threads=None) -> dict:
    """Times the oracle in a fresh CPU-only process whose BLAS/OpenMP thread count is fixed (all
    the cores this process may use unless `threads` is given), so `cores` is the thread count
    actually used."""
    cores = threads or host_cores()
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[var] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    spec = json.dumps({"tokens": tokens, "decode_tokens": decode_tokens, "repeats": repeats,
                       "layer_ids": list(layer_ids), "router_bias": router_bias})
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", spec], env=env,
                         capture_output=True, text=True, check=True)
    data = json.loads(res.stdout.strip().splitlines()[-1])
    data["cores"] = cores
    return data


def cpu_baseline(args) -> dict:
    """The oracle on all the host's cores (the reported value) and on one thread (a smaller
    sample), with the host's core count, CPU model and machine."""
    rb = None if args.router_bias == "none" else args.router_bias
    tokens = 128
    d = run_oracle_sample(tokens, decode_tokens=4, repeats=1, layer_ids=[0], router_bias=rb)
    t_pre = statistics.mean(d["prefill_s"])
    t_dec = statistics.mean(d["decode_s"])
    t1 = 32
    d1 = run_oracle_sample(t1, decode_tokens=2, repeats=1, layer_ids=[0], router_bias=rb, threads=1)
    t1_pre = statistics.mean(d1["prefill_s"])
    t1_dec = statistics.mean(d1["decode_s"])
    return {"value": tokens / t_pre, "unit": UNIT, "cores": d["cores"], "kind": "oracle",
            "decode_us_per_layer": t_dec * 1e6,
            "sample": f"numpy fp64 oracle on layer 0 of the stack: one {tokens}-token prefill chunk "
                      f"({t_pre:.1f} s) and 4 single-token decodes ({t_dec:.2f} s each)",
            "single_thread": {"value": t1 / t1_pre, "unit": UNIT, "decode_us_per_layer": t1_dec * 1e6,
                              "sample": f"one {t1}-token prefill chunk ({t1_pre:.1f} s) and 2 single-token "
                                        f"decodes ({t1_dec:.2f} s each), 1 thread"},
            "host": host_info()}


def run_reference(args, config: dict) -> None:
    """Reference arm: the CPU oracle as it stands, same metric, unit and config, each step a
    bounded sample (one 16-token prefill chunk and one decode token of one layer)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    tokens = 16
    n = args.warmup + args.steps
    d = run_oracle_sample(tokens, decode_tokens=1, repeats=n, layer_ids=[0, 1, 2, 3],
                          router_bias=None if args.router_bias == "none" else args.router_bias)
    pre = d["prefill_s"][args.warmup:]
    dec = d["decode_s"][args.warmup:]
    value = tokens / statistics.mean(pre)
    step_ms = 1e3 * (statistics.mean(pre) + statistics.mean(dec))
    sample = (f"numpy fp64 oracle, each step one {tokens}-token prefill chunk and one decode token of "
              f"one layer (layers 0..3 in turn)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
            "decode_us_per_layer": 1e6 * statistics.mean(dec),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": d["cores"], "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# The GPU workload
# ------------------------------------------------------------------------------------------
class Workload:
    """Device-resident layers, per-layer prefill inputs and per-step decode inputs (pinned host
    copies kept for the end-to-end leg)."""

    def __init__(self, args, device, seed_offset: int = 0):
        import numpy as np
        import torch
        import quantized_grouped_gemm_router_gb300 as m
        from synthetic import FULL, make_layer, make_tokens
        self.m, self.shape, self.args = m, FULL, args
        L, T, S, d = args.layers, args.prefill_tokens, args.decode_steps, FULL.d
        rb = None if args.router_bias == "none" else args.router_bias
        self.layers = [m.upload_layer(make_layer(FULL, seed=seed_offset + l, router_bias=rb), device)
                       for l in range(L)]
        self.dims = self.layers[0].dims
        xp = np.stack([make_tokens(T, d, seed=seed_offset + l, stream=1) for l in range(L)]) if T else None
        xd = make_tokens(S * L, d, seed=seed_offset, stream=2).reshape(S, L, d) if S else None
        pin = lambda a: torch.from_numpy(a.view(np.int16)).pin_memory()  # noqa: E731
        self.xp_host = pin(xp) if T else None
        self.xd_host = pin(xd) if S else None
        self.xp = self.xp_host.to(device) if T else None
        self.xd = self.xd_host.to(device) if S else None
        self.yp = torch.empty_like(self.xp) if T else None
        self.yd = torch.empty_like(self.xd) if S else None
        self.yp_host = torch.empty_like(self.xp_host).pin_memory() if T else None
        self.yd_host = torch.empty_like(self.xd_host).pin_memory() if S else None
        self.ws_p = m.workspace(self.dims, max(T, 1), device)
        self.ws_d = m.workspace(self.dims, 1, device)

    def prefill_all(self, events=None):
        for l, layer in enumerate(self.layers):
            self.m.prefill(layer, self.xp[l], self.ws_p, y=self.yp[l], events=None if events is None else events.get(l))

    def decode_all(self, events=None):
        """events: {step: (start, end)} brackets the whole 40-layer decode step (one event before
        its first call, one after its last), so the event nodes do not sit between kernels."""
        L = len(self.layers)
        for s in range(self.args.decode_steps):
            pair = None if events is None else events.get(s)
            for l, layer in enumerate(self.layers):
                ev = None
                if pair is not None and (l == 0 or l == L - 1):
                    ev = [pair[0] if l == 0 else None, None, None, pair[1] if l == L - 1 else None]
                self.m.decode(layer, self.xd[s, l], self.ws_d, y=self.yd[s, l], events=ev)

    def launches_per_step(self) -> int:
        a = self.args
        # prefill: router GEMM, top-k, histogram, scatter, row placement, gate/up, down, cast;
        # decode: router GEMV, expert kernel (top-k, gate/up, SwiGLU), down kernel (with the combine)
        return (8 * a.layers if a.prefill_tokens else 0) + 3 * a.layers * a.decode_steps


def capture(W: Workload, ev_pre=None, ev_dec=None, graphs: bool = True):
    """Returns (run_prefill_step, run_decode_step): replays of CUDA graphs captured from the
    library calls (the timed launch configuration), or the eager calls."""
    import torch
    if not graphs:
        return (lambda: W.prefill_all(ev_pre)), (lambda: W.decode_all(ev_dec))
    g_pre, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    if W.args.prefill_tokens:
        with torch.cuda.graph(g_pre):
            W.prefill_all(ev_pre)
    if W.args.decode_steps:
        with torch.cuda.graph(g_dec):
            W.decode_all(ev_dec)
    W.graphs = (g_pre, g_dec)
    return g_pre.replay, g_dec.replay


def _new_events(n):
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()  # materialise the CUDA event so its handle can be handed to the library
    return evs


def run_ours(args, config: dict) -> None:
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    cpu = None
    if rank == 0 and not args.skip_cpu:
        cpu = cpu_baseline(args)           # CPU oracle sample, before any GPU work
    from quantized_grouped_gemm_router_gb300 import build as B
    B.build()
    W = Workload(args, device, seed_offset=1000 * rank)
    L, T, S = args.layers, args.prefill_tokens, args.decode_steps

    # events inside the timed region: per kernel on every 8th prefill layer; around every 16th
    # 40-layer decode step (kernels overlap through PDL, which an event between two kernels stops,
    # so most layers run without them and the decode unit is the whole layer)
    ev_pre = {l: _new_events(6) for l in range(0, L, 8)} if T else {}
    ev_dec = {s: tuple(_new_events(2)) for s in range(0, S, 16)}
    for _ in range(2):                     # eager warm-up (also initialises the library)
        if T:
            W.prefill_all()
        if S:
            W.decode_all()
    torch.cuda.synchronize()
    if W.m.read_device_status(W.ws_p) or W.m.read_device_status(W.ws_d):
        raise RuntimeError("device status set during warm-up")

    run_pre, run_dec = capture(W, ev_pre, ev_dec, graphs=not args.no_graph)
    for _ in range(args.warmup):
        if T:
            run_pre()
        if S:
            run_dec()
    torch.cuda.synchronize()

    names_pre = ["prefill_router_gemm", "prefill_route", "prefill_gate_up_gemm", "prefill_down_gemm", "prefill_cast"]
    names_dec = ["decode_layer"]
    ksum = {n: 0.0 for n in names_pre + names_dec}
    kcnt = {n: 0 for n in names_pre + names_dec}
    e0, e1, e2 = _new_events(3)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks_csv = args.clocks_csv.replace("{rank}", str(rank)) if args.clocks_csv else \
        os.path.join(tempfile.gettempdir(), f"moe_bench_clocks_{os.getpid()}_r{rank}.csv")
    if os.path.dirname(clocks_csv):
        os.makedirs(os.path.dirname(clocks_csv), exist_ok=True)
    barrier()
    torch.cuda.synchronize()
    clocks.start(clocks_csv)
    wall0 = time.perf_counter()
    pre_ms = dec_ms = 0.0
    for _ in range(args.steps):
        e0.record()
        if T:
            run_pre()
        e1.record()
        if S:
            run_dec()
        e2.record()
        e2.synchronize()                   # read this step's sampled kernel events
        pre_ms += e0.elapsed_time(e1)
        dec_ms += e1.elapsed_time(e2)
        for evs in ev_pre.values():
            for i, n in enumerate(names_pre):
                ksum[n] += evs[i].elapsed_time(evs[i + 1])
                kcnt[n] += 1
        for e_a, e_b in ev_dec.values():
            ksum["decode_layer"] += e_a.elapsed_time(e_b) / L
            kcnt["decode_layer"] += 1
    torch.cuda.synchronize()
    barrier()
    wall_s = time.perf_counter() - wall0
    clk = clocks.stop()
    st = W.m.read_device_status(W.ws_p) | W.m.read_device_status(W.ws_d)
    if st:
        raise RuntimeError(f"device status {st} set during the timed region")

    # end-to-end: host inputs in pinned memory, copies inside the timed region, eager calls
    e2e = None
    if not args.skip_e2e:
        e2e_pre, e2e_dec = end_to_end(W, args, e0, e1, e2)
        red = reduce_over_ranks({"pre": e2e_pre, "dec": e2e_dec}, "max")
        h2d = (W.xp_host.numel() * 2 if T else 0) + (W.xd_host.numel() * 2 if S else 0)
        e2e = {"value": world * L * T * args.steps / (red["pre"] / 1e3) if T else None, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": h2d,
               "decode_us_per_layer": 1e3 * red["dec"] / (args.steps * max(1, S * L)) if S else None,
               "prefill_ms_per_step": getattr(W, "e2e_prefill_ms_per_step", None),
               "how": "prefill: per layer, pinned host x copied in on a copy stream, an eager moe_prefill call "
                      "through the Python binding on the compute stream once its input has landed, y copied "
                      "back on a second copy stream, so layer l's copies overlap the neighbouring layers' "
                      "compute; decode: all inputs copied in, 256x40 eager moe_decode calls, outputs copied "
                      f"back, per step; {args.warmup} untimed steps first"}

    diag = decode_diagnostics(W) if S and not args.skip_diag else None
    probe = None
    if T and not args.skip_diag:  # the layer-stack workload's GEMMs against their read-only probes
        nl = min(L, 8)
        probe = gemm_read_probe(W.m, W.layers[:nl], [W.xp[l] for l in range(nl)], [W.yp[l] for l in range(nl)],
                                W.ws_p, {"gate_up": 1e3 * ksum["prefill_gate_up_gemm"] / kcnt["prefill_gate_up_gemm"],
                                         "down": 1e3 * ksum["prefill_down_gemm"] / kcnt["prefill_down_gemm"]},
                                W.shape.n_experts, expert_bytes(W.shape.d, W.shape.inter),
                                load_peaks()["hbm_gbs"], 4)
        if W.m.read_device_status(W.ws_p):
            raise RuntimeError("device status set during the read-only probes")
    configs = None if args.skip_configs else config_results(W, load_peaks())
    small = chunked = None
    if T and not args.skip_diag:
        small = small_batch_diagnostics(W, None if diag is None else diag["decode_us_per_layer"])
        chunked = chunked_prefill_diagnostics(W)

    red = reduce_over_ranks({"pre": pre_ms, "dec": dec_ms, "wall": wall_s}, "max")
    kavg = {n: ksum[n] / kcnt[n] for n in ksum if kcnt[n]}
    if rank != 0:
        return
    peaks = load_peaks()
    work = algorithmic_work(W.shape.d, W.shape.n_experts, W.shape.top_k, W.shape.inter, T)
    per_step_launches = {n: L for n in names_pre}  # the sampled layers' averages stand for all
    per_step_launches.update({n: L * S for n in names_dec})
    rooflines = []
    traffic = measured_traffic(T, args.router_bias)
    for n, ms in kavg.items():
        w = work.get(n)
        if not w:
            continue
        share_ms = ms * per_step_launches[n]
        if "flop" in w:
            ach = w["flop"] / (ms * 1e-3) / 1e12
            peak = peaks["bf16_tflops_sustained"]
            r = {"kernel": n, "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                 "frac": ach / peak, "per_launch": f"{w['flop'] / 1e9:.2f} GFLOP (real rows only)"}
        else:
            ach = w["bytes"] / (ms * 1e-3) / 1e9
            peak = peaks["hbm_gbs"]
            r = {"kernel": n, "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                 "per_launch": f"{w['bytes'] / 1e6:.3f} MB (router + k+1 active experts + x, y) per layer; "
                               "router, expert and down (+ combine) kernels overlap through PDL"}
        r.update({"avg_launch_us": ms * 1e3, "ms_per_step": share_ms,
                  "peak_source": f"{peaks['source']} ({'sustained bf16 = fp16 dense' if 'flop' in w else 'HBM copy'})",
                  "traffic": traffic.get(n)})
        rooflines.append(r)
    rooflines.sort(key=lambda r: -r["ms_per_step"])
    value = world * L * T * args.steps / (red["pre"] / 1e3) if T else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": (red["pre"] + red["dec"]) / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic", "config": config,
        "decode_us_per_layer": 1e3 * red["dec"] / (args.steps * S * L) if S else None,
        "prefill_us_per_layer": 1e3 * red["pre"] / (args.steps * L) if T else None,
        "roofline": dict(rooflines[0]) if rooflines else None, "rooflines": rooflines,
        "cpu_baseline": cpu, "e2e": e2e, "configs": configs, "decode_diagnostics": diag,
        "small_batch_diagnostics": small, "chunked_prefill_diagnostics": chunked, "prefill_read_probe": probe,
        "gpu_launches": W.launches_per_step() * args.steps,
        "clocks": clk, "wall_s_timed": red["wall"], "graphs": not args.no_graph,
        "device": device_info(device), "sources": {k: src_sha(*v) for k, v in KERNEL_SOURCES.items()},
    }
    print(json.dumps(line), flush=True)


def decode_diagnostics(W, steps: int = 8) -> dict:
    """The page's two decode ablations (section "What didn't work"), after the timed region:
    the decode chain with the GEMV arithmetic deleted, and a read-only probe of the expert kernel's
    weight copies alone, each captured in a CUDA graph over the stack's layers like the timed
    decode. The fraction is the decode's weight-read rate over the probe's (the page reports 90.3%
    for its GEMV); the arithmetic share is the time the arithmetic adds to the chain."""
    L, S = len(W.layers), W.args.decode_steps
    m = W.m

    def one(mode):
        def body():
            for s in range(steps):
                for l, layer in enumerate(W.layers):
                    if mode == 0:
                        m.decode(layer, W.xd[s % S, l], W.ws_d, y=W.yd[s % S, l])
                    else:
                        m.decode_diag(layer, W.xd[s % S, l], W.ws_d, mode, y=W.yd[s % S, l])
        return _graph_time_ms(body) * 1e3 / (steps * L)

    t_dec, t_nomath, t_read = one(0), one(m.DECODE_DIAG_NO_MATH), one(m.DECODE_DIAG_READ_ONLY)
    if m.read_device_status(W.ws_d):
        raise RuntimeError("device status set during the decode diagnostics")
    sh = W.shape
    expert_bytes = (sh.top_k + 1) * (3 * sh.inter * sh.d // 2 + 3 * (sh.inter * sh.d // 64) * 4)
    return {"decode_us_per_layer": t_dec, "no_math_us_per_layer": t_nomath, "read_only_us_per_layer": t_read,
            "expert_bytes_per_layer": expert_bytes, "read_only_GBps": expert_bytes / (t_read * 1e3),
            "decode_weight_GBps": expert_bytes / (t_dec * 1e3), "frac_of_read_only_rate": t_read / t_dec,
            "arithmetic_share": 1.0 - t_nomath / t_dec,
            "how": f"{L} layers x {steps} steps per CUDA graph, best of 3 replays; read-only probe: the "
                   "expert kernel's weight copies for experts 0..k-1 and the shared expert, launched alone"}


def _graph_time_ms(body, reps: int = 3, eager: bool = True) -> float:
    """Best of `reps` replays of a CUDA graph captured from body() (after one eager run, unless
    `eager` is false, and one untimed replay), in milliseconds. A body that hands events to the
    library records them as graph nodes, so it is only captured, never run eagerly."""
    import torch
    if eager:
        body()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    g.replay()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(reps):
        a.record()
        g.replay()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return min(ts)


def small_batch_diagnostics(W, decode_us: float | None, sizes=(1, 2, 3, 4, 5, 8)) -> dict:
    """T = 1..8 token rows at once (the shape of verifying a few draft tokens, which the page's
    section "What didn't work" found awkward): per-layer time over the stack in a CUDA graph of the
    small-batch decode (moe_decode_batch, which reads each distinct selected expert once) and of the
    prefill path, against T batch-1 decodes; and the distinct experts the T rows select, i.e. the
    expert bytes one such step must read."""
    import torch
    m, L, sh = W.m, len(W.layers), W.shape
    eb = expert_bytes(sh.d, sh.inter)
    one_expert = eb["gate_up"] + eb["down"]
    rows = []
    for T in sizes:
        if T > W.xp.shape[1]:
            break
        ys = torch.empty((L, T, sh.d), dtype=torch.int16, device=W.xp.device)

        def body():
            for l, layer in enumerate(W.layers):
                m.prefill(layer, W.xp[l, :T], W.ws_p, y=ys[l])
        us = 1e3 * _graph_time_ms(body) / L

        def body_batch():
            for l, layer in enumerate(W.layers):
                m.decode_batch(layer, W.xp[l, :T], W.ws_p, y=ys[l])
        us_b = 1e3 * _graph_time_ms(body_batch) / L
        distinct = 0
        for l, layer in enumerate(W.layers):
            out = m.route(layer, W.xp[l, :T], T, W.ws_p, out=m.route_out_tensors(W.dims, T, W.xp.device,
                                                                                  want=("counts",)))
            distinct += int((out["counts"] > 0).sum())
        distinct /= L
        nbytes = (distinct + 1) * one_expert + sh.n_experts * sh.d * 2
        rows.append({"T": T, "decode_batch_us_per_layer": us_b, "prefill_us_per_layer": us,
                     "T_decodes_us_per_layer": None if decode_us is None else T * decode_us,
                     "distinct_experts": distinct, "weight_MB": nbytes / 1e6,
                     "decode_batch_weight_GBps": nbytes / (us_b * 1e3), "prefill_weight_GBps": nbytes / (us * 1e3)})
    if m.read_device_status(W.ws_p):
        raise RuntimeError("device status set during the small-batch diagnostics")
    return {"rows": rows, "how": f"moe_decode_batch and moe_prefill on the first T rows of each layer's prefill "
                                 f"input, {L} layers per CUDA graph, best of 3 replays; T_decodes = T x the batch-1 "
                                 "decode time per layer"}


def chunked_prefill_diagnostics(W, prompt_chunks: int = 4, chunks=(512, 1024, 2048, 4096)) -> dict:
    """Bounded-chunk prefill (moe_prefill_chunked) of one long prompt per layer, made of
    `prompt_chunks` layers' prefill inputs back to back, with a workspace sized for the largest
    chunk only: per-layer time and token rate for several chunk sizes."""
    import torch
    m, L, sh = W.m, len(W.layers), W.shape
    T0 = W.xp.shape[1]
    n = min(prompt_chunks, L) * T0
    x = W.xp.view(-1, sh.d)[:n]
    y = torch.empty_like(x)
    chunks = [c for c in chunks if c <= T0]
    rows = []
    for c in chunks:
        def body():
            for layer in W.layers:
                m.prefill_chunked(layer, x, W.ws_p, c, y=y)
        us = 1e3 * _graph_time_ms(body) / L
        rows.append({"chunk_tokens": c, "us_per_layer": us, "tok_per_s_per_layer": n / (us * 1e-6),
                     "workspace_MB": m.workspace_bytes(W.dims, c) / 1e6})
    if m.read_device_status(W.ws_p):
        raise RuntimeError("device status set during the chunked prefill diagnostics")
    return {"prompt_tokens": n, "single_call_workspace_MB": m.workspace_bytes(W.dims, n) / 1e6, "rows": rows,
            "how": f"{L} layers per CUDA graph, each prefilling the same {n}-token prompt in chunks, best of 3 replays"}


def end_to_end(W, args, e0, e1, e2):
    """The same workload through the public binding with host buffers: (prefill ms, decode ms)
    summed over args.steps steps, after args.warmup untimed ones. Prefill overlaps each layer's host copies with the neighbouring
    layers' compute (copy-in stream, compute stream, copy-out stream); decode copies all inputs in,
    runs the eager calls and copies all outputs back."""
    import gc
    import torch
    L, T, S = args.layers, args.prefill_tokens, args.decode_steps
    compute = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    # as timeit does: no garbage-collection pause of the enqueuing thread inside a timed step (the
    # 10,240 eager decode calls of a step leave garbage behind that a collection would otherwise
    # sweep while the next step's prefill calls are being enqueued, leaving the GPU idle)
    gc.collect()
    gc.disable()
    try:
        pre, dec = _end_to_end_steps(W, args, e0, e1, e2, compute, s_in, s_out, L, T, S)
    finally:
        gc.enable()
    return pre, dec


def _end_to_end_steps(W, args, e0, e1, e2, compute, s_in, s_out, L, T, S):
    import torch
    ev_in = [torch.cuda.Event() for _ in range(L)]
    ev_done = [torch.cuda.Event() for _ in range(L)]
    pre = dec = 0.0
    per_step = []
    for step in range(args.warmup + args.steps):  # the first `warmup` steps are not counted
        e0.record(compute)
        if T:
            s_in.wait_stream(compute)      # the copies belong to the timed region
            s_out.wait_stream(compute)
            for l, layer in enumerate(W.layers):
                with torch.cuda.stream(s_in):
                    W.xp[l].copy_(W.xp_host[l], non_blocking=True)
                    ev_in[l].record(s_in)
                compute.wait_event(ev_in[l])
                W.m.prefill(layer, W.xp[l], W.ws_p, y=W.yp[l])
                ev_done[l].record(compute)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done[l])
                    W.yp_host[l].copy_(W.yp[l], non_blocking=True)
            compute.wait_stream(s_out)
        e1.record(compute)
        if S:
            W.xd.copy_(W.xd_host, non_blocking=True)
            W.decode_all()
            W.yd_host.copy_(W.yd, non_blocking=True)
        e2.record(compute)
        compute.synchronize()
        if step < args.warmup:
            continue
        pre += e0.elapsed_time(e1)
        dec += e1.elapsed_time(e2)
        per_step.append(round(e0.elapsed_time(e1), 2))
    W.e2e_prefill_ms_per_step = per_step
    return pre, dec


def _l2_bytes(device) -> int:
    import torch
    try:
        return int(torch.cuda.get_device_properties(device).L2_cache_size)
    except Exception:
        return 128 << 20


def config_results(W, peaks: dict, reps: int = 8) -> dict:
    """Per-workload sub-results on this GPU, after the timed region, each with its roofline:
      decode      single-layer batch-1 decode with a cold L2 (a buffer of twice the L2 size is
                  written before every call, the layer and x change every call): HBM fraction of
                  the router + k+1 active experts' bytes;
      prefill512  512-token prefill, near-uniform routing (all experts hit), layers rotated so no
                  weights stay in L2: HBM fraction of the bytes one layer must read, and the tensor
                  fraction of the expert GEMMs;
      skew2048    2048-token prefill with the Zipf router bias (a few experts with hundreds of rows,
                  most with few or none), eight layers rotated: tensor fraction of the grouped
                  gate/up + down GEMMs (the target the pages' design is held to) and of the layer.
    Layer times come from a CUDA graph of the plain calls (the timed launch configuration, best of
    3 replays); kernel times from events recorded by the library at its kernel boundaries in a
    second graph, where each event node also stops the PDL overlap of the kernels around it (so
    the kernel times and their sum, `layer_with_events`, are upper bounds). Peaks: the burst
    figures (kernels timed alone)."""
    import numpy as np
    import torch
    from synthetic import make_tokens, zipf_router_bias
    m, sh, dev = W.m, W.shape, W.xp.device if W.xp is not None else W.xd.device
    d, E, k, I = sh.d, sh.n_experts, sh.top_k, sh.inter
    eb = expert_bytes(d, I)
    one_expert = eb["gate_up"] + eb["down"]
    hbm, tf = peaks["hbm_gbs"], peaks["bf16_tflops"]
    out = {}

    # ---- single-layer decode, cold L2
    nl = min(len(W.layers), 8)
    flush = torch.empty(2 * _l2_bytes(dev), dtype=torch.uint8, device=dev)
    x1 = torch.from_numpy(make_tokens(reps, d, seed=77, stream=5).view(np.int16)).to(dev)
    y1 = torch.empty_like(x1)
    ws1 = m.workspace(W.dims, 1, dev)
    ev = [_new_events(2) for _ in range(reps)]

    def dec_body():
        for r in range(reps):
            flush.fill_(r & 0x7F)
            m.decode(W.layers[r % nl], x1[r], ws1, y=y1[r], events=[ev[r][0], None, None, ev[r][1]])
    _graph_time_ms(dec_body, reps=1, eager=False)
    us = statistics.median(1e3 * a.elapsed_time(b) for a, b in ev)
    nbytes = algorithmic_work(d, E, k, I, 1)["decode_layer"]["bytes"]
    out["decode"] = {"workload": "single MoE layer, batch-1 decode (T=1), cold L2", "us_per_layer": us,
                     "roofline": {"bound": "hbm", "achieved": nbytes / (us * 1e3), "peak": hbm, "unit": "GB/s",
                                  "frac": nbytes / (us * 1e3) / hbm, "per_launch_bytes": nbytes}}

    def prefill_config(T, layers, seed_stream, arms):
        xs = [torch.from_numpy(make_tokens(T, d, seed=i, stream=seed_stream).view(np.int16)).to(dev)
              for i in range(len(layers))]
        ys = [torch.empty_like(x) for x in xs]
        ws = m.workspace(W.dims, T, dev)
        evs = [[_new_events(6) for _ in layers] for _ in range(reps)]

        def body():
            for r in range(reps):
                for i, layer in enumerate(layers):
                    m.prefill(layer, xs[i], ws, y=ys[i], events=evs[r][i])
        _graph_time_ms(body, reps=1, eager=False)

        def plain():
            for _ in range(reps):
                for i, layer in enumerate(layers):
                    m.prefill(layer, xs[i], ws, y=ys[i])
        # the layer time without events: an event node between two kernels stops the PDL overlap
        layer_us = 1e3 * _graph_time_ms(plain) / (reps * len(layers))
        abl = {}
        for arm in arms:
            abl[arm] = prefill_ablation_arm(m, arm, layers, xs, ys, ws, reps)
        names = ["router", "route", "gate_up", "down", "cast"]
        per = {n: statistics.mean(1e3 * e[j].elapsed_time(e[j + 1]) for row in evs for e in row)
               for j, n in enumerate(names)}
        per["layer_with_events"] = statistics.mean(1e3 * e[0].elapsed_time(e[5]) for row in evs for e in row)
        hit = []
        for i, layer in enumerate(layers):
            o = m.route(layer, xs[i], T, ws, out=m.route_out_tensors(W.dims, T, dev, want=("counts",)))
            hit.append(int((o["counts"] > 0).sum()))
        probe = gemm_read_probe(m, layers, xs, ys, ws, per, statistics.mean(hit), eb, hbm, reps)
        if m.read_device_status(ws):
            raise RuntimeError("device status set during the per-workload sub-results")
        return layer_us, per, statistics.mean(hit), abl, probe

    def gemm_flop(T):
        return 2.0 * (T * k + T) * 3 * I * d

    # ---- 512-token prefill, near-uniform routing
    lay = W.layers[:min(len(W.layers), 4)]
    T = 512
    layer_us, per, hit, abl, probe = prefill_config(T, lay, 3, ("host_routing", "dense", "wide_cfg"))
    nbytes = (hit + 1) * one_expert + E * d * 2 + 2 * T * d * 2
    gemm_us = per["gate_up"] + per["down"]
    out["prefill512"] = {
        "workload": "512-token prefill, one layer, near-uniform routing", "us_per_layer": layer_us,
        "tok_per_s": T / (layer_us * 1e-6), "kernels_us": per, "experts_hit": hit,
        "roofline": {"bound": "hbm", "achieved": nbytes / (layer_us * 1e3), "peak": hbm, "unit": "GB/s",
                     "frac": nbytes / (layer_us * 1e3) / hbm, "per_launch_bytes": nbytes},
        "gemm_tensor_frac": gemm_flop(T) / (gemm_us * 1e-6) / 1e12 / tf, "ablations": abl, "read_probe": probe}

    # ---- 2048-token prefill, Zipf router bias
    rb = torch.from_numpy(zipf_router_bias(E)).to(dev)
    lay = [m.Layer(W.dims, L.router_w, rb, L.packed) for L in W.layers[:min(len(W.layers), 8)]]
    T = 2048
    layer_us, per, hit, abl, probe = prefill_config(T, lay, 4, ("host_routing", "tile32", "narrow_cfg"))
    gemm_us = per["gate_up"] + per["down"]
    ach = gemm_flop(T) / (gemm_us * 1e-6) / 1e12
    out["skew2048"] = {
        "workload": "2048-token prefill, one layer, Zipf(1.1) router bias", "us_per_layer": layer_us,
        "tok_per_s": T / (layer_us * 1e-6), "kernels_us": per, "experts_hit": hit,
        "roofline": {"bound": "tensor", "kernel": "grouped gate/up + down GEMMs", "achieved": ach, "peak": tf,
                     "unit": "TFLOP/s", "frac": ach / tf, "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                     "per_launch_flop": gemm_flop(T)},
        "layer_tensor_frac": (gemm_flop(T) + 2.0 * T * E * d) / (layer_us * 1e-6) / 1e12 / tf, "ablations": abl,
        "read_probe": probe}
    out["how"] = (f"CUDA graphs of {reps} repetitions; prefill layer times from the plain calls (best of 3 "
                  f"replays), kernel times from events recorded by moe_prefill_timed at the kernel boundaries "
                  f"in a second graph (an event node stops the PDL overlap: upper bounds); decode: events "
                  f"around each moe_decode_timed call; peaks: {peaks['source']} burst (HBM copy, bf16 dense = "
                  f"fp16 dense)")
    return out


def gemm_read_probe(m, layers, xs, ys, ws, per: dict, hit: float, eb: dict, hbm: float, reps: int) -> dict:
    """The grouped GEMMs against their read-only probes (moe_prefill_diag: the same grid, work list,
    copies and ring depths, no arithmetic), timed like the GEMMs (events at the kernel boundaries
    in a CUDA graph of `reps` passes over the layers). per: the GEMMs' own times (us) on the same
    inputs; hit: experts with at least one row. frac_of_read_ceiling = probe time / GEMM time,
    i.e. the GEMM's read rate as a fraction of the fastest rate its own access pattern sustains;
    probe_weight_gbs = packed weights of the hit experts and the shared expert / probe time."""
    import torch
    evp = [[_new_events(6) for _ in layers] for _ in range(reps)]

    def body():
        for r in range(reps):
            for i, layer in enumerate(layers):
                m.prefill_diag(layer, xs[i], ws, m.PREFILL_DIAG_READ_ONLY, y=ys[i], events=evp[r][i])
    _graph_time_ms(body, reps=1, eager=False)
    torch.cuda.synchronize()
    res = {}
    for j, n in ((2, "gate_up"), (3, "down")):
        us = statistics.mean(1e3 * e[j].elapsed_time(e[j + 1]) for row in evp for e in row)
        wb = (hit + 1) * eb[n]
        res[n] = {"probe_us": us, "gemm_us": per[n], "frac_of_read_ceiling": us / per[n],
                  "probe_weight_gbs": wb / (us * 1e3), "probe_weight_frac_of_hbm": wb / (us * 1e3) / hbm}
    return res


def prefill_ablation_arm(m, arm: str, layers, xs, ys, ws, reps: int) -> dict:
    """One ablation arm of the page's prefill design against the product path, on the same layers
    and inputs (section "Prefill: keep routing on the GPU, dequantize in flight"):
      host_routing  the block map built on the host after a stream synchronisation, against the
                    GPU-resident routing: both called eagerly and timed per call on the host clock
                    (the arm cannot be graph-captured); `speedup` = arm time / product time, the
                    page's "+89%" at 512 tokens is a speedup of 1.89;
      tile32        32-row block-map tiles against tiles of up to moe_tile_rows() rows, both replayed
                    from CUDA graphs; `speedup` = arm time / product time (the page: +13.2% for its
                    32-row tiles over 16-row ones at 2K tokens);
      dense         the selected experts' weights expanded to fp16 in a buffer first, then dense
                    GEMMs, against in-tile dequantization, both from CUDA graphs (the page: +77.4%
                    at 512 tokens for in-tile dequantization over materialised bf16 weights);
      wide_cfg / narrow_cfg  the GEMM configuration moe_prefill did not pick for this token count
                    (tiles of up to 192 rows / 32-row tiles with deeper copy rings), forced."""
    import torch
    n = len(layers)
    aux = None
    if arm == "host_routing":
        def wall(fn):
            fn(0)
            torch.cuda.synchronize()
            ts = []
            for r in range(reps):
                for i in range(n):
                    t0 = time.perf_counter()
                    fn(i)
                    torch.cuda.synchronize()
                    ts.append(time.perf_counter() - t0)
            return 1e6 * statistics.median(ts)
        base = wall(lambda i: m.prefill(layers[i], xs[i], ws, y=ys[i]))
        t = wall(lambda i: m.prefill_ablation(layers[i], xs[i], ws, m.PREFILL_ARM_HOST_ROUTING, y=ys[i]))
        how = "eager calls, host clock per call with a synchronize, median"
    else:
        def graph(fn):
            def body():
                for _ in range(reps):
                    for i in range(n):
                        fn(i)
            return 1e3 * _graph_time_ms(body) / (reps * n)
        code = {"tile32": m.PREFILL_ARM_TILE32, "dense": m.PREFILL_ARM_DENSE, "wide_cfg": m.PREFILL_ARM_WIDE_TILES,
                "narrow_cfg": m.PREFILL_ARM_NARROW_TILES}[arm]
        n_aux = m.ablation_aux_bytes(layers[0].dims, code)
        aux = torch.empty(n_aux, dtype=torch.uint8, device=xs[0].device) if n_aux else None
        base = graph(lambda i: m.prefill(layers[i], xs[i], ws, y=ys[i]))
        t = graph(lambda i: m.prefill_ablation(layers[i], xs[i], ws, code, y=ys[i], aux=aux))
        how = "CUDA graphs over the rotated layers, best of 3 replays"
    del aux
    return {"arm_us_per_layer": t, "product_us_per_layer": base, "speedup": t / base, "how": how}


def spawn_ranks(args, argv) -> None:
    """`--gpus N` (N > 1) outside a launcher: re-executes this command under torch.distributed.run
    with N ranks on this node (rendezvous on 127.0.0.1). Inside a launcher the world size must be N."""
    import socket
    if "WORLD_SIZE" in os.environ:
        world = int(os.environ["WORLD_SIZE"])
        if world != args.gpus:
            print(json.dumps({"error": f"--gpus {args.gpus} but WORLD_SIZE={world}"}), flush=True)
            sys.exit(2)
        return
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    sys.stdout.flush()
    os.execv(sys.executable, cmd)


def rank_check() -> None:
    """Starts the process group (NCCL with GPUs, gloo without), sums one value over the ranks and
    prints the world size from rank 0."""
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    backend = "gloo"
    if world > 1:
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            backend = "nccl"
        dist.init_process_group(backend)
    total = reduce_over_ranks({"one": 1.0}, "sum")["one"]
    if rank == 0:
        print(json.dumps({"rank_check": True, "world": world, "ranks_summed": total, "backend": backend}), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(argv)
    if args.oracle_child is not None:
        _oracle_child(args.oracle_child)
        return
    if args.gpus > 1:
        spawn_ranks(args, argv)
    if args.rank_check:
        rank_check()
        return
    config = {"workload": f"layer stack: {args.layers} independent MoE layers x ({args.prefill_tokens}-token "
                          f"prefill + {args.decode_steps} batch-1 decode steps)",
              "layers": args.layers, "prefill_tokens": args.prefill_tokens, "decode_steps": args.decode_steps,
              "d": 2048, "experts": 256, "top_k": 8, "inter": 512, "shared_inter": 512,
              "weights": "Q4 affine, group 64, bf16 scale+bias", "router_bias": args.router_bias,
              "l2": "no flush: inputs larger than L2 (40 layers of packed weights, 18.2 GB)",
              "parallelism": f"replicas x{args.gpus}"}
    if args.impl == "reference":
        run_reference(args, config)
    else:
        run_ours(args, config)


if __name__ == "__main__":
    main()
