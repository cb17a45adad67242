"""Benchmark of the exact attention forward pass on one GB300 (per process).

One step = one call of the library's attention forward over the whole workload
(all of the hot path: tile schedule, TMA loads, Q K^T, masked online softmax,
P V, epilogue) with inputs resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload cfg3] [--impl ours|reference]
                  [--pass fwd|bwd]

--pass bwd times the backward instead (one step = one attn_bwd call: D prep, dQ
pass, dK/dV pass) on O and LSE from one untimed forward and a seeded dO; its
work is counted as 2.5x the forward's (five N x N x d products instead of two).

Multi-GPU: the forward pass of independent problems has no exchange step, so
N > 1 runs N independent replicas (one per rank, launched by torchrun); value is
the work of all ranks divided by the slowest rank's time.

--impl reference times the fp64 CPU oracle (the only other implementation
there is) on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import os

# The CPU-baseline leg uses numpy's BLAS; pin its thread count so the number of
# cores it uses is known.
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_tiled_attention_16_gb300 import synth  # noqa: E402

METRIC = "attention fwd TFLOP/s on 1 GB300 and % of dense BF16/FP8 tensor peak"
METRIC_BWD = "attention bwd TFLOP/s on 1 GB300 (counted as 2.5x forward flops) and % of dense BF16 tensor peak"
BWD_FLOP_RATIO = 2.5
L2_BYTES = 126 * 1024 * 1024
CSRC = os.path.join(ROOT, "exact_tiled_attention_16_gb300", "csrc")
# tensor-core work per SM clock: a 128 x 128 x 16 kind::f16 MMA occupies the pipe
# 64 cycles (measured), 8192 flops per cycle; the e4m3 Q K^T at the nominal 2x
ALL_WORKLOADS = ["cfg1", "cfg2n", "cfg2c", "cfg3", "cfg4", "cfg5", "cfg5p", "decode",
                 "custom:1,32,4096,128,0", "custom:1,32,8192,128,0", "custom:1,32,16384,128,0",
                 "custom:1,16,8192,128,0,e4m3", "bwd:cfg3", "bwd:cfg4"]
BF16_FLOP_PER_CLK_SM = 8192.0
FP8_FLOP_PER_CLK_SM = 16384.0
WORKLOAD_TEXT = {
    "cfg1": "bf16 B1 H2 N128 d64 non-causal",
    "cfg2n": "bf16 B4 H16 N2048 d128 non-causal",
    "cfg2c": "bf16 B4 H16 N2048 d128 causal",
    "cfg3": "bf16 B1 H32 N16384 d128 causal (long sequence, small batch)",
    "cfg4": "bf16 B16 H16 N4096 d64 non-causal, 2 shared Q/K outlier channels x20",
    "cfg5": "e4m3 block-scaled B2 H16 N8192 d128 non-causal, rotated Q/K",
    "cfg5p": "Direct-P FP4: cfg5's Q/K (e4m3) with V in MXFP4 (e2m1, E8M0 per 32 keys), B2 H16 N8192 d128",
    "decode": "bf16 B2 H16 Nq512 Nk65536 d128 non-causal, split-K/V forward + merge",
}
DECODE = dict(B=2, H=16, Nq=512, Nk=65536, d=128, seed=6)


def kernel_sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".inc")))


def kernel_hash() -> str:
    """Hash of every CUDA source of the library (what a profile was taken on)."""
    h = hashlib.sha256()
    for f in kernel_sources():
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def kernel_instance(dtype: str, d: int, partial: bool = False, causal: bool = False, table: bool = False,
                    pair_tail: bool = False) -> str:
    """The forward kernel's template instance as ncu names it, read from the
    instance table of attn_api.cu (D, K stages, V stages, fp8, partial, fp4, the
    TMA store of O, which the non-causal BF16 launches use, the unit table, which
    BF16 launches use when every CTA's rounds fit in it, and the pair tail, a
    non-causal last round split over CTA pairs, in BF16 table launches and FP8
    launches: `table` and `pair_tail` from the library's schedule diagnostic)."""
    import re
    text = open(os.path.join(CSRC, "attn_api.cu")).read()
    inst = dict(re.findall(r"#define (ATTN_\w+_D\d+) (\d+, \d+, \d+, (?:true|false))", text))
    key = {"bf16": f"ATTN_BF16_D{d}", "e4m3": f"ATTN_FP8_D{d}", "e4m3_e2m1": f"ATTN_FP4_D{d}"}[dtype]
    if key not in inst:
        return "attn::attn_fwd_kernel<?>"
    D, nk, nv, fp8 = (x.strip() for x in inst[key].split(","))
    fp4 = dtype == "e4m3_e2m1"
    tma_o = dtype == "bf16" and not partial and not causal
    tab = dtype == "bf16" and not partial and table
    tail = pair_tail and not partial and ((tab and tma_o) or dtype == "e4m3")
    args = [D, nk, nv, "1" if fp8 == "true" else "0", "1" if partial else "0", "1" if fp4 else "0",
            "1" if tma_o else "0", "1" if tab else "0", "1" if tail else "0"]
    return "attn::attn_fwd_kernel<" + ", ".join(args) + ">"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def traffic_for(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm = float(f[1])
                mx = float(f[2])
            except ValueError:
                continue
            sms.append(sm)
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        # samples taken while the GPU was loaded: the upper half of the clock samples
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


def max_over_ranks(dist, value: float, device=None) -> float:
    """The largest of `value` across the ranks of the default process group (the
    slowest rank's time); `dist` is torch.distributed or None for one process."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, world: int, steps: int, slowest_ms: float) -> float:
    """TFLOP/s of the whole job: the work of all ranks over the slowest rank's time."""
    return flops_per_step * world * steps / (slowest_ms * 1e-3) / 1e12


def make_decode_workload():
    """Few queries against a long K/V: the K/V rows of a seeded draw and, as
    queries, its last Nq rows (non-causal)."""
    c = DECODE
    w = synth.make_bf16(c["B"], c["H"], c["Nk"], c["d"], False, seed=c["seed"], name="decode")
    w.q = np.ascontiguousarray(w.q[:, :, c["Nk"] - c["Nq"]:])
    w.meta["Nq"] = c["Nq"]
    return w


def _blas_threads() -> int:
    return int(os.environ.get("OPENBLAS_NUM_THREADS", str(_CORES)))


def make_workload(args):
    """The synthetic workload the flags name (seeded; see synth.py)."""
    if args.custom:
        f = args.custom.split(",")
        B, H, N, d, c = (int(x) for x in f[:5])
        kind = f[5] if len(f) > 5 else "bf16"
        name = f"custom_B{B}H{H}N{N}d{d}{'c' if c else 'n'}"
        if kind == "e4m3":  # cfg5's recipe (outlier channels x10, rotated Q/K) on another shape
            return synth.make_fp8(B, H, N, d, bool(c), seed=3, outlier_frac=0.01, outlier_mult=10.0,
                                  name=name + "_e4m3")
        if kind != "bf16":
            raise SystemExit(f"--custom: unknown element type {kind!r} (bf16 or e4m3)")
        return synth.make_bf16(B, H, N, d, bool(c), seed=3, name=name)
    if args.workload == "decode":
        return make_decode_workload()
    return synth.make_config(args.workload)


def cpu_row_probe(args):
    """(run in a child process with the BLAS thread count pinned by its
    environment) times the oracle on sampled rows and prints one JSON object."""
    w = make_workload(args)
    fn = cpu_oracle_bwd_rate if args.bwd_pass == "bwd" else cpu_oracle_rate
    val, desc, secs, rows = fn(w, args.cpu_budget, rows_per_head=args.probe_rows)
    print(json.dumps({"value": val, "ms_per_row": secs * 1e3 / max(rows, 1), "rows": rows, "seconds": secs,
                      "threads": _blas_threads(), "sample": desc}), flush=True)


def cpu_rows_one_thread(args):
    """ms per query row of the oracle with one BLAS thread (child process)."""
    env = dict(os.environ)
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-row-probe", "--cpu-budget", str(args.cpu_budget / 3),
           "--probe-rows", "32", "--pass", args.bwd_pass]
    cmd += ["--custom", args.custom] if args.custom else ["--workload", args.workload]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError, OSError):
        return None


def run_all(args):
    """One JSON line per workload of ALL_WORKLOADS (each its own child process)."""
    for spec in ALL_WORKLOADS:
        cmd = [sys.executable, os.path.abspath(__file__), "--steps", str(args.steps), "--warmup", str(args.warmup),
               "--cpu-budget", str(args.cpu_budget)]
        if spec.startswith("custom:"):
            cmd += ["--custom", spec.split(":", 1)[1]]
        elif spec.startswith("bwd:"):
            cmd += ["--workload", spec.split(":", 1)[1], "--pass", "bwd"]
        else:
            cmd += ["--workload", spec]
        r = subprocess.run(cmd, capture_output=True, text=True)
        lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
        if r.returncode != 0 or not lines:
            print(json.dumps({"workload": spec, "error": (r.stderr or r.stdout)[-400:]}), flush=True)
            continue
        print(lines[-1], flush=True)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_oracle_rate(w: synth.Workload, budget_s: float, rows_per_head: int = 256, max_heads=None):
    """Times the fp64 oracle on sampled rows of successive heads until budget_s
    seconds of oracle time have passed; returns (TFLOP/s in the workload's
    counting convention, sample description, seconds)."""
    from oracle.attention import attention_head
    from oracle.direct_p import direct_p_head
    head_fn = direct_p_head if w.dtype == "e4m3_e2m1" else attention_head
    flops = 0.0
    elapsed = 0.0
    heads = 0
    rows_done = 0
    for b in range(w.B):
        for h in range(w.H):
            q, k, v = w.head_f64(b, h)
            rows = synth.sample_rows(q.shape[0], rows_per_head, w.seed, b, h)
            t0 = time.perf_counter()
            head_fn(q, k, v, w.causal, w.scale, rows=rows)
            elapsed += time.perf_counter() - t0
            vis = (rows + 1) if w.causal else np.full(len(rows), w.N)
            flops += float(4.0 * w.d * vis.sum())
            heads += 1
            rows_done += len(rows)
            if elapsed >= budget_s or (max_heads and heads >= max_heads):
                break
        if elapsed >= budget_s or (max_heads and heads >= max_heads):
            break
    what = "Direct-P oracle: " if w.dtype == "e4m3_e2m1" else ""
    desc = (f"{what}{rows_done} query rows ({rows_per_head} seeded rows per head x {heads} heads) against all "
            f"visible keys of {w.name}; fp64 numpy, {_blas_threads()} BLAS threads")
    return flops / elapsed / 1e12, desc, elapsed, rows_done


def cpu_oracle_bwd_rate(w: synth.Workload, budget_s: float, rows_per_head: int = 128, max_heads=None):
    """Times the fp64 gradient oracle's dq on sampled query rows of successive
    heads until budget_s seconds have passed.  Each row is counted as its share of
    the backward's work (2.5x its forward flops), so the rate is in the same
    units as the GPU number."""
    from oracle.attention_bwd import attention_bwd_query_rows
    flops = elapsed = 0.0
    heads = rows_done = 0
    done = False
    for b in range(w.B):
        for h in range(w.H):
            q, k, v = w.head_f64(b, h)
            do = synth.bf16_bits_to_f64(synth.make_grad_out(1, 1, w.N, w.d, seed=w.seed + 1000 * b + h)[0, 0])
            rows = synth.sample_rows(q.shape[0], rows_per_head, w.seed, b, h)
            t0 = time.perf_counter()
            attention_bwd_query_rows(q, k, v, do, w.causal, w.scale, rows)
            elapsed += time.perf_counter() - t0
            vis = (rows + 1) if w.causal else np.full(len(rows), w.N)
            flops += BWD_FLOP_RATIO * float(4.0 * w.d * vis.sum())
            heads += 1
            rows_done += len(rows)
            done = elapsed >= budget_s or bool(max_heads and heads >= max_heads)
            if done:
                break
        if done:
            break
    desc = (f"dq of {rows_done} query rows ({rows_per_head} seeded rows per head x {heads} heads) of "
            f"{w.name}, each counted as 2.5x its forward flops; fp64 numpy, {_blas_threads()} BLAS threads")
    return flops / elapsed / 1e12, desc, elapsed, rows_done


def run_reference(args, world, rank):
    """The oracle timed per step on a bounded sample (rank 0 only)."""
    if rank != 0:
        return
    if args.small:
        w = synth.make_bf16(1, 2, 1024, 128, True, 3)
    elif args.workload == "decode":
        w = make_decode_workload()
    else:
        w = synth.make_config(args.workload)
    from oracle.attention import attention_head
    from oracle.attention_bwd import attention_bwd_query_rows
    from oracle.direct_p import direct_p_head
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    rows_per_step = 32
    bwd = args.bwd_pass == "bwd"

    def step(i):
        b, h = heads[i % len(heads)]
        q, k, v = w.head_f64(b, h)
        rows = synth.sample_rows(q.shape[0], rows_per_step, w.seed + i, b, h)
        if bwd:
            do = synth.bf16_bits_to_f64(synth.make_grad_out(1, 1, w.N, w.d, seed=w.seed + i)[0, 0])
        t0 = time.perf_counter()
        if bwd:
            attention_bwd_query_rows(q, k, v, do, w.causal, w.scale, rows)
        elif w.dtype == "e4m3_e2m1":
            direct_p_head(q, k, v, w.causal, w.scale, rows=rows)
        else:
            attention_head(q, k, v, w.causal, w.scale, rows=rows)
        dt = time.perf_counter() - t0
        vis = (rows + 1) if w.causal else np.full(len(rows), w.N)
        return dt, float(4.0 * w.d * vis.sum()) * (BWD_FLOP_RATIO if bwd else 1.0)

    for i in range(args.warmup):
        step(i)
    tot_t = 0.0
    tot_f = 0.0
    for i in range(args.steps):
        dt, f = step(args.warmup + i)
        tot_t += dt
        tot_f += f
    value = tot_f / tot_t / 1e12
    sample = (f"each step: {'dq of ' if bwd else ''}{rows_per_step} seeded query rows of one head against all "
              f"visible keys (fp64 numpy oracle, {_CORES} BLAS threads)")
    line = {
        "impl": "reference", "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(args, w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle", "sample": sample,
                         "ms_per_row_all_cores": tot_t * 1e3 / (args.steps * rows_per_step), "nproc": os.cpu_count()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(args, w):
    in_bytes = w.q.nbytes + w.k.nbytes + w.v.nbytes
    extra = {"Nq": int(w.q.shape[2]), "splits": args.splits} if w.name == "decode" else {}
    what = "backward of " if getattr(args, "bwd_pass", "fwd") == "bwd" else ""
    return {"workload": f"{what}{w.name}: {WORKLOAD_TEXT.get(w.name, '')}", "B": w.B, "H": w.H, "N": w.N, "d": w.d,
            **extra,
            "causal": w.causal, "scale": w.scale, "seed": w.seed,
            "l2": (f"inputs larger than L2 ({in_bytes / 2**20:.0f} MiB > {L2_BYTES / 2**20:.0f} MiB); no flush"
                   if in_bytes > L2_BYTES else
                   "inputs smaller than L2: a 252 MiB buffer is written between steps; value from launch times"),
            "parallelism": "replicas" if getattr(args, "gpus", 1) > 1 else "1 GPU"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="cfg3", choices=sorted(synth.CONFIGS) + ["decode"])
    ap.add_argument("--splits", type=int, default=16, help="key-range splits of the decode workload")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--pass", dest="bwd_pass", default="fwd", choices=["fwd", "bwd"],
                    help="time the forward (default) or the backward of the workload")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--small", action="store_true", help="(reference arm only) a small sample workload")
    ap.add_argument("--custom", default=None,
                    help="B,H,N,d,causal[,e4m3]: a seeded bf16 (or block-scaled e4m3, cfg5's recipe) "
                         "workload of that shape instead of --workload (for profiling captures on a "
                         "reduced case)")
    ap.add_argument("--all", action="store_true",
                    help="one JSON line for each workload (cfg1-cfg5, Direct-P, decode, the non-causal "
                         "d=128 points N=4096/8192/16384, FP8 B1 H16 N8192 (its last round split over CTA "
                         "pairs), the backward of cfg3 and cfg4)")
    ap.add_argument("--cpu-row-probe", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--probe-rows", type=int, default=256, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.cpu_row_probe:
        cpu_row_probe(args)
        return
    if args.all:
        run_all(args)
        return

    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    import exact_tiled_attention_16_gb300 as pkg

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    decode = args.workload == "decode" and not args.custom
    w = make_workload(args)
    fp4 = w.dtype == "e4m3_e2m1"
    fp8 = w.dtype == "e4m3" or fp4
    bwd = args.bwd_pass == "bwd"
    if bwd and (fp8 or decode):
        raise SystemExit("--pass bwd runs on the bf16 square workloads (not the e4m3 one or decode)")
    if fp8:
        q_h, k_h, v_h = (torch.from_numpy(np.ascontiguousarray(x)).pin_memory() for x in (w.q, w.k, w.v))
        sc_h = [torch.from_numpy(np.ascontiguousarray(x)).pin_memory() for x in (w.q_scale, w.k_scale, w.v_scale)]
        scales = [t.to(dev) for t in sc_h]
    else:
        q_h, k_h, v_h = (torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).pin_memory()
                         for x in (w.q, w.k, w.v))
        sc_h, scales = [], []
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    Nq = q.shape[2]
    o = torch.empty((w.B, w.H, Nq, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, Nq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = w.flops() * (BWD_FLOP_RATIO if bwd else 1.0)
    launches_per_step = 2 if decode else (3 if bwd else 1)
    if bwd:
        do_h = torch.from_numpy(synth.make_grad_out(w.B, w.H, w.N, w.d, seed=w.seed).view(np.int16)).view(
            torch.bfloat16).pin_memory()
        dout = do_h.to(dev)
        pkg.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, o=o, lse=lse)
        grads = [torch.empty_like(q) for _ in range(3)]
        bws = torch.empty(pkg.bwd_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8, device=dev)
    if decode:
        ws = torch.empty(pkg.splitkv_workspace_bytes(w.B, w.H, Nq, w.d, args.splits), dtype=torch.uint8,
                         device=dev)

    def forward(qq, kk, vv, ss, oo=None, dd=None, ll=None):
        if fp4:
            pkg.attn_fwd_fp4p(qq, kk, vv, *ss, causal=w.causal, scale=w.scale, o=o, lse=lse)
        elif bwd:
            pkg.attn_bwd(qq, kk, vv, o if oo is None else oo, dout if dd is None else dd, lse if ll is None else ll,
                         causal=w.causal, scale=w.scale, dq=grads[0], dk=grads[1], dv=grads[2], workspace=bws)
        elif decode:
            pkg.attn_fwd_splitkv(qq, kk, vv, args.splits, causal=w.causal, scale=w.scale, o=o, lse=lse,
                                 workspace=ws)
        elif fp8:
            pkg.attn_fwd_fp8(qq, kk, vv, *ss, causal=w.causal, scale=w.scale, o=o, lse=lse)
        else:
            pkg.attn_fwd(qq, kk, vv, causal=w.causal, scale=w.scale, o=o, lse=lse)

    in_bytes = q.nbytes + k.nbytes + v.nbytes + ((o.nbytes + dout.nbytes) if bwd else 0)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if in_bytes <= L2_BYTES else None

    def step():
        if flush is not None:
            flush.fill_(1.0)  # evicts the inputs from L2 (outside the kernel's own events)
        forward(q, k, v, scales)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    rc, where = pkg.check_device_errors()
    if rc != 0:
        raise SystemExit(f"device error after warm-up (wait {where})")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_begin.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(1.0)
            starts[i].record(stream)
            forward(q, k, v, scales)
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    total_ms = t_begin.elapsed_time(t_end)
    kern_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    rc, where = pkg.check_device_errors()
    if rc != 0:
        raise SystemExit(f"device error in the timed region (wait {where})")
    total_ms = max_over_ranks(pg, total_ms, dev)
    avg_kernel_ms = sum(kern_ms) / len(kern_ms)
    if flush is not None:
        # the L2 flush between steps is not part of the step: time the launches only
        total_ms = max_over_ranks(pg, avg_kernel_ms, dev) * args.steps
    ms_per_step = total_ms / args.steps
    value = job_throughput(flops, world, args.steps, total_ms)
    achieved = flops / (avg_kernel_ms * 1e-3) / 1e12

    # end to end through the public API: pinned host inputs -> device, the pass,
    # its results back to pinned host memory, every step.  Forward: Q, K, V in,
    # O and LSE out; backward: Q, K, V, O, dO, LSE in, dQ, dK, dV out (one call of
    # the matching host-buffer entry point, which pipelines the transfers with the
    # kernels; decode: copies, the pass, copies on one stream).
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 20))
    qd, kd, vd = (torch.empty_like(t) for t in (q, k, v))
    sd = [torch.empty_like(t) for t in scales]
    if bwd:
        o_in_h = o.cpu().pin_memory()
        l_in_h = lse.cpu().pin_memory()
        od, dd, ld = torch.empty_like(o), torch.empty_like(dout), torch.empty_like(lse)
        outs = grads
        in_host = [q_h, k_h, v_h, o_in_h, do_h, l_in_h]
    else:
        outs = [o, lse]
        in_host = [q_h, k_h, v_h] + list(sc_h)
    outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]

    # the BF16, FP8 and Direct-P FP4 forwards and the backward: the library's
    # pipelined host-buffer entry points
    host_api = not decode
    if host_api:
        need = (pkg.bwd_host_workspace_bytes if bwd else pkg.fp4p_host_workspace_bytes if fp4
                else pkg.fp8_host_workspace_bytes if fp8 else pkg.fwd_host_workspace_bytes)(w.B, w.H, Nq, w.d)
        hws = torch.empty(need, dtype=torch.uint8, device=dev)

    def e2e_step():
        if host_api and bwd:
            pkg.attn_bwd_host(q_h, k_h, v_h, o_in_h, do_h, l_in_h, causal=w.causal, scale=w.scale,
                              dq=outs_h[0], dk=outs_h[1], dv=outs_h[2], workspace=hws)
            return
        if host_api and fp4:
            pkg.attn_fwd_fp4p_host(q_h, k_h, v_h, *sc_h, causal=w.causal, scale=w.scale, o=outs_h[0],
                                   lse=outs_h[1], workspace=hws)
            return
        if host_api and fp8:
            pkg.attn_fwd_fp8_host(q_h, k_h, v_h, *sc_h, causal=w.causal, scale=w.scale, o=outs_h[0],
                                  lse=outs_h[1], workspace=hws)
            return
        if host_api:
            pkg.attn_fwd_host(q_h, k_h, v_h, causal=w.causal, scale=w.scale, o=outs_h[0], lse=outs_h[1],
                              workspace=hws)
            return
        qd.copy_(q_h, non_blocking=True)
        kd.copy_(k_h, non_blocking=True)
        vd.copy_(v_h, non_blocking=True)
        for dst, src in zip(sd, sc_h):
            dst.copy_(src, non_blocking=True)
        if bwd:
            od.copy_(o_in_h, non_blocking=True)
            dd.copy_(do_h, non_blocking=True)
            ld.copy_(l_in_h, non_blocking=True)
            forward(qd, kd, vd, sd, od, dd, ld)
        else:
            forward(qd, kd, vd, sd)
        for dst, src in zip(outs_h, outs):
            dst.copy_(src, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(pg, e0.elapsed_time(e1), dev)
    e2e_value = job_throughput(flops, world, e2e_steps, e2e_ms)

    peaks, peak_src = measured_peaks()
    # FP8 peak = measured bf16 x 2 (the nominal dense fp8/bf16 ratio, 4.5 / 2.25 PFLOP/s)
    ratio = 2.0 if fp8 and not fp4 else 1.0
    peak = float(peaks["bf16_tflops"]) * ratio
    src = (f"{peak_src} bf16 burst (cuBLAS 8192^3, MEASURED_PEAKS.json)" if peak_src == "measured"
           else "fallback 1.9 PFLOP/s bf16") + (" x 2 (nominal fp8/bf16 ratio)" if fp8 else "")
    if bwd:
        kname = (f"attn::attn_bwd_prep_kernel<{w.d}> + attn::attn_bwd_dq_kernel + attn::attn_bwd_dkdv_kernel "
                 "(whole step)")
    elif decode:
        kname = kernel_instance(w.dtype, w.d, partial=True) + " + attn::attn_merge_kernel"
    else:
        sched = {}
        if w.dtype in ("bf16", "e4m3"):
            sched = pkg.diag_fwd_schedule(w.B * w.H, w.N, w.N, w.causal, d=w.d, fp8=w.dtype == "e4m3",
                                          num_sms=torch.cuda.get_device_properties(dev).multi_processor_count)[0]
        kname = kernel_instance(w.dtype, w.d, causal=w.causal, table=bool(sched.get("table")),
                                pair_tail=bool(sched.get("pair_tail")))
    clocks = clk.summary()
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": traffic_for(w.name + (":bwd" if bwd else "")), "peak_source": src,
            "frac_of_sustained": achieved / (float(peaks.get("bf16_tflops_sustained", peak)) * ratio),
            "kernel": kname, "kernel_hash": kernel_hash(), "avg_launch_ms": avg_kernel_ms, "flops_per_launch": flops}
    # Two more ceilings at the clock the SMs ran at during the timed region:
    #  * the tensor pipe's own rate (the measured 128x128x16 MMA time; e4m3 Q K^T
    #    at the nominal 2x), which cuBLAS's measured peak stays below;
    #  * the special-function unit: one ex2 per score (two in the backward, whose
    #    passes both recompute P) against 4 d counted flops per score (10 d in the
    #    backward), at the ex2 rate measured on this GPU now.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks.get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    hz = mhz * 1e6
    if fp4:
        pipe_fpc = 1.0 / (0.5 / FP8_FLOP_PER_CLK_SM + 0.5 / (3.0 * FP8_FLOP_PER_CLK_SM))
    elif fp8:
        pipe_fpc = 1.0 / (0.5 / FP8_FLOP_PER_CLK_SM + 0.5 / BF16_FLOP_PER_CLK_SM)
    else:
        pipe_fpc = BF16_FLOP_PER_CLK_SM
    roof["pipe_peak"] = pipe_fpc * sms * hz / 1e12
    roof["frac_of_pipe_peak"] = achieved / roof["pipe_peak"]
    roof["pipe_peak_source"] = (f"{pipe_fpc:.0f} flop/clk/SM x {sms} SMs x {mhz:.0f} MHz (median SM clock of the "
                                "timed region); 8192 = a 128x128x16 bf16 MMA per 64 cycles, measured"
                                + ("; e4m3 Q K^T at the nominal 2x" if fp8 else ""))
    try:
        sfu_rate, poly_rate = pkg.measure_exp2_rates()
        exps, fl = (2.0, 10.0 * w.d) if bwd else (1.0, 4.0 * w.d)
        roof["sfu_ceiling"] = fl / exps * sfu_rate * sms * hz / 1e12
        roof["sfu_ceiling_source"] = (f"ex2.approx measured {sfu_rate:.2f}/clk/SM (FMA-pipe polynomial "
                                      f"{poly_rate:.2f}); {exps:.0f} exponential(s) per score against "
                                      f"{fl:.0f} counted flops per score")
    except Exception as e:  # the ceiling is context; its absence must not void the line
        roof["sfu_ceiling"] = None
        roof["sfu_ceiling_source"] = f"not measured: {e}"
    if fp4:
        # Q K^T on the fp8 path (2x bf16), P V on the FP4 path (6x bf16: nominal
        # 13.5 / 2.25 PFLOP/s): the roof of that mix is 1 / (0.5/fp8 + 0.5/fp4)
        b16 = float(peaks["bf16_tflops"])
        mixed = 1.0 / (0.5 / (2.0 * b16) + 0.5 / (6.0 * b16))
        roof["peak"] = mixed
        roof["frac"] = achieved / mixed
        roof["peak_source"] = src + " x 3 (mixed roof: Q K^T at the nominal fp8 ratio 2, P V at the fp4 ratio 6)"
        roof["frac_of_sustained"] = achieved / (float(peaks.get("bf16_tflops_sustained", b16)) * 3.0)
    elif fp8:
        # Q K^T runs on the fp8 tensor path and P V on the 16-bit one: the roof of
        # that mix is flops / (flops/2 / fp8_peak + flops/2 / bf16_peak).
        mixed = 1.0 / (0.5 / peak + 0.5 / float(peaks["bf16_tflops"]))
        roof["peak_mixed_fp8_qk_f16_pv"] = mixed
        roof["frac_of_mixed"] = achieved / mixed

    line = {
        "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded N(0,1) inputs)",
        "config": config_block(args, w),
        "pct_of_peak": 100.0 * value / world / roof["peak"],
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "steps": e2e_steps,
                "h2d_bytes_per_step": int(sum(t.nbytes for t in in_host)),
                "d2h_bytes_per_step": int(sum(t.nbytes for t in outs_h)),
                "api": ((("attn_bwd_host" if bwd else "attn_fwd_fp4p_host" if fp4 else "attn_fwd_fp8_host" if fp8
                          else "attn_fwd_host")
                         + ": pinned host buffers, chunked copies overlapped with the kernels")
                        if host_api else "pinned host copies in, the pass, copies out, on one stream")},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, desc, secs, rows = (cpu_oracle_bwd_rate if bwd else cpu_oracle_rate)(w, args.cpu_budget)
        one = cpu_rows_one_thread(args)
        line["cpu_baseline"] = {"value": val, "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle",
                                "sample": desc, "seconds": secs,
                                "ms_per_row_all_cores": secs * 1e3 / max(rows, 1),
                                "ms_per_row_1_thread": one["ms_per_row"] if one else None,
                                "sample_1_thread": one["sample"] if one else "not measured",
                                "nproc": os.cpu_count()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
