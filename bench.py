"""Throughput of the chunkwise gated delta-rule forward on GB300 (one JSON line on stdout).

A step is one forward call -- the whole path: decay cumsum, rescaling, WY
build, state scan and output.  The default workload is KDA at B=4, T=4096,
H=16, dk=dv=128, bf16 inputs, fp32 state, initial state given (one
kda_chunk_fwd call per step).  --workload picks another of the seeded
workloads: the GDN / DeltaNet / GLA sweep at B=8, T=2048, H=32, d=128 (same
entry point) or general DPLR at B=2, T=8192, H=16, d=128 (one dplr_chunk_fwd
call per step; the line also carries the transition-norm report).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

--impl ours (default): the CUDA library through its C ABI.  `value` is tokens/s
with the inputs resident in HBM; `e2e` is the same metric with pinned host
inputs copied in and o / ht copied out inside the timed region, every step
(the host runner overlaps one step's copies with the previous step's call on
separate streams, as a serving loop would); `roofline`
compares the kernel's algorithmic bytes per launch against the measured HBM
copy bandwidth; `cpu_baseline` times the float64 oracle on a bounded sample
of the same workload on the host cores.
--impl reference: the float64 oracle (the only reference this method has) on
the host cores, on a bounded sample per step.

Under torchrun (N > 1) every rank runs its own replica of the workload: the
(batch, head) scans are independent, so there is no collective on the data
path ("scaling": "weak").  Rank 0 prints the line; times are the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

WORKLOAD = "kda_bf16_b4t4096h16d128"
METRIC = "tokens/s KDA chunk fwd(+bwd) B4·T4096·H16·d128 bf16; % of roofline"
CSRC = os.path.join(ROOT, "chunkwise_gated_delta_gb300", "csrc")

# kernel that runs each variant's step: (name, source file)
KERNELS = {"kda": ("kda_fwd_tc", "kda_fwd_tc.cu"), "gdn": ("kda_fwd_tc", "kda_fwd_tc.cu"),
           "deltanet": ("kda_fwd_tc", "kda_fwd_tc.cu"), "gla": ("kda_fwd_tc", "kda_fwd_tc.cu"),
           "dplr": ("dplr_fwd_simt", "dplr_fwd_simt.cu"), "kda_bwd": ("kda_bwd_simt", "kda_bwd_simt.cu"),
           "dplr_bwd": ("dplr_bwd_simt", "dplr_bwd_simt.cu")}
LAUNCHES_PER_STEP = {"kda": 2, "gdn": 2, "deltanet": 2, "gla": 2, "dplr": 2, "kda_bwd": 4,
                     "dplr_bwd": 4}   # kernels one step launches (bf16 forward: its two-kernel form)


def forward_form(w, d, o, ht, gate, scale_v):
    """Which form the library runs for this forward: 'single' (one kernel, the status word as
    workspace) or 'records' (chunk-record kernel + scan), read from its workspace query."""
    import ctypes

    from chunkwise_gated_delta_gb300 import _lib, api
    a = api.make_args(d["q"], d["k"], d["v"], d.get("g"), d.get("beta"), d.get("h0"), o, ht, gate=gate,
                      scale_v=scale_v)
    return "single" if _lib.load().kda_chunk_fwd_workspace(ctypes.byref(a)) <= 256 else "records"


def kind_of(w) -> str:
    if w.grads:
        return "dplr_bwd" if w.variant == "dplr" else "kda_bwd"
    return w.variant
GATES = {"kda": "channel", "gla": "channel", "dplr": "channel", "gdn": "scalar", "deltanet": "none"}


def metric_for(w) -> str:
    if w.name == WORKLOAD:
        return METRIC
    shape = f"B{w.B}·T{w.T}·H{w.H}·d{w.dk}"
    if w.grads:
        return f"tokens/s {'DPLR' if w.variant == 'dplr' else 'KDA'} chunk bwd {shape} bf16; % of roofline"
    return f"tokens/s {w.variant.upper() if w.variant != 'deltanet' else 'DeltaNet'} chunk fwd {shape} bf16; % of roofline"


def algorithmic_bytes(w) -> int:
    """Inputs read once and outputs written once (bf16 sequences, fp32 states).

    KDA: q, k, g (dk wide), v, o (dv wide), beta, h0, ht.  GDN: g is one value
    per token and head.  DeltaNet: no g.  GLA: no beta.  DPLR: q, k, a, b, g
    (dk wide), v, o (dv wide), h0 when given, ht.
    """
    bth = w.B * w.T * w.H
    es = 2 if w.dtype == torch.bfloat16 else 4
    state = w.B * w.H * w.dv * w.dk * 4
    states = state * (2 if w.h0 else 1)
    if w.grads and w.variant == "dplr":
        # reads q, k, a, b, g, v, dO, h0 when given, dht; writes dq, dk, da, db, dg, dv, dh0
        reads = bth * (5 * w.dk + 2 * w.dv) * es + state * (2 if w.h0 else 1)
        writes = bth * (5 * w.dk + w.dv) * es + state
        return reads + writes
    if w.grads:
        # reads q, k, v, g, beta, h0, dO, dht; writes dq, dk, dv, dg, dbeta, dh0
        reads = bth * (3 * w.dk + 2 * w.dv + 1) * es + state * (2 if w.h0 else 1)
        writes = bth * (3 * w.dk + w.dv + 1) * es + state
        return reads + writes
    if w.variant == "dplr":
        return bth * (5 * w.dk + 2 * w.dv) * es + states
    seq = bth * (2 * w.dk + 2 * w.dv) * es
    g = {"kda": bth * w.dk, "gla": bth * w.dk, "gdn": bth, "deltanet": 0}[w.variant] * es
    beta = 0 if w.variant == "gla" else bth * es
    return seq + g + beta + states


def traffic_file(w) -> str:
    shape = w.name.split("_")[-1]
    return os.path.join(ROOT, "profiles", f"{KERNELS[kind_of(w)][0]}_{w.variant}_{shape}_traffic.txt")


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def traffic_per_launch(w):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel source."""
    try:
        src = os.path.join(CSRC, KERNELS[kind_of(w)][1])
        src_hash = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        vals = {}
        for line in open(traffic_file(w)):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        if vals.get("kernel_source_sha256_16") != src_hash:
            return None
        return int(vals["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while a region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [r for t, r in self.rows if self.t0 is not None and self.t0 - 0.15 <= t <= self.t1 + 0.15]
        if not rows and self.rows:
            rows = [min(self.rows, key=lambda tr: abs(tr[0] - (self.t1 or tr[0])))[1]]
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_sample(w, x, heads, T):
    """Time the float64 oracle on `heads` (b, h) pairs over the first T tokens."""
    import oracle
    f = lambda n: (x[n][:, :T].double().numpy() if n in x else None)
    q, k, v, g, beta, a, b = (f(n) for n in ("q", "k", "v", "g", "beta", "a", "b"))
    h0 = x["h0"].double().numpy() if "h0" in x else None
    cores = len(os.sched_getaffinity(0))
    kw = dict(h0=h0, heads=heads, threads=cores)
    t0 = time.perf_counter()
    if w.grads:
        dht = x["dht"].double().numpy() if "dht" in x else None
        if w.variant == "dplr":
            oracle.dplr_bwd(q, k, v, a, b, g, f("do"), dht=dht, **kw)
        else:
            oracle.kda_bwd(q, k, v, g, beta, f("do"), dht=dht, **kw)
    elif w.variant == "kda":
        oracle.kda_fwd(q, k, v, g, beta, **kw)
    elif w.variant == "gdn":
        oracle.gdn_fwd(q, k, v, g, beta, **kw)
    elif w.variant == "deltanet":
        oracle.deltanet_fwd(q, k, v, beta, **kw)
    elif w.variant == "gla":
        oracle.gla_fwd(q, k, v, g, **kw)
    else:
        oracle.dplr_fwd(q, k, v, a, b, g, **kw)
    dt = time.perf_counter() - t0
    tokens = len(heads) * T / w.H              # head-tokens expressed as workload tokens
    return tokens, dt, cores


def cpu_baseline_leg(w, x, budget_s=12.0):
    """Oracle on a bounded sample: as many (b, h) pairs over the full T as fit the budget."""
    cores = len(os.sched_getaffinity(0))
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    probe = pairs[:min(cores, len(pairs))]
    tokens, dt, _ = oracle_sample(w, x, probe, w.T)
    n = len(probe)
    scale = max(1, int(budget_s / max(dt, 1e-3)))
    n = min(len(pairs), n * scale)
    if n > len(probe):
        tokens, dt, _ = oracle_sample(w, x, pairs[:n], w.T)
    return {"value": tokens / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {len(pairs)} (batch, head) pairs over the full T={w.T}, float64 token "
                      f"recurrence{' reverse mode' if w.grads else ''} in C, {cores} threads; tokens counted as "
                      f"head-tokens / H; {dt:.1f} s"}


def run_reference(args, rank, world):
    from chunkwise_gated_delta_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[args.workload]
    if rank != 0:
        return
    x = make_inputs(w, seed=0)
    cores = len(os.sched_getaffinity(0))
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    heads = pairs[:min(cores, len(pairs))]
    # size each step so the whole run stays within about a minute
    tokens, dt, _ = oracle_sample(w, x, heads, 256)
    per_step_budget = max(0.05, 60.0 / max(1, args.steps + args.warmup))
    T = int(min(w.T, max(64, 256 * per_step_budget / max(dt, 1e-4))))
    for _ in range(args.warmup):
        oracle_sample(w, x, heads, T)
    tot_tokens, tot_dt = 0.0, 0.0
    for _ in range(args.steps):
        tk, dt, _ = oracle_sample(w, x, heads, T)
        tot_tokens += tk
        tot_dt += dt
    value = tot_tokens / tot_dt
    sample = (f"{len(heads)} (batch, head) pairs x {T} tokens per step, float64 token recurrence in C, "
              f"{cores} threads; tokens counted as head-tokens / H")
    line = {
        "impl": "reference", "metric": metric_for(w), "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(w):
    inputs = {"kda": "bf16 q,k,v,g,beta", "gdn": "bf16 q,k,v,beta, g [B,T,H]", "deltanet": "bf16 q,k,v,beta",
              "gla": "bf16 q,k,v,g; beta = 0, v unscaled", "dplr": "bf16 q,k,v,a,b,g"}[w.variant]
    if w.grads and w.variant == "dplr":
        inputs += ", dO; fp32 dht, no h0; outputs bf16 dq,dk,dv,da,db,dg, fp32 dh0"
    elif w.grads:
        inputs += ", dO; fp32 h0, dht; outputs bf16 dq,dk,dv,dg,dbeta, fp32 dh0"
    else:
        inputs += "; fp32 h0/ht" if w.h0 else "; fp32 ht, no h0"
    return {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
            "chunk": 16 if kind_of(w) == "dplr_bwd" else 32 if (w.variant == "dplr" or w.grads) else w.chunk, "h0": w.h0, "inputs": inputs,
            "l2": f"no flush: inputs larger than L2 ({algorithmic_bytes(w) / 1e6:.1f} MB per step vs 129 MB)",
            "parallelism": "replicas (independent (batch, head) scans, no collective)"}


def run_ours(args, rank, world, local):
    from chunkwise_gated_delta_gb300 import (HostRunner, dplr_chunk_bwd, dplr_chunk_fwd, dplr_factor_norms,
                                             kda_chunk_bwd, kda_chunk_fwd)
    from chunkwise_gated_delta_gb300.inputs import WORKLOADS, make_inputs
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    x = make_inputs(w, seed=rank)
    x = {k: v for k, v in x.items() if k in ("q", "k", "v", "g", "beta", "h0", "a", "b", "do", "dht", "scale_v")}
    d = {k: v.to(dev) for k, v in x.items() if isinstance(v, torch.Tensor)}
    o = torch.empty(w.B, w.T, w.H, w.dv, dtype=w.dtype, device=dev)
    ht = torch.empty(w.B, w.H, w.dv, w.dk, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    gate = GATES[w.variant]

    if kind_of(w) == "dplr_bwd":
        grads = {n: torch.empty_like(d[src]) for n, src in (("dq", "q"), ("dk", "k"), ("dv", "v"), ("da", "a"),
                                                            ("db", "b"), ("dg", "g"))}
        grads["dh0"] = torch.empty(w.B, w.H, w.dv, w.dk, dtype=torch.float32, device=dev)

        def step():
            dplr_chunk_bwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["g"], d.get("h0"), d["do"], d["dht"],
                           gate=gate, grads=grads, stream=stream)
    elif w.grads:
        grads = {"dq": torch.empty_like(d["q"]), "dk": torch.empty_like(d["k"]), "dv": torch.empty_like(d["v"]),
                 "dg": torch.empty_like(d["g"]), "dbeta": torch.empty_like(d["beta"]),
                 "dh0": torch.empty(w.B, w.H, w.dv, w.dk, dtype=torch.float32, device=dev)}

        def step():
            kda_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("h0"), d["do"], d["dht"], gate=gate,
                          scale_v=x["scale_v"], grads=grads, stream=stream)
    elif w.variant == "dplr":
        def step():
            dplr_chunk_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d.get("g"), d.get("h0"), gate=gate,
                           o=o, ht=ht, stream=stream)
    else:
        def step():
            kda_chunk_fwd(d["q"], d["k"], d["v"], d.get("g"), d.get("beta"), d.get("h0"), gate=gate,
                          scale_v=x["scale_v"], o=o, ht=ht, stream=stream)

    launches = LAUNCHES_PER_STEP.get(kind_of(w), 1)
    form = None
    if kind_of(w) in ("kda", "gdn", "deltanet", "gla"):
        form = forward_form(w, d, o, ht, gate, x["scale_v"])
        # single: the kernel, then (gated variants) the launch that redoes a call whose decay
        # passed the one-product Gram's range and otherwise exits at once; records: Z + scan
        launches = (1 if gate == "none" else 2) if form == "single" else 2

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark_begin()
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = t_all0.elapsed_time(t_all1)
    launch_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    launch_ms = max_over_ranks(launch_ms, world)

    # end to end from pinned host buffers
    e2e = None
    if not args.no_e2e:
        runner = HostRunner(x, device=dev, scale_v=x["scale_v"], gate=gate,
                            kind=kind_of(w) if kind_of(w) in ("dplr", "kda_bwd", "dplr_bwd") else "kda")
        runner.begin(stream)
        for _ in range(max(3, min(args.warmup, 10))):
            runner.run(stream)
        runner.finish(stream)
        torch.cuda.synchronize()
        e2e_steps = max(3, min(args.steps, 50))
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        runner.begin(stream)            # the copy streams start after e0 ...
        for _ in range(e2e_steps):
            runner.run(stream)          # every step copies its inputs in and its results out
        runner.finish(stream)           # ... and e1 waits for the last read-back
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
        barrier(world)
        e2e = {"value": world * w.B * w.T / (e2e_ms * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": runner.h2d_bytes, "d2h_bytes_per_step": runner.d2h_bytes}

    tokens = w.B * w.T
    peaks, peak_kind = measured_peaks()
    abytes = algorithmic_bytes(w)
    achieved = abytes / (launch_ms * 1e-3) / 1e9
    line = {
        "metric": metric_for(w),
        "value": world * tokens * args.steps / (elapsed_ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": config_dict(w),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic_per_launch(w),
                     "kernel": KERNELS[kind_of(w)][0],
                     "form": form,
                     "scope": f"whole step: {launches} kernel launch(es) per step, "
                              "timed together between CUDA events",
                     "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)",
                     "algorithmic_bytes_per_launch": abytes, "kernel_ms_per_launch": launch_ms},
        "e2e": e2e,
        "gpu_launches": args.steps * launches,
        "clocks": clk,
    }
    if kind_of(w) == "dplr":
        # transition-norm report (outside the timed region), without and with the eq. (7) clip
        _, _, mx = dplr_factor_norms(d["a"], d["b"], d.get("g"), gate=gate, stream=stream)
        _, _, mxc = dplr_factor_norms(d["a"], d["b"], d.get("g"), gate=gate, clip=True, stream=stream)
        torch.cuda.synchronize()
        line["factor_norms"] = {"max_rho_eq4": float(mx[0]), "max_factor_norm": float(mx[1]),
                                "max_factor_norm_clipped": float(mxc[1]), "tokens": w.B * w.T * w.H}
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline_leg(w, x)
        print(json.dumps(line), flush=True)


def free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def relaunch_ranks(n_gpus: int, argv) -> int:
    """`--gpus N` (N > 1) started without a rank environment: run N ranks of this same command.

    One process per GPU through torch.distributed.run on 127.0.0.1; rank 0 prints the line and
    the return code is the launcher's."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n_gpus}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["kda_fp32_b1t256h1d64", "kda_bf16_b4t4096h16d128", "gdn_bf16_b8t2048h32d128", "deltanet_bf16_b8t2048h32d128",
                             "gla_bf16_b8t2048h32d128", "dplr_bf16_b2t8192h16d128", "kda_bwd_bf16_b4t4096h16d128",
                             "dplr_bwd_bf16_b2t8192h16d128"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    args = ap.parse_args()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(relaunch_ranks(args.gpus, sys.argv[1:]))
    if int(os.environ.get("WORLD_SIZE", "1")) != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={os.environ.get('WORLD_SIZE', '1')}")
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
