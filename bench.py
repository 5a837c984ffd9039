#!/usr/bin/env python
"""Benchmark of one RACE attention layer, forward + backward, on GB300.

A step is one forward and one backward pass (every kernel of the path) over one synthetic batch
of the named workload, through the library's C ABI.  Inputs are resident in HBM when the timed
region starts; every input tensor is larger than L2 for the default workload, so no flush is
needed between steps.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

--impl reference times the float64 CPU oracle on the host cores (a bounded token prefix of the
same workload per step) and prints the same line with "impl": "reference".
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RACE attn fwd+bwd tokens/sec at 1 GB300 (H=4,d=128); achieved HBM GB/s vs peak"
DEFAULT_WORKLOAD = "c5_bf16_causal_12m"
SMI_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

# Compulsory HBM bytes per (token, head) of each kernel, as (multiples of d * elem_bytes, extra
# bytes, feature rows): the token tensors it must read or write once, per-token float32 scalars,
# and rows of bf16 bucket features (L R values padded to a multiple of 8) it writes or reads.
KERNEL_BYTES = {
    "sketch_keys": (2, 0, 0),        # reads K, V
    "sketch_grad": (2, 8, 0),        # reads Q, dO and {1/den, dO.O}
    "readout": (2, 0, 0),            # reads Q, writes O
    "bwd_query": (3, 8, 0),          # reads Q, dO; writes dQ and {1/den, dO.O}
    "bwd_key": (4, 0, 0),            # reads K, V; writes dK, dV
    "causal_fwd": (4, 0, 0),         # reads Q, K, V; writes O
    "causal_bwd_q": (5, 8, 0),       # reads Q, K, V, dO; writes dQ and {1/den, dO.O}
    "causal_bwd_kv": (6, 8, 0),      # reads Q, K, V, dO and {1/den, dO.O}; writes dK, dV
    "tc5_sketch_keys": (2, 0, 0),    # reads K, V
    "tc5_sketch_grad": (2, 8, 0),    # reads Q, dO and {1/den, dO.O}
    "tc5_readout": (2, 0, 0),        # reads Q, writes O
    "tc5_bwd_query": (3, 8, 0),      # reads Q, dO; writes dQ and {1/den, dO.O}
    "tc5_bwd_key": (4, 0, 0),        # reads K, V; writes dK, dV
    "tc5_causal_fwd": (3, 0, 1),     # reads Q, phi(K) rows, V; writes O
    "tc5_causal_bwd_q": (4, 8, 2),   # reads Q, phi(K) rows, V, dO; writes dQ, {1/den, dO.O} and F'_Q
    "tc5_causal_bwd_kv": (5, 8, 1),  # reads F'_Q, K, V, dO and {1/den, dO.O}; writes dK, dV
}
# On the causal path the segment-sum pass also writes every key's phi(K) row.
CAUSAL_FEATURE_WRITERS = {"tc5_sketch_keys"}


def feature_row_bytes(w):
    """Bytes of one stored bucket-feature row: L R bf16 values padded to a multiple of 8."""
    return 2 * ((w.LR + 7) // 8 * 8)


def compulsory_bytes(name, w):
    mult, extra, feat = KERNEL_BYTES[name]
    if w.causal and name in CAUSAL_FEATURE_WRITERS:
        feat += 1
    return (mult * w.d * w.elem_bytes + extra + feat * feature_row_bytes(w)) * w.B * w.H * w.N


# Each kernel's share of the step's algorithmic bytes (12 d e per (token, head): the forward
# reads Q, K, V and writes O; the backward reads Q, K, V, O, dO and writes dQ, dK, dV), in
# multiples of d * elem_bytes: the token tensors of that list it is the one to read or write.
# Re-reads (the causal segment sums' K and V, the key side's Q and dO) are not algorithmic.
KERNEL_ALG_SHARE = {
    "sketch_keys": 2, "readout": 2, "bwd_query": 3, "sketch_grad": 0, "bwd_key": 4,
    "causal_fwd": 4, "causal_bwd_q": 3, "causal_bwd_kv": 4,
    "tc5_sketch_keys": 2, "tc5_readout": 2, "tc5_bwd_query": 3, "tc5_sketch_grad": 0, "tc5_bwd_key": 4,
    "tc5_causal_fwd": 4, "tc5_causal_bwd_q": 3, "tc5_causal_bwd_kv": 4,
}
# The causal path's segment-sum pass reads K and V but owns none of the algorithmic bytes.
CAUSAL_SEGMENT_SUMS = {"sketch_keys", "tc5_sketch_keys"}

# Other workloads timed after the headline one (each a few steps; no e2e line).
SIDE_CONFIGS = ["c2_bf16_65k", "c3_bf16_causal_lm", "c4_bf16_1m_lr256"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(ms, dist, device):
    """The slowest rank's time per step (every rank receives it): replicas run the same
    workload, so the job is done when the last one is."""
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_tokens_per_s(world, tokens_per_rank, ms):
    """Whole-job throughput of `world` replicas that each process `tokens_per_rank` tokens in
    `ms` milliseconds (the max over ranks)."""
    return world * tokens_per_rank / (ms / 1000.0)


# ------------------------------------------------------------------ host oracle timing

def oracle_sample_rate(w, target_s, cap_tokens=None, threads=None):
    """Time the float64 oracle (forward + backward) on a token prefix of workload w sized to take
    about target_s seconds; returns (tokens/s, threads used, description)."""
    import torch

    import oracle
    from linear_lsh_sketch_gb300.workloads import as_oracle_array, make_inputs

    if threads is None:
        threads = min(os.cpu_count() or 1, w.B * w.H)

    def run(n):
        ws = w.scaled(N=n)
        inp = make_inputs(ws, seed=0, device="cpu")
        a = {k: as_oracle_array(inp[k]) for k in ("Q", "K", "V", "dO")}
        W = inp["W"].double().numpy()
        t0 = time.perf_counter()
        oracle.forward(a["Q"], a["K"], a["V"], W, w.beta, w.causal, nthreads=threads)
        oracle.backward(a["Q"], a["K"], a["V"], a["dO"], W, w.beta, w.causal, nthreads=threads)
        return time.perf_counter() - t0

    n = min(w.N, 2048)
    dt = run(n)
    while dt < 0.5 and n < w.N:
        n = min(w.N, n * 4)
        dt = run(n)
    n_target = int(n * target_s / max(dt, 1e-6))
    n_final = max(1, min(w.N, n_target, cap_tokens or w.N))
    if n_final != n:
        dt = run(n_final)
        n = n_final
    rate = w.B * n / dt
    desc = ("first %d of %d tokens of each of the B*H=%d (batch, head) sequences, forward + backward, "
            "float64, %.1f s" % (n, w.N, w.B * w.H, dt))
    return rate, threads, desc, n, dt


def run_reference(args, w):
    rank, world, _ = env_rank()
    if rank != 0:
        return
    import oracle
    from linear_lsh_sketch_gb300.workloads import as_oracle_array, make_inputs

    threads = min(os.cpu_count() or 1, w.B * w.H)
    per_step = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    _, _, _, n, _ = oracle_sample_rate(w, per_step)
    ws = w.scaled(N=n)
    inp = make_inputs(ws, seed=0, device="cpu")
    a = {k: as_oracle_array(inp[k]) for k in ("Q", "K", "V", "dO")}
    W = inp["W"].double().numpy()
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.forward(a["Q"], a["K"], a["V"], W, w.beta, w.causal, nthreads=threads)
        oracle.backward(a["Q"], a["K"], a["V"], a["dO"], W, w.beta, w.causal, nthreads=threads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = w.B * n * len(times) / total
    sample = ("first %d of %d tokens of each of the B*H=%d sequences per step (float64 oracle, "
              "forward + backward)" % (n, w.N, w.B * w.H))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "host_cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def workload_config(w):
    return {"workload": w.describe(), "name": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "P": w.P,
            "L": w.L, "R": w.R, "beta": w.beta, "causal": w.causal, "io_dtype": w.dtype,
            "accumulate": "f32", "l2": "every input tensor (%.1f GB) is larger than L2; no flush"
            % (w.B * w.H * w.N * w.d * w.elem_bytes / 1e9)}


class ClockSampler:
    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, "--query-gpu=" + ",".join(SMI_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(SMI_FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_table(prof, w, hbm_peak):
    """Per kernel of the timed region: launches, total ms, share of the kernel time, ms per launch
    and, for the kernels in KERNEL_BYTES, two HBM fractions of the peak: `frac` against the
    kernel's own compulsory bytes (what it must move as written) and `alg_frac` against its share
    of the step's algorithmic bytes.  prof: {name: (launches, total ms)}."""
    total = sum(v[1] for v in prof.values())
    out = {}
    unit = w.d * w.elem_bytes * w.B * w.H * w.N
    for name, (nl, ms) in prof.items():
        row = {"launches": nl, "ms_total": ms, "share": ms / max(total, 1e-9),
               "ms_per_launch": ms / max(nl, 1)}
        if name in KERNEL_BYTES and nl > 0 and ms > 0:
            nbytes = compulsory_bytes(name, w)
            sec = row["ms_per_launch"] / 1000.0
            gbs = nbytes / sec / 1e9
            share = 0 if (w.causal and name in CAUSAL_SEGMENT_SUMS) else KERNEL_ALG_SHARE.get(name, 0)
            alg = share * unit
            row.update(achieved_gbs=gbs, frac=gbs / hbm_peak, compulsory_bytes=nbytes, alg_bytes=alg,
                       alg_gbs=alg / sec / 1e9, alg_frac=alg / sec / 1e9 / hbm_peak)
        out[name] = row
    return out


def step_roofline(w, ms, prof, hbm_peak, peak_kind):
    """The step's roofline: 12 d e algorithmic bytes per (token, head) over the step time, with the
    dominant kernel (largest share of the kernel time) and its own fractions beside it."""
    step_bytes = 12 * w.d * w.elem_bytes * w.B * w.H * w.N
    gbs = step_bytes / (ms / 1000.0) / 1e9
    roof = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
            "peak_kind": peak_kind + " (copy bandwidth)", "algorithmic_bytes_per_step": step_bytes,
            "basis": "12 * d * elem_bytes per (token, head) over ms_per_step: the forward reads Q, K, V and "
                     "writes O; the backward reads Q, K, V, O, dO and writes dQ, dK, dV",
            "traffic": traffic_for_step(w, prof)}
    table = kernel_table(prof, w, hbm_peak) if prof else {}
    if table:
        name = max(table, key=lambda k: table[k]["ms_total"])
        k = table[name]
        roof["dominant_kernel"] = {
            "name": name, "ms_per_launch": k["ms_per_launch"], "alg_bytes_per_launch": k.get("alg_bytes"),
            "alg_frac": k.get("alg_frac"), "compulsory_bytes_per_launch": k.get("compulsory_bytes"),
            "compulsory_frac": k.get("frac"), "traffic": traffic_for(name, w)}
    return roof, table


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import linear_lsh_sketch_gb300 as race
    from linear_lsh_sketch_gb300.workloads import CONFIGS, make_inputs

    rank, world, local = env_rank()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    race.load_library()
    hbm_peak, tc_peak, peak_kind = load_peaks()

    # host baseline first (rank 0 only), before the GPU is busy
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, threads, desc, _, _ = oracle_sample_rate(w, args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "host_cores": os.cpu_count(),
               "kind": "oracle", "sample": desc,
               "note": "the oracle runs one thread per (batch, head) problem, so it uses min(host cores, B*H) "
                       "threads"}

    inp = make_inputs(w, seed=rank, device=dev)
    Q, K, V, dO, W = inp["Q"], inp["K"], inp["V"], inp["dO"], inp["W"]
    shape = race.make_shape(w.B, w.H, w.N, w.d, w.torch_dtype)
    state = torch.empty(race.race_attn_state_bytes(shape, w.L, w.P, w.causal), dtype=torch.uint8, device=dev)
    ws_bytes = max(race.race_attn_workspace_bytes(shape, w.L, w.P, w.causal, b) for b in (0, 2 if args.dW else 1))
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    O, dQ, dK, dV = (torch.empty_like(Q) for _ in range(4))
    stream = torch.cuda.current_stream(dev)

    dbeta = torch.empty((w.B, w.H), dtype=torch.float32, device=dev) if args.dbeta else None
    dW = torch.empty((w.B, w.H, w.L, w.P, w.d), dtype=torch.float32, device=dev) if args.dW else None

    def step():
        race.race_attn_fwd(Q, K, V, W, w.beta, w.L, w.P, w.causal, O=O, state=state, workspace=workspace)
        race.race_attn_bwd(Q, K, V, W, w.beta, w.L, w.P, w.causal, dO, O=O, dQ=dQ, dK=dK, dV=dV, state=state,
                           workspace=workspace, dbeta=dbeta, dW=dW)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    uuid = torch.cuda.get_device_properties(dev).uuid
    uuid = "GPU-" + str(uuid) if not str(uuid).startswith("GPU-") else str(uuid)
    race.race_attn_profile_reset()
    race.race_attn_profile(True)
    n0 = race.race_attn_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(uuid) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    ms = e0.elapsed_time(e1) / args.steps
    launches = race.race_attn_launch_count() - n0
    race.race_attn_profile(False)
    prof = race.race_attn_profile_read()
    if world > 1:
        ms = max_over_ranks(ms, dist, dev)

    tokens = w.B * w.N
    value = weak_scaling_tokens_per_s(world, tokens, ms)

    roof, kernels = step_roofline(w, ms, prof, hbm_peak, peak_kind)
    clocks = clk.summary()

    e2e = None
    if rank == 0 and not args.no_e2e:
        try:
            e2e = measure_e2e_pipelined(args, w, race, inp) if w.B * w.H > 1 else None
        except Exception as exc:  # keep the sequential measurement
            print("pipelined e2e failed (%s); sequential copies instead" % exc, file=sys.stderr)
            e2e = None
        if e2e is None:
            e2e = measure_e2e(args, w, race, inp, state, workspace)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": dict(workload_config(w), dbeta=bool(args.dbeta), dW=bool(args.dW)), "clocks": clocks,
            "roofline": roof,
            "kernels": kernels, "gpu_launches": launches, "cpu_baseline": cpu, "e2e": e2e,
        }
        if world == 1 and not args.no_configs and not args.tokens:
            del Q, K, V, dO, W, O, dQ, dK, dV, state, workspace, inp
            torch.cuda.empty_cache()
            line["configs"] = {name: time_side_config(args, CONFIGS[name], race, dev, uuid, hbm_peak, peak_kind)
                               for name in SIDE_CONFIGS if name != w.name}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def traffic_for(name, w):
    """Measured DRAM bytes per launch from the committed ncu summary, if it covers this kernel
    and workload with the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except Exception:
        return None
    ent = table.get(name)
    if not ent or ent.get("workload") != w.name:
        return None
    if ent.get("sources_sha") != sources_sha():
        return None
    return ent.get("bytes_per_launch")


def traffic_for_step(w, prof):
    """Sum over the step's kernels of their measured DRAM bytes per launch times launches per step,
    when the committed ncu summary covers every one of them for this workload; else None."""
    if not prof:
        return None
    total = 0.0
    for name, (nl, _) in prof.items():
        if name in ("combine", "dbeta_combine", "dw_combine"):
            continue
        t = traffic_for(name, w)
        if t is None:
            return None
        total += t * nl
    return total


def _flush_l2(torch, buf):
    buf.add_(1)


def time_side_config(args, w, race, dev, uuid, hbm_peak, peak_kind):
    """ms per fwd+bwd step of workload w on resident synthetic inputs (CUDA events around each
    step; when the inputs fit in L2 a 512 MB buffer is rewritten before every step, outside the
    events), its step roofline and per-kernel table, the clocks, and the float64 oracle on the
    host cores (all threads it can use, and one thread) for the workloads the oracle finishes in
    seconds per thousand tokens."""
    import torch
    from linear_lsh_sketch_gb300.workloads import make_inputs

    inp = make_inputs(w, seed=0, device=dev)
    Q, K, V, dO, W = inp["Q"], inp["K"], inp["V"], inp["dO"], inp["W"]
    shape = race.make_shape(w.B, w.H, w.N, w.d, w.torch_dtype)
    state = torch.empty(race.race_attn_state_bytes(shape, w.L, w.P, w.causal), dtype=torch.uint8, device=dev)
    workspace = torch.empty(max(race.race_attn_workspace_bytes(shape, w.L, w.P, w.causal, b) for b in (0, 1)),
                            dtype=torch.uint8, device=dev)
    O, dQ, dK, dV = (torch.empty_like(Q) for _ in range(4))
    tensor_bytes = Q.numel() * Q.element_size()
    flush = 4 * tensor_bytes < 2 * L2_BYTES
    fbuf = torch.zeros(512 * 2 ** 20 // 4, dtype=torch.float32, device=dev) if flush else None
    stream = torch.cuda.current_stream(dev)

    def step():
        race.race_attn_fwd(Q, K, V, W, w.beta, w.L, w.P, w.causal, O=O, state=state, workspace=workspace)
        race.race_attn_bwd(Q, K, V, W, w.beta, w.L, w.P, w.causal, dO, O=O, dQ=dQ, dK=dK, dV=dV, state=state,
                           workspace=workspace)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    # enough steps to span about a second, so the clock sampler sees the timed region
    t0 = time.perf_counter()
    step()
    torch.cuda.synchronize(dev)
    est = time.perf_counter() - t0
    steps = int(max(3, args.side_steps, min(5000, 1.0 / max(est, 1e-6))))
    race.race_attn_profile_reset()
    race.race_attn_profile(True)
    n0 = race.race_attn_launch_count()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with ClockSampler(uuid) as clk:
        for e0, e1 in ev:
            if flush:
                _flush_l2(torch, fbuf)
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize(dev)
    race.race_attn_profile(False)
    prof = race.race_attn_profile_read()
    launches = race.race_attn_launch_count() - n0
    ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    roof, kernels = step_roofline(w, ms, prof, hbm_peak, peak_kind)
    out = {"workload": w.describe(), "ms_per_step": ms, "steps": steps, "value": w.B * w.N / (ms / 1000.0),
           "unit": "tokens/s", "roofline": roof, "kernels": kernels, "clocks": clk.summary(),
           "gpu_launches": launches,
           "l2": ("inputs fit in L2: a 512 MB buffer is rewritten before each step, outside the timed events"
                  if flush else "every input tensor is larger than L2; no flush")}
    del inp, Q, K, V, dO, W, O, dQ, dK, dV, state, workspace, fbuf
    torch.cuda.empty_cache()
    if not args.no_cpu_baseline and w.N * w.B <= 2 ** 17:
        rate, threads, desc, _, _ = oracle_sample_rate(w, args.side_cpu_seconds)
        rate1, _, desc1, _, _ = oracle_sample_rate(w, args.side_cpu_seconds, threads=1)
        out["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": threads, "host_cores": os.cpu_count(),
                               "kind": "oracle", "sample": desc, "one_thread": {"value": rate1, "sample": desc1}}
    return out


def sources_sha():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_lsh_sketch_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def measure_e2e_pipelined(args, w, race, inp):
    """The e2e metric with the host link's two directions overlapped: the (b, h) problems are
    independent, so each is one public-API call pair (forward + backward, B = H = 1) on a
    compute stream, fed by pinned host -> device copies on a second stream and drained by
    device -> host copies on a third; events order the three per (b, h)."""
    import torch

    dev = inp["Q"].device
    B, H, N, d = inp["Q"].shape
    host_in = {k: torch.empty(inp[k].shape, dtype=inp[k].dtype, pin_memory=True) for k in ("Q", "K", "V", "dO")}
    host_out = [torch.empty(inp["Q"].shape, dtype=inp["Q"].dtype, pin_memory=True) for _ in range(4)]
    for k in host_in:
        host_in[k].copy_(inp[k])
    dev_in = {k: torch.empty_like(inp[k]) for k in ("Q", "K", "V", "dO")}
    outs = [torch.empty_like(inp["Q"]) for _ in range(4)]
    W = inp["W"]
    one = race.make_shape(1, 1, N, d, w.torch_dtype)
    ws = torch.empty(max(race.race_attn_workspace_bytes(one, w.L, w.P, w.causal, b) for b in (0, 1)),
                     dtype=torch.uint8, device=dev)
    st = torch.empty(race.race_attn_state_bytes(one, w.L, w.P, w.causal), dtype=torch.uint8, device=dev)
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    heads = [(b, h) for b in range(B) for h in range(H)]
    ev_in = [torch.cuda.Event() for _ in heads]
    ev_cmp = [torch.cuda.Event() for _ in heads]

    def sl(t, b, h):
        return t[b:b + 1, h:h + 1]

    def step():
        for i, (b, h) in enumerate(heads):
            with torch.cuda.stream(s_in):
                for k in dev_in:
                    sl(dev_in[k], b, h).copy_(sl(host_in[k], b, h), non_blocking=True)
                ev_in[i].record(s_in)
        for i, (b, h) in enumerate(heads):
            s_cmp.wait_event(ev_in[i])
            q, k_, v, g = (sl(dev_in[x], b, h) for x in ("Q", "K", "V", "dO"))
            o, dq, dk, dv = (sl(x, b, h) for x in outs)
            race.race_attn_fwd(q, k_, v, W, w.beta, w.L, w.P, w.causal, O=o, state=st, workspace=ws,
                               stream=s_cmp)
            race.race_attn_bwd(q, k_, v, W, w.beta, w.L, w.P, w.causal, g, O=o, dQ=dq, dK=dk, dV=dv,
                               state=st, workspace=ws, stream=s_cmp)
            ev_cmp[i].record(s_cmp)
            s_out.wait_event(ev_cmp[i])
            with torch.cuda.stream(s_out):
                for hd, dd in zip(host_out, outs):
                    sl(hd, b, h).copy_(sl(dd, b, h), non_blocking=True)

    step()
    torch.cuda.synchronize(dev)
    steps = max(1, args.e2e_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for _ in range(steps):
        s_in.wait_stream(s_out)  # a step starts when the previous one's results are home
        step()
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    nbytes = inp["Q"].numel() * inp["Q"].element_size()
    return {"value": w.B * w.N / (ms / 1000.0), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": 4 * nbytes, "d2h_bytes_per_step": 4 * nbytes,
            "schedule": "per (b, h): H2D, compute and D2H on three streams, overlapped"}


def measure_e2e(args, w, race, inp, state, workspace):
    """Same metric end to end through the public API: per step, pinned host -> device copies of
    Q, K, V, dO, forward + backward, and device -> host copies of O, dQ, dK, dV."""
    import torch

    dev = inp["Q"].device
    try:
        host_in = {k: torch.empty(inp[k].shape, dtype=inp[k].dtype, pin_memory=True) for k in ("Q", "K", "V", "dO")}
        host_out = [torch.empty(inp["Q"].shape, dtype=inp["Q"].dtype, pin_memory=True) for _ in range(4)]
    except Exception as exc:  # pinned memory unavailable
        return {"value": None, "unit": "tokens/s", "error": "pinned allocation failed: %s" % exc}
    for k in host_in:
        host_in[k].copy_(inp[k])
    dev_in = {k: torch.empty_like(inp[k]) for k in ("Q", "K", "V", "dO")}
    W = inp["W"]
    outs = [torch.empty_like(inp["Q"]) for _ in range(4)]
    stream = torch.cuda.current_stream(dev)

    def step():
        for k in dev_in:
            dev_in[k].copy_(host_in[k], non_blocking=True)
        race.race_attn_fwd(dev_in["Q"], dev_in["K"], dev_in["V"], W, w.beta, w.L, w.P, w.causal, O=outs[0],
                           state=state, workspace=workspace)
        race.race_attn_bwd(dev_in["Q"], dev_in["K"], dev_in["V"], W, w.beta, w.L, w.P, w.causal, dev_in["dO"],
                           O=outs[0], dQ=outs[1], dK=outs[2], dV=outs[3], state=state, workspace=workspace)
        for h, d in zip(host_out, outs):
            h.copy_(d, non_blocking=True)

    step()
    torch.cuda.synchronize(dev)
    steps = max(1, args.e2e_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    nbytes = inp["Q"].numel() * inp["Q"].element_size()
    return {"value": w.B * w.N / (ms / 1000.0), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": 4 * nbytes, "d2h_bytes_per_step": 4 * nbytes}


L2_BYTES = 129 * 2 ** 20
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12  # SMs x FP32 lanes x 2 (FMA) x max SM clock


def _timed(torch, dev, uuid, fn, warmup, steps, race):
    """Mean ms per call of fn over `steps` calls (CUDA events on the current stream, after
    `warmup` untimed calls), the clocks seen meanwhile and the library launches counted."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = race.race_attn_launch_count()
    with ClockSampler(uuid) as clk:
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / steps, clk.summary(), race.race_attn_launch_count() - n0


def run_row(args, w):
    """One JSON line for a widening row: the causal decode step or exact angular attention."""
    import torch

    import linear_lsh_sketch_gb300 as race

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    race.load_library()
    hbm_peak, _, peak_kind = load_peaks()
    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    common = {"n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
              "scaling": "weak", "vs_baseline": None, "data": "synthetic",
              "dtype": "bf16" if w.dtype == "bf16" else "f32"}
    LR = w.L << w.P
    if args.row == "decode":
        per_head = LR * (w.d + 1) * 4
        heads = max(args.heads, -(-2 * L2_BYTES // per_head))  # state at least twice L2: no flush
        q, k, v = (torch.randn((1, heads, 1, w.d), generator=g, device=dev).to(w.torch_dtype) for _ in range(3))
        W = torch.randn((w.L, w.P, w.d), generator=g, device=dev)
        state = torch.randn((1, heads, LR, w.d + 1), generator=g, device=dev).abs_()
        o = torch.empty_like(q)
        ms, clocks, launches = _timed(torch, dev, uuid, lambda: race.race_attn_decode(
            q, k, v, W, w.beta, w.L, w.P, state, o=o), args.warmup, args.steps, race)
        alg = heads * (2 * per_head + 4 * w.d * w.elem_bytes)  # state read + write; q, k, v, o
        gbs = alg / (ms / 1000.0) / 1e9
        line = dict(common, metric="RACE causal decode step tokens/s (one token per (b, h))",
                    value=heads / (ms / 1000.0), unit="tokens/s", ms_per_step=ms,
                    config={"workload": "decode, %d heads, d %d, (P, L) = (%d, %d), state %.2f GB > L2, "
                            "no flush" % (heads, w.d, w.P, w.L, heads * per_head / 1e9),
                            "heads": heads, "d": w.d, "P": w.P, "L": w.L, "io_dtype": w.dtype},
                    roofline={"bound": "hbm", "kernel": "decode", "achieved": gbs, "peak": hbm_peak,
                              "unit": "GB/s", "frac": gbs / hbm_peak, "peak_kind": peak_kind,
                              "algorithmic_bytes_per_launch": alg, "traffic": None},
                    clocks=clocks, gpu_launches=launches)
    else:
        n = args.tokens or 8192
        ws = w.scaled(N=n)
        Q, K, V = (torch.randn((ws.B, ws.H, n, ws.d), generator=g, device=dev).to(ws.torch_dtype)
                   for _ in range(3))
        O = torch.empty_like(Q)
        gamma = float(ws.P)
        ms, clocks, launches = _timed(torch, dev, uuid, lambda: race.race_attn_angular(
            Q, K, V, gamma, ws.causal, O=O), args.warmup, args.steps, race)
        pairs = ws.B * ws.H * (n * (n + 1) // 2 if ws.causal else n * n)
        flops = pairs * 8 * ws.d  # |a - b|^2, |a + b|^2 (6 d) and the weighted value sum (2 d)
        tf = flops / (ms / 1000.0) / 1e12
        line = dict(common, metric="exact angular attention (gamma = P) pair evaluations/s",
                    value=pairs / (ms / 1000.0), unit="pairs/s", ms_per_step=ms,
                    config={"workload": "angular attention, B %d H %d N %d d %d gamma %g causal %s" %
                            (ws.B, ws.H, n, ws.d, gamma, ws.causal), "io_dtype": ws.dtype,
                            "l2": "O(N^2) arithmetic on L2-resident rows; no flush"},
                    roofline={"bound": "alu", "kernel": "angular", "achieved": tf, "peak": FP32_ALU_TFLOPS,
                              "unit": "TFLOP/s", "frac": tf / FP32_ALU_TFLOPS,
                              "peak_kind": "FP32 CUDA-core FMA rate from unit counts and the 2070 MHz clock",
                              "flops_per_launch": flops, "traffic": None},
                    clocks=clocks, gpu_launches=launches)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--e2e-steps", type=int, default=2)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override N (sequence length) of the workload, e.g. for a small profiling capture")
    ap.add_argument("--dbeta", action="store_true", help="the backward also writes d(loss)/d(beta)")
    ap.add_argument("--dW", action="store_true", help="the backward also writes d(loss)/d(W)")
    ap.add_argument("--row", choices=["step", "decode", "angular"], default="step",
                    help="decode: one causal decode step per (b, h) of --heads heads; angular: exact angular "
                         "attention at the workload's d and --tokens (default 8192) tokens")
    ap.add_argument("--heads", type=int, default=1024, help="(b, h) problems of the decode batch")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads timed after the headline one (the `configs` key)")
    ap.add_argument("--side-steps", type=int, default=10, help="timed steps of each other workload")
    ap.add_argument("--side-cpu-seconds", type=float, default=4.0,
                    help="seconds of oracle time per host-baseline sample of the small workloads")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # timing rule: at least three untimed warm-up steps
    from linear_lsh_sketch_gb300.workloads import CONFIGS
    w = CONFIGS[args.workload]
    if args.tokens:
        w = w.scaled(N=args.tokens, name="%s_N%d" % (w.name, args.tokens))
    if args.row != "step":
        run_row(args, w)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
