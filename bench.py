#!/usr/bin/env python
"""Benchmark: batched Nystrom decode throughput (group-steps/s) on GB300.

Default workload ``batch64``: 64 sequences x 28 layers x 8 KV groups = 14336
group states (heads_per_kv=2, d=dv=128, m=32, w=128, sink=4, Aggregate),
sealed on a 256-token synthetic prompt, then decoded with one
``nys_step_batch`` launch per token over all 14336 groups.  One benchmark
step = one such token launch (all of the decode path: ring insert/evict, far
insert, near and far read, rectifier, joint division).  The seal is timed once
and reported beside it.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
on the same workload and metric instead.  Under torchrun each rank runs an
independent replica of the workload on its own GPU (the states shard with no
exchange), and ``value`` counts the group-steps of all ranks.
"""
from __future__ import annotations

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    __import__("os").environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("Nyström decode group-steps/s at batch 64, 28 layers; "
          "achieved HBM GB/s vs peak")
UNIT = "group-steps/s"
FALLBACK_HBM_GBS = 6800.0
STEP_SOURCE = os.path.join(ROOT, "streaming_nystr_landmark_gb300", "csrc", "nys_step_tma.cu")
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "step_kernel_batch64.txt")


def algorithmic_bytes(wl) -> int:
    """Bytes one group-step must move at minimum, counting the method's own
    fp32 state (nystrom.rs, NystromGroup / NystromHead): the window read, the
    sinks, K~, the new k/v read and written into the ring; per head Q~, M,
    T^ read and written, Z^ and m_max read and written, q and the output."""
    f, H, m, w, s, d, dv = 4, wl.heads_per_kv, wl.m, wl.w, wl.sink, wl.d, wl.dv
    shared = f * (w * (d + dv) + s * (d + dv) + m * d + 2 * (d + dv))
    head = f * (m * d + m * m + 2 * m * dv + 4 * m + d + dv)
    return shared + H * head


def state_overhead_bytes(wl) -> int:
    """Bytes per group-step beyond the method's fp32 state that this
    implementation moves: the compensation (low) parts of the far
    accumulators, T^ lo (bf16) and Z^ lo (fp32), each read and written."""
    H, m, dv = wl.heads_per_kv, wl.m, wl.dv
    return H * (2 * 2 * m * dv + 2 * 4 * m)


def workload_config(wl, extra=None):
    cfg = {
        "workload": (f"{wl.name}: {wl.seqs} seq x {wl.layers} layers x "
                     f"{wl.kv_groups} KV groups = {wl.n_groups} group states, "
                     f"heads_per_kv={wl.heads_per_kv}, d={wl.d}, dv={wl.dv}, "
                     f"m={wl.m}, w={wl.w}, sink={wl.sink}, "
                     f"rect={'aggregate' if wl.rect == 0 else 'fm'}, "
                     f"prompt t={wl.t}"),
        "groups_per_launch": wl.n_groups,
        "heads_per_kv": wl.heads_per_kv,
        "prompt_len": wl.t,
        "inputs": "synthetic fp32 N(0,1), k mean " + wl.k_mean,
        "l2": ("state per launch far above the 126 MB L2 (no flush needed)"
               if (algorithmic_bytes(wl) + state_overhead_bytes(wl)) * wl.n_groups > 512e6 else
               "state fits in L2: latency-bound, roofline fraction not meaningful"),
    }
    if extra:
        cfg.update(extra)
    return cfg


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic():
    """dram read+write bytes per launch of the step kernel from the committed
    ncu summary, or None when that summary was taken on another version of
    the kernel source."""
    try:
        src = hashlib.sha256(open(STEP_SOURCE, "rb").read()).hexdigest()[:16]
        fields = {}
        for line in open(TRAFFIC_PROFILE):
            if ":" in line:
                key, val = line.split(":", 1)
                fields[key.strip()] = val.strip()
        if fields.get("step_source_sha256_16") != src:
            return None
        return int(fields["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="nys_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap")
        reasons = sorted({n for r in rows for n, val in zip(names, r[5:9])
                          if val.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ dist
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_rate(world, groups_per_rank, steps, seconds):
    """Whole-job group-steps/s: every rank steps its own replica of the
    workload, and the job takes as long as its slowest rank (`seconds` is the
    max over ranks)."""
    return world * groups_per_rank * steps / seconds


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle
def host_cores() -> int:
    """Cores this process may run on (the affinity mask, else cpu_count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_decode(wl, groups, steps, warmup, budget_s, start=None):
    """Seal `groups` with the fp64 oracle (untimed), wait at `start` if
    given, then time decode tokens round-robin over them.  Returns
    (group_steps, seconds, tokens_timed)."""
    from oracle import NystromOracle
    from streaming_nystr_landmark_gb300.workloads import GroupInputs
    states = []
    for g in groups:
        gi = GroupInputs(wl, g)
        q, k, v = gi.prompt()
        o = NystromOracle(wl.m, wl.w, wl.sink, wl.heads_per_kv, wl.rect)
        o.prefill(q, k, v)
        states.append((o, gi))
    n = 0
    for _ in range(warmup):
        for o, gi in states:
            o.step(*gi.token(n))
        n += 1
    if start is not None:
        start.wait()
    t0 = time.perf_counter()
    done = 0
    while done < steps:
        for o, gi in states:
            o.step(*gi.token(n))
        n += 1
        done += 1
        if budget_s is not None and time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done * len(groups), dt, done


def _oracle_worker(wl, groups, steps, warmup, budget_s, start, results):
    results.put(_oracle_decode(wl, groups, steps, warmup, budget_s, start))


def time_oracle(wl, groups, steps, warmup=0, budget_s=None, procs=1):
    """The oracle's decode rate on `procs` host cores: the groups are dealt
    round-robin to `procs` processes (spawned, one numpy thread each), every
    process seals its groups untimed, all start decoding together, and the
    rate is all group-steps over the slowest process's time.  Returns
    (group_steps, seconds, tokens_timed_by_the_slowest)."""
    if procs <= 1:
        return _oracle_decode(wl, groups, steps, warmup, budget_s)
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    start = ctx.Barrier(procs)
    results = ctx.Queue()
    workers = [ctx.Process(target=_oracle_worker,
                           args=(wl, groups[i::procs], steps, warmup, budget_s,
                                 start, results))
               for i in range(procs)]
    for w in workers:
        w.start()
    got = [results.get() for _ in workers]
    for w in workers:
        w.join()
    gs = sum(r[0] for r in got)
    dt = max(r[1] for r in got)
    return gs, dt, min(r[2] for r in got)


def oracle_groups(wl, count):
    """`count` distinct groups spread evenly over the workload."""
    count = max(1, min(count, wl.n_groups))
    return sorted({round(i * (wl.n_groups - 1) / max(count - 1, 1))
                   for i in range(count)})


def run_reference(args, wl):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    cores = host_cores()
    # Enough groups per core that every process times >= ~256 group-steps
    # even for a small --steps (short windows are dominated by start skew).
    per_core = min(32, max(args.ref_groups, -(-256 // max(args.steps, 1))))
    groups = oracle_groups(wl, cores * per_core)
    gs, dt, done = time_oracle(wl, groups, args.steps, args.warmup,
                               budget_s=args.ref_budget, procs=cores)
    value = gs / dt
    sample = (f"{len(groups)} of {wl.n_groups} groups ({per_core} per "
              f"core), sealed untimed on the t={wl.t} prompt, then "
              f"{args.warmup} untimed + at least {done} timed decode tokens "
              f"each (at most {args.steps}, {args.ref_budget:.0f} s budget); "
              f"fp64 numpy oracle (streaming form), {cores} processes x 1 "
              "thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": done, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / max(done, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(wl, {"sampled_groups": len(groups)}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ours
def run_ours(args, wl):
    import torch
    from streaming_nystr_landmark_gb300.nys import NystromStates
    from streaming_nystr_landmark_gb300.workloads import DeviceFill

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    G, H = wl.n_groups, wl.heads_per_kv
    st = NystromStates(wl.m, wl.w, wl.sink, H, wl.d, wl.dv, G, wl.rect, dev)
    fill = DeviceFill(wl, dev, seed=1000 + rank)

    # ---- seal (timed once)
    q = torch.empty((G, H, wl.t, wl.d), device=dev)
    k = torch.empty((G, wl.t, wl.d), device=dev)
    v = torch.empty((G, wl.t, wl.dv), device=dev)
    fill.prompt_into(q, k, v)
    seal_times = []
    for _ in range(3):   # the first seal is cold, the others warm
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        s0.record()
        st.seal(q, k, v)
        s1.record()
        torch.cuda.synchronize(dev)
        seal_times.append(s0.elapsed_time(s1))
    seal_ms, seal_warm_ms = seal_times[0], min(seal_times[1:])
    del q, k, v
    torch.cuda.empty_cache()

    # ---- decode inputs resident in HBM before timing
    total = args.warmup + args.steps
    pool = min(total, args.pool)
    tq = torch.empty((pool, G, H, wl.d), device=dev)
    tk = torch.empty((pool, G, wl.d), device=dev)
    tv = torch.empty((pool, G, wl.dv), device=dev)
    chunk = 64
    for c0 in range(0, pool, chunk):
        c1 = min(pool, c0 + chunk)
        fill.tokens_into(tq[c0:c1], tk[c0:c1], tv[c0:c1])
    out = torch.empty((G, H, wl.dv), device=dev)
    step_i = 0
    for _ in range(args.warmup):
        j = step_i % pool
        st.step(tq[j], tk[j], tv[j], out)
        step_i += 1
    torch.cuda.synchronize(dev)
    barrier(world)

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0.record()
    for _ in range(args.steps):
        j = step_i % pool
        st.step(tq[j], tk[j], tv[j], out)
        step_i += 1
    e1.record()
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    dt = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    value = aggregate_rate(world, G, args.steps, dt)
    launch_s = dt / args.steps
    finite = bool(torch.isfinite(out).all().item())
    del tq, tk, tv

    # ---- end to end through pinned host buffers
    pe = 4
    hq = [torch.empty((G, H, wl.d), pin_memory=True) for _ in range(pe)]
    hk = [torch.empty((G, wl.d), pin_memory=True) for _ in range(pe)]
    hv = [torch.empty((G, wl.dv), pin_memory=True) for _ in range(pe)]
    for i in range(pe):
        hq[i].normal_()
        hk[i].normal_()
        hv[i].normal_()
    hout = torch.empty((G, H, wl.dv), pin_memory=True)
    pipe = st.host_pipeline()
    e2e_steps = args.steps
    for i in range(2):
        pipe.submit(hq[i], hk[i], hv[i], hout)
    pipe.synchronize()
    barrier(world)
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record()
    pipe.copy.wait_event(e2)  # the first token's input copy starts the clock
    for i in range(e2e_steps):
        pipe.submit(hq[i % pe], hk[i % pe], hv[i % pe], hout)
    # The timed region ends when the last token's outputs are on the host.
    pipe.down.wait_stream(torch.cuda.current_stream(dev))
    e3.record(pipe.down)
    pipe.synchronize()
    barrier(world)
    dt_e2e = max_over_ranks(e2.elapsed_time(e3) / 1e3, world, dev)
    e2e = {"value": aggregate_rate(world, G, e2e_steps, dt_e2e), "unit": UNIT,
           "h2d_bytes_per_step": 4 * G * (H * wl.d + wl.d + wl.dv),
           "d2h_bytes_per_step": 4 * G * H * wl.dv}
    st.close()

    if rank != 0:
        return
    peak, peak_kind = measured_peak()
    alg, over = algorithmic_bytes(wl), state_overhead_bytes(wl)
    per_launch = alg * G
    achieved = per_launch / launch_s / 1e9
    achieved_all = (alg + over) * G / launch_s / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": profiled_traffic(),
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_group_step": alg,
                "algorithmic_bytes_per_launch": per_launch,
                "state_overhead_bytes_per_group_step": over,
                "achieved_incl_state_overhead": achieved_all,
                "frac_incl_state_overhead": achieved_all / peak,
                "kernel": "step_tma_kernel (one persistent launch per token)"}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cores = host_cores()
        groups = oracle_groups(wl, 3 * cores)
        gs, cdt, done = time_oracle(wl, groups, 10 ** 9, budget_s=args.cpu_budget,
                                    procs=cores)
        g1 = oracle_groups(wl, 3)
        gs1, cdt1, done1 = time_oracle(wl, g1, 10 ** 9, budget_s=args.cpu_budget / 2)
        cpu = {"value": gs / cdt, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": (f"{len(groups)} of {G} groups (3 per core) sealed untimed, "
                          f"then >= {done} decode tokens each in {cdt:.1f} s; fp64 numpy "
                          f"oracle (streaming form), {cores} processes x 1 thread"),
               "single_core": {"value": gs1 / cdt1, "cores": 1,
                               "sample": (f"{len(g1)} groups, {done1} decode tokens each "
                                          f"in {cdt1:.1f} s, 1 thread")}}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(wl, {"parallelism": f"replicas x{world}",
                                       "seal_ms": seal_ms,
                                       "seal_warm_ms": seal_warm_ms,
                                       "decode_input_pool": pool,
                                       "outputs_finite": finite}),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if world == 1 and not args.no_secondary:
        # Driver-visible figures of two other paths (not part of `value`).
        line["secondary"] = {"long_decode": secondary_long_decode(dev),
                             "per_layer_graph": secondary_layers_graph(dev)}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def secondary_long_decode(dev, steps=300, warmup=5):
    """The eight-head long-context decode (512 groups: 128 sequences x 4 KV
    heads, H=8, m=64, d=128), timed like the main line.  The decode state's
    shape and byte count do not depend on the prompt length once m_eff = m,
    so a 1024-token prompt stands in for the 32K one (the seal of the full
    prompt is timed by --mode seal --workload long)."""
    import torch
    from streaming_nystr_landmark_gb300.nys import NystromStates
    from streaming_nystr_landmark_gb300.workloads import WORKLOADS, DeviceFill
    wl = WORKLOADS["long"].with_(t=1024)
    G, H = wl.n_groups, wl.heads_per_kv
    st = NystromStates(wl.m, wl.w, wl.sink, H, wl.d, wl.dv, G, wl.rect, dev)
    fill = DeviceFill(wl, dev, seed=3000)
    q = torch.empty((G, H, wl.t, wl.d), device=dev)
    k = torch.empty((G, wl.t, wl.d), device=dev)
    v = torch.empty((G, wl.t, wl.dv), device=dev)
    fill.prompt_into(q, k, v)
    st.seal(q, k, v)
    del q, k, v
    pool = 64
    tq = torch.empty((pool, G, H, wl.d), device=dev)
    tk = torch.empty((pool, G, wl.d), device=dev)
    tv = torch.empty((pool, G, wl.dv), device=dev)
    fill.tokens_into(tq, tk, tv)
    out = torch.empty((G, H, wl.dv), device=dev)
    for i in range(warmup):
        st.step(tq[i % pool], tk[i % pool], tv[i % pool], out)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record()
    for i in range(steps):
        st.step(tq[i % pool], tk[i % pool], tv[i % pool], out)
    e1.record()
    torch.cuda.synchronize(dev)
    st.close()
    ms = e0.elapsed_time(e1) / steps
    peak, _ = measured_peak()
    alg, over = algorithmic_bytes(wl), state_overhead_bytes(wl)
    return {"workload": ("long decode: 128 seq x 4 KV groups = 512 group states, "
                         "heads_per_kv=8, d=dv=128, m=64, w=128, sink=4 (1024-token "
                         "prompt: same decode state as the 32K one)"),
            "steps": steps, "ms_per_step": ms, "group_steps_per_s": G / (ms / 1e3),
            "frac": alg * G / (ms / 1e3) / 1e9 / peak,
            "frac_incl_state_overhead": (alg + over) * G / (ms / 1e3) / 1e9 / peak}


def secondary_layers_graph(dev, reps=25):
    """batch64 decoded as a model runs it: 28 per-layer handles (512 groups
    each), one launch per layer per token, 8 tokens per CUDA graph replay."""
    import torch
    from streaming_nystr_landmark_gb300.nys import NystromStates
    from streaming_nystr_landmark_gb300.workloads import WORKLOADS, DeviceFill
    wl = WORKLOADS["batch64"]
    L, H, per = wl.layers, wl.heads_per_kv, wl.seqs * wl.kv_groups
    fill = DeviceFill(wl.with_(layers=1), dev, seed=4000)
    layers = []
    for _ in range(L):
        st = NystromStates(wl.m, wl.w, wl.sink, H, wl.d, wl.dv, per, wl.rect, dev)
        q = torch.empty((per, H, wl.t, wl.d), device=dev)
        k = torch.empty((per, wl.t, wl.d), device=dev)
        v = torch.empty((per, wl.t, wl.dv), device=dev)
        fill.prompt_into(q, k, v)
        st.seal(q, k, v)
        layers.append(st)
        del q, k, v
    T = 8
    tq = torch.empty((T, L, per, H, wl.d), device=dev)
    tk = torch.empty((T, L, per, wl.d), device=dev)
    tv = torch.empty((T, L, per, wl.dv), device=dev)
    for i in range(T):
        fill.tokens_into(tq[i], tk[i], tv[i])
    out = torch.empty((L, per, H, wl.dv), device=dev)

    def token(i):
        for l, st in enumerate(layers):
            st.step(tq[i, l], tk[i, l], tv[i, l], out[l])

    for i in range(3):
        token(i % T)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(T):
            token(i)
    graph.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    for st in layers:
        st.close()
    ms = e0.elapsed_time(e1) / (reps * T)
    return {"workload": ("batch64 as 28 per-layer launches per token (512 groups each), "
                         "replayed from a CUDA graph"),
            "tokens": reps * T, "ms_per_token": ms,
            "group_steps_per_s": L * per / (ms / 1e3), "launches_per_token": L}


def run_layers(args, wl):
    """Decode as a model runs it: one handle per layer (batch x KV groups
    each), one launch per layer per token -- 28 dependent launches instead of
    one fused launch -- eagerly or replayed from a CUDA graph."""
    import torch
    from streaming_nystr_landmark_gb300.nys import NystromStates
    from streaming_nystr_landmark_gb300.workloads import DeviceFill

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    L, H = wl.layers, wl.heads_per_kv
    per = wl.seqs * wl.kv_groups
    lw = wl.with_(layers=1)
    layers = []
    fill = DeviceFill(lw, dev, seed=2000 + rank)
    seal_ms = 0.0
    for _ in range(L):
        st = NystromStates(wl.m, wl.w, wl.sink, H, wl.d, wl.dv, per, wl.rect, dev)
        q = torch.empty((per, H, wl.t, wl.d), device=dev)
        k = torch.empty((per, wl.t, wl.d), device=dev)
        v = torch.empty((per, wl.t, wl.dv), device=dev)
        fill.prompt_into(q, k, v)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        st.seal(q, k, v)
        b.record()
        torch.cuda.synchronize(dev)
        seal_ms += a.elapsed_time(b)
        del q, k, v
        layers.append(st)
    torch.cuda.empty_cache()
    T = 8  # distinct decode tokens in the pool (and in one graph)
    tq = torch.empty((T, L, per, H, wl.d), device=dev)
    tk = torch.empty((T, L, per, wl.d), device=dev)
    tv = torch.empty((T, L, per, wl.dv), device=dev)
    for i in range(T):
        fill.tokens_into(tq[i], tk[i], tv[i])
    out = torch.empty((L, per, H, wl.dv), device=dev)

    def token(i):
        for l, st in enumerate(layers):
            st.step(tq[i, l], tk[i, l], tv[i, l], out[l])

    for i in range(args.warmup):
        token(i % T)
    torch.cuda.synchronize(dev)
    graph = None
    if args.mode == "layers-graph":
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(T):
                token(i)
        graph.replay()
        torch.cuda.synchronize(dev)
    reps = max(1, args.steps // T) if graph is not None else args.steps
    steps = reps * T if graph is not None else args.steps
    barrier(world)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    if graph is not None:
        for _ in range(reps):
            graph.replay()
    else:
        for i in range(steps):
            token(i % T)
    e1.record()
    host_s = time.perf_counter() - t0
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    dt = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    for st in layers:
        st.close()
    if rank != 0:
        return
    G = L * per
    peak, _ = measured_peak()
    launch_s = dt / steps
    achieved = algorithmic_bytes(wl) * G / launch_s / 1e9
    line = {
        "metric": METRIC, "value": aggregate_rate(world, G, steps, dt), "unit": UNIT,
        "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * launch_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(wl, {
            "mode": args.mode, "launches_per_token": L,
            "groups_per_launch": per, "seal_ms_all_layers": seal_ms,
            "host_enqueue_ms_per_token": 1e3 * host_s / steps,
            "decode_input_pool": T}),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None},
        "gpu_launches": steps * L,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_seal(args, wl):
    """Time the seal: one uniform batch at the workload's prompt length, and
    one ragged batch of the same groups whose lengths are spread uniformly
    over [t/2, 3t/2] (about the same number of prompt tokens)."""
    import numpy as np
    import torch
    from streaming_nystr_landmark_gb300.nys import NystromStates

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    G, H = wl.n_groups, wl.heads_per_kv
    gen = torch.Generator(device=dev)
    gen.manual_seed(77)
    rng = np.random.default_rng(77)
    ts = rng.integers(wl.t // 2, 3 * wl.t // 2 + 1, size=G).astype(np.int32)
    ts = np.maximum(ts, wl.w + wl.sink + 9)
    res = {}
    for kind, total in (("uniform", G * wl.t), ("ragged", int(ts.sum()))):
        st = NystromStates(wl.m, wl.w, wl.sink, H, wl.d, wl.dv, G, wl.rect, dev)
        q = torch.randn((H * total, wl.d), device=dev, generator=gen)
        k = torch.randn((total, wl.d), device=dev, generator=gen)
        v = torch.randn((total, wl.dv), device=dev, generator=gen)
        times = []
        for rep in range(args.warmup + 3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            if kind == "uniform":
                st.seal(q.view(G, H, wl.t, wl.d), k.view(G, wl.t, wl.d),
                        v.view(G, wl.t, wl.dv))
            else:
                st.seal_ragged(ts.tolist(), q, k, v)
            b.record()
            torch.cuda.synchronize(dev)
            if rep >= args.warmup:
                times.append(a.elapsed_time(b))
        res[kind] = {"ms": min(times), "prompt_tokens": total,
                     "tokens_per_s": total / (min(times) / 1e3)}
        st.close()
        del q, k, v
        torch.cuda.empty_cache()
    # Roofline of the uniform seal: its fp32-equivalent arithmetic (replay
    # logits and P V over the evicted keys, the pinv's landmark products,
    # A^T A, Cholesky and solves) against the fp32 FMA peak derived from
    # the unit counts and the maximum clock (SMs x 128 lanes x 2 x 2.07 GHz).
    m_eff = min(max(wl.t // 8, 4), wl.m)
    n_ev = max(wl.t - wl.w - wl.sink, 0)
    flop_head = (n_ev * m_eff * 2 * (wl.d + wl.dv)
                 + 2 * m_eff * m_eff * wl.d + m_eff ** 3 + m_eff ** 3 // 3 + 2 * m_eff ** 3)
    seal_flop = G * H * flop_head
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = sms * 128 * 2 * 2.07e9 / 1e12
    achieved = seal_flop / (res["uniform"]["ms"] / 1e3) / 1e12
    roofline = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": None,
                "peak_source": f"derived: {sms} SMs x 128 fp32 lanes x 2 x 2.07 GHz",
                "flop_per_seal": seal_flop,
                "note": "fp32-equivalent work; the replay runs on tensor cores for prompts "
                        "folding >= 256 keys, the pinv's f64-accurate parts in f64 and "
                        "double-float"}
    line = {"metric": "Nyström seal ms per batch (uniform vs ragged prompts)",
            "value": res["ragged"]["ms"], "unit": "ms", "higher_is_better": False,
            "n_gpus": 1, "steps": 3, "warmup": args.warmup, "dtype": "f32+f64",
            "data": "synthetic", "roofline": roofline,
            "config": workload_config(wl, {"ragged_t_range": [int(ts.min()), int(ts.max())],
                                           "uniform": res["uniform"],
                                           "ragged": res["ragged"]})}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_seal_rate(wl, args.cpu_budget)
    print(json.dumps(line), flush=True)


def oracle_seal_rate(wl, budget_s):
    """The fp64 oracle's seal (prefill) rate in prompt tokens per second:
    whole groups sealed one after another, from the host-drawn inputs of
    groups 0, 1, ..., until the time budget is spent (at least one group)."""
    from oracle import NystromOracle
    from streaming_nystr_landmark_gb300.workloads import GroupInputs
    tokens, spent, groups = 0, 0.0, 0
    while groups == 0 or (spent < budget_s and groups < wl.n_groups):
        q, k, v = GroupInputs(wl, groups).prompt()
        o = NystromOracle(m=wl.m, w=wl.w, sink=wl.sink, heads=wl.heads_per_kv, rect=wl.rect,
                          d=wl.d, dv=wl.dv)
        t0 = time.perf_counter()
        o.prefill(q, k, v)
        spent += time.perf_counter() - t0
        tokens += wl.t
        groups += 1
    return {"value": tokens / spent, "unit": "prompt tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{groups} group(s) of {wl.t} tokens sealed in {spent:.1f} s; fp64 numpy "
                      f"oracle (streaming form), 1 thread"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="batch64")
    ap.add_argument("--pool", type=int, default=256,
                    help="distinct decode-token batches kept in HBM (cycled)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the long-context and per-layer graph figures")
    ap.add_argument("--ref-groups", type=int, default=3,
                    help="oracle groups per host core in --impl reference")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="seconds of timed oracle decode in --impl reference")
    ap.add_argument("--mode", choices=("fused", "layers", "layers-graph", "seal"),
                    default="fused",
                    help="fused: one launch per token over every layer's groups; "
                         "layers: one launch per layer per token; layers-graph: "
                         "the same launches replayed from a CUDA graph")
    ap.add_argument("--groups", type=int, default=0,
                    help="override the workload's group count (profiling on a "
                         "smaller case); 0 keeps the workload's own")
    ap.add_argument("--prompt", type=int, default=0,
                    help="override the workload's prompt length (profiling the "
                         "decode step without the full prompt); 0 keeps it")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    from streaming_nystr_landmark_gb300.workloads import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.groups:
        wl = wl.with_(name=f"{wl.name}[{args.groups} groups]", seqs=1, layers=1,
                      kv_groups=args.groups)
    if args.prompt:
        wl = wl.with_(name=f"{wl.name}[prompt {args.prompt}]", t=args.prompt)
    if args.impl == "reference":
        run_reference(args, wl)
    elif args.mode == "seal":
        run_seal(args, wl)
    elif args.mode != "fused":
        run_layers(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
