"""Benchmark of the walk-resident serial draft head.

Metric: microseconds per gamma = 16 draft walk (B = 1, V = 151,936, r = 256, greedy Markov head) and the
fraction of the on-chip-bandwidth roofline. One "step" of this benchmark is one whole walk (one kernel
launch) over synthetic inputs that are resident in HBM; the L2 cache is flushed (256 MB write) before
every timed walk, outside the timed interval. Per-walk times come from CUDA events on the walk's stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

With N > 1 (torchrun) every rank runs an independent replica (no data-path collective); the job's value
is the slowest rank's timed total divided by all walks of all ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "us per gamma=16 draft walk (B=1, V=152k, greedy) & % of on-chip-BW roofline"
DEFAULT_WORKLOAD = "markov_v151936_r256_b1_g16"

# Per-SM on-chip figures for the roofline (bytes per SM clock), measured live by the probe library when it
# loads; these are the fallbacks (shared memory: 32 banks x 4 B; tensor memory: tcgen05.ld measured on GB300).
SMEM_B_PER_CLK = 128.0
TMEM_B_PER_CLK = 428.0
TMEM_BYTES = 128 * 512 * 4
# Registers this kernel family can dedicate to W: one 16-row group per warp, 12 warps.
RF_W_BYTES_CAP = 12 * 16 * 512


def recorded_traffic():
    """DRAM bytes per walk launch from the committed ncu summary, if it was taken on the current kernel source."""
    import hashlib
    import re
    src = os.path.join(ROOT, "speculative_decoding_serial_gb300", "csrc", "walk_kernel.cuh")
    prof = os.path.join(ROOT, "profiles", "walk_kernel_markov_v151936_r256_b1_g16.md")
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        m = re.search(r"traffic_bytes_per_launch: (\d+) \(walk_kernel.cuh sha256 prefix ([0-9a-f]+)\)",
                      open(prof).read())
        if m and m.group(2) == h:
            return int(m.group(1))
    except OSError:
        pass
    return None


def probe_onchip():
    """Shared/tensor-memory bytes per SM clock, mma.sync and thin-N tcgen05.mma clocks per op, grid-exchange clocks,
    and the clocks of tcgen05.mma and mma.sync run alone and side by side (do they share the tensor pipe)."""
    import ctypes
    from speculative_decoding_serial_gb300 import build
    try:
        L = ctypes.CDLL(build.PROBE_LIB)
        out = (ctypes.c_double * 9)()
        rc = L.whead_probe_onchip(out)
        if rc != 0:
            return None
        return {"smem_b_per_clk": out[0], "tmem_b_per_clk": out[1], "mma_m16n8k16_clk_per_sm": out[2],
                "grid_exchange_clk": out[3], "tcgen05_m128n16k16_clk_1_issuer": out[4],
                "tcgen05_m128n16k16_clk_4_issuers": out[5],
                "tcgen05_beside_mma_sync_clk": {"tcgen05_alone": out[6], "mma_sync_alone": out[7],
                                                "mma_sync_with_tcgen05": out[8]}}
    except OSError:
        return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        # raw samples go to WHEAD_CLOCK_LOG_DIR when set (to keep them with other run output), else a temp dir
        import tempfile
        log_dir = os.environ.get("WHEAD_CLOCK_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"whead_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", self.gpu_id, "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        smax = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons, "samples": len(rows)}


def gpu_selector(torch, dev):
    try:
        p = torch.cuda.get_device_properties(dev)
        bus = getattr(p, "pci_bus_id", None)
        dom = getattr(p, "pci_domain_id", None)
        devid = getattr(p, "pci_device_id", None)
        if bus is not None and dom is not None and devid is not None:
            return f"{dom:08x}:{bus:02x}:{devid:02x}.0"
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[dev]
    return str(dev)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_walk_time(d, gamma_sample, repeats, threads=1):
    """Wall time of the oracle on `repeats` samples of `gamma_sample` steps of the workload, with the rows of each
    step's projection split over `threads` host threads (the results do not depend on the count)."""
    from oracle import oracle as O
    base = d["base"][:, :gamma_sample].copy()
    O.set_threads(threads)
    try:
        t = time.perf_counter()
        for _ in range(repeats):
            O.walk(d["kind"], d["W"], d["E"], base, d["s0"], A=d["A"], c=d["c"], T=d["T"], want_gap=False)
        return (time.perf_counter() - t) / repeats
    finally:
        O.set_threads(1)


def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline(d, gamma, name, seconds):
    """The oracle timed on this host: on all allotted cores (the reported value) and on one thread, each for
    about half of `seconds` of wall time."""
    from oracle import oracle as O
    cores = O.set_threads(host_cores())
    O.set_threads(1)
    out = {}
    for label, threads in (("all", cores), ("one", 1)):
        one = oracle_walk_time(d, gamma, 1, threads)
        reps = max(1, min(200, int(math.ceil(seconds / 2 / max(one, 1e-3)))))
        out[label] = (oracle_walk_time(d, gamma, reps, threads), reps, threads)
    per, reps, threads = out["all"]
    per1, reps1, _ = out["one"]
    return {"value": per * 1e6, "unit": "us/walk", "cores": threads, "kind": "oracle",
            "sample": f"{reps} full walks of {name} on {threads} host threads (rows of each step split over "
                      f"the threads); single thread: {reps1} walks",
            "single_thread": {"value": per1 * 1e6, "unit": "us/walk", "cores": 1}}


def trace_phases(torch, head, base, s0, tok, w, plan, flush, stream, dev, walks=20, advance=True):
    """Per-step phase durations from the kernel's phase stamps (median over walks, steps 1.., and CTAs).
    advance=False: a fixed-latent walk, whose steps end at the exchange (no advance stamp)."""
    gamma, G = w["gamma"], plan["grid"]
    S = 4 + 8 * gamma
    buf = torch.zeros((G, S), dtype=torch.int64, device=dev)
    head.set_trace(buf)
    rows = []
    for _ in range(walks):
        flush.zero_()
        head.walk(base, s0, T=w["T"], seed=0, out_tokens=tok)
        torch.cuda.synchronize(dev)
        rows.append(buf.cpu().numpy().copy())
    head.set_trace(None)
    import numpy as np
    a = np.stack(rows).astype(np.int64)            # walks x G x S
    half = S // 2
    clk, ns = a[:, :, :half], a[:, :, half:]
    st = lambda t, i: 2 + 4 * t + i
    proj, exch, adv, skew, step_ns, step_clk = [], [], [], [], [], []
    for t in range(1, gamma):
        proj.append(clk[:, :, st(t, 1)] - clk[:, :, st(t, 0)])
        exch.append(clk[:, :, st(t, 2)] - clk[:, :, st(t, 1)])
        if advance and t < gamma - 1:  # the last step has no advance unless the states are asked for
            adv.append(clk[:, :, st(t, 3)] - clk[:, :, st(t, 2)])
        done = ns[:, :, st(t, 1)]
        skew.append(done.max(axis=1) - done.min(axis=1))
        step_ns.append(ns[:, :, st(t, 0)].max(axis=1) - ns[:, :, st(t - 1, 0)].max(axis=1))
        step_clk.append(clk[:, :, st(t, 0)] - clk[:, :, st(t - 1, 0)])
    med = lambda x: float(np.median(np.concatenate([np.ravel(v) for v in x]))) if x else None
    p90 = lambda x: float(np.percentile(np.concatenate([np.ravel(v) for v in x]), 90)) if x else None
    entry_ns = ns[:, :, 1] - ns[:, :, 0]
    last = st(gamma - 1, 2)  # every walk stamps the end of its last exchange
    span_clk, span_ns = clk[:, :, last] - clk[:, :, 0], ns[:, :, last] - ns[:, :, 0]
    ok = span_ns > 0
    mhz = float(np.median(span_clk[ok] / span_ns[ok] * 1e3)) if ok.any() else None
    phase_sum = med(proj) + med(exch) + (med(adv) if adv else 0.0) if proj else None
    return {"walks": walks, "kernel_sm_mhz": mhz, "proj_select_clk": med(proj), "proj_select_clk_p90": p90(proj),
            "exchange_clk": med(exch), "advance_clk": med(adv), "step_clk": med(step_clk),
            "arrival_skew_ns": med(skew), "step_ns": med(step_ns), "entry_ns_median": float(np.median(entry_ns)),
            "entry_ns_max": float(np.median(entry_ns.max(axis=1))),
            "exchange_share": (med(exch) / phase_sum) if proj else None}


def central_mean(xs, cut=0.1):
    """Mean of the middle 80 % of a list of walk times. CUDA event times advance in steps of about a microsecond,
    so a median lands on one of those steps; the mean of many walks, outliers cut, resolves below a step."""
    v = sorted(xs)
    k = int(len(v) * cut)
    v = v[k:len(v) - k] or v
    return sum(v) / len(v)


def fit_line(xs, ys):
    """Least-squares slope and intercept (Fig. 11's method: slope = per-step cost, intercept = entry)."""
    xm, ym = sum(xs) / len(xs), sum(ys) / len(ys)
    sl = sum((a - xm) * (b - ym) for a, b in zip(xs, ys)) / sum((a - xm) ** 2 for a in xs)
    return sl, ym - sl * xm


def fixed_latent(args):
    """Fig. 13b of the pages on GB300: complete calls and disjoint per-step costs of the Markov (16 steps) and
    recurrent (15 steps) heads, each with the state advance and as the fixed-latent probe (WHEAD_FLAG_FIXED_LATENT:
    projection and selection repeated on the unchanged initial state). Per-step cost = least-squares slope of the
    walk time over gamma in {1, 7, gamma}; phases from the kernel's stamps. One JSON line per head and mode."""
    import numpy as np
    import torch

    import whead_inputs as I
    from speculative_decoding_serial_gb300 import build
    from speculative_decoding_serial_gb300 import whead as wh

    build.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for name in ("markov_v151936_r256_b1_g16", "recurrent_v151936_r256_b1_g15"):
        w = I.WORKLOADS[name]
        d = I.workload_inputs(name)
        B, G16 = w["B"], w["gamma"]
        W = torch.from_numpy(d["W"].view(np.int16)).view(torch.bfloat16).to(dev)
        E = torch.from_numpy(d["E"].view(np.int16)).view(torch.bfloat16).to(dev)
        base = torch.from_numpy(d["base"]).to(dev)
        s0 = torch.from_numpy(d["s0"]).to(dev)
        A = None if d["A"] is None else torch.from_numpy(d["A"]).to(dev)
        c = None if d["c"] is None else torch.from_numpy(d["c"]).to(dev)
        gammas = [1, 7, G16]
        for mode, flags in (("walk", 0), ("fixed_latent", wh.FLAG_FIXED_LATENT)):
            head = wh.Head(W, E, kind=w["kind"], A=A, c=c, max_B=B, max_gamma=G16, stream=stream, flags=flags)
            plan = head.plan(B)
            ys = []
            for g in gammas:
                bg = base[:, :g].contiguous()
                tok = torch.empty((B, g), dtype=torch.int32, device=dev)
                for _ in range(3):
                    head.walk(bg, s0, T=w["T"], out_tokens=tok)
                ts = []
                for _ in range(args.sweep_walks):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    head.walk(bg, s0, T=w["T"], out_tokens=tok)
                    e1.record(stream)
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1e3)
                ys.append(central_mean(ts))
            tok = torch.empty((B, G16), dtype=torch.int32, device=dev)
            phases = trace_phases(torch, head, base, s0, tok, w, plan, flush, stream, dev, advance=(flags == 0))
            status = head.status()
            head.close()
            sl, ic = fit_line(gammas, ys)
            print(json.dumps({"fig13b": mode, "workload": name, "status": status, "gammas": gammas,
                              "us_per_walk": ys, "us_per_step_slope": sl, "entry_intercept_us": ic,
                              "phases": phases, "placement": plan}), flush=True)


def sharded_measure(walk, merge_once, steps, warmup, world, timer):
    """Rank logic of the sharded leg. walk(): one whole walk of this rank's shard (all ranks call it together;
    returns the tokens); merge_once(): one all-reduce of a step's packed keys; timer(fn) -> seconds that fn took
    on this rank's device (CUDA events) or host. Returns seconds per walk and per merge, each the maximum over
    ranks, and the last walk's tokens."""
    for _ in range(warmup):
        walk()
    out = {}
    barrier(world)
    out["walk_s"] = max_over_ranks(timer(lambda: [out.__setitem__("tokens", walk()) for _ in range(steps)]),
                                   world) / steps
    barrier(world)
    out["merge_s"] = max_over_ranks(timer(lambda: [merge_once() for _ in range(steps)]), world) / steps
    return out


def sharded(args, world, rank, local):
    """Vocabulary sharding (the one exchange the method has across GPUs: Fig. 8's packed selection taken over
    ranks). With N > 1 ranks (torchrun, NCCL) rank k holds rows shard_bounds(V, N, k) of W and walks them step by
    step: a one-step walk of its shard, an all-reduce MAX of B packed keys, the state advanced on its GPU. With
    one process, --shards K shards of the vocabulary run in lockstep on the one GPU (their keys merged on the
    device), which measures the protocol's per-step cost without the link. One JSON line (rank 0)."""
    import numpy as np
    import torch

    import whead_inputs as I
    from speculative_decoding_serial_gb300 import build
    from speculative_decoding_serial_gb300 import sharded as S
    from speculative_decoding_serial_gb300 import whead as wh

    if rank == 0 or not build.needs_build():
        build.build()
    barrier(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    name = args.workload
    w = I.WORKLOADS[name]
    d = I.workload_inputs(name)
    B, gamma, V, r = w["B"], w["gamma"], w["V"], w["r"]
    W = torch.from_numpy(d["W"].view(np.int16)).view(torch.bfloat16).to(dev)
    E = torch.from_numpy(d["E"].view(np.int16)).view(torch.bfloat16).to(dev)
    base = torch.from_numpy(d["base"]).to(dev)
    s0 = torch.from_numpy(d["s0"]).to(dev)
    A = None if d["A"] is None else torch.from_numpy(d["A"]).to(dev)
    c = None if d["c"] is None else torch.from_numpy(d["c"]).to(dev)
    nshards = world if world > 1 else max(1, args.shards)
    mine = [rank] if world > 1 else list(range(nshards))
    heads, bases, bounds = [], [], []
    for k in mine:
        lo, hi = S.shard_bounds(V, nshards, k)
        heads.append(wh.Head(W[lo:hi].contiguous(), E, kind=w["kind"], A=A, c=c, max_B=B, max_gamma=1, v_offset=lo,
                             e_rows=V, stream=stream))
        bases.append([base[:, t:t + 1, lo:hi].contiguous() for t in range(gamma)])
        bounds.append((lo, hi))
    keys = torch.empty((B, 1), dtype=torch.int64, device=dev)
    tok1 = torch.empty((B, 1), dtype=torch.int32, device=dev)
    merge = S.allreduce_max() if world > 1 else (lambda v: v)

    def step(t, s):
        got = []
        for h, bs in zip(heads, bases):
            h.walk_keys(bs[t], s, T=w["T"], seed=0, t0=t, out_tokens=tok1, out_keys=keys)
            got.append(S.to_ordered(keys[:, 0]))
        local_max = got[0] if len(got) == 1 else torch.stack(got).max(dim=0).values
        return S.from_ordered(local_max)

    def advance(x, s):
        return heads[0].advance(x.contiguous(), s, torch.empty_like(s))

    proto = S.ShardedWalk(step, merge, advance)
    probe = torch.zeros((B,), dtype=torch.int64, device=dev)

    def timer(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e-3

    m = sharded_measure(lambda: proto.walk(s0, gamma)[0], lambda: merge(probe), args.steps, max(3, args.warmup),
                        world, timer)
    status = max(h.status() for h in heads)
    tokens = m["tokens"].cpu().numpy()
    # the unsharded walk of the same inputs, for the tokens and the comparison
    full = wh.Head(W, E, kind=w["kind"], A=A, c=c, max_B=B, max_gamma=gamma, stream=stream)
    ref_tok = full.walk(base, s0, T=w["T"], seed=0).cpu().numpy()
    full.close()
    for h in heads:
        h.close()
    if rank != 0:
        return
    print(json.dumps({
        "sharded": name, "n_gpus": world, "shards": nshards, "mode": "ranks (NCCL)" if world > 1 else
        "shards in lockstep on one GPU", "rows_per_shard": [b[1] - b[0] for b in bounds] if world == 1 else
        [S.shard_bounds(V, world, k)[1] - S.shard_bounds(V, world, k)[0] for k in range(world)],
        "us_per_walk": m["walk_s"] * 1e6, "us_per_step": m["walk_s"] * 1e6 / gamma,
        "allreduce_us_per_step": m["merge_s"] * 1e6 if world > 1 else None, "walks": args.steps,
        "tokens_equal_unsharded_walk": bool((tokens == ref_tok).all()), "status": status,
        "launches_per_walk": gamma * (len(heads) + 1)}), flush=True)


def reference_arm(args, world, rank):
    """The oracle, as it stands, on this host's cores: each step is one walk step of the workload."""
    if rank != 0:
        return
    import whead_inputs as I
    from oracle import oracle as O
    w = I.WORKLOADS[args.workload]
    d = I.workload_inputs(args.workload)
    cores = O.set_threads(host_cores())  # rows of each step over every allotted core (same results)
    base1 = d["base"][:, :1].copy()
    for _ in range(args.warmup):
        O.walk(d["kind"], d["W"], d["E"], base1, d["s0"], A=d["A"], c=d["c"], T=d["T"], want_gap=False)
    t = time.perf_counter()
    for k in range(args.steps):
        s0 = d["s0"]
        O.walk(d["kind"], d["W"], d["E"], d["base"][:, k % w["gamma"]:k % w["gamma"] + 1].copy(), s0, A=d["A"],
               c=d["c"], T=d["T"], t0=k % w["gamma"], want_gap=False)
    per_step = (time.perf_counter() - t) / args.steps
    O.set_threads(1)
    value = per_step * w["gamma"] * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "us/walk", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, **{k: w[k] for k in ("V", "r", "B", "gamma", "T")}},
        "cpu_baseline": {"value": value, "unit": "us/walk", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} single walk steps of the workload (x{w['gamma']} for a walk), "
                                   f"rows of each step split over {cores} host threads"},
        "e2e": {"value": value, "unit": "us/walk", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def ours(args, world, rank, local):
    import numpy as np
    import torch

    import whead_inputs as I
    from speculative_decoding_serial_gb300 import build
    from speculative_decoding_serial_gb300 import whead as wh

    if rank == 0 or not build.needs_build():
        build.build()
    barrier(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = I.WORKLOADS[args.workload]
    d = I.workload_inputs(args.workload)
    B, gamma, V, r = w["B"], w["gamma"], w["V"], w["r"]
    W = torch.from_numpy(d["W"].view(np.int16)).view(torch.bfloat16).to(dev)
    E = torch.from_numpy(d["E"].view(np.int16)).view(torch.bfloat16).to(dev)
    base = torch.from_numpy(d["base"]).to(dev)
    s0 = torch.from_numpy(d["s0"]).to(dev)
    A = None if d["A"] is None else torch.from_numpy(d["A"]).to(dev)
    c = None if d["c"] is None else torch.from_numpy(d["c"]).to(dev)
    stream = torch.cuda.current_stream(dev)
    wflags = wh.FLAG_W_E4M3 if w.get("w") == "e4m3" else 0
    head = wh.Head(W, E, kind=w["kind"], A=A, c=c, max_B=B, max_gamma=gamma, stream=stream, flags=wflags)
    plan = head.plan(B)
    tok = torch.empty((B, gamma), dtype=torch.int32, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def timed_walks(n, g, flush_l2=True):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        bg = base[:, :g].contiguous() if g != gamma else base
        tk = tok[:, :g].contiguous() if g != gamma else tok
        for k in range(n):
            if flush_l2:
                flush.zero_()
            ev[k][0].record(stream)
            head.walk(bg, s0, T=w["T"], seed=0, out_tokens=tk)
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in ev]

    timed_walks(args.warmup, gamma)
    assert head.status() == 0

    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(gpu_selector(torch, local)) as clk:
        times_ms = timed_walks(args.steps, gamma)
        torch.cuda.synchronize(dev)
    barrier(world)
    st = head.status()
    if st != 0:
        raise RuntimeError(f"device status {st} during the timed walks")
    total_ms = max_over_ranks(sum(times_ms), world)
    us_per_walk = total_ms * 1e3 / (args.steps * world)
    clocks = clk.summary()

    # per-step cost: least-squares slope over gamma in {1, 7, 16}; intercept = entry cost
    fit_g, fit_t = [], []
    for g in (1, 7, 16):
        if g > gamma:
            continue
        ts = timed_walks(max(20, min(200, args.steps)), g)
        fit_g.append(g)
        fit_t.append(central_mean(ts) * 1e3)
    # the same walk with L2 warm (back to back, no flush): W, E and the base logits partly in L2 already
    warm_ms = timed_walks(max(20, min(200, args.steps)), gamma, flush_l2=False)
    l2_warm = {"walk_us": central_mean(warm_ms) * 1e3, "walks": len(warm_ms)}
    slope = intercept = None
    if len(fit_g) >= 2:
        gm, tm = sum(fit_g) / len(fit_g), sum(fit_t) / len(fit_t)
        slope = sum((a - gm) * (b - tm) for a, b in zip(fit_g, fit_t)) / sum((a - gm) ** 2 for a in fit_g)
        intercept = tm - slope * gm

    phases = trace_phases(torch, head, base, s0, tok, w, plan, flush, stream, dev)
    clocks["kernel_sm_mhz"] = phases.pop("kernel_sm_mhz")
    clocks["kernel_sm_mhz_source"] = ("clock64 / globaltimer stamps of every CTA over the traced walks run right "
                                      "after the timed region (the timed region is shorter than one nvidia-smi "
                                      "sample)")
    traffic = recorded_traffic() if args.workload == DEFAULT_WORKLOAD else None

    # roofline (on-chip operand bandwidth for the steps, HBM for the one-time shard load)
    hbm_gbs, peak_kind = load_peaks()
    onchip = probe_onchip()
    smem_bpc = onchip["smem_b_per_clk"] if onchip else SMEM_B_PER_CLK
    tmem_bpc = onchip["tmem_b_per_clk"] if onchip else TMEM_B_PER_CLK
    sm = plan["sm_count"]
    wbytes = V * r * 2
    w_per_sm = plan["groups_per_cta"] * 16 * r * 2
    smem_min = max(0, w_per_sm - TMEM_BYTES - RF_W_BYTES_CAP)
    tmem_used = min(TMEM_BYTES, w_per_sm)
    t_star_clk = max(smem_min / smem_bpc, tmem_used / tmem_bpc)
    # the same bound for the placement the library actually ships for this walk (its shared and tensor-memory groups)
    group_bytes = 16 * r * 2
    t_star_shipped_clk = max(plan["smem_groups"] * group_bytes / smem_bpc, plan["tmem_groups"] * group_bytes / tmem_bpc)
    # cycles to time at the clock the kernel ran at (its own stamps), else the sampled one
    mhz = clocks["kernel_sm_mhz"] or clocks["sm_mhz"] or 1447.0
    clock_source = "kernel stamps" if clocks["kernel_sm_mhz"] else ("nvidia-smi" if clocks["sm_mhz"] else "fallback")
    t_star_us = t_star_clk / mhz
    t_entry_us = wbytes / (hbm_gbs * 1e3)
    t_roof_us = t_entry_us + gamma * t_star_us
    alg_bytes = wbytes + gamma * wbytes + B * gamma * V * 4 + gamma * B * r * 2
    achieved = alg_bytes / (us_per_walk * 1e3)
    peak = alg_bytes / (t_roof_us * 1e3)


    # end to end through the host-buffer entry point: pinned inputs copied in, tokens copied out
    base_h = torch.from_numpy(d["base"]).pin_memory()
    s0_h = torch.from_numpy(d["s0"]).pin_memory()
    tok_h = torch.empty((B, gamma), dtype=torch.int32).pin_memory()
    for _ in range(5):
        head.walk_host(base_h, s0_h, T=w["T"], out_tokens=tok_h)
    n_e2e = max(20, min(200, args.steps))
    e2e = []
    for _ in range(n_e2e):
        flush.zero_()
        torch.cuda.synchronize(dev)
        t = time.perf_counter()
        head.walk_host(base_h, s0_h, T=w["T"], out_tokens=tok_h)
        e2e.append(time.perf_counter() - t)
    # the mean of the middle 80 % of the calls: a host call now and then waits on the machine (measured: a whole
    # run's mean once came out 1.7 times the others'), and the trimmed mean keeps one such stretch from deciding it
    e2e_us = max_over_ranks(central_mean(e2e) * 1e6, world)
    e2e_spread = [float(np.percentile(e2e, q)) * 1e6 for q in (10, 50, 90)] if e2e else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(d, gamma, args.workload, args.cpu_seconds)

    head.close()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": us_per_walk, "unit": "us/walk", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us_per_walk / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "V": V, "r": r, "B": B, "gamma": gamma, "T": w["T"],
                   "l2": "flushed (256 MB write) before every timed walk", "placement": plan},
        "roofline": {"bound": "onchip", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": t_roof_us / us_per_walk,
                     "traffic": traffic,
                     "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch, from the "
                                        "committed profile taken on this kernel source (sha-matched)")
                     if traffic is not None else None,
                     "t_roof_us": t_roof_us, "t_entry_us": t_entry_us, "t_star_clk_per_step": t_star_clk,
                     "hbm_peak_gbs": hbm_gbs, "hbm_peak_kind": peak_kind, "clock_mhz": mhz, "clock_source": clock_source,
                     "onchip_measured": onchip,
                     "onchip_kind": "measured" if onchip else "fallback (128 B/clk shared, 428 B/clk tensor memory)"},
        "per_step": {"slope_us": slope, "intercept_us": intercept, "gammas": fit_g, "walk_us": fit_t,
                     "t_star_shipped_placement_clk": t_star_shipped_clk,
                     "frac_of_shipped_placement_bound": (t_star_shipped_clk / mhz / slope) if slope else None,
                     "t_star_us": t_star_us,
                     "frac_of_onchip_roofline": (t_star_us / slope) if slope else None},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_us, "unit": "us/walk", "h2d_bytes_per_step": B * gamma * V * 4 + B * r * 4,
                "d2h_bytes_per_step": B * gamma * 4, "calls": len(e2e), "p10_p50_p90_us": e2e_spread},
        "clocks": clocks,
        "phases": phases,
        "l2_warm": l2_warm,
        "gpu_launches": args.steps,
    }
    print(json.dumps(line))


def sweep(args):
    """Latency of every workload of the pages (one JSON line each): the small case, the B x gamma x T sweep at
    V = 151,936, partial residency at V = 248,064 and the recurrent head. Not part of the default run."""
    import numpy as np
    import torch

    import whead_inputs as I
    from speculative_decoding_serial_gb300 import build
    from speculative_decoding_serial_gb300 import whead as wh

    build.build()
    dev = torch.device("cuda", 0)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    cases = []
    for name in ("markov_v4096_r64_b1_g4", "markov_v248064_r256_b1_g16", "markov_v248064_r256_b4_g16",
                 "recurrent_v151936_r256_b1_g15", "markov_v151936_r256_b1_g16_e4m3",
                 "markov_v248064_r256_b1_g16_e4m3", "markov_v248064_r256_b4_g16_e4m3"):
        w = I.WORKLOADS[name]
        cases.append((name, w["kind"], w["V"], w["r"], w["B"], w["gamma"], w["T"], w.get("w", "bf16")))
    sw = I.SWEEP
    for B in sw["Bs"]:
        for g in sw["gammas"]:
            for T in sw["Ts"]:
                cases.append((f"sweep_v{sw['V']}_b{B}_g{g}_t{int(T)}", sw["kind"], sw["V"], sw["r"], B, g, T, "bf16"))
    cache = {}
    for name, kind, V, r, B, g, T, wfmt in cases:
        key = (kind, V, r, B, g)
        if key not in cache:
            cache.clear()
            d = I.make_inputs(kind, V, r, B, g, seed=0)
            cache[key] = d
        d = cache[key]
        W = torch.from_numpy(d["W"].view(np.int16)).view(torch.bfloat16).to(dev)
        E = torch.from_numpy(d["E"].view(np.int16)).view(torch.bfloat16).to(dev)
        base = torch.from_numpy(d["base"]).to(dev)
        s0 = torch.from_numpy(d["s0"]).to(dev)
        A = None if d["A"] is None else torch.from_numpy(d["A"]).to(dev)
        c = None if d["c"] is None else torch.from_numpy(d["c"]).to(dev)
        head = wh.Head(W, E, kind=kind, A=A, c=c, max_B=B, max_gamma=g, stream=stream,
                       flags=wh.FLAG_W_E4M3 if wfmt == "e4m3" else 0)
        tok = torch.empty((B, g), dtype=torch.int32, device=dev)
        for _ in range(5):
            head.walk(base, s0, T=T, out_tokens=tok)
        ts = []
        for _ in range(args.sweep_walks):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            head.walk(base, s0, T=T, out_tokens=tok)
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        st = head.status()
        print(json.dumps({"case": name, "kind": "recurrent" if kind else "markov", "w": wfmt, "V": V, "r": r, "B": B,
                          "gamma": g, "T": T, "us_per_walk": central_mean(ts), "status": st,
                          "placement": head.plan(B)}), flush=True)
        head.close()


def ablation(args):
    """Fusion versus residency on GB300 (Figs. 4 and 11 of the pages): complete-call latency over gamma in
    {1, 7, 16} and its least-squares slope (us/step) and intercept (entry) for (a) the resident megakernel,
    (b) the same fused walk with every row of W re-read from L2/HBM each step, and (c) step-wise execution,
    one launch per step (each launch loads W again). One JSON line per variant."""
    import numpy as np
    import torch

    import whead_inputs as I
    from speculative_decoding_serial_gb300 import build
    from speculative_decoding_serial_gb300 import whead as wh

    build.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    w = I.WORKLOADS[args.workload]
    d = I.workload_inputs(args.workload)
    B, G16, V, r = w["B"], w["gamma"], w["V"], w["r"]
    W = torch.from_numpy(d["W"].view(np.int16)).view(torch.bfloat16).to(dev)
    E = torch.from_numpy(d["E"].view(np.int16)).view(torch.bfloat16).to(dev)
    base = torch.from_numpy(d["base"]).to(dev)
    s0 = torch.from_numpy(d["s0"]).to(dev)
    A = None if d["A"] is None else torch.from_numpy(d["A"]).to(dev)
    c = None if d["c"] is None else torch.from_numpy(d["c"]).to(dev)
    gammas = [g for g in (1, 7, 16) if g <= G16]

    def timed(fn, n):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(n):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return central_mean(ts)

    def fit(xs, ys):
        xm, ym = sum(xs) / len(xs), sum(ys) / len(ys)
        sl = sum((a - xm) * (b - ym) for a, b in zip(xs, ys)) / sum((a - xm) ** 2 for a in xs)
        return sl, ym - sl * xm

    variants = {}
    for name, flags in (("resident", 0), ("fused_streaming", wh.FLAG_FORCE_STREAM)):
        head = wh.Head(W, E, kind=w["kind"], A=A, c=c, max_B=B, max_gamma=G16, stream=stream, flags=flags)
        plan = head.plan(B)
        ys = []
        for g in gammas:
            bg = base[:, :g].contiguous()
            tok = torch.empty((B, g), dtype=torch.int32, device=dev)
            ys.append(timed(lambda: head.walk(bg, s0, T=w["T"], out_tokens=tok), args.sweep_walks))
        assert head.status() == 0
        head.close()
        variants[name] = (ys, plan)
    # step-wise: one launch per step, the state handed over through device memory
    head = wh.Head(W, E, kind=w["kind"], A=A, c=c, max_B=B, max_gamma=1, stream=stream)
    steps_base = [base[:, t:t + 1].contiguous() for t in range(G16)]
    st = torch.empty((G16 + 1, B, r), dtype=torch.float32, device=dev)
    tok1 = torch.empty((B, 1), dtype=torch.int32, device=dev)
    ys = []
    for g in gammas:
        def stepwise(g=g):
            cur = s0
            for t in range(g):
                head.walk_ex(steps_base[t], cur, T=w["T"], t0=t, out_tokens=tok1, out_state=st[t + 1])
                cur = st[t + 1]
        ys.append(timed(stepwise, max(10, args.sweep_walks // 4)))
    assert head.status() == 0
    variants["step_wise"] = (ys, head.plan(B))
    head.close()
    for name, (ys, plan) in variants.items():
        sl, ic = fit(gammas, ys)
        print(json.dumps({"ablation": name, "workload": args.workload, "gammas": gammas, "us_per_walk": ys,
                          "us_per_step_slope": sl, "entry_intercept_us": ic, "placement": plan}), flush=True)


def placement(args):
    """Placement sweep on GB300 (Fig. 12 of the pages): per-step cost and entry for chosen splits of a CTA's
    16-row groups over shared memory, tensor memory and registers, the rest streamed from L2/HBM every step
    (WHEAD_FLAG_PLACEMENT_CAPS). Complete-call latency over gamma in {1, 7, 16}, least-squares slope and
    intercept, as for the ablation. One JSON line per split."""
    import numpy as np
    import torch

    import whead_inputs as I
    from speculative_decoding_serial_gb300 import build
    from speculative_decoding_serial_gb300 import whead as wh

    build.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    w = I.WORKLOADS[args.workload]
    d = I.workload_inputs(args.workload)
    B, G16 = w["B"], w["gamma"]
    W = torch.from_numpy(d["W"].view(np.int16)).view(torch.bfloat16).to(dev)
    E = torch.from_numpy(d["E"].view(np.int16)).view(torch.bfloat16).to(dev)
    base = torch.from_numpy(d["base"]).to(dev)
    s0 = torch.from_numpy(d["s0"]).to(dev)
    A = None if d["A"] is None else torch.from_numpy(d["A"]).to(dev)
    c = None if d["c"] is None else torch.from_numpy(d["c"]).to(dev)
    gammas = [g for g in (1, 7, 16) if g <= G16]
    # (shared, tensor, register) caps; None = the planner's own (fully resident) split
    splits = [None, (64, 64, 0), (64, 16, 8), (64, 0, 8), (13, 64, 8), (0, 64, 8), (0, 0, 8), (0, 0, 0)]
    for caps in splits:
        head = wh.Head(W, E, kind=w["kind"], A=A, c=c, max_B=B, max_gamma=G16, stream=stream, caps=caps)
        plan = head.plan(B)
        ys = []
        for g in gammas:
            bg = base[:, :g].contiguous()
            tok = torch.empty((B, g), dtype=torch.int32, device=dev)
            for _ in range(3):
                head.walk(bg, s0, T=w["T"], out_tokens=tok)
            ts = []
            for _ in range(args.sweep_walks):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                head.walk(bg, s0, T=w["T"], out_tokens=tok)
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3)
            ys.append(central_mean(ts))
        status = head.status()
        head.close()
        xm, ym = sum(gammas) / len(gammas), sum(ys) / len(ys)
        sl = sum((a - xm) * (b - ym) for a, b in zip(gammas, ys)) / sum((a - xm) ** 2 for a in gammas)
        print(json.dumps({"placement_caps": caps, "workload": args.workload, "status": status, "gammas": gammas,
                          "us_per_walk": ys, "us_per_step_slope": sl, "entry_intercept_us": ym - sl * xm,
                          "placement": plan}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sweep", action="store_true", help="latency of every workload of the pages (one line each)")
    ap.add_argument("--sweep-walks", type=int, default=100)
    ap.add_argument("--ablation", action="store_true", help="fusion vs residency (resident / fused streaming / step-wise)")
    ap.add_argument("--placement", action="store_true", help="placement sweep over shared/tensor/register tiers")
    ap.add_argument("--fixed-latent", action="store_true",
                    help="per-step cost with and without the state advance (Markov and recurrent heads)")
    ap.add_argument("--sharded", action="store_true",
                    help="vocabulary sharded over the ranks (or --shards K shards in lockstep on one GPU)")
    ap.add_argument("--shards", type=int, default=2)
    args = ap.parse_args()
    if args.placement:
        placement(args)
        return
    if args.fixed_latent:
        fixed_latent(args)
        return
    if args.sweep:
        sweep(args)
        return
    if args.ablation:
        ablation(args)
        return
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_setup(args)
    if args.sharded:
        sharded(args, world, rank, local)
    elif args.impl == "reference":
        reference_arm(args, world, rank)
    else:
        ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
