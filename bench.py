#!/usr/bin/env python3
"""Throughput of the fused sample / verify call on GB300.

One step = one ss_verify call over the mixed serving batch (B = 512 rows,
V = 151936 fp32 logits, 60% single-step rows and 40% verify rows with ragged
gamma in 1..7, every logits processor on): the one workload whose single
call runs every step of the path (prelude, tile top-128, merge, truncation,
Gumbel sampling, accept test, residual and bonus tokens).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is rows per second over all ranks,
timed with CUDA events around K calls replayed from CUDA graphs with the
inputs already resident in HBM (the last G calls carry per-kernel events,
which give the kernel durations of the roofline); `e2e` is the same metric with each step's
inputs copied from pinned host memory and its tokens copied back inside the
timed region.  Under torchrun each rank runs its own batch (weak scaling,
no collective on the data path).  `--impl reference` times the CPU oracle
on every host core (four rows per core per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "rows/sec and achieved HBM GB/s (% of GB300 peak) per fused sample/verify call"
FALLBACK_HBM_GBS = 6800.0
STAGE1_SOURCES = ["spec_verification_gb300/csrc/ss_stage1.cuh", "spec_verification_gb300/csrc/ss_common.cuh"]


def workload(name: str):
    from spec_verification_gb300 import workloads as W
    table = {
        "c5": (W.config5, "mixed serving batch: B=512, V=151936 fp32, 60% single-step / 40% verify "
                          "(gamma 1..7), all processors, per-row flags from seed 5"),
        "c2": (W.config2, "single-step heterogeneous: B=64, V=131072 bf16, all processors"),
        "c3": (W.config3, "single-step top-k stress: B=256, V=262144 fp32, half near-flat rows"),
        "c4": (W.config4, "speculative verification: B=32, gamma=4, V=131072 bf16 target and draft probs"),
        "c1": (W.config1, "single-step: B=4, V=32000 fp32, 2 greedy + 2 stochastic rows"),
        "c4_onehot": (lambda: W.with_one_hot_drafts(W.config4()),
                      "speculative verification: B=32, gamma=4, V=131072 bf16 target, drafts without "
                      "probabilities (one-hot q)"),
        "c2_exact": (lambda: W.with_exact_sampling(W.config2()),
                     "single-step heterogeneous: B=64, V=131072 bf16, all processors, stochastic rows "
                     "untruncated and sampled over the whole vocabulary (exact sampling)"),
        "c4_bounded": (lambda: W.with_bounded_p(W.config4()),
                       "speculative verification: B=32, gamma=4, V=131072 bf16 target and draft probs, "
                       "stochastic rows verified against the 128-candidate softmax"),
    }
    fn, desc = table[name]
    return fn(), desc


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def stage1_source_hash() -> str:
    h = hashlib.sha256()
    for s in STAGE1_SOURCES:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(wname: str):
    """DRAM bytes per stage-1 launch from the committed ncu summary, if it was
    taken on the current stage-1 source (else None)."""
    path = os.path.join(ROOT, "profiles", f"stage1_{wname}_ncu.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"stage1_source_sha256_16:\s*([0-9a-f]+)", text)
    t = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not m or not t or m.group(1) != stage1_source_hash():
        return None
    return float(t.group(1))


class Clocks:
    """nvidia-smi sampler of SM clocks and throttle reasons."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "20", "-i", str(self.index)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


_CUDART = None


def event_ms(a, b) -> float:
    """Milliseconds between two timing events recorded by the library (inside
    a captured graph), read with cudaEventElapsedTime."""
    try:
        return a.elapsed_time(b)
    except (RuntimeError, ValueError):
        pass
    global _CUDART
    import ctypes
    if _CUDART is None:
        for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
            try:
                _CUDART = ctypes.CDLL(name)
                break
            except OSError:
                continue
    f = ctypes.c_float()
    rc = _CUDART.cudaEventElapsedTime(ctypes.byref(f), ctypes.c_void_p(a.cuda_event), ctypes.c_void_p(b.cuda_event))
    if rc != 0:
        raise RuntimeError(f"cudaEventElapsedTime failed ({rc})")
    return f.value


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest x over the ranks (the slowest rank's time); x itself on one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, rows: int, steps: int, ms: float) -> float:
    """Rows per second over all ranks: each rank runs its own copy of the
    workload (replicas, weak scaling) and the job takes the slowest rank's time."""
    return world * rows * steps / (ms / 1e3)


def num_segments(npos: int, z: int, ctas: int) -> int:
    """Segments of the stage-1 split: with two or more CTAs per position each
    position is cut into kk = ceil(z / ceil(z / k)) ranges (k = ctas // npos),
    one segment each; otherwise the npos * z tiles are cut into
    g = min(ctas, npos * z) contiguous runs (run c starts at c * T // g) and
    each (run, position) overlap is one segment."""
    if npos <= 0:
        return 0
    k = ctas // npos
    if k >= 2:
        lr = -(-z // k)
        return npos * (-(-z // lr))
    T = npos * z
    g = min(ctas, T)
    starts = [c * T // g for c in range(g)]
    # a run that starts inside a position (not at its first tile) adds a segment
    return npos + sum(1 for s in starts[1:] if s % z != 0)


def stage1_alg_bytes(w, tile: int, ctas: int) -> int:
    """Bytes stage 1 must move per launch: each position's logits and (when
    its row applies the grammar mask) its bitmask row are read once; each
    segment writes 128 packed 8-byte candidates plus 12 bytes of metadata."""
    import numpy as np
    from spec_verification_gb300 import workloads as W
    z = -(-w.V // tile)
    s = 2 if w.dtype == "bf16" else 4
    offs = w.position_offsets()
    mask_rows = (w.rows["flags"] & W.MASK) != 0
    per_pos_mask = np.repeat(mask_rows, np.diff(offs)) if w.bitmask is not None else np.zeros(w.n_positions, bool)
    n = w.n_positions * w.V * s + num_segments(w.n_positions, z, ctas) * (128 * 8 + 12)
    n += int(per_pos_mask.sum()) * 4 * (-(-w.V // 32))
    return int(n)


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class RowSubsets:
    """Row r of a workload as a workload of its own, built on access."""

    def __init__(self, w):
        self.w = w

    def __len__(self):
        return self.w.B

    def __getitem__(self, r):
        from spec_verification_gb300.workloads import subset
        return subset(self.w, [int(r)])


def oracle_rows_parallel(subs, cores: int, budget_s: float | None = None, ex=None):
    """The oracle, as it stands, on the one-row workloads `subs` over `cores`
    threads pulling rows from one queue in the given order; each thread calls
    the single-threaded oracle (a ctypes call, which releases the GIL).  With
    budget_s no row starts after that many seconds.  Returns (rows done,
    target positions done, wall seconds)."""
    import concurrent.futures as cf
    from oracle import oracle
    oracle.lib()
    t0 = time.perf_counter()

    def one(i):
        if budget_s is not None and time.perf_counter() - t0 >= budget_s:
            return 0, 0
        s = subs[i]
        (oracle.verify if s.is_verify else oracle.sample)(s)
        return 1, s.n_positions

    if ex is None:
        with cf.ThreadPoolExecutor(max_workers=cores) as own:
            res = list(own.map(one, range(len(subs))))
    else:
        res = list(ex.map(one, range(len(subs))))
    return sum(a for a, _ in res), sum(b for _, b in res), time.perf_counter() - t0


def cpu_baseline(w, desc_name: str, budget_s: float = 12.0) -> dict:
    """The oracle, as it stands (bounded k = 128 mode, one thread): one
    warm-up row, then three repetitions over the first rows of the same
    workload, each about budget_s / 3 seconds of CPU work, and the median
    rate; beside it, the same oracle with the rows spread over every host
    core for about half budget_s of wall time."""
    from oracle import oracle
    from spec_verification_gb300.workloads import subset
    oracle.lib()
    first = subset(w, [0])
    (oracle.verify if first.is_verify else oracle.sample)(first)  # warm-up
    reps = []
    for _ in range(3):
        done_rows, npos, t_total = 0, 0, 0.0
        r = 0
        while t_total < budget_s / 3 and r < w.B:
            s = subset(w, [r])
            t0 = time.perf_counter()
            (oracle.verify if s.is_verify else oracle.sample)(s)
            t_total += time.perf_counter() - t0
            done_rows += 1
            npos += s.n_positions
            r += 1
        reps.append((done_rows / t_total, done_rows, npos, t_total))
    rate, done_rows, npos, t_total = sorted(reps)[1]
    cores = host_cores()
    n_all, npos_all, wall = oracle_rows_parallel(RowSubsets(w), cores, budget_s / 2)
    return {"value": rate, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": f"median of 3 repetitions, each the first {done_rows} rows ({npos} target positions) "
                      f"of {desc_name} in about {t_total:.1f} s; oracle bounded k=128 mode, single-threaded",
            "all_cores": {"value": n_all / wall, "unit": "rows/s", "cores": cores,
                          "sample": f"{n_all} rows ({npos_all} target positions) of {desc_name} pulled by "
                                    f"{cores} threads from one queue, {wall:.1f} s wall"}}


def run_reference(args, w, desc):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import concurrent.futures as cf
    from oracle import oracle
    from spec_verification_gb300.workloads import subset
    oracle.lib()
    cores = host_cores()
    n_rows = min(w.B, 64)
    subs = [subset(w, [r]) for r in range(n_rows)]

    per_step = 4 * cores

    def step(i, ex):
        # four rows per host core, cycling over the first n_rows rows, pulled
        # from one queue longest first so that no core idles behind a long row
        rows = [subs[(i * per_step + k) % n_rows] for k in range(per_step)]
        rows.sort(key=lambda s: -s.n_positions)
        oracle_rows_parallel(rows, cores, ex=ex)

    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        for i in range(args.warmup):
            step(i, ex)
        t0 = time.perf_counter()
        for i in range(args.steps):
            step(args.warmup + i, ex)
        dt = time.perf_counter() - t0
    value = args.steps * per_step / dt
    sample = (f"{per_step} rows (all their target positions) of {args.workload} per step on {cores} host "
              f"cores (one queue, longest row first), cycling over the first {n_rows} rows; oracle bounded "
              f"k=128 mode, single-threaded per row")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": desc, "name": args.workload, "B": w.B, "V": w.V},
            "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": sample, "value": value, "unit": "rows/s"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def input_copies(call_bytes: int, l2_bytes: int, G: int) -> int:
    """Resident copies of a call's streamed inputs (logits, draft probs) so
    that consecutive passes over them hold at least twice the L2 size: 2
    when two copies already do, else the next multiple of the G calls per
    graph."""
    need = max(2, -(-2 * l2_bytes // max(1, call_bytes)))
    return 2 if need <= 2 else -(-need // G) * G


def graph_copies(R: int, G: int) -> list:
    """The copy each call of each captured graph uses: call i of graph j
    takes copy (j * G + i) mod R, so replaying the R / gcd(R, G) graphs in
    turn walks through every copy in order."""
    import math
    NG = R // math.gcd(R, G)
    return [[(j * G + i) % R for i in range(G)] for j in range(NG)]


def time_device(args, w, dev, world, K, Wm, tile=0):
    """Graph-replayed timing of K calls of workload w with inputs resident in
    HBM (after Wm warm-up calls): returns the run, the slowest rank's time of
    the K calls (ms), the per-kernel durations of the last G calls (us) and
    the clock record of the timed region."""
    import torch
    import torch.distributed as dist
    from spec_verification_gb300.runner import DeviceRun

    run = DeviceRun(w, device=str(dev), candidates=False, tile=tile)
    G = max(d for d in range(1, min(10, K) + 1) if K % d == 0)
    # resident copies of the streamed inputs, walked in turn so that nothing
    # is served from L2 (together at least twice its size)
    call_bytes = sum(t.numel() * t.element_size() for t in (run.d["logits"], run.d.get("draft_probs"))
                     if t is not None)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20))
    R = input_copies(call_bytes, l2, G)
    lg = [run.d["logits"]] + [run.d["logits"].clone() for _ in range(R - 1)]
    qq = [run.d.get("draft_probs")] + [run.d["draft_probs"].clone() if "draft_probs" in run.d else None
                                       for _ in range(R - 1)]
    plan = graph_copies(R, G)
    NG = len(plan)
    j_ev = (K // G - 1) % NG  # the timed region's last replay, the one with events
    stream = torch.cuda.Stream(device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(G)]
    for row in ev:  # torch creates the underlying cudaEvent_t at the first record
        for e in row:
            e.record(stream)
    with torch.cuda.stream(stream):
        for i in range(2):
            run(logits=lg[i % 2], draft_probs=qq[i % 2])
    stream.synchronize()
    # Graphs of G calls: one per set of copies in `graphs`, without
    # instrumentation, and `graph_ev` with an event before, between and after
    # the kernels of each call.  Event nodes cost about 15 us per call here,
    # so the timed region replays `graphs` in turn for all but its last G
    # calls, which come from `graph_ev` (on the copies next in turn) and give
    # the per-kernel durations (measured inside the timed region).
    graphs = []
    for cp in plan:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                run(logits=lg[cp[i]], draft_probs=qq[cp[i]])
        graphs.append(g)
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=stream):
        for i in range(G):
            run(logits=lg[plan[j_ev][i]], draft_probs=qq[plan[j_ev][i]], events=ev[i])
    with torch.cuda.stream(stream):
        for t in range(max(1, -(-Wm // G))):
            graphs[t % NG].replay()
        graph_ev.replay()
    stream.synchronize()

    clocks = Clocks(dev.index or 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.05)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for t in range(K // G - 1):
            graphs[t % NG].replay()
        graph_ev.replay()
        t_end.record(stream)
    torch.cuda.synchronize(dev)
    ck = clocks.stop()
    if world > 1:
        dist.barrier()
    ms = t_start.elapsed_time(t_end)
    stages = {"stage1": 1e3 * statistics.mean(event_ms(ev[i][0], ev[i][1]) for i in range(G)),
              "stage2": 1e3 * statistics.mean(event_ms(ev[i][1], ev[i][2]) for i in range(G)),
              "residual": 1e3 * statistics.mean(event_ms(ev[i][2], ev[i][3]) for i in range(G)) if w.is_verify else 0.0}
    ms_max = max_over_ranks(ms, world, dev)
    info = {"R": R, "call_bytes": call_bytes, "l2": l2, "G": G, "NG": NG}
    del graphs, graph_ev, lg, qq
    return run, ms_max, stages, ck, info


def roofline_of(w, run, stages, ms_max, K, peak, peak_kind, traffic=None) -> tuple:
    """The stage-1 roofline and the whole call's counted-byte rate."""
    alg1 = stage1_alg_bytes(w, run.plan.tile, run.plan.stage1_ctas)
    achieved = alg1 / (stages["stage1"] / 1e6) / 1e9
    # a call without a stage-2 launch ran stage 2 inside stage 1 (the fused
    # form: stage 1, plus the residual pass of a verification call)
    fused = run.plan.last_launches() == (2 if w.is_verify else 1)
    roof = {"bound": "hbm", "kernel": "stage1 with stage 2 fused into it" if fused else "stage1",
            "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic, "alg_bytes_per_launch": alg1}
    counted = w.counted_bytes(8192)  # the metric's definition: staging of 8192-token tiles
    s_call = ms_max / K / 1e3
    hbm = {"counted_bytes_per_call": counted, "counted_gbs": counted / s_call / 1e9,
           "counted_frac": counted / s_call / 1e9 / peak,
           "read_bytes_per_call": alg1 + stage2_read_bytes(w, run),
           "read_frac": (alg1 + stage2_read_bytes(w, run)) / s_call / 1e9 / peak,
           "note": ("counted = logits + bitmask + draft probabilities + staging write and read of 8192-token "
                    "tiles per call, the metric's definition; the kernels read only q(d) of each draft and the q "
                    "rows of rejected untruncated positions, so counted_frac overstates the bytes moved when q "
                    "is large.  read = stage-1 algorithmic bytes + the staging lists stage 2 reads: the bytes "
                    "the call must move")}
    return roof, hbm


def stage2_read_bytes(w, run) -> int:
    """Bytes stage 2 reads: each segment's 128 packed candidates and its metadata."""
    z = run.plan.num_tiles
    return num_segments(w.n_positions, z, run.plan.stage1_ctas) * (128 * 8 + 12)


def h2d_copy_rate(dev, nbytes: int, streams: int) -> float:
    """GB/s of a plain pinned host -> device copy of nbytes, split over
    `streams` streams (the link's rate for the inputs of one call)."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ss = [torch.cuda.Stream(device=dev) for _ in range(streams)]
    main = torch.cuda.current_stream(dev)

    def once():
        ev0 = torch.cuda.Event()
        ev0.record(main)
        for i, st in enumerate(ss):
            st.wait_event(ev0)
            a, b = nbytes * i // streams, nbytes * (i + 1) // streams
            with torch.cuda.stream(st):
                d[a:b].copy_(h[a:b], non_blocking=True)
        for st in ss:
            e = torch.cuda.Event()
            e.record(st)
            main.wait_event(e)

    once()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    for _ in range(5):
        once()
    b.record(main)
    torch.cuda.synchronize(dev)
    rate = 5 * nbytes / (a.elapsed_time(b) / 1e3) / 1e9
    del h, d
    return rate


CONFIG_SWEEP = ["c1", "c2", "c3", "c4"]


def run_ours(args, w, desc):
    import torch
    import torch.distributed as dist
    from spec_verification_gb300 import build
    from spec_verification_gb300.runner import DeviceRun

    world, rank, local = dist_setup()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    verify = w.is_verify
    K, Wm = args.steps, args.warmup
    run, ms_max, stages, ck, info = time_device(args, w, dev, world, K, Wm, tile=args.tile)
    R, call_bytes, l2, G, NG = info["R"], info["call_bytes"], info["l2"], info["G"], info["NG"]

    # end to end: inputs from pinned host memory, tokens back, every step;
    # the streamed inputs are copied in row ranges over 4 copy streams, into
    # one of two sets of device buffers in turn, so that a step's upload
    # overlaps the previous step's kernels (each step still copies all of
    # its inputs and reads its tokens back inside the timed region)
    e2e = None
    if not args.no_e2e:
        hruns = [DeviceRun(w, device=str(dev), candidates=False, tile=args.tile, pinned_host=True)
                 for _ in range(2)]
        hrun = hruns[0]
        E = max(3, min(K, args.e2e_steps))
        outs = {"tokens": torch.empty(hrun.tokens.shape, dtype=torch.int32, pin_memory=True),
                "row_status": torch.empty(hrun.row_status.shape, dtype=torch.int32, pin_memory=True)}
        if verify:
            outs["num_accepted"] = torch.empty(hrun.num_accepted.shape, dtype=torch.int32, pin_memory=True)
        stream = torch.cuda.Stream(device=dev)
        copy_streams = [torch.cuda.Stream(device=dev) for _ in range(4)]
        up_ev = [[torch.cuda.Event() for _ in range(len(copy_streams) + 1)] for _ in hruns]
        done_ev = [torch.cuda.Event() for _ in hruns]  # the last step that read each buffer set
        step_no = [0]

        def e2e_step():
            i = step_no[0] % 2
            step_no[0] += 1
            h = hruns[i]
            h.upload_split(stream, copy_streams, up_ev[i], after=done_ev[i])
            with torch.cuda.stream(stream):
                h(stream=stream)
                done_ev[i].record(stream)
                outs["tokens"].copy_(h.tokens, non_blocking=True)
                outs["row_status"].copy_(h.row_status, non_blocking=True)
                if verify:
                    outs["num_accepted"].copy_(h.num_accepted, non_blocking=True)

        for ev in done_ev:
            ev.record(stream)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for st in copy_streams:
            st.wait_event(a)
        for _ in range(E):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ems = max_over_ranks(a.elapsed_time(b), world, dev)
        h2d = hrun.input_bytes()
        e2e = {"value": whole_job_rate(world, w.B, E, ems), "unit": "rows/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hrun.output_bytes(),
               "steps": E, "ms_per_step": ems / E, "h2d_gbs": h2d / (ems / E / 1e3) / 1e9,
               "copy_streams": len(copy_streams), "input_buffers": len(hruns),
               "plain_h2d_copy_gbs": {"1_stream": h2d_copy_rate(dev, h2d, 1), "4_streams": h2d_copy_rate(dev, h2d, 4)},
               "note": "h2d_gbs: the step's input bytes over the step time; plain_h2d_copy_gbs: a pinned host -> "
                       "device copy of the same bytes alone, the link's rate (the bound on e2e); two sets of "
                       "input buffers, so that a step's upload overlaps the previous step's kernels"}
        del hrun, hruns

    diag = run.diag()
    peak, peak_kind = read_peaks()
    tile = run.plan.tile
    roof, hbm = roofline_of(w, run, stages, ms_max, K, peak, peak_kind, profiled_traffic(args.workload))
    value = whole_job_rate(world, w.B, K, ms_max)
    n_ctas, n_tiles = run.plan.stage1_ctas, run.plan.num_tiles
    # kernels per call, as the library recorded its launch decisions (one or
    # two stage-1 forms, stage 2 unless fused, the residual pass of ss_verify)
    launches_per_call = run.plan.last_launches()
    del run
    torch.cuda.empty_cache()

    # the other configurations, each timed the same way (graph replays,
    # resident inputs larger than L2, per-kernel events, clocks sampled)
    configs = None
    if not args.no_configs and args.workload == "c5":
        configs = {}
        K2 = max(10, min(K, 500) // 10 * 10)
        for name in CONFIG_SWEEP:
            wc, dc = workload(name)
            rc_, msc, stc, ckc, _ = time_device(args, wc, dev, world, K2, max(Wm, 3), tile=args.tile)
            roofc, hbmc = roofline_of(wc, rc_, stc, msc, K2, peak, peak_kind, profiled_traffic(name))
            configs[name] = {"workload": dc, "value": whole_job_rate(world, wc.B, K2, msc), "unit": "rows/s",
                             "ms_per_step": msc / K2, "steps": K2, "stages_us": stc, "roofline": roofc,
                             "hbm": hbmc, "clocks": ckc, "positions": wc.n_positions, "V": wc.V,
                             "dtype": "f32" if wc.dtype == "f32" else "bf16",
                             "gpu_launches": K2 * rc_.plan.last_launches()}
            del rc_
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w, args.workload, args.cpu_seconds)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K, "warmup": Wm,
            "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if w.dtype == "f32" else "bf16", "data": "synthetic",
            "config": {"workload": desc, "name": args.workload, "B": w.B, "V": w.V,
                       "positions": w.n_positions, "tile": tile, "tiles_per_row": n_tiles,
                       "stage1_ctas": n_ctas,
                       "l2": f"inputs larger than L2: {R} resident copies walked in turn "
                             f"({R * call_bytes / 1e6:.0f} MB against {l2 / 1e6:.0f} MB of L2)",
                       "graph": f"{G} calls per CUDA graph ({NG} graphs over the copies), {K // G} replays, "
                                f"the last with per-kernel events", "parallelism": f"replicas{world}"},
            "roofline": roof,
            "stages_us": stages,
            "hbm": hbm,
            "clocks": ck,
            "e2e": e2e,
            "gpu_launches": K * launches_per_call,
            # stage-1 counters over every call of the run: stages replaced by
            # their exact top-128, candidate buffers cut back to their exact
            # top-128, and bulk copies that did not land within the wait limit
            # (nonzero: the run's results are not valid)
            "self_check": {"stage_fallbacks": int(diag[0]), "buffer_compactions": int(diag[4]),
                           "copy_timeouts": int(diag[3])},
            "configs": configs,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c5", choices=["c5", "c2", "c3", "c4", "c1", "c4_onehot", "c4_bounded", "c2_exact"])
    ap.add_argument("--tile", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-configs", action="store_true",
                    help="time only the main workload (by default a c5 run also times c1-c4)")
    args = ap.parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: relaunch under torch.distributed.run
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
        os.execv(sys.executable, cmd)
    if "WORLD_SIZE" in os.environ and int(os.environ["WORLD_SIZE"]) != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={os.environ['WORLD_SIZE']}")
    if args.impl == "ours":
        args.warmup = max(args.warmup, 3)
    w, desc = workload(args.workload)
    if args.impl == "reference":
        run_reference(args, w, desc)
    else:
        run_ours(args, w, desc)


if __name__ == "__main__":
    main()
