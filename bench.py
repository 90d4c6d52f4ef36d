"""Benchmark of the MoE permute + FP8 group-quant + combine hot path on GB300.

One step = one compact dispatch (route plan + group-128 UE8M0 quantisation +
scatter + m_indices) followed by one top-k weighted combine, on the prefill
workload: T = 8192 tokens, hidden 7168, 256 local experts, top-8 routing with a
Zipf(1.2) popularity and >= 10 empty experts, block_e = 128, packed UE8M0
scales. The metric is algorithmic bytes moved per second (dispatch + combine),
with the dispatch and combine figures, routed tokens/s, the roofline of the
dominant kernel against the measured HBM copy bandwidth, the CPU oracle as a
reported baseline, and the other hot-path rows timed on their own workloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 launch with torchrun; every rank runs an independent replica of the
workload (no collective on the data path) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "dispatch+quant & combine GB/s and % of GB300 HBM peak; routed tokens/s"
UNIT = "GB/s"
WORKLOAD = "prefill compact: T=8192 H=7168 E=L=256 top8 Zipf(1.2) block_e=128 g128 packed-UE8M0"
L2_FLUSH_BYTES = 512 << 20


class L2Flush:
    """Evict L2 between timed steps: write a buffer larger than L2, then read
    another one, so the step starts with an L2 of clean, unrelated lines and
    is not charged for writing back the flush buffer's dirty lines."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.zeros(L2_FLUSH_BYTES // 2, dtype=torch.int32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.max()


# ---------------------------------------------------------------------------
# algorithmic bytes (what the definition must read and write, once)
# ---------------------------------------------------------------------------

def dispatch_bytes(T, H, K, L, b, g, kept):
    """x read once; ids read; payload + packed scales written per kept slot;
    m_indices over the static bound; src2dst written."""
    G = H // g
    bound = b * (min(T * K, L) + (T * K - min(T * K, L)) // b)
    return (T * H * 2 + T * K * 4 + kept * H + kept * ((G + 3) // 4) * 4 + bound * 4 + T * K * 4)


def combine_bytes(T, H, K, kept):
    """one bf16 row read per kept slot; src2dst and weights read; out written."""
    return kept * H * 2 + T * K * 4 + T * K * 4 + T * H * 2


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampling
# ---------------------------------------------------------------------------

class Clocks:
    def __init__(self, gpu_index: int):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        self.p.wait()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample of the same workload)
# ---------------------------------------------------------------------------

_PREFILL_CACHE = {}


def prefill_inputs(seed=0):
    if seed not in _PREFILL_CACHE:
        _PREFILL_CACHE[seed] = synth.prefill(seed)
    return _PREFILL_CACHE[seed]


def oracle_sample(tokens: int, reps: int, start: int = 0):
    import oracle as ref
    d = prefill_inputs(0)
    c = d["cfg"]
    T, H, K, L, b, g = tokens, c["H"], c["K"], c["L"], c["block_e"], c["g"]
    sl = slice(start, start + T)
    x, ids, w = d["x"][sl].copy(), d["topk_ids"][sl].copy(), d["topk_weights"][sl].copy()
    bound = ref.compact_bound(T * K, L, b)
    y = synth.expert_outputs(np.random.default_rng(11), bound, H)
    xq = np.zeros((bound, H), np.uint8)
    sc, ld = ref.scale_buffer("packed", bound, H // g)
    mi = np.zeros(bound, np.int32)
    s2d = np.zeros((T, K), np.int32)
    cnt, st, ps = (np.zeros(L, np.int32) for _ in range(3))
    tot = np.zeros(1, np.int32)
    kept = int(((ids >= 0) & (ids < L)).sum())
    nbytes = dispatch_bytes(T, H, K, L, b, g, kept) + combine_bytes(T, H, K, kept)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        ref.dispatch_compact(x, T, T, H, ids, w, K, L, b, g, "packed", xq, sc, ld, mi, bound, s2d,
                             cnt, st, ps, tot)
        ref.combine_f32(y, s2d, w, T, K, H)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    return dict(value=nbytes / t / 1e9, unit=UNIT, cores=1, kind="oracle",
                sample=f"first {T} of 8192 prefill tokens (all H=7168 columns), dispatch + "
                       f"combine, median of {reps}, single-threaded C oracle",
                seconds=t, tokens_per_s=T / t)


def _oracle_core_worker(i, tokens, barrier, cmd, out):
    """One host core: build the inputs once, then for every "run" command wait
    for all cores and run the oracle once on this core's own token window."""
    start = (i * tokens) % (8192 - tokens + 1)
    prefill_inputs(0)
    oracle_sample(tokens, 1, start=start)   # warm (oracle load, caches)
    while cmd.get() is not None:
        barrier.wait(timeout=600)
        t0 = time.perf_counter()
        r = oracle_sample(tokens, 1, start=start)
        out.put((t0, time.perf_counter(), r["value"] * r["seconds"]))


class OracleCores:
    """The oracle as it stands on every host core at once: one spawned process
    per core (spawn: this process may already hold a CUDA context), each on its
    own window of `tokens` prefill tokens (16 cores x 512 tokens cover the whole
    8192-token batch). step() runs every core once and returns (GB/s, seconds):
    all bytes / the span from the first start to the last end."""

    def __init__(self, tokens: int = 512):
        import multiprocessing as mproc
        self.n = len(os.sched_getaffinity(0))
        self.tokens = tokens
        ctx = mproc.get_context("spawn")
        # held for the pool's lifetime: the workers open these by name
        self.barrier, self.out = ctx.Barrier(self.n), ctx.Queue()
        self.cmd = [ctx.Queue() for _ in range(self.n)]
        self.procs = [ctx.Process(target=_oracle_core_worker,
                                  args=(i, tokens, self.barrier, self.cmd[i], self.out), daemon=True)
                      for i in range(self.n)]
        for p in self.procs:
            p.start()

    def step(self):
        import queue
        for q in self.cmd:
            q.put("run")
        res, waited = [], 0.0
        while len(res) < self.n:
            try:
                res.append(self.out.get(timeout=5))
            except queue.Empty:
                waited += 5
                if waited > 900 or any(p.exitcode is not None for p in self.procs):
                    raise RuntimeError("an oracle worker process stopped")
        span = max(r[1] for r in res) - min(r[0] for r in res)
        return sum(r[2] for r in res) / span, span

    def close(self):
        for q in self.cmd:
            q.put(None)
        for p in self.procs:
            p.join(timeout=60)
            if p.exitcode is None:
                p.terminate()


def oracle_all_cores(tokens: int = 512, reps: int = 3):
    """One warm-up step of OracleCores, then the median of `reps` steps."""
    pool = OracleCores(tokens)
    try:
        pool.step()
        runs = sorted(pool.step() for _ in range(reps))
    finally:
        pool.close()
    v, span = runs[len(runs) // 2]
    return dict(value=v, cores=pool.n, seconds=span, tokens=pool.n * tokens)


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def step_config(world, T=None):
    """The workload's `config`, identical in both arms (the reference arm runs
    the same workload on the host, so the GPU arm's L2 flush is named for what
    it is). T overrides the token count (--tokens)."""
    c = synth.PREFILL
    T = c["T"] if T is None else T
    H, K, E, L, b, g = c["H"], c["K"], c["E"], c["L"], c["block_e"], c["g"]
    work = WORKLOAD if T == c["T"] else WORKLOAD.replace(f"T={c['T']}", f"T={T}")
    return {"workload": work, "T": T, "H": H, "K": K, "E": E, "L": L, "block_e": b,
            "group": g, "scales": "packed UE8M0",
            "bound_rows": b * (min(T * K, L) + (T * K - min(T * K, L)) // b),
            "l2": (f"GPU arm: flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write + "
                   f"{L2_FLUSH_BYTES >> 20} MiB read, outside the events); CPU arm: no flush"),
            "parallelism": f"replicas x{world} (no collective on the data path)"}


# ---------------------------------------------------------------------------
# reference arm: the oracle as it stands, on host cores
# ---------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return
    pool = OracleCores(512)
    try:
        for _ in range(args.warmup):
            pool.step()
        runs = [pool.step() for _ in range(args.steps)]
    finally:
        pool.close()
    v = statistics.median(r[0] for r in runs)
    secs = [r[1] for r in runs]
    sample = (f"{pool.n} processes, one per host core, each running the single-threaded C oracle "
              f"(dispatch + combine) on its own window of {pool.tokens} prefill tokens per step "
              f"({pool.n * pool.tokens} tokens per step)")
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(secs) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3",
        "data": "synthetic (seeded numpy: Zipf top-8 routing, N(0,1) activations)",
        "config": step_config(args.gpus),
        "sample_tokens_per_step": pool.n * pool.tokens,
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": pool.n, "kind": "oracle",
                         "sample": sample, "cpu": cpu_model()},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import combine_fp8_quant_gb300 as mp
    from combine_fp8_quant_gb300 import build as cuda_build

    if rank == 0:
        cuda_build.build()
    if world > 1:
        dist.barrier()
    mp.load()
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)

    d = synth.prefill(rank, T=args.tokens)
    c = d["cfg"]
    T, H, K, E, L, b, g = c["T"], c["H"], c["K"], c["E"], c["L"], c["block_e"], c["g"]
    x_h = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16)
    ids_h = torch.from_numpy(d["topk_ids"])
    w_h = torch.from_numpy(d["topk_weights"])
    x, ids, w = x_h.to(dev), ids_h.to(dev), w_h.to(dev)
    bound = mp.moe_compact_bound(T * K, L, b)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7000 + rank)
    y = torch.randn((bound, H), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    kept = int(((d["topk_ids"] >= 0) & (d["topk_ids"] < L)).sum())
    db = dispatch_bytes(T, H, K, L, b, g, kept)
    cb = combine_bytes(T, H, K, kept)

    ws = mp.Workspace(T, K, L, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    xq = torch.empty((bound, H), dtype=torch.uint8, device=dev)
    sc, ld = mp.scale_tensor("packed", bound, H, g, dev)
    mi = torch.empty(bound, dtype=torch.int32, device=dev)
    s2d = torch.empty((T, K), dtype=torch.int32, device=dev)
    cnt, sts, ps = (torch.empty(L, dtype=torch.int32, device=dev) for _ in range(3))
    tot = torch.empty(1, dtype=torch.int32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)

    def dispatch(xx, ii):
        code = mp.moe_dispatch_compact(xx, H, T, None, H, ii, None, K, E, L, b, g, "packed", xq, sc,
                                       ld, mi, bound, s2d, cnt, sts, ps, tot, None, ws.buf,
                                       ws.nbytes, st)
        assert code == 0, code

    def combine(yy, ww, oo):
        code = mp.moe_combine(yy, H, bound, s2d, ww, T, None, K, H, oo, st)
        assert code == 0, code

    # -- device-resident timing ----------------------------------------------
    # The step (the dispatch call then the combine call) is captured once in a
    # CUDA graph: the calls launch fixed grids that depend only on scalar
    # arguments. Every timed step flushes L2 (outside the events) and replays
    # the graph between two CUDA events. The per-call split comes from a
    # second loop that replays one graph per call with an event between them
    # (that event itself costs a few microseconds per step), and the same
    # steps through direct calls follow, reported beside it.
    for _ in range(max(args.warmup, 3)):
        dispatch(x, ids)
        combine(y, w, out)
    torch.cuda.synchronize()
    assert mp.moe_status_sync(st) == 0
    g_step, g_disp, g_comb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        dispatch(x, ids)
        combine(y, w, out)
    with torch.cuda.graph(g_disp):
        dispatch(x, ids)
    with torch.cuda.graph(g_comb):
        combine(y, w, out)
    for _ in range(max(args.warmup, 3)):
        g_step.replay()
        g_disp.replay()
        g_comb.replay()
    torch.cuda.synchronize()
    assert mp.moe_status_sync(st) == 0
    K_steps = args.steps

    def timed_whole(run_step):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K_steps)]
        for i in range(K_steps):
            flush()                             # L2 flush between timed steps (outside the events)
            ev[i][0].record()
            run_step()
            ev[i][1].record()
        torch.cuda.synchronize()
        return sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(K_steps)) / K_steps

    def timed_steps(run_disp, run_comb):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K_steps)]
        for i in range(K_steps):
            flush()
            ev[i][0].record()
            run_disp()
            ev[i][1].record()
            run_comb()
            ev[i][2].record()
        torch.cuda.synchronize()
        t_disp = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K_steps)]
        t_comb = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K_steps)]
        return sum(t_disp) / K_steps, sum(t_comb) / K_steps

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device() if world == 1 else local_rank)
    ms_step = timed_whole(g_step.replay)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms_step = max_over_ranks([ms_step], world, dev)[0]
    ms_disp, ms_comb = timed_steps(g_disp.replay, g_comb.replay)
    ms_disp, ms_comb = max_over_ranks([ms_disp, ms_comb], world, dev)
    assert mp.moe_status_sync(st) == 0
    torch.cuda.synchronize()
    ms_disp_direct, ms_comb_direct = timed_steps(lambda: dispatch(x, ids), lambda: combine(y, w, out))
    ms_disp_direct, ms_comb_direct = max_over_ranks([ms_disp_direct, ms_comb_direct], world, dev)
    # Each call alone after an L2 flush. Inside the step the combine starts
    # while the dispatch's last payload writes (tens of MB) still drain from
    # L2, so the step's split charges that write-back to the combine.
    us_disp_alone = time_call(lambda: dispatch(x, ids), flush)
    us_comb_alone = time_call(lambda: combine(y, w, out), flush)
    us_disp_alone, us_comb_alone = max_over_ranks([us_disp_alone, us_comb_alone], world, dev)
    assert mp.moe_status_sync(st) == 0

    if args.only_step:
        if rank == 0:
            hbm, _ = peaks()
            print(json.dumps({"only_step": True, "T": T, "ms_per_step": ms_step,
                              "dispatch_us": ms_disp * 1e3, "combine_us": ms_comb * 1e3,
                              "dispatch_gbs": db / (ms_disp * 1e-3) / 1e9,
                              "combine_gbs": cb / (ms_comb * 1e-3) / 1e9, "hbm_peak": hbm,
                              "direct_calls": {"dispatch_us": ms_disp_direct * 1e3,
                                               "combine_us": ms_comb_direct * 1e3},
                              "clocks": clk}), flush=True)
        return

    # -- end to end through the C ABI with host buffers -------------------------
    # Every step copies its inputs (x, ids, weights, expert outputs y) from
    # pinned host memory, runs the two calls and reads the combined output
    # back. Two device buffer sets alternate between steps, so step i+1's
    # host->device copies (the bulk of the time, at the host link's rate,
    # measured on its own below as h2d_link_gbs) overlap step i's compute and
    # its device->host read; y is copied in two halves on two streams.
    x_p, ids_p, w_p = x_h.pin_memory(), ids_h.pin_memory(), w_h.pin_memory()
    y_p = y.cpu().pin_memory()
    out_p = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    sets = [dict(x=torch.empty_like(x), ids=torch.empty_like(ids), w=torch.empty_like(w),
                 y=torch.empty_like(y), out=torch.empty_like(out)) for _ in range(2)]
    del y
    h2d = x_p.numel() * 2 + ids_p.numel() * 4 + w_p.numel() * 4 + y_p.numel() * 2
    d2h = out_p[0].numel() * 2

    main = torch.cuda.current_stream()
    up = [torch.cuda.Stream(), torch.cuda.Stream()]     # host -> device
    down = torch.cuda.Stream()                           # device -> host
    half = y_p.shape[0] // 2
    y_halves = [slice(0, half), slice(half, y_p.shape[0])]
    inputs_in = [[torch.cuda.Event(), torch.cuda.Event()] for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]   # the set's inputs are no longer read
    produced = [torch.cuda.Event() for _ in range(2)]   # the set's output is complete
    read_back = [torch.cuda.Event() for _ in range(2)]  # the set's output reached the host
    for i in range(2):
        consumed[i].record(main)
        read_back[i].record(main)

    def e2e_step(i):
        bset, b = sets[i % 2], i % 2
        for j, (sl, stream) in enumerate(zip(y_halves, up)):
            stream.wait_event(consumed[b])
            with torch.cuda.stream(stream):
                bset["y"][sl].copy_(y_p[sl], non_blocking=True)
                if j == 0:
                    bset["x"].copy_(x_p, non_blocking=True)
                    bset["ids"].copy_(ids_p, non_blocking=True)
                    bset["w"].copy_(w_p, non_blocking=True)
                inputs_in[b][j].record(stream)
        main.wait_event(inputs_in[b][0])
        dispatch(bset["x"], bset["ids"])
        main.wait_event(inputs_in[b][1])
        main.wait_event(read_back[b])
        combine(bset["y"], bset["w"], bset["out"])
        consumed[b].record(main)
        produced[b].record(main)
        down.wait_event(produced[b])
        with torch.cuda.stream(down):
            out_p[b].copy_(bset["out"], non_blocking=True)
            read_back[b].record(down)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    # the host link on its own: the pinned expert outputs (the bulk of each
    # step's host->device bytes) copied to the device on one stream
    lk0, lk1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    lk0.record(main)
    sets[0]["y"].copy_(y_p, non_blocking=True)
    lk1.record(main)
    torch.cuda.synchronize()
    link_gbs = y_p.numel() * 2 / (lk0.elapsed_time(lk1) * 1e-3) / 1e9
    e2e_steps = max(4, min(K_steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for i in range(e2e_steps):
        e2e_step(i)
    main.wait_stream(down)
    e1.record(main)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1) / e2e_steps
    ms_e2e = max_over_ranks([ms_e2e], world, dev)[0]
    assert mp.moe_status_sync(st) == 0
    del sets

    # -- other hot-path rows on their own workloads --------------------------------
    rows = other_rows(mp, dev, flush) if rank == 0 else None

    if rank != 0:
        return
    hbm, peak_kind = peaks()
    step_bytes = (db + cb) * world
    value = whole_job_gbs(db + cb, world, ms_step)
    comb_gbs = cb / (ms_comb * 1e-3) / 1e9
    disp_gbs = db / (ms_disp * 1e-3) / 1e9
    traffic = load_traffic("combine")
    cpu = oracle_sample(2048, 3)
    cpu_all = oracle_all_cores(512)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K_steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3 (u8), fp32 accumulate",
        "data": "synthetic (seeded: numpy Zipf top-8 routing and N(0,1) x; torch N(0,1) expert outputs)",
        "config": step_config(world, T),
        "timing": "per step: L2 flush, then one CUDA-graph replay of the dispatch call and "
                  "the combine call between two CUDA events (mean of the steps); the "
                  "per-call split in detail comes from a second loop with an event between "
                  "the calls",
        "detail": {
            "dispatch": {"us": ms_disp * 1e3, "gbs": disp_gbs, "frac_of_peak": disp_gbs / hbm,
                         "algorithmic_bytes": db, "launches": 2},
            "combine": {"us": ms_comb * 1e3, "gbs": comb_gbs, "frac_of_peak": comb_gbs / hbm,
                        "algorithmic_bytes": cb, "launches": 1},
            "routed_tokens_per_s": T * world / (ms_step * 1e-3),
            "dispatch_tokens_per_s": T / (ms_disp * 1e-3),
            "assignments_per_s": kept * world / (ms_step * 1e-3),
            "frac_of_nominal_8TBs": value / world / 8000.0,
            "direct_calls": {
                "note": "the same steps through direct C-ABI calls instead of graph replays",
                "dispatch_us": ms_disp_direct * 1e3, "combine_us": ms_comb_direct * 1e3,
                "step_gbs": (db + cb) / ((ms_disp_direct + ms_comb_direct) * 1e-3) / 1e9},
            "each_call_alone": {
                "note": "each call timed on its own after an L2 flush (trimmed mean of 40); inside the "
                        "step the combine also absorbs the write-back of the dispatch's last payload "
                        "rows still dirty in L2",
                "dispatch_us": us_disp_alone, "dispatch_gbs": db / (us_disp_alone * 1e-6) / 1e9,
                "combine_us": us_comb_alone, "combine_gbs": cb / (us_comb_alone * 1e-6) / 1e9},
        },
        "roofline": {"bound": "hbm", "kernel": "combine_kernel", "achieved": comb_gbs, "peak": hbm,
                     "unit": "GB/s", "frac": comb_gbs / hbm, "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs (copy, burst)"},
        "roofline_dispatch": {"bound": "hbm", "kernel": "route_plan + quant_scatter",
                              "achieved": disp_gbs, "peak": hbm, "unit": "GB/s",
                              "frac": disp_gbs / hbm, "traffic": load_traffic("dispatch")},
        "cpu_baseline": {"value": cpu_all["value"], "unit": UNIT, "cores": cpu_all["cores"],
                         "kind": "oracle",
                         "sample": f"{cpu_all['cores']} processes, one per host core, each running the "
                                   f"single-threaded C oracle (dispatch + combine) on its own window "
                                   f"of 512 prefill tokens ({cpu_all['tokens']} tokens per step); all "
                                   f"bytes / the span from first start to last end; median of 3 "
                                   f"steps after one warm-up step",
                         "cpu": cpu_model(),
                         "single_core": {k: cpu[k] for k in ("value", "cores", "sample")}},
        "e2e": {"value": whole_job_gbs(db + cb, world, ms_e2e), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "api": "moe_dispatch_compact + moe_combine (C ABI), pinned host buffers; two "
                       "device buffer sets alternate so one step's host->device copies overlap "
                       "the previous step's compute and device->host read",
                "h2d_link_gbs": link_gbs,
                "h2d_link_note": "one pinned host->device copy of the expert outputs alone on this "
                                 "box; the step's host->device bytes / this rate bound the e2e step"},
        "gpu_launches": 3 * K_steps,
        "clocks": clk,
        "rows": rows,
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(values, world, device=None):
    """Element-wise max of per-rank timings (a barrier-free all-reduce); the
    whole job is as slow as its slowest replica."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_gbs(bytes_per_rank, world, ms):
    """Aggregate throughput: all ranks' algorithmic bytes over the max time."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


def kernel_source_sha(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "combine_fp8_quant_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(which):
    """DRAM bytes (read + write) per launch of a kernel (per call, for the
    two-launch dispatch) from the committed ncu summary
    profiles/dram_traffic_prefill.txt -- null when absent or when a source
    file of the kernel has changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "dram_traffic_prefill.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#") and parts[0] == which:
            files = parts[3].split(",")
            if parts[2] != kernel_source_sha(files):
                return None
            return int(parts[1])
    return None


class NvtxRange:
    """An NVTX range around a timed row, so that a profiler capture can select
    one row's launches (ncu --nvtx --nvtx-include "<name>/"); a no-op where
    NVTX is unavailable."""

    def __init__(self, name):
        self.name, self.pushed = name, False

    def __enter__(self):
        if self.name:
            try:
                import torch
                torch.cuda.nvtx.range_push(self.name)
                self.pushed = True
            except Exception:
                self.pushed = False
        return self

    def __exit__(self, *exc):
        if self.pushed:
            import torch
            torch.cuda.nvtx.range_pop()
        return False


def time_call(fn, flush, reps=40, name=None):
    """Device time of one call in us, L2 flushed before each: the mean of
    `reps` CUDA-event intervals with the top and bottom 10% dropped. Events on
    this GPU tick in steps of about 2 us, so a median would snap to a tick;
    the trimmed mean averages over the quantisation. `name` labels the calls
    with an NVTX range."""
    with NvtxRange(name):
        return _time_call(fn, flush, reps)


def _time_call(fn, flush, reps):
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ts.sort()
    cut = reps // 10
    kept = ts[cut:reps - cut]
    return sum(kept) / len(kept) * 1e3  # us


def other_rows(mp, dev, flush):
    """The other hot-path rows, each on its own workload (trimmed mean of 40,
    L2 flushed before each call): the decode chain -- masked dispatch with its
    expanded-layout psum, slab -> expanded, expanded -> slab, weighted combine
    from slab rows -- call by call and as one CUDA-graph replay; MXFP8
    live-row quant; the live-row quantiser on a full batch; requant; and
    expanded <-> slab on the requant workload."""
    import torch
    hbm, _ = peaks()
    res = {}

    def entry(us, nbytes):
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"us": us, "gbs": gbs, "frac_of_peak": gbs / hbm, "algorithmic_bytes": nbytes}

    # decode, masked layout
    dd = synth.decode(0)
    c = dd["cfg"]
    T, H, K, E, L, cap, g = c["T"], c["H"], c["K"], c["E"], c["L"], c["cap"], c["g"]
    x = torch.from_numpy(dd["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    ids = torch.from_numpy(dd["topk_ids"]).to(dev)
    w = torch.from_numpy(dd["topk_weights"]).to(dev)
    ws = mp.Workspace(T, K, L, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    xq = torch.empty((L, cap, H), dtype=torch.uint8, device=dev)
    sc, ld = mp.scale_tensor("packed", L * cap, H, g, dev, blocks=L)
    mm = torch.empty(L, dtype=torch.int32, device=dev)
    s2d = torch.empty((T, K), dtype=torch.int32, device=dev)
    kept = int(((dd["topk_ids"] >= 0) & (dd["topk_ids"] < L)).sum())
    live_tok = int((((dd["topk_ids"] >= 0) & (dd["topk_ids"] < L)).any(axis=1)).sum())

    align = c["align"]
    psum = torch.empty(L, dtype=torch.int32, device=dev)
    G4 = (H // g + 3) // 4
    R = mp.moe_compact_bound(T * K, L, align)     # static rows of the expanded layout
    exp = torch.empty((R, H), dtype=torch.uint8, device=dev)
    esc, ld_es = mp.scale_tensor("packed", R, H, g, dev)
    mi = torch.empty(R, dtype=torch.int32, device=dev)
    slab2 = torch.empty_like(xq)
    sc2 = torch.empty_like(sc)
    mm2 = torch.empty_like(mm)
    yslab = torch.randn((L * cap, H), device=dev).to(torch.bfloat16)
    outd = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

    def dec():
        assert mp.moe_dispatch_masked(x, H, T, None, H, ids, None, K, E, L, cap, g, "packed", xq, sc,
                                      ld, mm, s2d, None, psum, align, ws.buf, ws.nbytes, st) == 0

    def from_slab():
        assert mp.moe_expand_from_slab(xq, 1, H, sc, ld, psum, L, align, cap, "packed", g, None, exp,
                                       R, esc, ld_es, mi, st) == 0

    def to_slab():
        assert mp.moe_expand_to_slab(exp, 1, H, R, esc, ld_es, psum, L, align, cap, "packed", g,
                                     slab2, sc2, ld, mm2, st) == 0

    def decomb():
        assert mp.moe_combine(yslab, H, L * cap, s2d, w, T, None, K, H, outd, st) == 0

    # x rows of tokens with a local slot and ids read; payload + scale words per
    # kept slot, masked_m + psum and src2dst written
    nb_disp = live_tok * H * 2 + T * K * 4 + kept * (H + 4 * G4) + L * 8 + T * K * 4
    nb_repack = 2 * kept * (H + 4 * G4) + L * 4          # rows and scale words, read + written
    nb_from = nb_repack + R * 4                           # + m_indices over the expanded rows
    nb_to = nb_repack + L * 4                             # + masked_m
    nb_comb = kept * H * 2 + T * K * 8 + T * H * 2
    res["decode_masked_dispatch"] = entry(time_call(dec, flush, name="decode_masked_dispatch"), nb_disp)
    res["decode_slab_to_expand"] = entry(time_call(from_slab, flush, name="decode_slab_to_expand"), nb_from)
    res["decode_expand_to_slab"] = entry(time_call(to_slab, flush, name="decode_expand_to_slab"), nb_to)
    res["decode_combine_from_slab"] = entry(time_call(decomb, flush, name="decode_combine_from_slab"), nb_comb)
    # the whole decode chain, captured once, as one graph replay
    dec(), from_slab(), to_slab(), decomb()
    torch.cuda.synchronize()
    gchain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gchain):
        dec()
        from_slab()
        to_slab()
        decomb()
    res["decode_chain_graph"] = entry(time_call(gchain.replay, flush, name="decode_chain_graph"),
                                      nb_disp + nb_from + nb_to + nb_comb)
    res["decode_chain_graph"]["launches"] = 4
    res["decode_chain_graph"]["expanded_rows"] = R
    del gchain

    # MXFP8 sparse buffer: 112 live rows of 24576
    dm = synth.mxfp8(0)
    cm = dm["cfg"]
    xb = torch.from_numpy(dm["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    nl = torch.tensor([cm["n_live"]], dtype=torch.int32, device=dev)
    xqm = torch.empty((cm["T_cap"], cm["H"]), dtype=torch.uint8, device=dev)
    scm = torch.empty((cm["T_cap"], cm["H"] // 32), dtype=torch.uint8, device=dev)

    def mx():
        assert mp.moe_quant_group(xb, cm["H"], cm["T_cap"], nl, cm["H"], 32, "u8", xqm, scm,
                                  cm["H"] // 32, st) == 0
    us = time_call(mx, flush, name="mxfp8_live_quant")
    res["mxfp8_live_quant"] = entry(us, cm["n_live"] * cm["H"] * 3 + cm["n_live"] * 224)
    res["mxfp8_live_quant"]["capacity_rows"] = cm["T_cap"]
    # the same quantiser on a full prefill batch (8192 rows, group 128, packed)
    xf = torch.from_numpy(prefill_inputs(0)["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    Tq, Hq = xf.shape
    xqf = torch.empty((Tq, Hq), dtype=torch.uint8, device=dev)
    scf, ldf = mp.scale_tensor("packed", Tq, Hq, 128, dev)

    def qf():
        assert mp.moe_quant_group(xf, Hq, Tq, None, Hq, 128, "packed", xqf, scf, ldf, st) == 0
    res["quant_group_prefill"] = entry(time_call(qf, flush, name="quant_group_prefill"), Tq * Hq * 3 + Tq * (Hq // 128))
    res["quant_group_prefill"]["rows"] = Tq
    del xf, xqf, scf

    # requant and expand <-> slab on the 4096-row workload, and on the same
    # rows tiled 4x (16384 rows, 4x the expert blocks): the small workload is
    # dominated by launch and first-access latency, the larger one shows the
    # kernels' streaming rate.
    dr = synth.requant(0)
    cr = dr["cfg"]
    for tag, rep in (("", 1), ("_x4", 4)):
        q = torch.from_numpy(np.tile(dr["q"], (rep, 1))).to(dev)
        s = torch.from_numpy(np.tile(dr["s_tok"], rep)).to(dev)
        T, H = q.shape
        qo = torch.empty_like(q)
        S = torch.empty(1, dtype=torch.float32, device=dev)

        def rq():
            assert mp.fp8_requant_per_tensor(q, H, s, T, H, qo, S) == 0
        res["requant_per_tensor" + tag] = entry(time_call(rq, flush, name="requant_per_tensor" + tag), 2 * T * H + T * 4 + 4)
        res["requant_per_tensor" + tag]["rows"] = T

        counts = synth.repack_counts(np.random.default_rng(17 + rep), cr["L"], cr["blocks"] * rep,
                                     cr["align"])
        psum_l, prev = [], 0
        for cnt in counts:
            st0 = -(-prev // 128) * 128
            psum_l.append(st0 + int(cnt))
            prev = st0 + int(cnt)
        R = T
        capr = int(-(-counts.max() // 128) * 128)
        psum = torch.tensor(psum_l, dtype=torch.int32, device=dev)
        G = H // 128
        esc, ld_es = mp.scale_tensor("packed", R, H, 128, dev)
        slab = torch.empty((cr["L"] * capr, H), dtype=torch.uint8, device=dev)
        ssc, ld_ss = mp.scale_tensor("packed", cr["L"] * capr, H, 128, dev, blocks=cr["L"])
        mmr = torch.empty(cr["L"], dtype=torch.int32, device=dev)
        back = torch.empty_like(q)
        mi = torch.empty(R, dtype=torch.int32, device=dev)
        real = int(counts.sum())

        def to_slab():
            assert mp.moe_expand_to_slab(q, 1, H, R, esc, ld_es, psum, cr["L"], 128, capr, "packed",
                                         128, slab, ssc, ld_ss, mmr, st) == 0

        def from_slab():
            assert mp.moe_expand_from_slab(slab, 1, H, ssc, ld_ss, psum, cr["L"], 128, capr,
                                           "packed", 128, None, back, R, esc, ld_es, mi, st) == 0
        nb = 2 * real * (H + ((G + 3) // 4) * 4) + cr["L"] * 8
        res["expand_to_slab" + tag] = entry(time_call(to_slab, flush, name="expand_to_slab" + tag), nb)
        res["slab_to_expand" + tag] = entry(time_call(from_slab, flush, name="slab_to_expand" + tag), nb + R * 4)
        res["expand_to_slab" + tag]["real_rows"] = real
        del q, qo, slab, back
    torch.cuda.synchronize()
    assert mp.moe_status_sync(st) == 0
    return res


def layout_sweep(args):
    """Compact vs masked dispatch cost of these kernels over (T, L) -- the
    layout question the PR #33128 review raises (compact slower than masked
    below ~8192 tokens with 128 local experts), restricted to the permute /
    quantise step (no GEMM). Uniform top-8 routing over 256 experts of which
    the first L are local; the masked capacity is the largest expert's count
    rounded up to 128. One JSON line per point."""
    import torch
    import combine_fp8_quant_gb300 as mp
    from combine_fp8_quant_gb300 import build as cuda_build
    cuda_build.build()
    mp.load()
    dev = torch.device("cuda:0")
    flush = L2Flush(dev)
    H, K, E, g = 7168, 8, 256, 128
    for T in (128, 512, 2048, 8192):
        rng = np.random.default_rng(T)
        x = torch.from_numpy(synth.normal_bf16(rng, (T, H)).view(np.int16)).to(dev).view(torch.bfloat16)
        ids_np = synth.uniform_topk(rng, T, E, K)
        ids = torch.from_numpy(ids_np).to(dev)
        for L in (32, 128, 256):
            cnt = np.bincount(ids_np[ids_np < L].ravel(), minlength=L)
            cap = max(128, int(-(-cnt.max() // 128) * 128))
            ws = mp.Workspace(T, K, L, dev)
            st = torch.zeros(1, dtype=torch.int32, device=dev)
            bound = mp.moe_compact_bound(T * K, L, 128)
            xq = torch.empty((bound, H), dtype=torch.uint8, device=dev)
            sc, ld = mp.scale_tensor("packed", bound, H, g, dev)
            mi = torch.empty(bound, dtype=torch.int32, device=dev)
            s2d = torch.empty((T, K), dtype=torch.int32, device=dev)
            c3 = [torch.empty(L, dtype=torch.int32, device=dev) for _ in range(3)]
            tot = torch.empty(1, dtype=torch.int32, device=dev)
            xqm = torch.empty((L, cap, H), dtype=torch.uint8, device=dev)
            scm, ldm = mp.scale_tensor("packed", L * cap, H, g, dev, blocks=L)
            mm = torch.empty(L, dtype=torch.int32, device=dev)

            def compact():
                assert mp.moe_dispatch_compact(x, H, T, None, H, ids, None, K, E, L, 128, g, "packed",
                                               xq, sc, ld, mi, bound, s2d, *c3, tot, None, ws.buf,
                                               ws.nbytes, st) == 0

            def masked():
                assert mp.moe_dispatch_masked(x, H, T, None, H, ids, None, K, E, L, cap, g, "packed",
                                              xqm, scm, ldm, mm, s2d, None, None, 128, ws.buf,
                                              ws.nbytes, st) == 0
            uc, um = time_call(compact, flush), time_call(masked, flush)
            torch.cuda.synchronize()
            assert mp.moe_status_sync(st) == 0
            print(json.dumps({"layout_sweep": True, "T": T, "L": L, "E": E, "kept_slots": int(cnt.sum()),
                              "compact_rows": bound, "masked_rows": L * cap, "compact_us": uc,
                              "masked_us": um, "masked_over_compact": um / uc}), flush=True)
            del xq, sc, mi, xqm, scm


def shape_sweep(args):
    """The dispatch + combine step on other MoE shapes (hidden size, experts,
    top-k, tokens), all experts local, Zipf(1.2) routing with 12 empty experts
    where there are enough experts, group-128 packed UE8M0 scales, block_e
    128. Each call and the whole step are timed as CUDA-graph replays after
    an L2 flush (trimmed mean of 40). One JSON line per shape."""
    import torch
    import combine_fp8_quant_gb300 as mp
    from combine_fp8_quant_gb300 import build as cuda_build
    cuda_build.build()
    mp.load()
    dev = torch.device("cuda:0")
    flush = L2Flush(dev)
    hbm, _ = peaks()
    g, b = 128, 128
    for T, H, E, K in ((8192, 7168, 256, 8), (32768, 7168, 256, 8), (8192, 4096, 128, 8),
                       (8192, 5120, 160, 6), (16384, 2048, 64, 6), (4096, 7168, 256, 8)):
        L = E
        rng = np.random.default_rng(T + H + E + K)
        x = torch.from_numpy(synth.normal_bf16(rng, (T, H)).view(np.int16)).to(dev).view(torch.bfloat16)
        ids_np = synth.zipf_topk(rng, T, E, K, n_empty=min(12, E - K))
        ids = torch.from_numpy(ids_np).to(dev)
        w = torch.from_numpy(synth.softmax_weights(rng, T, K)).to(dev)
        kept = int(((ids_np >= 0) & (ids_np < L)).sum())
        db, cbytes = dispatch_bytes(T, H, K, L, b, g, kept), combine_bytes(T, H, K, kept)
        ws = mp.Workspace(T, K, L, dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        bound = mp.moe_compact_bound(T * K, L, b)
        xq = torch.empty((bound, H), dtype=torch.uint8, device=dev)
        sc, ld = mp.scale_tensor("packed", bound, H, g, dev)
        mi = torch.empty(bound, dtype=torch.int32, device=dev)
        s2d = torch.empty((T, K), dtype=torch.int32, device=dev)
        c3 = [torch.empty(L, dtype=torch.int32, device=dev) for _ in range(3)]
        tot = torch.empty(1, dtype=torch.int32, device=dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(T)
        y = torch.randn((bound, H), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

        def disp():
            assert mp.moe_dispatch_compact(x, H, T, None, H, ids, None, K, E, L, b, g, "packed", xq, sc,
                                           ld, mi, bound, s2d, *c3, tot, None, ws.buf, ws.nbytes, st) == 0

        def comb():
            assert mp.moe_combine(y, H, bound, s2d, w, T, None, K, H, out, st) == 0
        disp()
        comb()
        torch.cuda.synchronize()
        graphs = {}
        for name, fns in (("step", (disp, comb)), ("dispatch", (disp,)), ("combine", (comb,))):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                for fn in fns:
                    fn()
            graphs[name] = gr
        us = {name: time_call(gr.replay, flush) for name, gr in graphs.items()}
        torch.cuda.synchronize()
        assert mp.moe_status_sync(st) == 0
        line = {"shape_sweep": True, "T": T, "H": H, "E": E, "K": K, "kept_slots": kept}
        for name, nbytes in (("step", db + cbytes), ("dispatch", db), ("combine", cbytes)):
            gbs = nbytes / (us[name] * 1e-6) / 1e9
            line[name] = {"us": us[name], "gbs": gbs, "frac_of_peak": gbs / hbm}
        print(json.dumps(line), flush=True)
        del graphs, y, xq, x


def only_dispatch(args):
    """The prefill dispatch call alone (route plan + quantise/scatter), W
    warm-up calls then K calls through the C ABI, with no expert outputs
    allocated (about 0.8 GB on the device): the case profiler captures of the
    dispatch kernels run on. Prints one JSON line."""
    import torch

    import combine_fp8_quant_gb300 as mp
    from combine_fp8_quant_gb300 import build as cuda_build
    cuda_build.build()
    mp.load()
    dev = torch.device("cuda:0")
    d = synth.prefill(0, T=args.tokens)
    c = d["cfg"]
    T, H, K, E, L, b, g = c["T"], c["H"], c["K"], c["E"], c["L"], c["block_e"], c["g"]
    x = torch.from_numpy(d["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    ids = torch.from_numpy(d["topk_ids"]).to(dev)
    bound = mp.moe_compact_bound(T * K, L, b)
    ws = mp.Workspace(T, K, L, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    xq = torch.empty((bound, H), dtype=torch.uint8, device=dev)
    sc, ld = mp.scale_tensor("packed", bound, H, g, dev)
    mi = torch.empty(bound, dtype=torch.int32, device=dev)
    s2d = torch.empty((T, K), dtype=torch.int32, device=dev)
    c3 = [torch.empty(L, dtype=torch.int32, device=dev) for _ in range(3)]
    tot = torch.empty(1, dtype=torch.int32, device=dev)
    for _ in range(args.warmup + args.steps):
        assert mp.moe_dispatch_compact(x, H, T, None, H, ids, None, K, E, L, b, g, "packed", xq, sc, ld,
                                       mi, bound, s2d, *c3, tot, None, ws.buf, ws.nbytes, st) == 0
    torch.cuda.synchronize()
    assert mp.moe_status_sync(st) == 0
    print(json.dumps({"only_dispatch": True, "T": T, "calls": args.warmup + args.steps}), flush=True)


def only_rows(args):
    """The other hot-path rows alone (no prefill step, e2e or CPU baseline),
    each labelled with an NVTX range; for profiler captures of their kernels."""
    import torch
    import combine_fp8_quant_gb300 as mp
    from combine_fp8_quant_gb300 import build as cuda_build
    cuda_build.build()
    mp.load()
    dev = torch.device("cuda:0")
    rows = other_rows(mp, dev, L2Flush(dev))
    print(json.dumps({"only_rows": True, "rows": rows}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only-step", action="store_true",
                    help="time the dispatch + combine step only (no e2e, other rows or CPU "
                         "baseline); used for profiler captures")
    ap.add_argument("--only-dispatch", action="store_true",
                    help="run W + K prefill dispatch calls and nothing else; for profiler "
                         "captures of the dispatch kernels")
    ap.add_argument("--only-rows", action="store_true",
                    help="time the other hot-path rows only, each in an NVTX range named after its "
                         "row; for profiler captures of their kernels")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T of the prefill workload (profiling smaller cases)")
    ap.add_argument("--layout-sweep", action="store_true",
                    help="compact vs masked dispatch cost over (T, L); one JSON line per point")
    ap.add_argument("--shape-sweep", action="store_true",
                    help="the dispatch + combine step on other (T, H, E, K) shapes; one JSON line per shape")
    args = ap.parse_args()
    if args.only_dispatch:
        only_dispatch(args)
        return
    if args.only_rows:
        only_rows(args)
        return
    if args.layout_sweep:
        layout_sweep(args)
        return
    if args.shape_sweep:
        shape_sweep(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
