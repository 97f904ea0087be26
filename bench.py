#!/usr/bin/env python3
"""Benchmark of the FP8 paged-KV decode-pool hot path on GB300.

One step = one decode step of one layer over one batch: quantise-on-append of
every request's new K/V token into its page, the separate batched page-tag
check, and split-KV decode attention over the e4m3 cache (all of it in
libfp8kv's kernels).  The BF16-cache variant of the same step runs on the
identical values for comparison.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload b32_8k]
  python bench.py --impl reference ...     # the CPU oracle, timed on host cores
  python bench.py --capacity [--kv-budget-gib 4]   # admission curve, BF16 vs FP8 cache
  python bench.py --gemv [--gemv-n 28672 --gemv-k 8192]   # INT4 vs e4m3 weight decode GEMV

Multi-GPU (torchrun): every rank runs an independent replica (its own requests
and pool); nothing on the data path is exchanged, only the timing is reduced.
"""
from __future__ import annotations

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

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = ("decode-attention tokens/s and achieved HBM GB/s (% of GB300 peak), FP8 vs BF16 KV")
UNIT = "tokens/s"


# ---------------------------------------------------------------------------
# distributed plumbing (timing only)
# ---------------------------------------------------------------------------
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# algorithmic bytes (what the method must move per step)
# ---------------------------------------------------------------------------
def attention_bytes(wl, step: int, fp8: bool) -> int:
    """KV bytes of every context token, page-table entries, queries and outputs."""
    lens = wl.seq_lens_after(step).astype(np.int64)
    b = 1 if fp8 else 2
    kv = int(lens.sum()) * 2 * wl.Hkv * wl.D * b
    pages = int((-(-lens // wl.page_size)).sum())
    table = pages * 4
    q = wl.B * wl.Hq * wl.D * 2
    out = wl.B * wl.Hq * (wl.D + 1) * 4
    return kv + table + q + out


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# the sources compiled into the attention kernel's translation unit
KERNEL_SOURCES = ("decode_attn.cu", "attn_plan.cuh", "common.cuh", "step_ops.cuh", "quant.cuh")


def _strip_comments(src: str) -> str:
    """C/C++ source without comments, every run of whitespace made one space
    (a comment marker inside a string or character literal is not a comment)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_digest(read=None) -> str:
    """sha256 prefix of the attention kernel's sources with comments and
    whitespace removed: it changes when the compiled code can, not when a
    comment does.  read(name) -> text overrides where the files come from."""
    import hashlib
    csrc = os.path.join(ROOT, "fp8_paged_kv_gb300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                return f.read()
    body = "\n".join(_strip_comments(read(n)) for n in KERNEL_SOURCES)
    return hashlib.sha256(body.encode("utf-8")).hexdigest()[:16]


def read_profile_traffic(workload: str, tag: str = "fp8"):
    """Per-launch DRAM bytes (read + write) of the attention kernel from the committed
    ncu record, or None when there is none or the kernel source changed since."""
    p = os.path.join(ROOT, "profiles", f"paged_decode_attn_{tag}_{workload}.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if kernel_source_digest() != d.get("source_sha256_16"):
        return None
    return d.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_segment_problem(wl, r: int, h: int, step: int):
    """One (request, kv head) segment as a compact single-head-group problem for
    the oracle: that request's pages with only kv head h, renumbered 0..P-1."""
    import oracle
    L = int(wl.seq_lens_after(step)[r])
    ps, D, G = wl.page_size, wl.D, wl.G
    P = -(-L // ps)
    a, b = int(wl.cu_prompt[r]), int(wl.cu_prompt[r + 1])
    kv = np.full(2 * P * ps * D, 0x7F, np.uint8)
    pt = np.arange(P, dtype=np.int32)[None, :]
    k = np.ascontiguousarray(wl.k_prompt[a:b, h:h + 1])
    v = np.ascontiguousarray(wl.v_prompt[a:b, h:h + 1])
    oracle.kv_prefill(k, v, np.array([0, b - a], np.int32), kv, wl.k_scale, wl.v_scale, pt,
                      None, None, None, fp8=True, Hkv=1, D=D, page_size=ps, num_pages=P)
    kn, vn = wl.step_tokens(step)
    q = np.ascontiguousarray(wl.step_query(step)[r:r + 1, h * G:(h + 1) * G])
    return dict(kn=np.ascontiguousarray(kn[r:r + 1, h:h + 1]), vn=np.ascontiguousarray(vn[r:r + 1, h:h + 1]),
                kv=kv, pt=pt, lens=np.array([L], np.int32), q=q, P=P,
                tags=np.zeros(P, np.uint32), exp=np.zeros((1, P), np.uint32))


def oracle_params(wl) -> dict:
    """The scalars of a workload that the oracle's segment step needs (small
    enough to send to worker processes)."""
    return dict(k_scale=float(wl.k_scale), v_scale=float(wl.v_scale), sm_scale=float(wl.sm_scale),
                page_size=int(wl.page_size), D=int(wl.D))


def oracle_segment_step(par: dict, prob) -> None:
    """The oracle's decode step on one segment: append, tag check, fp64 attention."""
    import oracle
    ps = par["page_size"]
    k_scale, v_scale = np.float32(par["k_scale"]), np.float32(par["v_scale"])
    oracle.kv_append(prob["kn"], prob["vn"], prob["kv"], k_scale, v_scale,
                     prob["pt"], prob["lens"], prob["tags"], prob["exp"], None, fp8=True, Hkv=1,
                     D=par["D"], page_size=ps, num_pages=prob["P"])
    mask, _ = oracle.page_tags_validate(prob["pt"], prob["exp"], prob["lens"], prob["tags"],
                                        prob["P"], ps)
    oracle.paged_attention(prob["q"], prob["kv"], prob["pt"], prob["lens"], fp8=True,
                           k_scale=k_scale, v_scale=v_scale, abort_mask=mask,
                           sm_scale=par["sm_scale"], Hkv=1, page_size=ps, num_pages=prob["P"])


def _oracle_worker(job):
    """One host core: segment steps over its problems, round robin, until the
    time budget is spent (or `rounds` steps); returns (segments, seconds)."""
    par, probs, budget_s, rounds = job
    done, t0 = 0, time.perf_counter()
    while (rounds is None and time.perf_counter() - t0 < budget_s) or (rounds is not None and done < rounds):
        oracle_segment_step(par, probs[done % len(probs)])
        done += 1
    return done, time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_threads(n: int):
    """n host threads for the oracle.  Its work runs in C called through ctypes,
    which releases the interpreter lock, so the threads run on n cores."""
    import concurrent.futures as cf
    return cf.ThreadPoolExecutor(max_workers=n)


def cpu_baseline(wl, budget_s: float = 10.0):
    """Oracle throughput on a bounded sample: (request, kv head) segments, on
    every host core at once (one thread per core, ~budget_s of work each) and
    on one core; one segment is 1/Hkv token."""
    import oracle
    oracle.build()
    par = oracle_params(wl)
    g = np.random.default_rng(0)
    n = host_cores()
    probs = [oracle_segment_problem(wl, int(g.integers(0, wl.B)), int(g.integers(0, wl.Hkv)), 0)
             for _ in range(2 * n)]
    one, t_one = _oracle_worker((par, probs[:2], budget_s / 4, None))
    with oracle_threads(n) as pool:
        t0 = time.perf_counter()
        res = list(pool.map(_oracle_worker, [(par, probs[2 * i:2 * i + 2], budget_s, None) for i in range(n)]))
        wall = time.perf_counter() - t0
    done = sum(d for d, _ in res)
    return {"value": done / wl.Hkv / wall, "unit": UNIT, "cores": n, "kind": "oracle",
            "single_core_value": one / wl.Hkv / t_one,
            "sample": f"{done} (request, kv head) segments of {wl.name} (append + tag check + fp64 "
                      f"attention each) on {n} threads, {wall:.1f} s wall; one thread: {one} "
                      f"segments in {t_one:.1f} s"}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, on the host cores (one
    thread per core, each step one segment per thread)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    from workloads import WORKLOADS
    wl = WORKLOADS[args.workload]()
    par = oracle_params(wl)
    n = host_cores()
    g = np.random.default_rng(1)
    probs = [oracle_segment_problem(wl, int(g.integers(0, wl.B)), int(g.integers(0, wl.Hkv)), 0)
             for _ in range(n)]
    jobs = [(par, [probs[i]], 0.0, 1) for i in range(n)]
    with oracle_threads(n) as pool:
        for _ in range(args.warmup):
            list(pool.map(_oracle_worker, jobs))
        t0 = time.perf_counter()
        for _ in range(args.steps):
            list(pool.map(_oracle_worker, jobs))
        dt = time.perf_counter() - t0
    tokens = args.steps * n / wl.Hkv
    value = tokens / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": n, "kind": "oracle",
                             "sample": f"each step: {n} (request, kv head) segments of {wl.name} "
                                       f"(append + tag check + fp64 attention), one per host thread"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(wl):
    return {"workload": f"{wl.name}: B={wl.B}, Hq={wl.Hq}, Hkv={wl.Hkv}, D={wl.D}, "
                        f"page_size={wl.page_size}, contexts {int(wl.seq_lens_after(0).min())}.."
                        f"{int(wl.seq_lens_after(0).max())}, pool {wl.num_pages} pages",
            "batch": wl.B, "layers": 1, "step": "append + page-tag validate + split-KV attention",
            "l2": "inputs larger than L2 (KV pool > 129 MB)"}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def time_steps(pool, steps: int, warmup: int, validate: bool = True):
    """Device time of `steps` decode steps; also the attention and validation kernels' own
    event times (events recorded between launches on the launching stream)."""
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        pool.step(validate=validate)
    torch.cuda.synchronize()
    # the step as DecodePool.step runs it (write + tag check in one launch, then
    # attention); events bracket each launch on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s)
    for i in range(steps):
        e = ev[i]
        e[0].record(s)
        if validate:
            pool.append_check(stream=s)
        else:
            pool.append(stream=s)
        e[1].record(s)
        e[2].record(s)
        pool.attend(use_mask=validate, stream=s)
        e[3].record(s)
    end.record(s)
    torch.cuda.synchronize()
    total_ms = start.elapsed_time(end)
    attn = [e[2].elapsed_time(e[3]) for e in ev]
    app = [e[0].elapsed_time(e[1]) for e in ev]
    return total_ms, statistics.mean(attn), statistics.mean(app)


def capture_step(pool, validate: bool = True, io=None):
    """One decode step (and, for io=(h2d, d2h) callables, its host copies) as a CUDA graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            if io:
                io[0]()
            pool.step(validate=validate)
            if io:
                io[1]()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        if io:
            io[0]()
        pool.step(validate=validate)
        if io:
            io[1]()
    torch.cuda.synchronize()
    return g


def time_graph(g, steps: int, warmup: int) -> float:
    """Device ms per replay of a captured step (events on the replay stream)."""
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(steps):
        g.replay()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def capture_steps_sequence(pool, nsteps: int):
    """Decode steps 0..nsteps-1 of a growing workload as ONE graph: before each
    step its context lengths, new K/V rows and query are copied on the device
    from arrays staged once (they are the workload's inputs, not results)."""
    wl = pool.wl
    dev = pool.device
    from fp8_paged_kv_gb300.pool import to_device
    lens = to_device(np.stack([wl.seq_lens_after(s) for s in range(nsteps)]), dev)
    kn, vn, qs = [], [], []
    for s in range(nsteps):
        k, v = wl.step_tokens(s)
        kn.append(k)
        vn.append(v)
        qs.append(wl.step_query(s) if s < 4 else wl.step_query(s % 4))
    K = to_device(np.stack(kn), dev)
    V = to_device(np.stack(vn), dev)
    Q = to_device(np.stack(qs), dev)

    def io(s):
        pool.seq_lens.copy_(lens[s])
        pool.k_new.copy_(K[s])
        pool.v_new.copy_(V[s])
        pool.q.copy_(Q[s])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for s in range(2):
            io(s)
            pool.step(validate=True)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for s in range(nsteps):
            io(s)
            pool.step(validate=True)
    torch.cuda.synchronize()
    return g, (K, V, Q, lens)


def time_prefill(pool, reps: int = 5):
    """The bulk prompt write into the FP8 pages and the device amax -> scale
    reduction over K and V, with the whole prompt resident on the device.  The
    write reuses the pool's own scales, so the cache contents do not change."""
    import fp8_paged_kv_gb300 as fpk
    from fp8_paged_kv_gb300.pool import to_device
    wl = pool.wl
    dev = pool.device
    k = to_device(wl.k_prompt, dev)
    v = to_device(wl.v_prompt, dev)
    cu = to_device(wl.cu_prompt.astype(np.int32), dev)
    ks = torch.empty(1, dtype=torch.float32, device=dev)
    vs = torch.empty(1, dtype=torch.float32, device=dev)
    scratch = torch.zeros(2, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream(dev)

    def write():
        fpk.fpk_kv_prefill_fp8(k, v, cu, pool.kv_pool, pool.k_scale, pool.v_scale, pool.page_table,
                               pool.live_tags, pool.expected_tags, None, **pool.kw)

    def amax():
        fpk.fpk_amax_scale_bf16(k, ks, scratch)
        fpk.fpk_amax_scale_bf16(v, vs, scratch)

    res = []
    for fn in (write, amax):
        fn()
        torch.cuda.synchronize(dev)
        t = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            torch.cuda.synchronize(dev)
            t.append(a.elapsed_time(b))
        res.append(statistics.median(t))
    n = int(wl.k_prompt.size)  # bf16 elements of K (and of V)
    write_bytes = 2 * n * 2 + 2 * n          # read K, V bf16; write their e4m3 codes
    amax_bytes = 2 * n * 2                   # read K and V
    del k, v
    return {"tokens": int(wl.cu_prompt[-1]), "write_us": res[0] * 1e3,
            "write_gbs": write_bytes / (res[0] * 1e-3) / 1e9, "amax_scale_us": res[1] * 1e3,
            "amax_scale_gbs": amax_bytes / (res[1] * 1e-3) / 1e9}


def time_e2e(pool, steps: int, warmup: int, depth: int = 16):
    """The step through the public API with host buffers (DecodePool +
    HostPipeline): every step copies its own inputs (q, new K/V rows, context
    lengths: one buffer) in from pinned host memory and its results (out, lse,
    abort mask: one buffer) back out, with step i+1's copy-in and step i-1's
    copy-out under step i's kernels.  `depth` steps (each with its own host
    buffers) are captured as one CUDA graph and replayed."""
    from fp8_paged_kv_gb300.pool import HostPipeline
    src = pool.io_in.cpu()
    h_in = [src.clone().pin_memory() for _ in range(depth)]
    h_out = [torch.empty_like(pool.io_out, device="cpu").pin_memory() for _ in range(depth)]
    pipe = HostPipeline(pool, h_in, h_out, validate=True)
    h2d, d2h = pipe.bytes_per_step()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        pipe.run(depth)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pipe.run(depth)
    torch.cuda.synchronize()
    reps = max(1, -(-steps // depth))
    ms = time_graph(g, reps, max(1, -(-warmup // depth))) / depth
    return ms, h2d, d2h, reps * depth


class L2Flush:
    """Evicts L2 before a timed launch: a 512 MB write, then a 512 MB read, so the
    launch starts with a cold L2 that holds no dirty lines.  (After the write alone
    ~126 MB of dirty lines are written back while the timed kernel runs, 9-14 us
    on GB300, which no real decode step has: the kernels before attention mostly
    read weights.)"""
    NOTE = "flushed before every timed launch (512 MB write, then 512 MB read)"

    def __init__(self, dev):
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(512 << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.w.zero_()
        self.sink = self.r.sum(dtype=torch.int64)


def run_capacity(args, rank, world):
    """Admission at a fixed KV budget (one layer): how many 8192-token requests of
    the b32_8k shape (Hq=64, Hkv=8, D=128, page 16) fit in the pool with a BF16
    cache and with an e4m3 cache, and decode-attention tokens/s and GB/s at
    concurrencies up to each cap.  Cache values are random codes: only timing is
    taken here (the same kernels are parity-tested elsewhere).  L2 is flushed
    before every timed launch."""
    import fp8_paged_kv_gb300 as fpk
    from fp8_paged_kv_gb300 import build as fbuild
    if rank == 0 or world == 1:
        fbuild.build()
    barrier(world)
    fpk.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    Hq, Hkv, D, ps, L = 64, 8, 128, 16, 8192
    budget = int(args.kv_budget_gib * 2**30)
    ppr = L // ps
    g = torch.Generator(device=dev)
    g.manual_seed(7 + rank)
    flush = L2Flush(dev)
    s = torch.cuda.current_stream(dev)
    curves = {}
    with ClockSampler(local_rank()) as clk:
        for fp8 in (False, True):
            b = 1 if fp8 else 2
            page_bytes = 2 * Hkv * ps * D * b
            num_pages = budget // page_bytes
            cap = num_pages // ppr
            n = num_pages * page_bytes // b
            if fp8:
                pool = torch.randint(0, 0x7F, (n,), dtype=torch.uint8, device=dev, generator=g)
                pool |= torch.randint(0, 2, (n,), dtype=torch.uint8, device=dev, generator=g) << 7
            else:
                pool = torch.randn(n, device=dev, generator=g, dtype=torch.float32).to(torch.bfloat16)
            perm = torch.randperm(num_pages, device=dev, generator=g).to(torch.int32)
            conc = sorted({c for c in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024) if c <= cap} | {cap})
            pts = []
            for c in conc:
                pt = perm[:c * ppr].view(c, ppr).contiguous()
                lens = torch.full((c,), L, dtype=torch.int32, device=dev)
                q = torch.randn(c, Hq, D, device=dev, generator=g).to(torch.bfloat16)
                out = torch.empty(c, Hq, D, device=dev)
                lse = torch.empty(c, Hq, device=dev)
                ws = torch.zeros(fpk.fpk_decode_workspace_bytes(c, Hq, Hkv, D, 0), dtype=torch.uint8,
                                 device=dev)
                ks = torch.tensor([0.01], device=dev)
                kw = dict(Hkv=Hkv, page_size=ps, num_pages=num_pages, sm_scale=D ** -0.5)

                def run():
                    if fp8:
                        fpk.fpk_paged_decode_attn_fp8(q, pool, ks, ks, pt, lens, None, out, lse, ws, **kw)
                    else:
                        fpk.fpk_paged_decode_attn_bf16(q, pool, pt, lens, None, out, lse, ws, **kw)
                t = []
                for i in range(3 + args.capacity_reps):
                    flush()
                    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(s)
                    run()
                    e.record(s)
                    torch.cuda.synchronize(dev)
                    if i >= 3:
                        t.append(a.elapsed_time(e))
                ms = statistics.median(t)
                kv = c * L * 2 * Hkv * D * b
                pts.append({"requests": c, "attn_us": ms * 1e3, "tokens_per_s": c / (ms * 1e-3),
                            "gbs": (kv + c * ppr * 4 + c * Hq * D * 2 + c * Hq * (D + 1) * 4) / (ms * 1e-3) / 1e9})
                del ws, q, out, lse
            curves["fp8" if fp8 else "bf16"] = {"cap_requests": cap, "pool_pages": num_pages,
                                                "points": pts}
            del pool, perm
            torch.cuda.empty_cache()
    bf, f8 = curves["bf16"], curves["fp8"]
    line = {"mode": "capacity", "kv_budget_gib": args.kv_budget_gib, "context": L,
            "shape": f"Hq={Hq}, Hkv={Hkv}, D={D}, page_size={ps}, one layer",
            "bf16": bf, "fp8": f8,
            "fp8_over_bf16_cap": f8["cap_requests"] / max(1, bf["cap_requests"]),
            "fp8_at_cap_over_bf16_at_cap_tokens_per_s":
                f8["points"][-1]["tokens_per_s"] / bf["points"][-1]["tokens_per_s"],
            "l2": L2Flush.NOTE, "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_gemv(args, rank, world):
    """Weight-only quantised decode GEMV (the pages' second technique): INT4
    weights in groups of 128 against e4m3 weights with a row scale, for one
    N x K projection (random-init bf16 weights, synthetic activations) at
    decode batches of 1..16 tokens.  L2 is flushed before every timed launch
    (the INT4 weights alone would fit in it)."""
    import fp8_paged_kv_gb300 as fpk
    from fp8_paged_kv_gb300 import build as fbuild
    if rank == 0 or world == 1:
        fbuild.build()
    barrier(world)
    fpk.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    N, K = args.gemv_n, args.gemv_k
    g = torch.Generator(device=dev)
    g.manual_seed(11 + rank)
    w = (torch.randn(N, K, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    c4 = torch.empty(N * K // 2, dtype=torch.uint8, device=dev)
    s4 = torch.empty(N, K // 128, dtype=torch.bfloat16, device=dev)
    c8 = torch.empty(N * K, dtype=torch.uint8, device=dev)
    r8 = torch.empty(N, dtype=torch.float32, device=dev)
    fpk.fpk_w4_quantize(w, c4, s4)
    fpk.fpk_w8_quantize(w, c8, r8)
    del w
    flush = L2Flush(dev)
    s = torch.cuda.current_stream(dev)
    peak, peak_kind = measured_peaks()
    pts = []
    with ClockSampler(local_rank()) as clk:
        for B in (int(b) for b in args.gemv_batches.split(",")):
            x = torch.randn(B, K, device=dev, generator=g).to(torch.bfloat16)
            y = torch.empty(B, N, device=dev)
            row = {"batch": B}
            for name, fn, wbytes in (("int4", lambda: fpk.fpk_w4_gemv(x, c4, s4, y), N * K // 2 + N * (K // 128) * 2),
                                     ("fp8", lambda: fpk.fpk_w8_gemv(x, c8, r8, y), N * K + N * 4)):
                t = []
                for i in range(3 + args.capacity_reps):
                    flush()
                    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(s)
                    fn()
                    e.record(s)
                    torch.cuda.synchronize(dev)
                    if i >= 3:
                        t.append(a.elapsed_time(e))
                ms = statistics.median(t)
                nbytes = wbytes + B * K * 2 + B * N * 4
                row[name] = {"us": ms * 1e3, "gbs": nbytes / (ms * 1e-3) / 1e9,
                             "frac": nbytes / (ms * 1e-3) / 1e9 / peak, "bytes": nbytes}
            row["int4_speedup"] = row["fp8"]["us"] / row["int4"]["us"]
            pts.append(row)
    line = {"mode": "gemv", "shape": f"N={N}, K={K}, random-init bf16 weights", "points": pts,
            "peak_gbs": peak, "peak_source": peak_kind,
            "l2": L2Flush.NOTE, "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_profile(args):
    """One workload's attention kernel alone, for a profiler: the pool is written,
    one decode step runs (cache write and tag check, then the warp-level
    attention), then `--launches` attention launches of the chosen kernel
    (FP8 or BF16 warp-level, or the FP8 tensor-core variant)."""
    import fp8_paged_kv_gb300 as fpk
    from fp8_paged_kv_gb300 import build as fbuild
    from fp8_paged_kv_gb300.pool import DecodePool
    from workloads import WORKLOADS
    fbuild.build()
    fpk.load_library()
    wl = WORKLOADS[args.workload]()
    pool = DecodePool(wl, fp8=args.profile != "bf16", device=torch.device("cuda", torch.cuda.current_device()),
                      tensor_cores=args.profile == "tc")
    pool.prefill()
    pool.set_step(0)
    pool.step()
    for _ in range(args.launches):
        pool.attend(use_mask=True)
    torch.cuda.synchronize()
    print(json.dumps({"mode": "profile", "kernel": args.profile, "workload": wl.name,
                      "launches": args.launches, "status_word": fpk.fpk_decode_status(pool.workspace)}),
          flush=True)


def local_rank() -> int:
    return int(os.environ.get("LOCAL_RANK", "0"))


def validation_overhead(g_val, g_noval, pairs: int, replays: int):
    """Share of the step the tag check adds: the single-step graph with and
    without the check (same inputs, same kernels, the check's CTAs absent),
    timed as `pairs` interleaved pairs of `replays` replays each (the order
    inside a pair alternates).  Reports the median and quartiles of the
    per-pair relative differences."""
    d, tv, tn = [], [], []
    for i in range(pairs):
        if i % 2 == 0:
            a = time_graph(g_val, replays, 3)
            b = time_graph(g_noval, replays, 3)
        else:
            b = time_graph(g_noval, replays, 3)
            a = time_graph(g_val, replays, 3)
        tv.append(a)
        tn.append(b)
        d.append(100.0 * (a - b) / b)
    q1, med, q3 = (float(x) for x in np.percentile(d, [25, 50, 75]))
    return {"median_pct": med, "q1_pct": q1, "q3_pct": q3, "pairs": pairs, "replays_per_side": replays,
            "step_us_with": 1e3 * statistics.median(tv), "step_us_without": 1e3 * statistics.median(tn)}


def time_attention_b2b(pool, launches: int, reps: int = 5):
    """The attention launch's average duration: `launches` back-to-back launches
    (same inputs, KV far larger than L2) captured in one CUDA graph, replayed
    between two events on the current stream, median over `reps` replays.  Each
    launch's grid set-up overlaps the previous launch's tail, as in the decode
    step, which also runs as a graph.  (Eager launches of the same kernel run
    about 2 us slower once the process has captured any CUDA graph, whatever
    the graph holds; replayed launches do not.)"""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            pool.attend(use_mask=True)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(launches):
            pool.attend(use_mask=True)
    s = torch.cuda.current_stream()
    for _ in range(3):
        g.replay()
    t = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        g.replay()
        b.record(s)
        torch.cuda.synchronize()
        t.append(a.elapsed_time(b) / launches)
    del g
    return statistics.median(t)


def time_attention_sequence(pool, staged, nsteps: int):
    """Attention launches of decode steps 0..nsteps-1, each timed with events on
    its stream after that step's inputs were staged and its write + check ran;
    returns (mean attention ms, mean write + check ms)."""
    K, V, Q, lens = staged
    s = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nsteps)]
    for i in range(nsteps):
        pool.seq_lens.copy_(lens[i])
        pool.k_new.copy_(K[i])
        pool.v_new.copy_(V[i])
        pool.q.copy_(Q[i])
        ev[i][0].record(s)
        pool.append_check(stream=s)
        ev[i][1].record(s)
        ev[i][2].record(s)
        pool.attend(use_mask=True, stream=s)
        ev[i][3].record(s)
    torch.cuda.synchronize()
    return (statistics.mean(e[2].elapsed_time(e[3]) for e in ev),
            statistics.mean(e[0].elapsed_time(e[1]) for e in ev))


def roofline(abytes: float, attn_ms: float, name: str, peak: float, peak_kind: str):
    achieved = abytes / (attn_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": read_profile_traffic(name, "fp8"), "algorithmic_bytes": int(abytes),
            "kernel": "paged_decode attention (split-KV, FP8)",
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s"}


def measure_fp8(wl, args, world, local, headline: bool):
    """The FP8 decode step of one workload: step time (CUDA graph; a growing
    workload replays all its decode steps as one graph), the attention
    launch's own time and roofline, the tag check's share of the step, and for
    the headline workload also the end-to-end figure and the prompt write."""
    import fp8_paged_kv_gb300 as fpk
    from fp8_paged_kv_gb300.pool import DecodePool
    dev = torch.device("cuda", torch.cuda.current_device())
    pool = DecodePool(wl, fp8=True, device=dev)
    pool.prefill()
    pool.set_step(0)
    pool.step()
    torch.cuda.synchronize()
    live = int(wl.B - int(pool.abort_count.item()))
    # the decode step as one CUDA graph (cache write and tag check in one launch,
    # attention after it); the mismatch count is taken on the host from the abort
    # mask the step returns
    pool.count_aborts = False
    g_step = capture_step(pool, True)
    g_noval = capture_step(pool, False)
    seq_steps = wl.steps if wl.steps > 1 else 0
    g_seq = staged = None
    if seq_steps:
        g_seq, staged = capture_steps_sequence(pool, seq_steps)
    barrier(world)
    torch.cuda.synchronize()
    peak, peak_kind = measured_peaks()
    res = {}
    with ClockSampler(local) as clk:
        if g_seq is None:
            timed_steps = args.steps
            ms_step = time_graph(g_step, args.steps, args.warmup)
        else:
            reps = max(1, -(-args.steps // seq_steps))
            timed_steps = reps * seq_steps
            ms_step = time_graph(g_seq, reps, 1) / seq_steps
        barrier(world)
        ms_step = max_over_ranks(ms_step, world)
        # the attention launch alone: its average duration over back-to-back
        # launches at decode step 0 (the roofline's), and each launch timed on
        # its own between the step's launches (at step 0, or over every step
        # of a growing workload), which adds the launch's own latency
        if staged is None:
            pool.set_step(0)
            _, single_ms, app_ms = time_steps(pool, max(args.steps // 4, 20), 3)
            single_bytes = attention_bytes(wl, 0, True)
        else:
            single_ms, app_ms = time_attention_sequence(pool, staged, seq_steps)
            single_bytes = statistics.mean(attention_bytes(wl, s_, True) for s_ in range(seq_steps))
            pool.set_step(0)
            pool.append_check()
        attn_ms = time_attention_b2b(pool, 20)
        abytes = attention_bytes(wl, 0, True)
        # the same launch on the tcgen05 tensor cores (fpk_paged_decode_attn_fp8_tc)
        pool.tensor_cores = True
        tc_ms = time_attention_b2b(pool, 20)
        pool.tensor_cores = False
        val = validation_overhead(g_step, g_noval, args.val_pairs, args.val_replays)
        status = fpk.fpk_decode_status(pool.workspace)
        if headline:
            e2e_ms, h2d, d2h, e2e_steps = time_e2e(pool, max(args.steps, 64), 16)
            e2e_ms = max_over_ranks(e2e_ms, world)
    res.update({
        "workload": workload_config(wl)["workload"], "ms_per_step": ms_step, "timed_steps": timed_steps,
        "tokens_per_s": live * world / (ms_step * 1e-3),
        "step_launch": ("one CUDA graph per step" if g_seq is None
                        else f"all {seq_steps} decode steps as one CUDA graph (inputs staged on the device)"),
        "attn_us": attn_ms * 1e3, "append_and_check_us": app_ms * 1e3,
        "attn_timing": "average over 20 back-to-back launches replayed from one CUDA graph at decode step 0 (median of 5 replays)",
        "attn_us_single_launch": single_ms * 1e3,
        "single_launch_gbs": single_bytes / (single_ms * 1e-3) / 1e9,
        "single_launch_timing": ("each launch between two events, after the step's write + check launch"
                                 + (f", mean over all {seq_steps} steps" if staged is not None else "")),
        "attn_tokens_per_s": live * world / (attn_ms * 1e-3),
        "roofline": roofline(abytes, attn_ms, wl.name, peak, peak_kind),
        "tensor_cores": {"attn_us": tc_ms * 1e3, "attn_gbs": abytes / (tc_ms * 1e-3) / 1e9,
                         "frac": abytes / (tc_ms * 1e-3) / 1e9 / peak,
                         "kernel": "paged_decode_tc_kernel: tcgen05.mma kind::f8f6f4 (q and p as four e4m3 "
                                   "parts), accumulators in TMEM, K rows by tensor-map copies",
                         "attn_timing": "average over 20 back-to-back launches replayed from one CUDA graph at decode step 0 (median of 5 replays)"},
        "validation_overhead_pct": val["median_pct"], "validation_overhead": val,
        "status_word": status, "clocks": clk.summary(), "live_requests": live})
    if wl.num_splits:
        res["num_splits"] = wl.num_splits
    if headline:
        res["e2e"] = {"value": live * world / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "timed_steps": e2e_steps,
                      "api": "DecodePool + HostPipeline: pinned host buffers per step, copies on a second "
                             "stream overlapping the neighbouring steps' kernels, 16 steps per CUDA graph"}
        res["prefill"] = time_prefill(pool)
    if wl.name == "long128k":
        # the same launch with the automatic split count (one wave of CTAs)
        pool.set_step(0)
        pool.num_splits = 0
        pool.workspace = torch.zeros(max(256, fpk.fpk_decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.D, 0)),
                                     dtype=torch.uint8, device=dev)
        pool.append_check()
        a_auto = time_attention_b2b(pool, 20)
        res["attn_us_auto_splits"] = a_auto * 1e3
        res["roofline_auto_splits_frac"] = attention_bytes(wl, 0, True) / (a_auto * 1e-3) / 1e9 / peak
    del pool
    torch.cuda.empty_cache()
    return res


def capacity_summary(args, local):
    """Admission at a fixed one-layer KV budget, compactly: each cache's cap in
    8192-token requests of the headline shape and its decode-attention tokens/s
    at the cap and at 32 requests (where both fit).  Cache values are random
    codes (only timing is taken); L2 is flushed before every timed launch."""
    import fp8_paged_kv_gb300 as fpk
    from fp8_paged_kv_gb300.pool import admission_cap
    dev = torch.device("cuda", torch.cuda.current_device())
    Hq, Hkv, D, ps, L = 64, 8, 128, 16, 8192
    budget = int(args.kv_budget_gib * 2**30)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    flush = L2Flush(dev)
    s = torch.cuda.current_stream(dev)
    res = {"kv_budget_gib": args.kv_budget_gib, "context": L,
           "shape": f"Hq={Hq}, Hkv={Hkv}, D={D}, page_size={ps}, one layer", "l2": L2Flush.NOTE}
    with ClockSampler(local) as clk:
        for fp8 in (False, True):
            num_pages, ppr, cap = admission_cap(budget, L, Hkv=Hkv, D=D, page_size=ps, fp8=fp8)
            n = num_pages * 2 * Hkv * ps * D
            if fp8:
                pool = torch.randint(0, 0x7F, (n,), dtype=torch.uint8, device=dev, generator=g)
                pool |= torch.randint(0, 2, (n,), dtype=torch.uint8, device=dev, generator=g) << 7
            else:
                pool = torch.randn(n, device=dev, generator=g, dtype=torch.bfloat16)
            perm = torch.randperm(num_pages, device=dev, generator=g).to(torch.int32)
            pts = {}
            for c in sorted({32, cap}):
                if c > cap:
                    continue
                pt = perm[:c * ppr].view(c, ppr).contiguous()
                lens = torch.full((c,), L, dtype=torch.int32, device=dev)
                q = torch.randn(c, Hq, D, device=dev, generator=g).to(torch.bfloat16)
                out = torch.empty(c, Hq, D, device=dev)
                lse = torch.empty(c, Hq, device=dev)
                ws = torch.zeros(fpk.fpk_decode_workspace_bytes(c, Hq, Hkv, D, 0), dtype=torch.uint8,
                                 device=dev)
                ks = torch.tensor([0.01], device=dev)
                kw = dict(Hkv=Hkv, page_size=ps, num_pages=num_pages, sm_scale=D ** -0.5)
                t = []
                for i in range(3 + args.capacity_reps):
                    flush()
                    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(s)
                    if fp8:
                        fpk.fpk_paged_decode_attn_fp8(q, pool, ks, ks, pt, lens, None, out, lse, ws, **kw)
                    else:
                        fpk.fpk_paged_decode_attn_bf16(q, pool, pt, lens, None, out, lse, ws, **kw)
                    e.record(s)
                    torch.cuda.synchronize(dev)
                    if i >= 3:
                        t.append(a.elapsed_time(e))
                ms = statistics.median(t)
                kv = c * L * 2 * Hkv * D * (1 if fp8 else 2)
                nbytes = kv + c * ppr * 4 + c * Hq * D * 2 + c * Hq * (D + 1) * 4
                pts["at_cap" if c == cap else "at_32"] = {"requests": c, "attn_us": ms * 1e3,
                                                          "tokens_per_s": c / (ms * 1e-3),
                                                          "gbs": nbytes / (ms * 1e-3) / 1e9}
                if c == 32 and cap == 32:
                    pts["at_32"] = pts["at_cap"]
                del ws, q, out, lse
            res["fp8" if fp8 else "bf16"] = {"pool_pages": num_pages, "pages_per_request": ppr,
                                             "cap_requests": cap, **pts}
            del pool, perm
            torch.cuda.empty_cache()
    res["fp8_over_bf16_cap"] = res["fp8"]["cap_requests"] / max(1, res["bf16"]["cap_requests"])
    res["fp8_at_cap_over_bf16_at_cap_tokens_per_s"] = (res["fp8"]["at_cap"]["tokens_per_s"] /
                                                       res["bf16"]["at_cap"]["tokens_per_s"])
    res["clocks"] = clk.summary()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="b32_8k")
    ap.add_argument("--no-bf16", action="store_true", help="skip the BF16 comparison leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline leg")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads' objects and the capacity object")
    ap.add_argument("--extra", default="b64_var,long128k",
                    help="workloads measured beside the headline one (comma separated)")
    ap.add_argument("--val-pairs", type=int, default=10)
    ap.add_argument("--val-replays", type=int, default=100)
    ap.add_argument("--capacity", action="store_true",
                    help="admission curve at a fixed KV budget instead of the step benchmark")
    ap.add_argument("--kv-budget-gib", type=float, default=4.0)
    ap.add_argument("--capacity-reps", type=int, default=10)
    ap.add_argument("--gemv", action="store_true",
                    help="INT4 vs e4m3 weight-only decode GEMV instead of the step benchmark")
    ap.add_argument("--gemv-n", type=int, default=28672)
    ap.add_argument("--gemv-k", type=int, default=8192)
    ap.add_argument("--gemv-batches", default="1,2,4,8,16",
                    help="decode batches of the --gemv leg (comma separated)")
    ap.add_argument("--profile", choices=["fp8", "bf16", "tc"],
                    help="run only the workload's attention (one decode step, then --launches "
                         "attention launches), for a profiler")
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.capacity:
        run_capacity(args, rank, world)
        return
    if args.gemv:
        run_gemv(args, rank, world)
        return
    if args.profile:
        run_profile(args)
        return

    import fp8_paged_kv_gb300 as fpk
    from fp8_paged_kv_gb300 import build as fbuild
    from fp8_paged_kv_gb300.pool import DecodePool
    from workloads import WORKLOADS

    if rank == 0 or world == 1:
        fbuild.build()
    barrier(world)
    fpk.load_library()

    def make(name):
        return WORKLOADS[name](seed=100 + rank) if world > 1 else WORKLOADS[name]()

    wl = make(args.workload)
    # ---------------- FP8 cache: the measured path
    m = measure_fp8(wl, args, world, local, headline=True)
    ms_step = m["ms_per_step"]
    live = m["live_requests"]
    out = {
        "metric": METRIC, "value": m["tokens_per_s"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 cache; f16 MMA, fp32 softmax",
        "data": "synthetic", "config": workload_config(wl),
        "roofline": m["roofline"],
        "fp8": {"attn_us": m["attn_us"], "attn_timing": m["attn_timing"],
                "attn_us_single_launch": m["attn_us_single_launch"],
                "append_and_check_us": m["append_and_check_us"],
                "attn_tokens_per_s": m["attn_tokens_per_s"], "attn_gbs": m["roofline"]["achieved"],
                "step_launch": m["step_launch"],
                "validation_overhead_pct": m["validation_overhead_pct"],
                "validation_overhead": m["validation_overhead"],
                "algorithmic_bytes_per_attention": m["roofline"]["algorithmic_bytes"],
                "status_word": m["status_word"], "tensor_cores": m["tensor_cores"]},
        # per timed step: the cache write + tag check launch and the attention
        # launch (the split combine runs inside the attention kernel)
        "gpu_launches": 2 * m["timed_steps"], "clocks": m["clocks"],
        "e2e": m["e2e"], "prefill": m["prefill"],
    }

    # ---------------- BF16 cache on identical values
    if not args.no_bf16:
        peak = m["roofline"]["peak"]
        p16 = DecodePool(wl, fp8=False, device=torch.device("cuda", torch.cuda.current_device()))
        p16.prefill()
        p16.set_step(0)
        p16.count_aborts = False
        n16 = max(args.steps // 4, 20)
        _, a16_single, _ = time_steps(p16, n16, args.warmup)
        p16.append_check()
        a16 = time_attention_b2b(p16, 20)
        g16 = capture_step(p16, True)
        t16 = time_graph(g16, n16, args.warmup) * n16
        b16 = attention_bytes(wl, 0, False)
        out["bf16"] = {"value": live * world / (t16 / n16 * 1e-3), "ms_per_step": t16 / n16,
                       "attn_us": a16 * 1e3, "attn_us_single_launch": a16_single * 1e3,
                       "attn_gbs": b16 / (a16 * 1e-3) / 1e9,
                       "attn_frac": b16 / (a16 * 1e-3) / 1e9 / peak,
                       "fp8_over_bf16_step": (t16 / n16) / ms_step,
                       "traffic": read_profile_traffic(wl.name, "bf16")}
        del p16, g16
        torch.cuda.empty_cache()

    # ---------------- the other workloads, each as its own object
    if not args.no_extra:
        for name in [n for n in args.extra.split(",") if n and n != args.workload]:
            w2 = make(name)
            out[name] = measure_fp8(w2, args, world, local, headline=False)
            del w2
        out["capacity"] = capacity_summary(args, local)

    if rank == 0 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
