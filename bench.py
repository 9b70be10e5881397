#!/usr/bin/env python3
"""S2ANTA decode-step benchmark (one JSON line on rank 0).

A step is one pass of the whole operator (score pass, combine + thresholds,
sample + gather) over one decode step of the workload, through the C ABI on
device-resident inputs; for 16-bit caches it is a single cooperative launch.
Protocol (after "Stochastic Sparse Attention for Memory-Bound Inference",
App. Q): W untimed warm-up steps, then K timed steps, each bracketed by CUDA
events on the launching stream.  Inputs are larger than L2: the steps rotate
over R copies of the K/V cache (R * |K, V| >= 512 MiB), so every step reads its
cache from HBM; workloads too small for that flush L2 between steps instead.

    python bench.py [--steps K] [--warmup W] [--workload llama32k|qwen|ragged|tiny]
    python bench.py --impl reference      # the CPU oracle, timed on host cores
Multi-GPU (torchrun): every rank decodes its own copy of the workload
(independent replicas, no collective on the data path; scaling "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "S²ANTA decode-attn µs/step and achieved HBM GB/s vs peak, 32K ctx bf16"
UNIT = "us/step"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 * 1024 * 1024
MAX_REPLICAS = 64   # more copies than this: an L2 flush between steps instead
KERNEL_SOURCES = ["stochastic_sparse_decode_split_gb300/csrc/santa_fused.cuh",
                  "stochastic_sparse_decode_split_gb300/csrc/santa_fused.cu",
                  "stochastic_sparse_decode_split_gb300/csrc/santa_tma.cuh",
                  "stochastic_sparse_decode_split_gb300/csrc/santa_part.cuh",
                  "stochastic_sparse_decode_split_gb300/csrc/santa_grid.cuh",
                  "stochastic_sparse_decode_split_gb300/csrc/santa_fused_bf16.cu",
                  "stochastic_sparse_decode_split_gb300/csrc/santa_window.cuh",
                  "stochastic_sparse_decode_split_gb300/csrc/santa_common.cuh",
                  "stochastic_sparse_decode_split_gb300/csrc/santa_seq.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fused_decode_traffic.json")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama32k", choices=["llama32k", "qwen", "ragged", "tiny"])
    ap.add_argument("--nk", type=int, default=None, help="override keys per sequence (llama32k shape)")
    ap.add_argument("--S", type=int, default=None)
    ap.add_argument("--variant", default=None, choices=["iid", "stratified", "systematic"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample length")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sampler", choices=["global", "prop", "flash"], default="global",
                    help="global: the single-launch sampler (the benchmark line); prop / flash: the pages' "
                         "tile samplers S2ANTA-prop and S2ANTA-flash")
    ap.add_argument("--tile", type=int, default=256, help="keys per tile for --sampler prop / flash")
    ap.add_argument("--bernoulli", type=int, default=0,
                    help="Bernoulli qK^T (mean group query, stratified) with this many samples per feature "
                         "in front of the single-launch decode; 0: exact scores")
    ap.add_argument("--l2", choices=["auto", "replicas", "flush"], default="auto",
                    help="inputs larger than L2 (rotating K/V copies) or an L2 flush between steps; "
                         "auto: copies when the cache is at least 128 MiB")
    return ap.parse_args()


def make_workload(args):
    import synth
    if args.workload == "llama32k":
        wl = synth.llama32k(nk=args.nk or 32768, S=args.S or 256, variant=args.variant or "systematic")
    elif args.workload == "qwen":
        wl = synth.qwen_batched()
    elif args.workload == "ragged":
        wl = synth.ragged()
    else:
        wl = synth.tiny(args.variant or "systematic")
    return wl


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, device=None) -> float:
    """The largest of every rank's value (the whole job ends when its slowest
    replica does); the value itself on one rank.  Any process-group backend."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# peaks, clocks, traffic record
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for k in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
            if k in d and d[k]:
                return float(d[k]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.idx = device_index

    def start(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
            uuid = os.environ.get("SANTA_GPU_UUID")
            if uuid:
                cmd += ["--id=" + uuid]
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        os.unlink(self.out.name)
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9]
        if not rows:
            return None
        by_gpu = {}
        for r in rows:
            by_gpu.setdefault(r[0], []).append(r)
        # the busiest GPU (highest median power) is ours when several are listed
        def med_power(rs):
            vals = [float(r[3]) for r in rs if r[3].replace(".", "", 1).isdigit()]
            return statistics.median(vals) if vals else 0.0
        rs = max(by_gpu.values(), key=med_power)
        sm = [float(r[1]) for r in rs if r[1].replace(".", "", 1).isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rs:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rs[0][2]) if rs[0][2].replace(".", "", 1).isdigit() else None,
                "reasons": sorted(reasons), "samples": len(rs)}


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name):
    """dram read+write bytes per launch of the decode kernel from a committed
    ncu summary, only while the kernel source is unchanged since the capture."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_hash") != source_hash(KERNEL_SOURCES):
        return None
    if rec.get("workload") != workload_name:
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# byte model (algorithmic bytes)
# ---------------------------------------------------------------------------

def esize(dtype):
    return {"bf16": 2, "fp16": 2, "fp32": 4}[dtype]


def score_pass_bytes(inp):
    """K read once + q read + per-chunk (max, exp-sum) written.  The fp32
    score stash is written to L2 and read back by the sampler there; it is
    not counted (ncu dram bytes show whether it reaches HBM)."""
    wl = inp.wl
    es = esize(wl.dtype)
    B, H, d = inp.q.shape
    rows = int(inp.kv_offsets[-1])
    chunks = sum((int(n) + 15) // 16 for n in inp.nk_per_seq)
    return rows * wl.n_kv_heads * d * es + B * H * d * es + 2 * 4 * H * chunks


def step_bytes(inp, unique_rows):
    """Full K + deduplicated gathered V rows + q + out."""
    wl = inp.wl
    es = esize(wl.dtype)
    B, H, d = inp.q.shape
    rows = int(inp.kv_offsets[-1])
    return rows * wl.n_kv_heads * d * es + unique_rows * d * es + B * H * d * es + B * H * d * 4


def dense_bytes(inp):
    wl = inp.wl
    es = esize(wl.dtype)
    B, H, d = inp.q.shape
    rows = int(inp.kv_offsets[-1])
    return 2 * rows * wl.n_kv_heads * d * es + B * H * d * es + B * H * d * 4


def count_unique_rows(inp, idx):
    """Distinct (sequence, KV head, key) triples drawn by any head of a group."""
    import numpy as np
    B, H, _ = inp.q.shape
    G = inp.wl.group
    total = 0
    for b in range(B):
        S_b = inp.S_of(b)
        for kvh in range(inp.wl.n_kv_heads):
            total += np.unique(idx[b, kvh * G:(kvh + 1) * G, :S_b]).size
    return int(total)


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_threads():
    return max(1, os.cpu_count() or 1)


def time_oracle_full_steps(inp, variant, seconds):
    """Whole decode steps of the oracle (all heads, OpenMP over heads) until
    `seconds` of wall time have passed; returns (us_per_step, steps, threads)."""
    import oracle
    P = oracle.Problem.from_inputs(inp)
    n_thr = oracle_threads()
    steps = 0
    t0 = time.perf_counter()
    while True:
        oracle.decode(P, variant, inp.wl.S, seed=steps, S_per_seq=inp.S_per_seq, n_threads=n_thr)
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds or steps >= 1000:
            break
    return el / steps * 1e6, steps, n_thr


def l2_plan(kv_bytes, mode):
    """How the timed steps keep L2 from serving the cache: R replicas of the
    K/V cache used in turn (R = None: a flush between steps), and the note
    the JSON line carries.  Shared by both arms, so their configs agree."""
    R = max(2, -(-FLUSH_BYTES // kv_bytes))
    if mode == "replicas" or (mode == "auto" and R <= MAX_REPLICAS):
        return R, f"inputs larger than L2: {R} replicas of the K/V cache used in turn ({R * kv_bytes >> 20} MiB)"
    return None, "L2 flush between steps: write 512 MiB, then read 512 MiB (clean lines), outside each step's events"


def graph_replay_ms(fn, n, warm, world):
    """fn(i) for i < warm, untimed; then the n calls fn(0..n-1) captured once as
    a CUDA graph and replayed between two events on the launching stream
    (barrier and synchronize on both sides).  Returns the replay's ms."""
    import torch
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            fn(i)
    g.replay()   # graph upload, untimed
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0.record(s)
    g.replay()
    e1.record(s)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    del g
    return e0.elapsed_time(e1)


def run_reference(args):
    ws_, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    import synth
    oracle.build()
    wl = make_workload(args)
    inp = synth.generate(wl, 0)
    P = oracle.Problem.from_inputs(inp)
    B, H, _ = inp.q.shape
    heads = [(b, h) for b in range(B) for h in range(H)]
    # one head's cost sizes the per-step sample so that the whole run stays near two minutes
    t0 = time.perf_counter()
    oracle.decode_head(P, wl.variant, inp.S_of(0), 0, 0, 0)
    t_head = max(time.perf_counter() - t0, 1e-4)
    total_steps = args.steps + args.warmup
    per_step = int(max(1, min(len(heads), 120.0 / (total_steps * t_head))))
    times = []
    for i in range(total_steps):
        sel = [heads[(i * per_step + k) % len(heads)] for k in range(per_step)]
        t0 = time.perf_counter()
        for (b, h) in sel:
            oracle.decode_head(P, wl.variant, inp.S_of(b), i, b, h)
        el = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(el * len(heads) / per_step)   # scaled to a whole decode step
    us = statistics.mean(times) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "variant": wl.variant, "S": inp.S_max, "nk": wl.nk, "batch": B,
                   "n_q_heads": H, "n_kv_heads": wl.n_kv_heads, "head_dim": inp.q.shape[2],
                   "l2": l2_plan(inp.K.nbytes * 2, args.l2)[1],
                   "parallelism": "replicas" if args.gpus > 1 else "single GPU"},
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} of {len(heads)} heads per step (single host thread, "
                                   f"inputs in host memory), time scaled to all heads"},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import numpy as np
    import torch
    import synth
    import stochastic_sparse_decode_split_gb300 as santa

    world, rank, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    santa.library()   # fails loudly if the CUDA library was not built

    wl = make_workload(args)
    inp = synth.generate(wl, 0)
    t = synth.to_torch(inp, dev)
    ragged = wl.ragged is not None
    nk_bound = int(inp.nk_per_seq.max()) if ragged else None
    kw = dict(nk=nk_bound, kv_offsets=t["kv_offsets"] if ragged else None)
    S_max = inp.S_max
    B, H, d = inp.q.shape

    # Inputs larger than L2: R replicas of the K/V cache (identical contents at
    # different addresses) are used in turn, so every step reads its cache from
    # HBM, as every layer of a model does.  Workloads too small for that use a
    # flush instead: write 512 MiB, then read 512 MiB so that no dirty line of
    # the flush is written back inside the timed step.
    kv_bytes = t["K"].numel() * t["K"].element_size() * 2
    R, l2_note = l2_plan(kv_bytes, args.l2)
    if R:
        reps = [(t["K"], t["V"])] + [(t["K"].clone(), t["V"].clone()) for _ in range(R - 1)]
        flush = None
    else:
        reps = [(t["K"], t["V"])]
        flush = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    R = len(reps)
    decs = [santa.Decoder(t["q"], Kr, Vr, S=S_max, variant=wl.variant, seed=0, S_per_seq=t["S_per_seq"], **kw)
            for (Kr, Vr) in reps]
    dec = decs[0]
    # sampled rows of the timed step (same seed and step), for the byte model
    idx = torch.full((B, H, S_max), -1, dtype=torch.int32, device=dev)
    santa.santa_decode(t["q"], t["K"], t["V"], S=S_max, variant=wl.variant, seed=0, step=0,
                       S_per_seq=t["S_per_seq"], sample_idx=idx, **kw)
    torch.cuda.synchronize()
    unique_rows = count_unique_rows(inp, idx.cpu().numpy())
    if santa.get_error(dec.workspace):
        raise RuntimeError("device flagged bad metadata")

    stream = torch.cuda.current_stream()
    sink = torch.zeros(1, dtype=torch.float32, device=dev)

    def between_steps():
        if flush is not None:
            flush.add_(1.0)
            sink.copy_(flush.sum())

    def timed_loop(fn, n, warm):
        for i in range(warm):
            between_steps()
            fn(i)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        for i in range(n):
            between_steps()
            starts[i].record(stream)
            fn(i)
            ends[i].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # The timed region with replicas: W plain warm-up steps, then the K steps
    # captured once as a CUDA graph (one kernel node per step over the
    # rotating replicas) and replayed between two events on the launching
    # stream.  The replay removes the host's launch overhead, not any device
    # work.
    def graph_timed(fn, n, warm):
        for i in range(warm):
            between_steps()
            fn(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                between_steps()
                fn(i)
        g.replay()   # graph upload, untimed
        torch.cuda.synchronize()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0.record(s)
        g.replay()
        e1.record(s)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        del g
        return e0.elapsed_time(e1)

    def timed_region(fn, n, warm):
        """Replicas: graph replay of the n steps.  Flush: the flush stays
        outside the timing, so each step is timed by its own events."""
        if flush is None:
            return graph_timed(fn, n, warm)
        return sum(timed_loop(fn, n, warm))

    sampler = ClockSampler(local_rank).start()
    time.sleep(0.3)
    region_ms = timed_region(lambda i: decs[i % R](step=0), args.steps, args.warmup)
    clocks = sampler.stop()

    total_ms = max_over_ranks(region_ms, dev)
    mean_ms = total_ms / args.steps

    # per-stage times (events recorded between the stages, same stream)
    n_prof = min(args.steps, 1000)
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_prof)]
    for es in ev_sets:          # torch creates the underlying cudaEvent_t on first record
        for e in es:
            e.record(stream)
    for i in range(args.warmup):
        between_steps()
        decs[i % R].profiled(ev_sets[0])
    torch.cuda.synchronize()
    for i in range(n_prof):
        between_steps()
        decs[i % R].profiled(ev_sets[i])
    torch.cuda.synchronize()
    stage_ms = [statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev_sets) for k in range(3)]

    # duration of one decode launch, and of the staged path's score pass alone:
    # launches issued back to back over the rotating replicas between one pair
    # of events (launch latency overlapped)
    def back_to_back(fn, n):
        for i in range(args.warmup):
            fn(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    launch_ms = score_launch_ms = None
    read_probe = None
    if flush is None:
        n_back = min(args.steps, 400)
        launch_ms = back_to_back(lambda i: decs[i % R](step=0), n_back)
        score_launch_ms = back_to_back(lambda i: decs[i % R].score_pass(), n_back)
        # read ceiling of this transfer size: a plain streaming read of the K
        # bytes, launched back to back over the same replicas
        import ctypes
        lib = santa.library()
        sink = torch.empty(lib.santa_read_probe_sink_words(), dtype=torch.int32, device=dev)
        k_bytes = t["K"].numel() * t["K"].element_size()
        sid = ctypes.c_void_p(stream.cuda_stream)

        def read_k(i):
            if lib.santa_read_probe(ctypes.c_void_p(reps[i % R][0].data_ptr()), k_bytes,
                                    ctypes.c_void_p(sink.data_ptr()), sid) != 0:
                raise RuntimeError("santa_read_probe failed")

        probe_ms = back_to_back(read_k, n_back)
        read_probe = {"kernel": "read_probe_kernel (16-byte streaming read, no compute)", "bytes": k_bytes,
                      "us_per_read": probe_ms * 1e3, "GBps": k_bytes / (probe_ms * 1e-3) / 1e9}

    # warm L2: the same protocol on one replica only, so that a step may find
    # what the previous step read in L2 (context for the cold figure)
    warm_ms = None
    if R > 1 and flush is None:
        n_warm = min(args.steps, 400)
        warm_ms = graph_timed(lambda i: decs[0](step=0), n_warm, args.warmup) / n_warm

    # dense comparator, same protocol
    denses = [santa.Decoder(t["q"], Kr, Vr, S=1, variant=wl.variant, dense=True, **kw) for (Kr, Vr) in reps]
    n_dense = min(args.steps, 1000)
    dense_ms = timed_region(lambda i: denses[i % R](), n_dense, args.warmup) / n_dense

    # end to end through the public API with host buffers, the D2H of the
    # output inside the timed region, the cache's host copy in pinned memory
    # (R replicas used in turn, as on the device, so that no step finds data
    # it read before in L2).  e2e: q and K copied H2D, V read in place by
    # santa_decode_host_kv (only the drawn rows cross the host link).
    # e2e_in_place: K and V both read in place.  e2e_copy: q, K, V copied to the
    # device, then santa_decode on the copies.
    e2e = e2e_in_place = e2e_copy = None
    if not args.no_e2e:
        hq = t["q"].cpu().pin_memory()
        hout = torch.empty((B, H, d), dtype=torch.float32).pin_memory()
        dq = torch.empty_like(t["q"])
        dK, dV = torch.empty_like(t["K"]), torch.empty_like(t["V"])
        n_e2e = min(args.steps, 200)
        q_bytes = hq.numel() * hq.element_size()
        k_bytes = t["K"].numel() * t["K"].element_size()
        v_rows = unique_rows * d * t["V"].element_size()
        d2h = hout.numel() * hout.element_size()
        hreps = [(Kr.cpu().pin_memory(), Vr.cpu().pin_memory()) for (Kr, Vr) in reps]
        ws_h = santa.alloc_workspace(dec.workspace.numel(), dev)
        out_h = torch.empty((B, H, d), dtype=torch.float32, device=dev)

        def host_kv_step(copy_k):
            def step(i):
                hK, hV = hreps[i % len(hreps)]
                dq.copy_(hq, non_blocking=True)
                if copy_k:
                    dK.copy_(hK, non_blocking=True)
                santa.santa_decode_host_kv(dq, dK if copy_k else hK, hV, S=S_max, variant=wl.variant, seed=0,
                                           out=out_h, workspace=ws_h, S_per_seq=t["S_per_seq"], **kw)
                hout.copy_(out_h, non_blocking=True)
            return step

        def e2e_line(ms, h2d, mode):
            return {"value": statistics.mean(ms) * 1e3 / world, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "mode": mode, "replicas": len(hreps)}

        e2e = e2e_line(timed_loop(host_kv_step(True), n_e2e, 3), q_bytes + k_bytes + v_rows,
                       "q, K copied H2D; V in pinned host memory, drawn rows read in place (santa_decode_host_kv)")
        e2e_in_place = e2e_line(timed_loop(host_kv_step(False), n_e2e, 3), q_bytes + k_bytes + v_rows,
                                "K and V in pinned host memory, read in place (santa_decode_host_kv)")
        dec_e = santa.Decoder(dq, dK, dV, S=S_max, variant=wl.variant, seed=0, S_per_seq=t["S_per_seq"], **kw)

        def copy_step(i):
            hK, hV = hreps[i % len(hreps)]
            dq.copy_(hq, non_blocking=True)
            dK.copy_(hK, non_blocking=True)
            dV.copy_(hV, non_blocking=True)
            o = dec_e(step=0)
            hout.copy_(o, non_blocking=True)

        e2e_copy = e2e_line(timed_loop(copy_step, n_e2e, 3), q_bytes + 2 * k_bytes,
                            "q, K, V copied H2D, then santa_decode")
        # the host link's ceiling for this size: the same bytes as e2e (q + K +
        # the drawn V rows) in one pinned H2D copy, nothing else in the region
        link_bytes = q_bytes + k_bytes + v_rows
        hbuf = torch.empty(link_bytes, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(link_bytes, dtype=torch.uint8, device=dev)
        link_ms = statistics.mean(timed_loop(lambda i: dbuf.copy_(hbuf, non_blocking=True), n_e2e, 3))
        e2e["link_ceiling"] = {"us": link_ms * 1e3, "bytes": link_bytes,
                               "GBps": link_bytes / (link_ms * 1e-3) / 1e9,
                               "e2e_over_ceiling": e2e["value"] * world / (link_ms * 1e3),
                               "probe": "one pinned H2D cudaMemcpyAsync of the e2e bytes"}
        del hreps, hbuf, dbuf

    peak, peak_kind = hbm_peak()
    sb = score_pass_bytes(inp)
    stb = step_bytes(inp, unique_rows)
    single = wl.dtype != "fp32"          # 16-bit caches: the whole step is one launch
    kernel_ms = mean_ms   # the timed region holds only the step's launches, one after another
    achieved = stb / (kernel_ms * 1e-3) / 1e9
    step_achieved = stb / (mean_ms * 1e-3) / 1e9
    value_us = mean_ms * 1e3 / world   # whole job: time per decode step over all ranks' steps

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        us_cpu, n_cpu, thr = time_oracle_full_steps(inp, wl.variant, args.cpu_seconds)
        cpu_baseline = {"value": us_cpu, "unit": UNIT, "cores": thr, "kind": "oracle",
                        "sample": f"{n_cpu} whole decode steps of {wl.name} (float64, OpenMP over heads), "
                                  f"{args.cpu_seconds:.0f} s budget"}

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value_us, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "variant": wl.variant, "S": S_max, "nk": wl.nk, "batch": B,
                   "n_q_heads": H, "n_kv_heads": wl.n_kv_heads, "head_dim": d,
                   "l2": l2_note,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "plain_launch_us": launch_ms * 1e3 if launch_ms is not None else None,
        "warm_l2": ({"us_per_step": warm_ms * 1e3, "GBps": stb / (warm_ms * 1e-3) / 1e9,
                     "note": "one K/V replica reused every step (part of it may be served from L2)"}
                    if warm_ms is not None else None),
        "roofline": {"bound": "hbm", "kernel": "fused_decode_kernel" if single else "staged path",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": recorded_traffic(wl.name) if single else None,
                     "peak_kind": f"of {peak_kind}", "alg_bytes_per_launch": stb,
                     "us_per_launch": kernel_ms * 1e3,
                     "timing": ("graph replay of the K timed steps over rotating replicas, events on the "
                                "launching stream" if flush is None else
                                "events around each step on the launching stream (L2 flush between steps)")},
        "step": {"alg_bytes": stb, "unique_v_rows": unique_rows, "achieved_GBps": step_achieved,
                 "frac": step_achieved / peak},
        "read_probe": (dict(read_probe, frac_of_peak=read_probe["GBps"] / peak) if read_probe else None),
        "staged_path": {"stage_us": {"score": stage_ms[0] * 1e3, "combine": stage_ms[1] * 1e3,
                                     "sample_gather": stage_ms[2] * 1e3},
                        "score_pass_us_per_launch": score_launch_ms * 1e3 if score_launch_ms else None,
                        "score_pass_GBps": sb / (score_launch_ms * 1e-3) / 1e9 if score_launch_ms else None},
        "dense": {"us_per_step": dense_ms * 1e3, "alg_bytes": dense_bytes(inp),
                  "achieved_GBps": dense_bytes(inp) / (dense_ms * 1e-3) / 1e9,
                  "frac": dense_bytes(inp) / (dense_ms * 1e-3) / 1e9 / peak,
                  "timing": "graph replay, as the main line",
                  "speedup_santa_vs_dense": dense_ms / mean_ms},
        "cpu_baseline": cpu_baseline,
        "e2e": e2e,
        "e2e_in_place": e2e_in_place,
        "e2e_copy": e2e_copy,
        "gpu_launches": (1 if single else 3) * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_tiled(args):
    """S2ANTA-prop / S2ANTA-flash step times (score pass, tile budgets for
    prop, tile sampler, merge), launched back to back over rotating K/V
    copies, with the same byte model as the main line."""
    import ctypes
    import numpy as np
    import torch
    import synth
    import stochastic_sparse_decode_split_gb300 as santa

    world, rank, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = santa.library()
    wl = make_workload(args)
    inp = synth.generate(wl, 0)
    t = synth.to_torch(inp, dev)
    ragged = wl.ragged is not None
    nk = int(inp.nk_per_seq.max()) if ragged else None
    offs = t["kv_offsets"] if ragged else None
    S_max = inp.S_max
    B, H, d = inp.q.shape
    L = args.tile
    p = santa.make_params(t["q"], t["K"], S_max, 0, 0, nk, offs, t["S_per_seq"])
    nd = santa.tiled_max_draws(p, args.sampler, L)
    nbytes = santa.tiled_workspace_size(p, args.sampler, L)
    if nd <= 0 or nbytes == 0:
        raise SystemExit(f"invalid tile sampler arguments (tile {L})")
    kv_bytes = t["K"].numel() * t["K"].element_size() * 2
    R = max(2, -(-FLUSH_BYTES // kv_bytes))
    reps = [(t["K"], t["V"])] + [(t["K"].clone(), t["V"].clone()) for _ in range(R - 1)]
    ws = santa.alloc_workspace(nbytes, dev)
    out = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    sid = ctypes.c_void_p(stream.cuda_stream)
    code = santa.SAMPLERS[args.sampler]
    ptrs = [(ctypes.c_void_p(Kr.data_ptr()), ctypes.c_void_p(Vr.data_ptr())) for Kr, Vr in reps]
    qp, op, wp = (ctypes.c_void_p(x.data_ptr()) for x in (t["q"], out, ws))

    def step(i, idx=None):
        Kp, Vp = ptrs[i % R]
        st = lib.santa_decode_tiled(ctypes.byref(p), code, L, qp, Kp, Vp, op, wp, nbytes,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                    None if idx is None else ctypes.c_void_p(idx.data_ptr()))
        if st != 0:
            raise RuntimeError(f"santa_decode_tiled: status {st}")

    idx = torch.full((B, H, nd), -1, dtype=torch.int32, device=dev)
    step(0, idx)
    torch.cuda.synchronize()
    if santa.get_error(ws):
        raise RuntimeError("device flagged bad metadata")
    ih = idx.cpu().numpy()
    G = wl.group
    unique_rows = 0
    for b in range(B):
        for kvh in range(wl.n_kv_heads):
            r = ih[b, kvh * G:(kvh + 1) * G]
            unique_rows += np.unique(r[r >= 0]).size
    draws = int((ih >= 0).sum())

    sampler = ClockSampler(local_rank).start()
    time.sleep(0.3)
    region = graph_replay_ms(step, args.steps, args.warmup, world)
    clocks = sampler.stop()
    ms = max_over_ranks(region, dev) / args.steps
    peak, peak_kind = hbm_peak()
    stb = step_bytes(inp, unique_rows)
    achieved = stb / (ms * 1e-3) / 1e9
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": ms * 1e3 / world, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "sampler": args.sampler, "tile_len": L, "S": S_max, "nk": wl.nk,
                   "batch": B, "n_q_heads": H, "n_kv_heads": wl.n_kv_heads, "head_dim": d,
                   "l2": f"inputs larger than L2: {R} replicas of the K/V cache used in turn "
                         f"({R * kv_bytes >> 20} MiB)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": "step: score pass + " + ("tile budgets + " if code == 0 else "") +
                     "tile sampler + merge", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None, "peak_kind": f"of {peak_kind}",
                     "alg_bytes_per_launch": stb,
                     "timing": "graph replay of the K timed steps over rotating replicas"},
        "step": {"alg_bytes": stb, "unique_v_rows": unique_rows, "draws": draws},
        "cpu_baseline": None,
        "e2e": None,
        "gpu_launches": (4 if code == 0 else 3) * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_bernoulli(args):
    """Decode step on Bernoulli qK^T effective queries (one small kernel, then
    the single-launch decode), launched back to back over rotating K/V copies.
    The decode still reads every key feature: the bytes are the main line's;
    the share of features the groups need is reported beside them."""
    import ctypes
    import numpy as np
    import torch
    import synth
    import stochastic_sparse_decode_split_gb300 as santa

    world, rank, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = santa.library()
    wl = make_workload(args)
    inp = synth.generate(wl, 0)
    t = synth.to_torch(inp, dev)
    ragged = wl.ragged is not None
    nk = int(inp.nk_per_seq.max()) if ragged else None
    offs = t["kv_offsets"] if ragged else None
    S_max = inp.S_max
    B, H, d = inp.q.shape
    p = santa.make_params(t["q"], t["K"], S_max, 0, 0, nk, offs, t["S_per_seq"])
    nbytes = santa.bernoulli_workspace_size(p)
    kv_bytes = t["K"].numel() * t["K"].element_size() * 2
    R = max(2, -(-FLUSH_BYTES // kv_bytes))
    reps = [(t["K"], t["V"])] + [(t["K"].clone(), t["V"].clone()) for _ in range(R - 1)]
    ws = santa.alloc_workspace(nbytes, dev)
    out = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    sid = ctypes.c_void_p(stream.cuda_stream)
    ptrs = [(ctypes.c_void_p(Kr.data_ptr()), ctypes.c_void_p(Vr.data_ptr())) for Kr, Vr in reps]
    qp, op, wp = (ctypes.c_void_p(x.data_ptr()) for x in (t["q"], out, ws))
    var = santa.VARIANTS[wl.variant]

    def step(i, idx=None, cnt=None):
        Kp, Vp = ptrs[i % R]
        st = lib.santa_decode_bernoulli(ctypes.byref(p), var, args.bernoulli, 1, qp, Kp, Vp, op, wp, nbytes,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                        None if idx is None else ctypes.c_void_p(idx.data_ptr()),
                                        None if cnt is None else ctypes.c_void_p(cnt.data_ptr()))
        if st != 0:
            raise RuntimeError(f"santa_decode_bernoulli: status {st}")

    idx = torch.full((B, H, S_max), -1, dtype=torch.int32, device=dev)
    cnt = torch.zeros((B, wl.n_kv_heads, d), dtype=torch.int32, device=dev)
    step(0, idx, cnt)
    torch.cuda.synchronize()
    unique_rows = count_unique_rows(inp, idx.cpu().numpy())
    share = float((cnt.cpu().numpy() > 0).mean())
    sampler = ClockSampler(local_rank).start()
    time.sleep(0.3)
    region = graph_replay_ms(step, args.steps, args.warmup, world)
    clocks = sampler.stop()
    ms = max_over_ranks(region, dev) / args.steps
    peak, peak_kind = hbm_peak()
    stb = step_bytes(inp, unique_rows)
    achieved = stb / (ms * 1e-3) / 1e9
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": ms * 1e3 / world, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "variant": wl.variant, "bernoulli_samples": args.bernoulli,
                   "bernoulli": "stratified, mean group query", "S": S_max, "nk": wl.nk, "batch": B,
                   "n_q_heads": H, "n_kv_heads": wl.n_kv_heads, "head_dim": d,
                   "l2": f"inputs larger than L2: {R} replicas of the K/V cache used in turn "
                         f"({R * kv_bytes >> 20} MiB)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": "step: bernoulli_query_kernel + fused_decode_kernel",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                     "peak_kind": f"of {peak_kind}", "alg_bytes_per_launch": stb,
                     "timing": "graph replay of the K timed steps over rotating replicas"},
        "step": {"alg_bytes": stb, "unique_v_rows": unique_rows, "key_feature_share": share},
        "cpu_baseline": None,
        "e2e": None,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.sampler != "global":
        return run_tiled(args)
    if args.bernoulli:
        return run_bernoulli(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
