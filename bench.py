#!/usr/bin/env python3
"""CSA2 decode throughput on GB300: queries/s per layer group and its fraction
of the HBM roofline.

One step = one pass of the whole layer group (indexer scoring, hierarchical
pool, exact Top-K, sparse attention) over one decode query per sequence of
the workload's batch, replayed from a CUDA graph of one csa2_layer_group
call.  Default workload: the hierarchical Reindex layer at 128K context
(batch 64, 32,768 compressed entries, pool of 2,048 blocks, Top-512 + 128 SWA).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): every rank runs its own replica of
the workload (batch-parallel, no exchange: weak scaling); the timed region is
bracketed by barriers and the max over ranks is reported.

``--impl reference`` times the CPU oracle (there is no other implementation
of this method to run) on a bounded sample of the same workload on the host
cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_attention_decode_index_gb300 import workloads as W  # noqa: E402

METRIC = "CSA2 decode queries/sec per layer group at 128K ctx; % of GB300 HBM roofline"
FUSED_MAX_ROWS = 32768          # rows per query served by the fused flat scoring + Top-K (8 CTAs x 4,096)
UNIT = "queries/s"
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"
    return 6800.0, "fallback (6.8 TB/s, earlier GB300 measurement)"


def algorithmic_bytes(wl) -> dict:
    """Bytes the method must move per step (each distinct index set's KV counted once)."""
    sh = wl.shape
    e = 4 if sh.dtype == "f32" else 2
    row_kv = (sh.k_dim + sh.v_dim) * e
    total = {"indexer_blocks": 0, "indexer_tokens": 0, "selected_kv": 0, "swa_kv": 0, "q": 0, "out": 0}
    for b in range(sh.batch):
        nv = int(wl.n_valid[b])
        ns = int(wl.n_swa[b])
        nb = -(-nv // sh.block)
        for L in wl.layers:
            if L.mode in (W.FULL, W.REINDEX):
                if L.hier:
                    pb = min(sh.pool_blocks, nb)
                    total["indexer_blocks"] += nb * sh.idx_dim * e
                    ncand = min(pb * sh.block, nv)
                    total["indexer_tokens"] += pb * sh.block * sh.idx_dim * e
                else:
                    ncand = nv
                    total["indexer_tokens"] += nv * sh.idx_dim * e
                total["selected_kv"] += min(sh.topk, ncand) * row_kv
            total["swa_kv"] += ns * row_kv
            total["q"] += sh.q_heads * sh.k_dim * e
            total["out"] += sh.q_heads * sh.v_dim * 4
    total["total"] = sum(total.values())
    return total


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
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
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle timing

def _oracle_worker(conn):
    import oracle
    data = None
    while True:
        msg = conn.recv()
        if msg[0] == "data":
            data = msg[1]
            conn.send(("ok",))
        elif msg[0] == "run":
            t0 = time.perf_counter()
            for wl in data:
                oracle.run_group(wl)
            conn.send(("done", time.perf_counter() - t0))
        else:
            conn.send(("bye",))
            return


def slice_queries(wl, queries):
    """A workload holding only the given queries of ``wl`` (batch = len(queries), one token per
    sequence: with ``shape.tokens`` = T > 1 query q reads cache sequence q // T, whose caches the
    slice copies)."""
    import copy
    T = max(1, int(getattr(wl.shape, "tokens", 1)))
    seqs = [q // T for q in queries]
    sub = copy.copy(wl)
    sub.shape = W.Shape(**{**wl.shape.__dict__, "batch": len(queries), "tokens": 1})
    sub.k_main, sub.v_main, sub.k_idx = wl.k_main[seqs], wl.v_main[seqs], wl.k_idx[seqs]
    sub.n_valid, sub.n_swa = wl.n_valid[queries], wl.n_swa[queries]
    sub.layers = [W.Layer(mode=L.mode, hier=L.hier, q=L.q[queries], k_swa=L.k_swa[queries],
                          v_swa=L.v_swa[queries], q_idx=None if L.q_idx is None else L.q_idx[queries],
                          w_idx=None if L.w_idx is None else L.w_idx[queries]) for L in wl.layers]
    return sub


class OraclePool:
    """One spawned process per host core, each running the oracle on its share of a sample."""

    def __init__(self, wl, queries_per_worker: int = 1, workers: int = 0):
        self.workers = workers or max(1, (os.cpu_count() or 1))
        self.workers = min(self.workers, wl.shape.batch)
        ctx = mp.get_context("spawn")
        env_keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in env_keep:
            os.environ[k] = "1"      # one BLAS thread per worker process
        self.conns, self.procs = [], []
        try:
            for w in range(self.workers):
                a, b = ctx.Pipe()
                p = ctx.Process(target=_oracle_worker, args=(b,), daemon=True)
                p.start()
                self.conns.append(a)
                self.procs.append(p)
        finally:
            for k, v in env_keep.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        qs = list(range(wl.shape.batch))
        self.queries = 0
        for w, c in enumerate(self.conns):
            mine = qs[w::self.workers][:queries_per_worker]
            self.queries += len(mine)
            c.send(("data", [slice_queries(wl, [q]) for q in mine]))
        for c in self.conns:
            c.recv()

    def step(self) -> float:
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(("run",))
        for c in self.conns:
            c.recv()
        return time.perf_counter() - t0

    def close(self):
        for c in self.conns:
            try:
                c.send(("stop",))
                c.recv()
            except (EOFError, OSError, BrokenPipeError):
                pass
        for p in self.procs:
            p.join(timeout=10)


CPU_SAMPLE_SECONDS = 10.0       # wall time of the oracle sample (bounded: at most CPU_SAMPLE_PASSES passes)
CPU_SAMPLE_PASSES = 2000


def cpu_sample(pool, wl) -> dict:
    """Time the oracle pool on repeated passes over its sample for about CPU_SAMPLE_SECONDS."""
    try:
        times = [pool.step()]
        while sum(times) < CPU_SAMPLE_SECONDS and len(times) < CPU_SAMPLE_PASSES:
            times.append(pool.step())
    finally:
        pool.close()
    return {"value": pool.queries * len(times) / sum(times), "unit": UNIT, "cores": pool.workers, "kind": "oracle",
            "sample": f"{pool.queries} of the {wl.shape.batch} queries of {wl.name} (one per worker process, 1 BLAS "
                      f"thread each), {len(times)} passes, {sum(times):.1f} s wall"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    wl = W.named(args.workload)
    pool = OraclePool(wl)
    try:
        for _ in range(args.warmup):
            pool.step()
        times = [pool.step() for _ in range(args.steps)]
    finally:
        pool.close()
    total = sum(times)
    value = pool.queries * len(times) / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {k: v for k, v in config_of(wl, args).items() if k not in ("l2", "launch")},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.workers, "kind": "oracle",
                             "sample": f"{pool.queries} of {wl.shape.batch} queries per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def make_flusher(torch, nbytes, device):
    """L2 flush between timed steps: write a buffer larger than L2, then read it
    back, so the next step finds none of its inputs in L2 and no dirty lines
    whose write-back would be charged to it."""
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    view = buf.view(torch.int64)
    sink = torch.empty((), dtype=torch.int64, device=device)

    def flush():
        buf.fill_(1)
        torch.amax(view, dim=0, out=sink)
    return flush


def config_of(wl, args):
    sh = wl.shape
    spec = W.WORKLOADS.get(wl.name, {})
    return {"workload": wl.name, "batch": sh.batch, "context_tokens": spec.get("context"),
            "entries": sh.n_entries, "layers": [W.MODE_NAMES[L.mode] + ("+hier" if L.hier else "") for L in wl.layers],
            "pool_blocks": sh.pool_blocks, "topk": sh.topk, "swa": sh.swa, "q_heads": sh.q_heads,
            "k_dim": sh.k_dim, "v_dim": sh.v_dim, "idx_heads": sh.idx_heads, "idx_dim": sh.idx_dim,
            "l2": f"flushed between timed steps ({args.flush_mb} MB written then read back)",
            "launch": "CUDA graph replay"}


# ----------------------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    from sparse_attention_decode_index_gb300 import build as B
    from sparse_attention_decode_index_gb300 import csa2

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    B.build()
    csa2.lib()

    wl = W.named(args.workload, seed=rank)
    sh = wl.shape
    ab = algorithmic_bytes(wl)
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    pool = OraclePool(wl) if want_cpu else None          # spawned before the first GPU work

    d = csa2.upload(wl, device=dev)
    if any(L.hier for L in wl.layers):
        csa2.block_keys(sh, d["k_idx"], d["n_valid"], d["kb"], d["ws"], round_to_int=bool(wl.round_block_keys))
    call = csa2.LayerGroupCall(sh, d["layers"], d["k_main"], d["v_main"], d["k_idx"], d["kb"], d["n_valid"],
                               d["n_swa"], d["ws"])
    stream = torch.cuda.Stream(device=dev)
    flush = make_flusher(torch, args.flush_mb * 1024 * 1024, dev)
    with torch.cuda.stream(stream):
        call(stream)                                     # first call: attributes, validation
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        n0 = csa2.launch_count()
        with torch.cuda.graph(graph, stream=stream):
            call(stream)
        per_step_launches = csa2.launch_count() - n0
        for _ in range(args.warmup):
            flush()
            graph.replay()
        torch.cuda.synchronize()
        st, bits = csa2.read_device_error(d["ws"], stream)
        if st != 0:
            raise RuntimeError(f"device error word {bits:#x} after warm-up")

        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]

        def soak(seconds):
            # untimed replays of the same step so that nvidia-smi (200 ms period) sees the
            # clocks of this workload around the (short) timed region
            t_end = time.perf_counter() + seconds
            while time.perf_counter() < t_end:
                for _ in range(20):
                    flush()
                    graph.replay()
                torch.cuda.synchronize()

        with ClockSampler(dev.index) as clk:
            soak(args.clock_soak)
            barrier()
            torch.cuda.synchronize()
            for e0, e1 in evs:
                flush()
                e0.record(stream)
                graph.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            barrier()
            soak(args.clock_soak / 2)
        step_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    total_s = max_over_ranks(sum(step_ms) / 1e3, dev)
    value = sh.batch * world * args.steps / total_s
    ms_per_step = 1e3 * total_s / args.steps

    peak, peak_src = measured_peaks()
    roof = dominant_kernel_roofline(csa2, wl, d, stream, flush, args, peak, peak_src)
    step_gbs = ab["total"] / (ms_per_step / 1e3) / 1e9
    e2e = end_to_end(csa2, wl, d, graph, stream, flush, args, dev)
    append = append_timing(csa2, wl, stream, args)
    clocks = clk.summary()
    clocks["window"] = (f"nvidia-smi every 200 ms over the timed steps plus {args.clock_soak:.1f} s before and "
                        f"{args.clock_soak / 2:.1f} s after of untimed replays of the same step")

    cpu = cpu_sample(pool, wl) if pool is not None else None
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(wl, args),
                "roofline": roof,
                "step_roofline": {"bound": "hbm", "achieved": step_gbs, "peak": peak, "unit": "GB/s",
                                  "frac": step_gbs / peak, "alg_bytes_per_step": ab["total"],
                                  "alg_bytes_breakdown": ab, "peak_source": peak_src,
                                  "frac_of_nominal_8TBs": step_gbs / 8000.0},
                "cpu_baseline": cpu, "e2e": e2e, "append": append,
                "gpu_launches": per_step_launches * args.steps,
                "launches_per_step": per_step_launches, "clocks": clocks,
                "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)}}
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


# Sources whose hash a traffic record carries, per dominant-kernel kind.
KERNEL_SOURCES = {
    "index_select_pooled": ("fused.cu", "common.cuh", "internal.h"),
    "index_select_flat": ("fused.cu", "common.cuh", "internal.h"),
    "indexer_flat": ("indexer.cu", "common.cuh", "internal.h"),
}


def kernel_source_hash(kind: str) -> str:
    """First 16 hex digits of the SHA-256 of a dominant kernel's sources, with
    comments and blank lines left out (an edit of the documentation alone does not
    make a traffic capture stale)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "sparse_attention_decode_index_gb300", "csrc", name)) as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        for line in text.splitlines():
            code = re.sub(r"//.*$", "", line).rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(wl, kind: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu capture
    (profiles/<kind>__<workload>.traffic.json, written beside its summary), or None when no
    capture covers this workload or the kernel's sources changed since it was captured."""
    name = f"{kind}__{wl.name}.traffic.json"
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None, "no ncu capture of this workload's dominant kernel"
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_sha256_16") != kernel_source_hash(kind):
        return None, "kernel source changed since the ncu capture"
    return int(rec["dram_bytes_per_launch"]), "dram__bytes_read.sum + dram__bytes_write.sum, profiles/" + name


def dominant_kernel_roofline(csa2, wl, d, stream, flush, args, peak, peak_src):
    """Time the step's dominant kernel alone (CUDA events on its stream, L2 flushed between launches)."""
    import torch
    sh = wl.shape
    L0 = next(L for L in d["layers"] if L["mode"] in (W.FULL, W.REINDEX))
    hier = bool(L0.get("hier"))
    dev = d["k_idx"].device
    reps = max(args.steps, 10)
    idx = torch.empty((sh.batch, sh.topk), dtype=torch.int32, device=dev)
    fused_flat = sh.n_entries <= FUSED_MAX_ROWS
    with torch.cuda.stream(stream):
        if hier:
            pool = torch.empty((sh.batch, sh.pool_blocks), dtype=torch.int32, device=dev)
            n_pool = torch.empty(sh.batch, dtype=torch.int32, device=dev)
            csa2.index_blocks(sh, L0["q_idx"], L0["w_idx"], d["kb"], d["n_valid"], pool, n_pool, d["ws"], stream)

            def launch():
                csa2.index_topk(sh, L0["q_idx"], L0["w_idx"], d["k_idx"], d["n_valid"], sh.topk, idx, d["ws"],
                                pool=pool, n_pool=n_pool, stream=stream)
            name = ("index_select_kernel<pooled> (csa2_index_topk: pooled token scoring + exact Top-512, "
                    "one cluster per query)")
            n_rows = sum(min(sh.pool_blocks, -(-int(v) // sh.block)) * sh.block for v in wl.n_valid)
        elif fused_flat:
            def launch():
                csa2.index_topk(sh, L0["q_idx"], L0["w_idx"], d["k_idx"], d["n_valid"], sh.topk, idx, d["ws"],
                                stream=stream)
            name = "index_select_kernel<flat> (csa2_index_topk: flat token scoring + exact Top-512)"
            n_rows = int(sum(int(v) for v in wl.n_valid))
        else:
            scores = torch.empty((sh.batch, sh.n_entries), dtype=torch.float32, device=dev)

            def launch():
                csa2.index_tokens(sh, L0["q_idx"], L0["w_idx"], d["k_idx"], d["n_valid"], scores, d["ws"],
                                  stream=stream)
            name = ("indexer_mma_kernel<flat> (csa2_index_tokens: flat token scoring of the Full layer, "
                    "scores written to HBM)")
            n_rows = int(sum(int(v) for v in wl.n_valid))
        launch()
        torch.cuda.synchronize()
        ms = []
        for _ in range(reps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch()
            e1.record(stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
    e = 4 if sh.dtype == "f32" else 2
    alg = n_rows * sh.idx_dim * e
    if not hier and not fused_flat:
        alg += n_rows * 4                                 # the fp32 score of every row is written
    avg = sum(ms) / len(ms)
    gbs = alg / (avg / 1e3) / 1e9
    kind = "index_select_pooled" if hier else ("index_select_flat" if fused_flat else "indexer_flat")
    traffic, traffic_src = profiled_traffic(wl, kind)
    return {"bound": "hbm", "kernel": name, "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
            "traffic": traffic, "traffic_source": traffic_src, "alg_bytes_per_launch": alg, "launch_us": 1e3 * avg,
            "peak_source": peak_src,
            "timing": f"alone, {reps} launches, CUDA events on its stream, L2 flushed before each"}


def append_timing(csa2, wl, stream, args):
    """Decode-step cache maintenance at the workload's batch and dims: one new compressed
    entry per query (csa2_kv_append, block keys kept) and one token per query into one
    layer's SWA ring (csa2_swa_append), each timed alone on its stream: device time per call
    from CUDA graphs of back-to-back calls.
    Runs on buffers of its own (1,024-entry caches; the cost does not depend on the
    cache length), after every other measurement."""
    import torch
    sh = dataclasses.replace(wl.shape, n_entries=1024, tokens=1)   # appends are per sequence
    B, dev = sh.batch, torch.device("cuda")
    bf = torch.bfloat16
    k_main = torch.zeros((B, sh.n_entries, sh.k_dim), dtype=bf, device=dev)
    v_main = torch.zeros((B, sh.n_entries, sh.v_dim), dtype=bf, device=dev)
    k_idx = torch.zeros((B, sh.n_entries, sh.idx_dim), dtype=bf, device=dev)
    kb = torch.zeros((B, sh.n_entries // sh.block, sh.idx_dim), dtype=bf, device=dev)
    k_new = torch.ones((B, 1, sh.k_dim), dtype=bf, device=dev)
    v_new = torch.ones((B, 1, sh.v_dim), dtype=bf, device=dev)
    x_new = torch.ones((B, 1, sh.idx_dim), dtype=bf, device=dev)
    n_new = torch.ones(B, dtype=torch.int32, device=dev)
    n_valid = torch.zeros(B, dtype=torch.int32, device=dev)
    k_swa = torch.zeros((B, sh.swa, sh.k_dim), dtype=bf, device=dev)
    v_swa = torch.zeros((B, sh.swa, sh.v_dim), dtype=bf, device=dev)
    k_tok = torch.ones((B, sh.k_dim), dtype=bf, device=dev)
    v_tok = torch.ones((B, sh.v_dim), dtype=bf, device=dev)
    head = torch.zeros(B, dtype=torch.int32, device=dev)
    n_swa = torch.zeros(B, dtype=torch.int32, device=dev)
    ws = csa2.workspace(sh)
    reps = max(args.steps, 20)

    per = 16                                                     # calls per captured graph

    def timed(fn, reset):
        """Median device time per call: graphs of `per` back-to-back calls replayed with
        CUDA events around each replay (so host-side argument marshalling is not timed)."""
        with torch.cuda.stream(stream):
            reset()
            fn()                                                 # warm-up outside capture
            reset()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(per):
                fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        with torch.cuda.stream(stream):
            for i in range(3):
                reset()
                g.replay()
            for e0, e1 in evs:
                reset()
                e0.record(stream)
                g.replay()
                e1.record(stream)
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3 / per

    us_kv = timed(lambda: csa2.kv_append(sh, n_new, k_new, v_new, x_new, k_main, v_main, k_idx, kb, n_valid, ws,
                                         stream=stream), lambda: n_valid.zero_())
    us_swa = timed(lambda: csa2.swa_append(sh, [(k_tok, v_tok, k_swa, v_swa)], head, n_swa, ws, stream=stream),
                   lambda: (head.zero_(), n_swa.zero_()))
    st, bits = csa2.read_device_error(ws, stream)
    row = 2 * (sh.k_dim + sh.v_dim + sh.idx_dim)                 # one entry read and written
    kv_bytes = B * (row + sh.block * 2 * sh.idx_dim + 2 * sh.idx_dim)   # + block rows read, summary written
    swa_bytes = B * 2 * 2 * (sh.k_dim + sh.v_dim)
    return {"workload": f"batch {B}, one new compressed entry and one SWA token per query",
            "kv_append_us": us_kv, "kv_append_bytes": kv_bytes, "swa_append_us": us_swa,
            "swa_append_bytes": swa_bytes, "bound": "launch latency (one CTA per query, KBs per call)",
            "device_error_bits": bits}


def end_to_end(csa2, wl, d, graph, stream, flush, args, dev):
    """Same metric through the public API with pinned host buffers, run as a serving loop would:
    every step copies its query inputs host->device and its outputs device->host, on two copy
    streams, while the compute stream runs the group.  The steps themselves stay serialised on the
    compute stream; two sets of per-step device buffers alternate, so step i+1's inputs arrive
    while step i computes.  The main-KV, indexer-key and block-key caches stay resident.  No L2
    flush between steps when a step reads more than the 129 MB L2 (the headline reads ~198 MB)."""
    import torch
    sh = wl.shape
    k_in, k_out = ("q", "q_idx", "w_idx", "k_swa", "v_swa"), ("out", "lse", "idx_out")

    def tensors(layers, n_valid, n_swa):
        ins = [y[k] for y in layers for k in k_in if y.get(k) is not None] + [n_valid, n_swa]
        outs = [y[k] for y in layers for k in k_out if y.get(k) is not None]
        return ins, outs

    layers1 = [{k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in y.items()} for y in d["layers"]]
    nv1, ns1 = d["n_valid"].clone(), d["n_swa"].clone()
    call1 = csa2.LayerGroupCall(sh, layers1, d["k_main"], d["v_main"], d["k_idx"], d["kb"], nv1, ns1, d["ws"])
    with torch.cuda.stream(stream):
        call1(stream)
        torch.cuda.synchronize()
        graph1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph1, stream=stream):
            call1(stream)
    sets = [tensors(d["layers"], d["n_valid"], d["n_swa"]), tensors(layers1, nv1, ns1)]
    host_in = [t.cpu().pin_memory() for t in sets[0][0]]
    host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs] for _, outs in sets]
    h2d = sum(t.numel() * t.element_size() for t in sets[0][0])
    d2h = sum(t.numel() * t.element_size() for t in sets[0][1])
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def capture(fn, st):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            fn()
        return g

    g_in, g_out = [], []
    for i, (ins, outs) in enumerate(sets):
        g_in.append(capture(lambda ins=ins: [dd.copy_(hd, non_blocking=True) for hd, dd in zip(host_in, ins)], up))
        g_out.append(capture(lambda i=i, outs=outs: [hd.copy_(dd, non_blocking=True)
                                                     for hd, dd in zip(host_out[i], outs)], down))
    comp = [graph, graph1]
    n = args.warmup + args.steps
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(n)] for _ in range(3))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for i in range(n):
        s_ = i % 2
        if i >= 2:
            up.wait_event(ev_comp[i - 2])          # set s_'s inputs were read by step i-2
        if i == args.warmup:
            t0.record(up)                          # the first timed step's input copy starts here
        with torch.cuda.stream(up):
            g_in[s_].replay()
        ev_in[i].record(up)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])       # set s_'s outputs of step i-2 are on the host
        with torch.cuda.stream(stream):
            comp[s_].replay()
        ev_comp[i].record(stream)
        down.wait_event(ev_comp[i])
        with torch.cuda.stream(down):
            g_out[s_].replay()
        ev_out[i].record(down)
    t1.record(down)
    torch.cuda.synchronize()
    total = max_over_ranks(t0.elapsed_time(t1) / 1e3, dev)
    world = dist_env()[1]
    return {"value": sh.batch * world * args.steps / total, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * total / args.steps,
            "pipeline": "inputs of step i+1 copied in and outputs of step i copied out while step i computes; "
                        "two buffer sets; steps serialised on the compute stream; timed from the start of the "
                        "first timed step's input copy to the end of the last timed step's output copy",
            "l2": f"not flushed between steps: each step reads {algorithmic_bytes(wl)['total'] / 1e6:.0f} MB of "
                  "algorithmic bytes" + (", more than the 129 MB L2" if algorithmic_bytes(wl)["total"] > 129e6
                                         else " (fits in L2: later steps may hit it)"),
            "resident": "the main-KV, indexer-key and block-key caches stay on the device"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="reindex_b64_128k", choices=sorted(W.WORKLOADS))
    ap.add_argument("--flush-mb", type=int, default=512)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-soak", type=float, default=1.5,
                    help="seconds of untimed replays around the timed steps while clocks are sampled")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
