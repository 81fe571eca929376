"""Benchmark of the causal GQA hot path on GB300.

Headline (one JSON line on stdout, rank 0): causal-visible TFLOP/s of the
dense prefill at Q=8000 query rows bottom-right aligned to KV=40000 keys,
Hq=6, Hkv=1, D=256, scale 1/16, fp16 in/out ("[Kernel][SM70] Default
long-prefill GQA architecture", Purpose and Test Result).  One step = one
gqa_attn_prefill call (main kernel + split merge) on inputs resident in HBM;
L2 is flushed before every timed step.  The same line carries:

* ``roofline``: the step's algorithmic FLOPs / measured step time against the
  measured dense bf16 tensor peak (fp16 runs at the same nominal rate);
* ``e2e``: the same metric through the C ABI with pinned host buffers and the
  host<->device copies inside the timed region;
* ``cpu_baseline``: the FP64 CPU oracle on a bounded sample of query rows;
  ``cpu_baselines`` times it on the other workloads as well (the small
  prefill in full, the E4M3 tails in full, the sparse prefill in full at 64
  and 512 tokens and on 512 sampled rows at 2048);
* ``secondary``: the rest of the 12-shape KV sweep (40K..128K), two other
  head groupings and head size 128 of the headline shape, the paged E4M3
  verifier tail at ctx 261888 (HBM roofline; one call alone, and calls back
  to back over distinct caches as the layers of a model run them), a batch of
  variable-length tails, and the selected-block sparse prefill.

``--impl reference`` times the CPU oracle alone on the same workload (bounded
sample per step) and prints the same kind of line with "impl": "reference".
Under torchrun each rank runs its own independent problem (weak scaling);
rank 0 prints.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HQ, D, SCALE = 6, 256, 1.0 / 16
Q_MAIN, KV_MAIN = 8000, 40000
KV_SWEEP = list(range(40000, 128001, 8000))      # the 12 prefill shapes
TAIL_CAPACITY, TAIL_CTX = 262144, 261888          # the E4M3 verifier-tail workload


def tail_kv_bytes(ctx_len: int, Dh: int = D) -> int:
    """E4M3 K and V bytes a tail reads: one byte per element, Hkv = 1."""
    return 2 * ctx_len * Dh


def visible_pairs(Q: int, KV: int) -> int:
    return Q * (KV - Q) + Q * (Q + 1) // 2


def prefill_flops(Q: int, KV: int, Hq: int = HQ, Dh: int = D) -> float:
    # QK^T and PV: 2 FLOPs per multiply-add each, per query head, per visible pair.
    return 4.0 * Dh * Hq * visible_pairs(Q, KV)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j.get("hbm_gbs", 6800.0), "bf16_tflops": j.get("bf16_tflops", 1900.0),
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", 1700.0),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job throughput: the units every rank processed (each rank runs its
    own independent problem) divided by the slowest rank's step time."""
    return units_per_rank * world / (max_ms * 1e-3)


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- GPU arm

PREWARM_S = 0.25


def time_steps(fn, steps, warmup, flush, stream, prewarm_s=PREWARM_S):
    """Per-step CUDA-event times (ms) of fn() on `stream`, L2 flushed before each.

    Before the `warmup` counted warm-up steps, untimed steps run for at least
    prewarm_s seconds, so that a GPU that sat idle while the inputs were made
    on the host has its clocks up before the timed steps (without this the
    timed steps of a fresh process included one 18 % slower than the rest)."""
    import torch
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < prewarm_s:
        for _ in range(4):
            flush()
            fn()
        torch.cuda.synchronize()
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    times = []
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    for a, b in evs:
        times.append(a.elapsed_time(b))
    return times


def profiled_traffic(profile: str, source: str, key: str = "traffic_bytes_per_launch"):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) that
    the ncu summary profiles/<profile> records, or None when the summary is
    missing or was taken on a different version of the kernel source (its
    source_sha256 line does not match)."""
    import hashlib
    import re
    try:
        text = open(os.path.join(ROOT, "profiles", profile)).read()
        digest = hashlib.sha256(open(os.path.join(ROOT, source), "rb").read()).hexdigest()
    except OSError:
        return None
    vals = dict(re.findall(r"^(\w+):\s*(\S+)\s*$", text, re.M))
    if vals.get("source_sha256") != digest or key not in vals:
        return None
    return int(vals[key])


def make_flush(device):
    """L2 flush run before every timed step: write a 256 MB buffer (twice the
    L2), then read a second 256 MB buffer.  The read replaces the write's dirty
    lines, so their write-back happens here rather than inside the timed
    kernel, and L2 holds neither the step's inputs nor its previous outputs."""
    import torch
    n = 256 * 1024 * 1024 // 4
    buf = torch.empty(n, dtype=torch.float32, device=device)
    buf2 = torch.ones(n, dtype=torch.float32, device=device)
    sink = torch.empty((), dtype=torch.float32, device=device)

    def flush():
        buf.fill_(1.0)
        torch.sum(buf2, dim=0, out=sink)
    return flush


def bench_prefill(binding, Q, KV, steps, warmup, flush, device, seed=0, Hq=HQ, Hkv=1, Dh=D,
                  e4m3=False):
    import torch
    from long_context_causal_gqa_gb300 import inputs
    stream = torch.cuda.current_stream()
    if e4m3:
        d = inputs.dense_e4m3_inputs(Q, KV, seed=seed, Hq=Hq, Hkv=Hkv, D=Dh)
        q, k, v = d.q.to(device), d.k.to(device), d.v.to(device)
        ks = torch.tensor([d.kscale], dtype=torch.float32, device=device)
        vs = torch.tensor([d.vscale], dtype=torch.float32, device=device)
        out = torch.empty_like(q)
        binding.prefill_e4m3(q, k, v, ks, vs, SCALE, out=out)
        times = time_steps(lambda: binding.prefill_e4m3(q, k, v, ks, vs, SCALE, out=out), steps,
                           warmup, flush, stream)
        return times, (q, k, v, out, d)
    d = inputs.dense_inputs(Q, KV, seed=seed, Hq=Hq, Hkv=Hkv, D=Dh)
    q, k, v = d.q.to(device), d.k.to(device), d.v.to(device)
    out = torch.empty_like(q)
    binding.prefill(q, k, v, SCALE, out=out)
    times = time_steps(lambda: binding.prefill(q, k, v, SCALE, out=out), steps, warmup, flush,
                       stream)
    return times, (q, k, v, out, d)


def bench_e2e_prefill(binding, d, steps, warmup, device):
    """Prefill through the public API with pinned host inputs: H2D copies of
    q, k, v, the call, and the D2H copy of out are all inside the timed region."""
    import torch
    hq, hk, hv = d.q.pin_memory(), d.k.pin_memory(), d.v.pin_memory()
    hout = torch.empty_like(d.q).pin_memory()
    q = torch.empty_like(hq, device=device)
    k = torch.empty_like(hk, device=device)
    v = torch.empty_like(hv, device=device)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()

    def step():
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        binding.prefill(q, k, v, SCALE, out=out)
        hout.copy_(out, non_blocking=True)

    times = time_steps(step, steps, warmup, lambda: None, stream)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = hout.numel() * hout.element_size()
    return times, h2d, d2h


def bench_e2e_prefill_overlapped(binding, d, steps, warmup, device):
    """The same end-to-end step as a serving loop would run it: two device
    buffer sets; step i's H2D copies go on a copy-in stream while step i - 1's
    kernels run, and step i's D2H read goes on a copy-out stream while step
    i + 1's kernels run.  Every step's copies are inside the timed region;
    events order each buffer's reuse.  Returns the mean ms per step."""
    import torch
    hin = [t.pin_memory() for t in (d.q, d.k, d.v)]
    hout = [torch.empty_like(d.q).pin_memory() for _ in range(2)]
    dev_in = [[torch.empty_like(t, device=device) for t in hin] for _ in range(2)]
    dev_out = [torch.empty_like(d.q, device=device) for _ in range(2)]
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        for i in range(n):
            b = i & 1
            cin.wait_event(ev_done[b])           # buffer set b no longer read by step i - 2
            with torch.cuda.stream(cin):
                for dst, src in zip(dev_in[b], hin):
                    dst.copy_(src, non_blocking=True)
            ev_in[b].record(cin)
            comp.wait_event(ev_in[b])
            comp.wait_event(ev_out[b])           # out[b] already read back
            q, k, v = dev_in[b]
            binding.prefill(q, k, v, SCALE, out=dev_out[b], stream=comp)
            ev_done[b].record(comp)
            cout.wait_event(ev_done[b])
            with torch.cuda.stream(cout):
                hout[b].copy_(dev_out[b], non_blocking=True)
            ev_out[b].record(cout)
        comp.wait_stream(cout)

    run(warmup)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    run(steps)
    end.record(comp)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def bench_paged(binding, R, device, steps, warmup, flush, ctx_len=TAIL_CTX, seed=0, Dh=D):
    import torch
    from long_context_causal_gqa_gb300 import inputs
    p = inputs.paged_e4m3_inputs(R=R, ctx_len=ctx_len, capacity=TAIL_CAPACITY, seed=seed, D=Dh)
    q = p.q.to(device)
    kc, vc = p.kcache.to(device), p.vcache.to(device)
    ks = torch.tensor([p.kscale], dtype=torch.float32, device=device)
    vs = torch.tensor([p.vscale], dtype=torch.float32, device=device)
    bt = p.block_table.to(device)
    out = torch.empty_like(q)

    def call():
        binding.paged_e4m3(q, kc, vc, ks, vs, bt, ctx_len, SCALE, out=out)
    call()
    torch.cuda.synchronize()
    # Replay the tail from a CUDA graph, as a verifier round would.
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    times = time_steps(g.replay, steps, warmup, flush, torch.cuda.current_stream())
    return times, tail_kv_bytes(ctx_len, Dh), 4.0 * Dh * HQ * visible_pairs(R, ctx_len)


def bench_paged_layers(binding, R, device, steps, warmup, flush, layers=4, ctx_len=TAIL_CTX,
                       seed=0):
    """`layers` tail calls back to back in one CUDA graph, each over its own
    cache (a model's layers: 4 x 134 MB, so no call finds the previous one's
    bytes in L2), L2 flushed before each replay; returns per-call times."""
    import torch
    from long_context_causal_gqa_gb300 import inputs
    sets = []
    for l in range(layers):
        p = inputs.paged_e4m3_inputs(R=R, ctx_len=ctx_len, capacity=TAIL_CAPACITY,
                                     seed=seed * 16 + l)
        sets.append((p.q.to(device), p.kcache.to(device), p.vcache.to(device),
                     torch.tensor([p.kscale], dtype=torch.float32, device=device),
                     torch.tensor([p.vscale], dtype=torch.float32, device=device),
                     p.block_table.to(device)))
    outs = [torch.empty_like(st[0]) for st in sets]

    def call():
        for st, o in zip(sets, outs):
            binding.paged_e4m3(*st, ctx_len, SCALE, out=o)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    times = time_steps(g.replay, steps, warmup, flush, torch.cuda.current_stream())
    return [t / layers for t in times], tail_kv_bytes(ctx_len)


def bench_paged_batch(binding, device, steps, warmup, flush, B=8, R=2, max_ctx=65536, seed=0):
    """B verifier tails of seeded lengths (about 262K tokens in all) in one
    gqa_attn_paged_e4m3_batch call, replayed from a CUDA graph with the
    context lengths in device memory."""
    import numpy as np
    import torch
    from long_context_causal_gqa_gb300 import inputs
    rng = np.random.default_rng(seed)
    ctxs = [int(x) for x in rng.integers(8192, 57345, size=B)]
    bi = inputs.paged_e4m3_batch_inputs(ctxs, R, max_ctx, seed=seed)
    c = bi.cache
    q = bi.q.to(device)
    kc, vc = c.kcache.to(device), c.vcache.to(device)
    ks = torch.tensor([c.kscale], dtype=torch.float32, device=device)
    vs = torch.tensor([c.vscale], dtype=torch.float32, device=device)
    bt = bi.tables.to(device)
    cl = torch.tensor(ctxs, dtype=torch.int32, device=device)
    out = torch.empty_like(q)

    def call():
        binding.paged_e4m3_batch(q, kc, vc, ks, vs, bt, cl, max_ctx, SCALE, out=out)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    times = time_steps(g.replay, steps, warmup, flush, torch.cuda.current_stream())
    kv_bytes = sum(2 * x * D for x in ctxs)
    return times, kv_bytes, ctxs


def bench_sparse(binding, T, device, steps, warmup, flush, rows=4096, ctx_len=32768, seed=0,
                 e4m3=False, Dh=D):
    """Selected-block sparse prefill over an fp16 cache, or an E4M3 cache
    (the raw codes on the FP8 tensor cores)."""
    import torch
    from long_context_causal_gqa_gb300 import inputs
    if e4m3:
        s = inputs.sparse_e4m3_inputs(rows=rows, ctx_len=ctx_len, tokens=T, seed=seed, D=Dh)
        ks = torch.tensor([s.kscale], dtype=torch.float32, device=device)
        vs = torch.tensor([s.vscale], dtype=torch.float32, device=device)
        q, kc, vc, bt, si, sc = [x.to(device) for x in (s.q, s.kcache, s.vcache, s.block_table,
                                                         s.sel_idx, s.sel_cnt)]
        out = torch.empty_like(q)

        def call():
            binding.sparse_blocks_e4m3(q, kc, vc, ks, vs, bt, si, sc, ctx_len, SCALE, out=out)
    else:
        s = inputs.sparse_inputs(rows=rows, ctx_len=ctx_len, tokens=T, seed=seed, D=Dh)
        args = [x.to(device) for x in (s.q, s.kcache, s.vcache, s.block_table, s.sel_idx,
                                       s.sel_cnt)]
        out = torch.empty_like(args[0])

        def call():
            binding.sparse_blocks(*args, ctx_len, SCALE, out=out)
    call()
    times = time_steps(call, steps, warmup, flush, torch.cuda.current_stream())
    visible = 0
    for i in range(rows):
        p = ctx_len - rows + i
        n = int(s.sel_cnt[i])
        visible += 4 * n - (3 - p % 4)
    gathered = rows * T * 2 * Dh * (1 if e4m3 else 2)   # K and V bytes of the selected tokens
    return times, gathered, 4.0 * Dh * HQ * visible


def cpu_baseline_prefill(Q, KV, seconds_target=15.0, seed=0):
    """Times the FP64 oracle on sampled query rows of the dense workload."""
    import numpy as np
    import oracle
    from long_context_causal_gqa_gb300 import inputs
    d = inputs.dense_inputs(Q, KV, seed=seed)
    ncores = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    # Calibrate on a few rows, then size the sample to about seconds_target.
    rows = rng.choice(Q, ncores, replace=False).astype(np.int32)
    t0 = time.perf_counter()
    oracle.dense(d.q, d.k, d.v, SCALE, rows=rows, nthreads=ncores)
    dt = time.perf_counter() - t0
    n = int(max(ncores, min(Q, ncores * max(1, int(seconds_target / max(dt, 1e-3))))))
    rows = np.sort(rng.choice(Q, n, replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    oracle.dense(d.q, d.k, d.v, SCALE, rows=rows, nthreads=ncores)
    dt = time.perf_counter() - t0
    pairs = sum(KV - Q + int(r) + 1 for r in rows)
    flops = 4.0 * D * HQ * pairs
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": ncores, "kind": "oracle",
            "seconds": dt,
            "sample": f"{n} of {Q} query rows x {HQ} heads of Q={Q} KV={KV}, FP64 two-pass"}


def _timed(fn):
    t0 = time.perf_counter()
    r = fn()
    return r, time.perf_counter() - t0


def cpu_baselines_other(seed=0):
    """The FP64 oracle, as it stands, timed on the small prefill (in full), the
    E4M3 verifier tails at ctx 261888 (in full, R = 1, 2, 8) and the sparse
    prefill (in full at T = 64 and 512, 512 sampled rows at T = 2048).  The
    oracle runs one thread per query row, so `cores` is min(rows, host cores)."""
    import numpy as np
    import oracle
    from long_context_causal_gqa_gb300 import inputs
    ncores = os.cpu_count() or 1
    res = []
    d = inputs.dense_inputs(256, 1024, seed=seed)
    _, dt = _timed(lambda: oracle.dense(d.q, d.k, d.v, SCALE, nthreads=ncores))
    fl = prefill_flops(256, 1024)
    res.append({"what": "dense prefill Q=256 KV=1024 (full)", "seconds": round(dt, 3),
                "TFLOP/s": fl / dt / 1e12, "cores": min(ncores, 256), "kind": "oracle"})
    for R in (1, 2, 8):
        p = inputs.paged_e4m3_inputs(R=R, ctx_len=TAIL_CTX, capacity=TAIL_CAPACITY, seed=seed)
        _, dt = _timed(lambda: oracle.paged_e4m3(p.q, p.kcache, p.vcache, p.kscale, p.vscale,
                                                 p.block_table, p.ctx_len, SCALE,
                                                 nthreads=ncores))
        nbytes = tail_kv_bytes(TAIL_CTX)
        res.append({"what": f"paged E4M3 tail R={R} ctx={TAIL_CTX} (full)",
                    "seconds": round(dt, 3), "GB/s": nbytes / dt / 1e9,
                    "TFLOP/s": 4.0 * D * HQ * visible_pairs(R, TAIL_CTX) / dt / 1e12,
                    "cores": min(ncores, R), "kind": "oracle"})
    for T in (64, 512, 2048):
        s = inputs.sparse_inputs(rows=4096, ctx_len=32768, tokens=T, seed=seed)
        rows = None
        n_rows = 4096
        if T == 2048:
            rows = np.sort(np.random.default_rng(T).choice(4096, 512, replace=False)).astype(
                np.int32)
            n_rows = 512
        _, dt = _timed(lambda: oracle.sparse_blocks(s.q, s.kcache, s.vcache, s.block_table,
                                                    s.sel_idx, s.sel_cnt, s.ctx_len, SCALE,
                                                    rows=rows, nthreads=ncores))
        rr = range(4096) if rows is None else rows
        visible = sum(4 * int(s.sel_cnt[i]) - (3 - (32768 - 4096 + int(i)) % 4) for i in rr)
        res.append({"what": f"sparse blocks T={T} ctx=32768, "
                            + ("4096 rows (full)" if rows is None else "512 of 4096 rows"),
                    "seconds": round(dt, 3),
                    "TFLOP/s": 4.0 * D * HQ * visible / dt / 1e12,
                    "cores": min(ncores, n_rows), "kind": "oracle"})
    return res


def config_of(Q, KV, world):
    """The `config` both arms report for the headline workload."""
    return {"workload": f"dense causal GQA prefill Q={Q} KV={KV} Hq=6 Hkv=1 D=256 "
                        "scale=1/16 batch 1", "Q": Q, "KV": KV,
            "l2": "flushed before every timed GPU step (256 MB write, then 256 MB read of a "
                  "second buffer)",
            "parallelism": f"{world} independent problem(s), one per GPU"}


def run_gpu(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from long_context_causal_gqa_gb300 import binding, build_lib
    if not build_lib.up_to_date():
        if rank == 0:
            build_lib.build()
        barrier(world)
    binding.load()
    peaks = load_peaks()
    flush = make_flush(device)
    Q, KV = args.q, args.kv

    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    times, keep = bench_prefill(binding, Q, KV, args.steps, args.warmup, flush, device,
                                seed=rank)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    step_ms = statistics.mean(times)
    step_ms_max = max_over_ranks(step_ms, world, device)
    flops = prefill_flops(Q, KV)
    value = whole_job_rate(flops, world, step_ms_max) / 1e12
    launches_per_step = 2  # main kernel + split merge
    achieved = flops / (step_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]

    e2e_times, h2d, d2h = bench_e2e_prefill(binding, keep[4], args.steps, min(args.warmup, 3),
                                            device)
    e2e_ms = max_over_ranks(statistics.mean(e2e_times), world, device)
    ovl_ms = max_over_ranks(bench_e2e_prefill_overlapped(binding, keep[4], args.steps,
                                                         min(args.warmup, 3), device),
                            world, device)
    assert binding.device_error() == 0

    line = {
        "metric": "causal-visible TFLOP/s of dense causal GQA prefill (Q=8000, KV=40000, "
                  "Hq=6, Hkv=1, D=256); % of FP16 tensor-core peak",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
        "data": "synthetic: seeded i.i.d. N(0,1) fp16 q/k/v",
        "config": config_of(Q, KV, world),
        "timing": {"prewarm": f"untimed steps for >= {PREWARM_S} s before the W warm-up steps",
                   "clock": "CUDA events on the launching stream, mean over the K timed steps"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peaks['source']} bf16 dense burst (fp16 same nominal rate)",
                     "traffic": profiled_traffic("prefill_kernel_Q8000_KV40000.md",
                                                 "long_context_causal_gqa_gb300/csrc/prefill.cu")
                     if (Q, KV) == (Q_MAIN, KV_MAIN) else None,
                     "traffic_note": "DRAM bytes per launch of prefill_kernel from the ncu "
                                     "summary in profiles/, null if taken on other source",
                     "note": "achieved = causal-visible FLOPs / CUDA-event time of one step "
                             "(main kernel + merge)"},
        "e2e": {"value": round(whole_job_rate(flops, world, e2e_ms) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "overlapped": {"value": round(whole_job_rate(flops, world, ovl_ms) / 1e12, 2),
                               "ms_per_step": round(ovl_ms, 4),
                               "note": "informational: the same copies and calls pipelined "
                                       "over two buffer sets (next inputs and previous output "
                                       "copied on their own streams while the kernels run)"}},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "step_ms": {"min": round(min(times), 4), "median": round(statistics.median(times), 4),
                    "max": round(max(times), 4)},
    }
    secondary = []
    if not args.quick:
        # Prefill secondaries, each with the SM clock sampled while it runs: they
        # follow one another for tens of seconds, and under that sustained load
        # the GPU's power cap can lower the clock (reported, not corrected).
        def prefill_secondary(what, kv, **kw):
            clk2 = ClockSampler(local)
            clk2.start()
            t, _ = bench_prefill(binding, Q, kv, max(3, args.steps // 2), 2, flush, device, **kw)
            c2 = clk2.stop()
            ms = statistics.mean(t)
            fl = prefill_flops(Q, kv, kw.get("Hq", HQ), kw.get("Dh", D))
            return {"what": what, "ms": round(ms, 4), "TFLOP/s": round(fl / ms / 1e9, 1),
                    "frac_of_peak": round(fl / ms / 1e9 / peak, 4),
                    "sm_mhz": c2.get("sm_mhz"), "clock_reasons": c2.get("reasons")}
        for hq, hkv, dh in ((6, 2, D), (8, 1, D), (6, 1, 128)):
            # Other head groupings (every query head's tiles in one launch when
            # Hkv > 1) and head size 128.
            e = prefill_secondary(f"prefill Q={Q} KV={KV} Hq={hq} Hkv={hkv} D={dh}", KV,
                                  Hq=hq, Hkv=hkv, Dh=dh)
            e["traffic"] = (profiled_traffic("prefill_kernel_d128_Q8000_KV40000.md",
                                             "long_context_causal_gqa_gb300/csrc/prefill.cu")
                            if (hq, hkv, dh, Q, KV) == (6, 1, 128, Q_MAIN, KV_MAIN) else None)
            secondary.append(e)
        for kv in (KV, KV_SWEEP[-1]):
            # K / V stored as E4M3 codes (converted to fp16 in shared memory).
            e = prefill_secondary(f"prefill Q={Q} KV={kv}, E4M3 K/V cache", kv, e4m3=True)
            e["traffic"] = (profiled_traffic("prefill_kernel_e4m3_Q8000_KV40000.md",
                                             "long_context_causal_gqa_gb300/csrc/prefill.cu")
                            if (Q, kv) == (Q_MAIN, KV_MAIN) else None)
            e["device_error"] = binding.device_error()
            secondary.append(e)
        for kv in ([x for x in KV_SWEEP if x != KV] if not args.no_sweep else [KV_SWEEP[-1]]):
            secondary.append(prefill_secondary(f"prefill Q={Q} KV={kv}", kv))
        for R in (1, 2, 8):
            try:
                t, nbytes, fl = bench_paged(binding, R, device, 50, 5, flush)
                derr = binding.device_error()
            except Exception as e:  # a secondary failure must not lose the headline
                secondary.append({"what": f"paged_e4m3 R={R}", "error": str(e)[:200]})
                continue
            if derr:
                secondary.append({"what": f"paged_e4m3 R={R}", "error": f"device error {derr}"})
                continue
            us = statistics.median(t) * 1e3
            gbs = nbytes / (us * 1e-6) / 1e9
            secondary.append({"what": f"paged E4M3 tail R={R} ctx=261888 (graph replay)",
                              "us": round(us, 2), "GB/s": round(gbs, 1),
                              "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                              "TFLOP/s": round(fl / (us * 1e-6) / 1e12, 1),
                              "algorithmic_bytes": nbytes,
                              "traffic": profiled_traffic(
                                  "paged_split_kernel_ctx261888.md",
                                  "long_context_causal_gqa_gb300/csrc/paged_e4m3.cu",
                                  f"traffic_bytes_per_launch_R{R}")})
        for R in (1, 8):
            try:
                t, nbytes, fl = bench_paged(binding, R, device, 50, 5, flush, Dh=128)
                derr = binding.device_error()
                us = statistics.median(t) * 1e3
                gbs = nbytes / (us * 1e-6) / 1e9
                secondary.append({"what": f"paged E4M3 tail R={R} ctx=261888 D=128 (graph replay)",
                                  "us": round(us, 2), "GB/s": round(gbs, 1),
                                  "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                                  "algorithmic_bytes": nbytes, "device_error": derr})
            except Exception as e:  # a secondary failure must not lose the headline
                secondary.append({"what": f"paged_e4m3 D=128 R={R}", "error": str(e)[:200]})
        for R in (1, 8):
            try:
                t, nbytes = bench_paged_layers(binding, R, device, 30, 5, flush)
                derr = binding.device_error()
                us = statistics.median(t) * 1e3
                gbs = nbytes / (us * 1e-6) / 1e9
                secondary.append({"what": f"paged E4M3 tail R={R} ctx=261888, 4 calls back to "
                                          "back over 4 distinct caches (graph replay), per call",
                                  "us": round(us, 2), "GB/s": round(gbs, 1),
                                  "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                                  "device_error": derr})
            except Exception as e:  # a secondary failure must not lose the headline
                secondary.append({"what": f"paged_e4m3 layers R={R}", "error": str(e)[:200]})
        try:
            t, nbytes, ctxs = bench_paged_batch(binding, device, 50, 5, flush)
            derr = binding.device_error()
            us = statistics.median(t) * 1e3
            gbs = nbytes / (us * 1e-6) / 1e9
            secondary.append({"what": f"paged E4M3 batch of {len(ctxs)} tails, R=2, contexts "
                                      f"{min(ctxs)}..{max(ctxs)} ({sum(ctxs)} tokens), device "
                                      "context lengths, graph replay",
                              "us": round(us, 2), "GB/s": round(gbs, 1),
                              "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                              "device_error": derr})
        except Exception as e:  # a secondary failure must not lose the headline
            secondary.append({"what": "paged_e4m3_batch", "error": str(e)[:200]})
        for e4m3 in (False, True):
            for T in (64, 512, 2048):
                kind = "E4M3 cache" if e4m3 else "fp16 cache"
                try:
                    t, gathered, fl = bench_sparse(binding, T, device, 5, 2, flush, e4m3=e4m3)
                    derr = binding.device_error()
                except Exception as e:
                    secondary.append({"what": f"sparse {kind} T={T}", "error": str(e)[:200]})
                    continue
                if derr:
                    secondary.append({"what": f"sparse {kind} T={T}",
                                      "error": f"device error {derr}"})
                    continue
                ms = statistics.median(t)
                secondary.append({"what": f"sparse blocks 4096 rows T={T} ctx=32768, {kind}",
                                  "ms": round(ms, 4),
                                  "gathered_GB/s": round(gathered / (ms * 1e-3) / 1e9, 1),
                                  "TFLOP/s": round(fl / (ms * 1e-3) / 1e12, 2),
                                  "traffic": profiled_traffic(
                                      "sparse_kernel_T512_rows4096.md",
                                      "long_context_causal_gqa_gb300/csrc/sparse_blocks.cu",
                                      "traffic_bytes_per_launch_e4m3" if e4m3
                                      else "traffic_bytes_per_launch") if T == 512 else None})
        for e4m3 in (False, True):
            kind = "E4M3 cache" if e4m3 else "fp16 cache"
            try:
                t, gathered, fl = bench_sparse(binding, 512, device, 5, 2, flush, e4m3=e4m3,
                                               Dh=128)
                derr = binding.device_error()
                ms = statistics.median(t)
                secondary.append({"what": f"sparse blocks 4096 rows T=512 ctx=32768 D=128, {kind}",
                                  "ms": round(ms, 4),
                                  "gathered_GB/s": round(gathered / (ms * 1e-3) / 1e9, 1),
                                  "TFLOP/s": round(fl / (ms * 1e-3) / 1e12, 2),
                                  "device_error": derr})
            except Exception as e:
                secondary.append({"what": f"sparse D=128 {kind}", "error": str(e)[:200]})
    line["secondary"] = secondary
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_prefill(Q, KV, seconds_target=args.cpu_seconds)
        if not args.quick:
            try:
                line["cpu_baselines"] = cpu_baselines_other()
            except Exception as e:
                line["cpu_baselines"] = [{"error": str(e)[:200]}]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_case(args):
    """One secondary workload alone (for profiling): --case prefill|paged|paged_batch|sparse."""
    import torch
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    from long_context_causal_gqa_gb300 import binding, build_lib
    if not build_lib.up_to_date():
        build_lib.build()
    binding.load()
    peaks = load_peaks()
    flush = make_flush(device)
    if args.case == "prefill":
        t, _ = bench_prefill(binding, args.q, args.kv, args.steps, args.warmup, flush, device,
                             Hq=args.hq, Hkv=args.hkv, Dh=args.d, e4m3=args.e4m3)
        ms = statistics.median(t)
        fl = prefill_flops(args.q, args.kv, args.hq, args.d)
        line = {"case": f"prefill Q={args.q} KV={args.kv} Hq={args.hq} Hkv={args.hkv} D={args.d}"
                        + (" E4M3 K/V" if args.e4m3 else ""),
                "ms": round(ms, 4), "TFLOP/s": round(fl / ms / 1e9, 1),
                "frac_of_peak": round(fl / ms / 1e9 / peaks["bf16_tflops"], 4)}
    elif args.case == "paged_batch":
        t, nbytes, ctxs = bench_paged_batch(binding, device, args.steps, args.warmup, flush)
        us = statistics.median(t) * 1e3
        line = {"case": f"paged E4M3 batch of {len(ctxs)} tails R=2 ({sum(ctxs)} tokens)",
                "us": round(us, 2), "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1),
                "hbm_frac": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}
    elif args.case in ("paged", "paged_layers"):
        if args.case == "paged":
            t, nbytes, fl = bench_paged(binding, args.rows, device, args.steps, args.warmup, flush,
                                       Dh=args.d)
        else:
            t, nbytes = bench_paged_layers(binding, args.rows, device, args.steps, args.warmup,
                                           flush)
        us = statistics.median(t) * 1e3
        line = {"case": f"paged E4M3 tail R={args.rows} ctx=261888 D={args.d}"
                        + (", 4 calls back to back, per call" if args.case != "paged" else ""),
                "us": round(us, 2), "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1),
                "hbm_frac": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}
    else:
        e4m3 = args.case == "sparse_e4m3"
        t, gathered, fl = bench_sparse(binding, args.tokens, device, args.steps, args.warmup, flush,
                                       e4m3=e4m3, Dh=args.d)
        ms = statistics.median(t)
        line = {"case": f"sparse blocks 4096 rows T={args.tokens} D={args.d}" + (" E4M3 cache" if e4m3 else ""),
                "ms": round(ms, 4), "gathered_GB/s": round(gathered / (ms * 1e-3) / 1e9, 1)}
    line["device_error"] = binding.device_error()
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The reference arm: the FP64 oracle, as it stands, on the host cores.
    Each step times the oracle on a bounded sample of the headline workload's
    query rows; `value` is the causal-visible FLOP rate of that sampled work,
    and `ms_per_step` the mean time of a step as run (the time the whole
    problem would take at that rate is reported separately)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    Q, KV = args.q, args.kv
    for _ in range(args.warmup):
        cpu_baseline_prefill(Q, KV, seconds_target=1.0)
    vals, secs = [], []
    last = None
    for _ in range(args.steps):
        last = cpu_baseline_prefill(Q, KV, seconds_target=args.ref_seconds)
        vals.append(last["value"])
        secs.append(last["seconds"])
    value = statistics.mean(vals)
    ms_full = prefill_flops(Q, KV) / (value * 1e12) * 1e3
    line = {
        "impl": "reference",
        "metric": "causal-visible TFLOP/s of dense causal GQA prefill (Q=8000, KV=40000, "
                  "Hq=6, Hkv=1, D=256); % of FP16 tensor-core peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(statistics.mean(secs) * 1e3, 1),
        "ms_per_step_note": "wall time of one step as run: the oracle on the sampled rows",
        "ms_full_problem_extrapolated": round(ms_full, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded i.i.d. N(0,1) fp16 q/k/v",
        "config": config_of(Q, KV, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last["cores"],
                         "kind": "oracle", "sample": last["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--q", type=int, default=Q_MAIN)
    ap.add_argument("--kv", type=int, default=KV_MAIN)
    ap.add_argument("--no-sweep", action="store_true",
                    help="secondary: only KV=128000 of the 12-shape KV sweep")
    ap.add_argument("--quick", action="store_true", help="headline only, no secondary")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=10.0)
    ap.add_argument("--case", default="headline", choices=["headline", "prefill", "paged",
                                                           "paged_layers", "paged_batch",
                                                           "sparse", "sparse_e4m3"],
                    help="run one secondary workload alone (profiling)")
    ap.add_argument("--rows", type=int, default=8, help="--case paged: tail rows")
    ap.add_argument("--hq", type=int, default=HQ, help="--case prefill: query heads")
    ap.add_argument("--hkv", type=int, default=1, help="--case prefill: KV heads")
    ap.add_argument("--d", type=int, default=D, help="--case prefill|paged|sparse: head size (256 or 128)")
    ap.add_argument("--tokens", type=int, default=2048, help="--case sparse: tokens per row")
    ap.add_argument("--e4m3", action="store_true", help="--case prefill: E4M3 K/V cache")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.case != "headline":
        run_case(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
