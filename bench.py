#!/usr/bin/env python
"""Benchmark of context-parallel MLA prefill attention on GB300.

One step = the whole path over one batch: DualChunkSwap partition maps (built
once per batch, outside the device-timed region), partial attention of all P
virtual shards in one launch, then the global LSE merge with the sink and the
restore to global order.  Default workload: the mixed varlen batch -- 8
prefills of U[1024, 65536] tokens and 32 decode rows over contexts of
U[4096, 131072], 64 heads, P = 8, top-2048 sparse (the largest single-GPU
configuration of the metric).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl cuda|reference] [--no-cpu-baseline]

Prints one JSON line.  value = TFLOP/s of the step (2*576 + 2*512 flops per
attended (token, head, key)), inputs resident in HBM, L2 flushed between steps.
e2e = the same metric through the public API with pinned host buffers: host
partition, host->device copy of the step's inputs, attention, merge, and the
device->host copy of the output inside the timed region.
"""
import argparse
import atexit
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "CP-prefill MLA attention TFLOP/s + tokens/s (incl. merge), % of GB300 roofline"
# DRAM bytes (read + write) of one launch of the dominant kernel, from the ncu
# capture summarised in profiles/ (per workload and path; None = not captured
# for the current kernel).  Must be reset whenever that kernel changes.
NCU_TRAFFIC_BYTES = {("dense_s8192_h16_p2", "merged"): 162_865_408 + 95_957_760,
                     ("topk_s32k_k2048", "topk"): 2_245_461_504 + 257_710_080,
                     # 16002-token capture of the same shape (1.433 + 1.018 GB),
                     # scaled to the workload's 326209 tokens
                     ("varlen_p8_h64", "merged"): int((1.432820e9 + 1.018263e9) * 326209 / 16002),
                     # 12288-token capture (587.7 + 376.8 MB), scaled to 32768 tokens
                     ("sparse_s32k_h32_p4", "merged"): int((587.681280e6 + 376.763136e6) * 32768 / 12288),
                     # 16384-token capture (451.9 + 244.5 MB), scaled to 131072 tokens
                     ("sparse_s128k_h16_p2_fp8", "merged"): int((451.890176e6 + 244.510464e6) * 131072 / 16384)}
FLOPS_PER_KEY_HEAD = 2 * 576 + 2 * 512
L2_FLUSH_BYTES = 512 << 20


class L2Flush:
    """Evicts L2 between timed steps: writes a buffer larger than L2 (129 MB),
    then reads another, so the written lines are back in HBM before the next
    timed launch (after a bare write, the launch would also pay for writing
    back up to 129 MB of the flush buffer's dirty lines)."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.acc = torch.zeros((), dtype=torch.float32, device=dev)

    def __call__(self, v=1.0):
        self.w.fill_(v)
        torch.sum(self.r, dim=0, out=self.acc)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, every 50 ms from
    entry (started before the warm-up, since nvidia-smi takes a while to
    start); `window(t0, t1)` (time.time() seconds) keeps the samples that
    arrived while the timed steps ran."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def __enter__(self):
        if self.proc is not None:  # already sampling (started early by clock_sampler)
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self is _SAMPLER:  # the shared sampler runs until the process exits
            return
        self.stop()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines, where = self.lines, "whole run"
        if self.t0 is not None:
            # a sample is printed shortly after it is taken; a timed region
            # shorter than the sampling period takes its nearest samples
            for pad, name in ((0.05, "timed steps"), (0.25, "timed steps +- 0.25 s")):
                near = [x for x in self.lines if self.t0 - pad + 0.05 <= x[0] <= self.t1 + pad]
                if near:
                    lines, where = near, name
                    break
        for _, ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0, "over": where}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "over": where}


_SAMPLER = None


def clock_sampler(index):
    """The process's sampler, started on first use (early, so that samples
    already flow when a short timed region runs) and stopped at exit."""
    global _SAMPLER
    if _SAMPLER is None:
        _SAMPLER = ClockSampler(index)
        _SAMPLER.__enter__()
        atexit.register(_SAMPLER.stop)
    return _SAMPLER


def dist_setup(n_gpus, backend=None):
    """One process per GPU (torchrun's RANK/LOCAL_RANK/WORLD_SIZE); NCCL when
    CUDA is present, gloo otherwise (the CPU tests of the multi-rank path)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Largest value over the ranks (step time: the job runs at its slowest rank)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, step_ms, world):
    """Whole-job throughput of `world` replicas that each process
    `units_per_rank` per step: all ranks' units over the max-over-ranks time."""
    return world * units_per_rank / (step_ms * 1e-3)


KV_INSERT_WORKLOAD = "kv_insert_s128k_fp8"


def run_kv_insert(args, world, rank, local):
    """The latent KV-cache insertion, fp8 layout, of the 131072-token sparse
    workload's KV: one launch per step over every token, slots those of a
    paged cache (64-token pages in a seeded random page order).  Reports GB/s against the measured HBM
    copy bandwidth (bytes: the bf16 rows and slots read, codes + scales + rope
    written).  --impl reference times the oracle's insertion on a sample."""
    n, s_cache = 131072, 131072
    g = torch.Generator().manual_seed(args.seed)
    kv = (torch.randn((n, 576), generator=g) * torch.exp(torch.randn((n, 1), generator=g)))
    kv = kv.to(torch.bfloat16)
    # a paged cache's slot mapping: 64-token pages, pages in a seeded random order
    page = 64
    order = torch.randperm(s_cache // page, generator=g).to(torch.int64)
    slot = (order[:, None] * page + torch.arange(page)[None, :]).reshape(-1)[:n]
    bytes_step = n * (576 * 2 + 8 + 512 + 4 * 4 + 64 * 2)
    cfg = {"workload": KV_INSERT_WORKLOAD, "tokens": n, "cache_rows": s_cache, "kv_format": "fp8",
           "slots": "64-token pages in a seeded random page order",
           "l2": "flushed between steps (512 MiB write, then 512 MiB read)", "parallelism": "single GPU"}
    if args.impl == "reference":
        if rank == 0:
            from oracle import oracle as orc
            bits = kv.view(torch.int16).numpy().view(np.uint16)
            m = 8192
            t0 = time.perf_counter()
            for i in range(args.steps):
                orc.kv_insert(bits[:m], slot[:m].numpy(), fmt=1, s_cache=s_cache)
            dt = (time.perf_counter() - t0) / args.steps
            v = m * (576 * 2 + 8 + 512 + 16 + 128) / dt / 1e9
            print(json.dumps({"impl": "reference", "metric": "KV-cache insert GB/s (fp8)",
                              "value": round(v, 3), "unit": "GB/s", "n_gpus": world,
                              "steps": args.steps, "warmup": args.warmup,
                              "higher_is_better": True, "config": cfg,
                              "cpu_baseline": {"kind": "oracle", "cores": 1, "value": round(v, 3),
                                               "sample": "%d of %d tokens per step" % (m, n)},
                              "e2e": {"value": round(v, 3), "unit": "GB/s",
                                      "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                  flush=True)
        return
    from context_sparse_mla_gb300 import build as cbuild
    from context_sparse_mla_gb300 import cpmla
    cbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kv_d, slot_d = kv.to(dev), slot.to(dev)
    c8 = torch.zeros((s_cache, 512), dtype=torch.uint8, device=dev)
    cs = torch.zeros((s_cache, 4), dtype=torch.float32, device=dev)
    cr = torch.zeros((s_cache, 64), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        cpmla.mla_kv_cache_insert(kv_d, slot_d, cache_fp8=c8, cache_scale=cs, cache_rope=cr,
                                  stream=stream)

    with clock_sampler(local) as clk:
        for _ in range(args.warmup):
            flush(1.0)
            step()
        torch.cuda.synchronize()
        assert cpmla.device_status() == 0
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        t_clk0 = time.time()
        for i in range(args.steps):
            flush(float(i))
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        clk.window(t_clk0, time.time())
    ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps, world)
    # end to end: the rows and slots up from pinned memory, the cache rows down
    kv_h, slot_h = kv.pin_memory(), slot.pin_memory()
    c8_h = torch.empty_like(c8, device="cpu").pin_memory()
    cs_h = torch.empty_like(cs, device="cpu").pin_memory()
    cr_h = torch.empty_like(cr, device="cpu").pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        kv_d.copy_(kv_h, non_blocking=True)
        slot_d.copy_(slot_h, non_blocking=True)
        step()
        c8_h.copy_(c8, non_blocking=True)
        cs_h.copy_(cs, non_blocking=True)
        cr_h.copy_(cr, non_blocking=True)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.e2e_steps, world)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle's insertion of the first 16384 tokens (one host core),
        # checked byte for byte against the timed launch's cache rows
        from oracle import oracle as orc
        m = 16384
        bits = kv.view(torch.int16).numpy().view(np.uint16)
        t0 = time.perf_counter()
        want = orc.kv_insert(bits[:m], slot[:m].numpy(), fmt=1, s_cache=s_cache)
        dt = time.perf_counter() - t0
        rows = slot[:m].to(dev)
        assert np.array_equal(c8[rows].cpu().numpy(), want["kv_fp8"][slot[:m].numpy()])
        v = m * (576 * 2 + 8 + 512 + 16 + 128) / dt / 1e9
        cpu = {"kind": "oracle", "cores": 1, "value": round(v, 4), "unit": "GB/s",
               "sample": "the first %d of %d tokens (%.1f s)" % (m, n, dt)}
    pk = peaks()
    gbs = world * bytes_step / (ms * 1e-3) / 1e9
    out = {"metric": "KV-cache insert GB/s (fp8)", "value": round(gbs, 1), "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3",
           "data": "synthetic (seeded N(0,1) rows with per-token log-normal magnitude)",
           "config": cfg,
           "roofline": {"bound": "hbm", "achieved": round(gbs / world, 1), "peak": pk["hbm"],
                        "unit": "GB/s", "frac": round(gbs / world / pk["hbm"], 4),
                        # DRAM read + write of one launch of this workload (ncu)
                        "traffic": 152071168 + 52147968, "kernel": "kv_insert_kernel",
                        "peak_source": pk["source"] + " HBM copy"},
           "e2e": {"value": round(world * bytes_step / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                   "ms_per_step": round(e2e_ms, 3),
                   "h2d_bytes_per_step": n * (576 * 2 + 8),
                   "d2h_bytes_per_step": s_cache * (512 + 16 + 128)},
           "gpu_launches": args.steps, "clocks": clk.summary(),
           "device_status": cpmla.device_status(), "cpu_baseline": cpu}
    if rank == 0:
        print(json.dumps(out), flush=True)


TOPK_WORKLOADS = {"topk_s32k_k2048": 32768, "topk_s8k_k2048": 8192}


def run_topk(args, world, rank, local):
    """The indexer's top-k selection over one causal request: logits fp32
    [S, S] (row t holds the scores of query t against keys 0..t), k = 2048.
    Reports GB/s of algorithmic bytes (the causal logits of rows longer than
    k read once, the row lengths read, the index lists written) against the
    measured HBM copy bandwidth.  --impl reference times the oracle on rows."""
    S, k = TOPK_WORKLOADS[args.workload], 2048
    rl_h = torch.arange(1, S + 1, dtype=torch.int32)
    n = rl_h.to(torch.int64)
    bytes_step = int(4 * n[n > k].sum()) + 4 * S + 4 * S * k
    cfg = {"workload": args.workload, "rows": S, "k": k, "logits": "fp32 [S, S], causal rows",
           "l2": "flushed between steps (512 MiB write, then 512 MiB read); the logits read exceed L2",
           "parallelism": "replicas (one full workload per GPU)" if world > 1 else "single GPU"}
    metric = "indexer top-k selection GB/s"
    data = "synthetic (seeded N(0,1) fp32 logits standing in for indexer scores)"
    if args.impl == "reference":
        if rank == 0:
            from oracle import oracle as orc
            rows = np.arange(S - 64, S)  # the longest rows
            x = synth_logits(args.workload, rows, args.seed)
            vals = []
            for i in range(args.warmup + args.steps):
                t0 = time.perf_counter()
                orc.topk_select(x, rl_h[rows].numpy(), k)
                if i >= args.warmup:
                    vals.append(rows_bytes(rl_h[rows], k) / (time.perf_counter() - t0) / 1e9)
            v = statistics.median(vals)
            print(json.dumps({"impl": "reference", "metric": metric, "value": round(v, 4),
                              "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
                              "warmup": args.warmup, "higher_is_better": True, "config": cfg,
                              "cpu_baseline": {"kind": "oracle", "cores": 1, "value": round(v, 4),
                                               "sample": "the 64 longest rows per step"},
                              "e2e": {"value": round(v, 4), "unit": "GB/s",
                                      "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                  flush=True)
        return
    from context_sparse_mla_gb300 import build as cbuild
    from context_sparse_mla_gb300 import cpmla, synth
    cbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = synth.indexer_logits(S, S, seed=args.seed, device=dev)
    rl = rl_h.to(dev)
    out = torch.empty((S, k), dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        cpmla.mla_topk_select(x, rl, k, out=out, stream=stream)

    with clock_sampler(local) as clk:
        for _ in range(args.warmup):
            flush(1.0)
            step()
        torch.cuda.synchronize()
        assert cpmla.device_status() == 0
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        t_clk0 = time.time()
        for i in range(args.steps):
            flush(float(i))
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        clk.window(t_clk0, time.time())
    ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps, world)
    # last step's lists on a few rows against the oracle (outside the timing)
    check_rows = torch.tensor([k, S // 2, S - 1], device=dev)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import oracle as orc
        want = orc.topk_select(x[check_rows].cpu().numpy(), rl_h[check_rows.cpu()].numpy(), k)
        assert np.array_equal(out[check_rows].cpu().numpy(), want), "top-k check failed"
        rows = np.arange(S - 256, S)
        xs = x[torch.as_tensor(rows, device=dev)].cpu().numpy()
        t0 = time.perf_counter()
        orc.topk_select(xs, rl_h[rows].numpy(), k)
        dt = time.perf_counter() - t0
        v = rows_bytes(rl_h[rows], k) / dt / 1e9
        cpu = {"kind": "oracle", "cores": 1, "value": round(v, 4), "unit": "GB/s",
               "sample": "the 256 longest rows (%.1f s)" % dt}
    # end to end: the logits and row lengths up from pinned memory, the lists down
    x_h = torch.empty((S, S), dtype=torch.float32).pin_memory()
    x_h.copy_(x)
    rl_p = rl_h.pin_memory()
    out_h = torch.empty((S, k), dtype=torch.int32).pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        x.copy_(x_h, non_blocking=True)
        rl.copy_(rl_p, non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.e2e_steps, world)
    pk = peaks()
    gbs = world * bytes_step / (ms * 1e-3) / 1e9
    res = {"metric": metric, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": data, "config": cfg,
           "roofline": {"bound": "hbm", "achieved": round(gbs / world, 1), "peak": pk["hbm"],
                        "unit": "GB/s", "frac": round(gbs / world / pk["hbm"], 4),
                        "traffic": NCU_TRAFFIC_BYTES.get((args.workload, "topk")),
                        "kernel": "topk_select_kernel",
                        "peak_source": pk["source"] + " HBM copy"},
           "e2e": {"value": round(world * bytes_step / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                   "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": 4 * S * S + 4 * S,
                   "d2h_bytes_per_step": 4 * S * k},
           "gpu_launches": args.steps, "clocks": clk.summary(),
           "device_status": cpmla.device_status(), "cpu_baseline": cpu}
    if rank == 0:
        print(json.dumps(res), flush=True)


def rows_bytes(row_len, k):
    """Algorithmic bytes of the selection of these rows (as in run_topk)."""
    n = row_len.to(torch.int64)
    return int(4 * n[n > k].sum()) + 4 * len(n) + 4 * len(n) * k


def synth_logits(workload, rows, seed):
    """Rows of the workload's logits, drawn as the GPU arm draws them (on the
    GPU when there is one, else the same generator on the host)."""
    from context_sparse_mla_gb300 import synth
    S = TOPK_WORKLOADS[workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = synth.indexer_logits(S, S, seed=seed, device=dev)
    return x[torch.as_tensor(rows, device=dev)].cpu().numpy()


def workload_config(name, prob, world):
    return {"workload": name, "tokens": prob.T, "heads": prob.H, "pcp": prob.P,
            "topk": prob.topk, "kv_format": prob.kv_format,
            "l2": "flushed between steps (512 MiB write, then 512 MiB read)",
            "parallelism": ("replicas (one full workload per GPU)" if world > 1
                            else "single GPU, %d virtual PCP shards" % prob.P)}


def cpu_oracle_sample(prob, target_s=25.0, max_tokens=4096, seed=0, min_tokens=None):
    """Time the fp64 oracle on a bounded seeded sample of the workload's tokens
    (all heads each): max_tokens of them (all when the workload has fewer),
    fewer only when that would take far longer than target_s; returns
    (TFLOP/s, tokens/s, n_tokens, seconds, cores)."""
    from oracle import oracle as orc
    from tests import parity_util as pu
    orc.build()
    kvh = pu.kv_host(prob)
    pos_all = prob.token_pos().numpy()
    rng = np.random.default_rng(seed)

    def run(n):
        toks = np.sort(rng.choice(prob.T, size=min(n, prob.T), replace=False))
        keys = np.minimum(pos_all[toks].astype(np.int64) + 1, prob.topk) if prob.topk else \
            pos_all[toks].astype(np.int64) + 1
        t0 = time.perf_counter()
        pu.oracle_tokens(prob, toks, kvh=kvh)
        dt = time.perf_counter() - t0
        return len(toks), float(keys.sum()) * prob.H * FLOPS_PER_KEY_HEAD, dt

    want = min(max_tokens, prob.T) if min_tokens is None else min(min_tokens, prob.T)
    n0, f0, d0 = run(16)
    # the full sample unless the calibration says it would take over twice
    # the target (the 16-token run includes thread start-up, so it overestimates)
    n = want if 16 * 2 * target_s / max(d0, 1e-3) >= want else \
        int(max(16, 16 * 2 * target_s / max(d0, 1e-3)))
    n1, f1, d1 = run(n)
    cores = os.cpu_count()
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        pass
    omp = os.environ.get("OMP_NUM_THREADS")
    if omp:
        cores = min(cores, int(omp))
    return f1 / d1 / 1e12, n1 / d1, n1, d1, cores


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="varlen_p8_h64")
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    # end-to-end steps timed back to back: the pipeline's fill (the first
    # upload) and drain (the last download) are inside the timed region once,
    # so more steps come closer to the rate a caller streaming batches sees
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--path", default="merged", choices=["merged", "two-launch"],
                    help="merged: one launch, the single-partial merge with the sink in the "
                         "attention epilogue; two-launch: partial attention, then the merge kernel")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    world, rank, local = dist_setup(args.gpus)
    from context_sparse_mla_gb300 import synth
    if args.impl == "cuda" and torch.cuda.is_available():
        clock_sampler(local)  # nvidia-smi starts while the inputs are built

    if args.workload == KV_INSERT_WORKLOAD:
        run_kv_insert(args, world, rank, local)
        return
    if args.workload in TOPK_WORKLOADS:
        run_topk(args, world, rank, local)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    from context_sparse_mla_gb300 import build as cbuild
    from context_sparse_mla_gb300 import cpmla
    cbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    prob = synth.make_problem(args.workload, device=dev, seed=args.seed)
    flops = synth.attended_keys(prob) * prob.H * FLOPS_PER_KEY_HEAD
    tokens = prob.T
    merged = args.path == "merged"
    plan = cpmla.plan_for(prob, device=dev)          # two-launch (partials + merge kernel)
    plan_m = cpmla.plan_for(prob, device=dev, merged=True)
    kvk = cpmla.kv_kwargs(prob)
    o_out = torch.empty((prob.T, prob.H, 512), dtype=torch.bfloat16, device=dev)
    lse_out = torch.empty((prob.T, prob.H), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None, two_launch=not merged):
        if ev:
            ev[0].record(stream)
        if two_launch:
            plan.attention(prob.q, softmax_scale=prob.scale, idx=prob.idx, stream=stream, **kvk)
        else:
            plan_m(prob.q, softmax_scale=prob.scale, sink=prob.sink, idx=prob.idx, o_out=o_out,
                   lse_out=lse_out, stream=stream, **kvk)
        if ev:
            ev[1].record(stream)
        if two_launch:
            plan.merge(o_out, lse_out, sink=prob.sink, stream=stream)
        if ev:
            ev[2].record(stream)

    def timed(n, two_launch, clk=None):
        for _ in range(args.warmup):
            flush(1.0)
            step(two_launch=two_launch)
        torch.cuda.synchronize()
        assert cpmla.device_status() == 0
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        barrier(world)
        torch.cuda.synchronize()
        t_wall0 = time.perf_counter()
        t_clk0 = time.time()
        for i in range(n):
            flush(float(i))  # evict L2 between steps (outside the events)
            step(evs[i], two_launch=two_launch)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
        if clk is not None:
            clk.window(t_clk0, time.time())
        barrier(world)
        a = [e[0].elapsed_time(e[1]) for e in evs]
        m = [e[1].elapsed_time(e[2]) for e in evs]
        return sum(a) / n, sum(m) / n, t_wall

    # the two-launch path, for the partial-attention and merge kernels' own
    # figures (outside the reported step when the merged path is timed)
    tl_attn, tl_merge, _ = timed(min(args.steps, 20) if merged else 1, True)
    with clock_sampler(local) as clk:
        attn_avg, merge_avg, t_wall = timed(args.steps, not merged, clk)
    if not merged:
        tl_attn, tl_merge = attn_avg, merge_avg
    status = cpmla.device_status()
    step_ms = max_over_ranks(attn_avg + merge_avg, world)

    # the decode rows alone through split-KV (each row's keys in P parts, one
    # per shard that holds a replica), for their share of the step
    decode = None
    n_dec = int(prob.is_decode.sum())
    if n_dec:
        plan_d = cpmla.plan_for(prob, device=dev, merged=True, split_decode=True)
        o_d = torch.empty_like(o_out)
        l_d = torch.empty_like(lse_out)

        def dstep():
            plan_d.decode(prob.q, o_d, l_d, softmax_scale=prob.scale, sink=prob.sink,
                          idx=prob.idx, stream=stream, **kvk)
        for _ in range(args.warmup):
            flush(1.0)
            dstep()
        dev_ = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(10)]
        for i in range(10):
            flush(float(i))
            dev_[i][0].record(stream)
            dstep()
            dev_[i][1].record(stream)
        torch.cuda.synchronize()
        assert cpmla.device_status() == 0
        dec_ms = sum(e[0].elapsed_time(e[1]) for e in dev_) / 10
        # the same rows' result in the timed step, bit for bit up to the split
        dt = plan_d.dec["tokens"].long()
        assert (o_d[dt].float() - o_out[dt].float()).abs().max().item() < 0.05
        dec_keys = int(torch.clamp(prob.token_pos()[dt.cpu()].long() + 1,
                                   max=prob.topk if prob.topk else 1 << 62).sum())
        decode = {"tokens": n_dec, "n_split": prob.P, "ms": round(dec_ms, 4),
                  "share_of_step": round(dec_ms / step_ms, 5),
                  "tflops": round(dec_keys * prob.H * FLOPS_PER_KEY_HEAD / (dec_ms * 1e-3) / 1e12,
                                  2),
                  "how": "mla_attn_split_kv over the decode rows alone (3 launches), CUDA "
                         "events, L2 flushed; in the timed step the owner replica of each "
                         "decode row computes it once inside the merged launch"}

    # ---------------- end to end through the public API with host buffers:
    # every step partitions its batch on the host, copies its inputs and the
    # partition maps up from pinned host memory and its result back down.
    # Two buffer sets and three streams pipeline the steps: step i's inputs
    # go up while step i-1 computes and step i-2's result comes down.
    q_h = prob.q.cpu().pin_memory()
    kv_h = {k: v.cpu().pin_memory() for k, v in kvk.items()}
    sink_h = prob.sink.cpu().pin_memory()
    idx_h = prob.idx.cpu().pin_memory() if prob.idx is not None else None
    cu, qs, dec, kvs = (prob.cu_seqlens.numpy(), prob.q_start_pos.numpy(), prob.is_decode.numpy(),
                        prob.kv_start.numpy())
    kvs_h = torch.from_numpy(np.ascontiguousarray(kvs, np.int64)).pin_memory()
    maps = ("rows", "pos", "req", "owner_row")
    part0 = cpmla.pcp_dualchunk_partition(prob.P, cu, qs, dec)
    sets = []
    for _ in range(2):
        st = {"q": torch.empty_like(prob.q), "kv": {k: torch.empty_like(v) for k, v in kvk.items()},
              "sink": torch.empty_like(prob.sink),
              "idx": torch.empty_like(prob.idx) if prob.idx is not None else None,
              "kv_start": torch.empty(len(kvs), dtype=torch.int64, device=dev),
              "o": torch.empty((prob.T, prob.H, 512), dtype=torch.bfloat16, device=dev),
              "lse": torch.empty((prob.T, prob.H), dtype=torch.float32, device=dev),
              "o_h": torch.empty((prob.T, prob.H, 512), dtype=torch.bfloat16).pin_memory(),
              "lse_h": torch.empty((prob.T, prob.H), dtype=torch.float32).pin_memory(),
              "maps_h": {k: torch.empty(len(part0[k]), dtype=torch.int32).pin_memory()
                         for k in maps},
              "maps_d": {k: torch.empty(len(part0[k]), dtype=torch.int32, device=dev)
                         for k in maps},
              "ev_in": torch.cuda.Event(), "ev_cp": torch.cuda.Event(),
              "ev_out": torch.cuda.Event()}
        if not merged:
            st["o_part"] = torch.empty((plan.n_rows, prob.H, 512), dtype=torch.float32, device=dev)
            st["lse_part"] = torch.empty((plan.n_rows, prob.H), dtype=torch.float32, device=dev)
        sets.append(st)
    s_in, s_cp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    maps_bytes = sum(len(part0[k]) * 4 for k in maps) + kvs_h.numel() * 8
    h2d = q_h.numel() * 2 + sum(v.numel() * v.element_size() for v in kv_h.values()) + \
        sink_h.numel() * 4 + maps_bytes
    if idx_h is not None:
        h2d += idx_h.numel() * 4
    d2h = prob.T * prob.H * (512 * 2 + 4)

    def e2e_step(i):
        st = sets[i % 2]
        part = cpmla.pcp_dualchunk_partition(prob.P, cu, qs, dec)  # host
        st["ev_in"].synchronize()  # the set's last upload has read its pinned maps
        for k in maps:
            st["maps_h"][k].numpy()[:] = part[k]
        with torch.cuda.stream(s_in):
            s_in.wait_event(st["ev_cp"])  # step i-2 has finished reading the set's inputs
            st["q"].copy_(q_h, non_blocking=True)
            for k in kv_h:
                st["kv"][k].copy_(kv_h[k], non_blocking=True)
            st["sink"].copy_(sink_h, non_blocking=True)
            if idx_h is not None:
                st["idx"].copy_(idx_h, non_blocking=True)
            st["kv_start"].copy_(kvs_h, non_blocking=True)
            for k in maps:
                st["maps_d"][k].copy_(st["maps_h"][k], non_blocking=True)
            st["ev_in"].record(s_in)
        s_cp.wait_event(st["ev_in"])
        s_cp.wait_event(st["ev_out"])  # the set's previous result is down
        m = st["maps_d"]
        if merged:
            cpmla.mla_attn_merged(st["q"], st["kv_start"], m["rows"], m["pos"], m["req"],
                                  m["owner_row"], st["o"], st["lse"], softmax_scale=prob.scale,
                                  sink=st["sink"], topk_idx=st["idx"], stream=s_cp, **st["kv"])
        else:
            if prob.topk:
                cpmla.mla_partial_attn_sparse(st["q"], st["kv_start"], m["rows"], m["pos"],
                                              m["req"], st["idx"], st["o_part"], st["lse_part"],
                                              softmax_scale=prob.scale, stream=s_cp, **st["kv"])
            else:
                cpmla.mla_partial_attn_dense(st["q"], st["kv_start"], m["rows"], m["pos"],
                                             m["req"], st["o_part"], st["lse_part"],
                                             softmax_scale=prob.scale, stream=s_cp, **st["kv"])
            cpmla.lse_merge_with_sink(st["o_part"], st["lse_part"], m["owner_row"], st["o"],
                                      st["lse"], sink=st["sink"], stream=s_cp)
        st["ev_cp"].record(s_cp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(st["ev_cp"])
            st["o_h"].copy_(st["o"], non_blocking=True)
            st["lse_h"].copy_(st["lse"], non_blocking=True)
            st["ev_out"].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    assert cpmla.device_status() == 0
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world)
    # the result of the last step, checked against the timed path's output
    # (the first and last 128 tokens)
    last = sets[(args.e2e_steps - 1) % 2]
    for sl in (slice(0, 128), slice(max(0, prob.T - 128), prob.T)):
        assert torch.equal(last["o_h"][sl].view(torch.int16), o_out[sl].cpu().view(torch.int16))

    # ---------------- roofline (attention kernel) and merge bandwidth
    pk = peaks()
    attn_tflops = flops / (attn_avg * 1e-3) / 1e12
    n_part = plan.n_rows
    merge_bytes = n_part * prob.H * (512 * 4 + 4) + prob.T * prob.H * (512 * 2 + 4) + \
        prob.T * 4 + prob.H * 4
    merge_gbs = merge_bytes / (tl_merge * 1e-3) / 1e9

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tf, tps, n_tok, secs, cores = cpu_oracle_sample(prob)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": "%d of %d tokens of the workload (all %d heads each), seeded, %.1f s; "
                         "%.1f tokens/s" % (n_tok, prob.T, prob.H, secs, tps)}

    value = job_throughput(flops, step_ms, world) / 1e12
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/KV, N(0,1) sink; no dataset or weights)",
        "config": workload_config(args.workload, prob, world),
        "tokens_per_s": round(job_throughput(tokens, step_ms, world), 1),
        "path": args.path,
        "attn_ms": round(attn_avg, 4), "merge_ms": round(merge_avg, 4),
        "two_launch": {"attn_ms": round(tl_attn, 4), "merge_ms": round(tl_merge, 4),
                       "ms_per_step": round(tl_attn + tl_merge, 4)},
        "roofline": {"bound": "tensor", "achieved": round(attn_tflops, 2),
                     "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": round(attn_tflops / pk["bf16"], 4),
                     "traffic": NCU_TRAFFIC_BYTES.get((args.workload, args.path)),
                     "kernel": "mla_dense_kernel" if not prob.topk else "mla_sparse_wide_kernel",
                     "peak_source": pk["source"] + " burst bf16"},
        "merge_roofline": {"bound": "hbm", "achieved": round(merge_gbs, 1), "peak": pk["hbm"],
                           "unit": "GB/s", "frac": round(merge_gbs / pk["hbm"], 4),
                           "bytes": merge_bytes, "kernel": "lse_merge_kernel (two-launch path)"},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "per step: host partition, inputs + maps up from pinned memory, one "
                       "path call, O + LSE down; steps pipelined over two buffer sets and "
                       "three streams; %d steps timed back to back, the pipeline's fill "
                       "and drain included" % args.e2e_steps},
        "decode_rows": decode,
        "gpu_launches": (1 if merged else 2) * args.steps,
        "clocks": clk.summary(),
        "device_status": status,
        "wall_s_timed": round(t_wall, 3),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args, world, rank):
    """The oracle as it stands on the host cores, on a bounded sample per step."""
    from context_sparse_mla_gb300 import synth
    if rank != 0:
        return
    prob = synth.make_problem(args.workload, device="cpu", seed=args.seed) \
        if args.workload in ("dense_s256_h4_p2", "dense_s8192_h16_p2") else \
        synth.make_problem(args.workload, device="cuda", seed=args.seed)
    per_step = []
    total_tf = []
    n_tok = 0
    for i in range(args.warmup + args.steps):
        tf, tps, n_tok, secs, cores = cpu_oracle_sample(prob, target_s=1.0, max_tokens=512,
                                                        seed=i)
        if i >= args.warmup:
            per_step.append(secs)
            total_tf.append(tf)
    value = statistics.median(total_tf)
    out = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * statistics.median(per_step), 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_config(args.workload, prob, 1), "impl": "reference",
           "cpu_baseline": {"kind": "oracle", "cores": cores, "value": round(value, 6),
                            "unit": "TFLOP/s",
                            "sample": "%d tokens per step (all heads), seeded" % n_tok},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
