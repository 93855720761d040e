#!/usr/bin/env python
"""Decode-step throughput of the GB300 HiSparse hot path; prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ctx128k] [--impl reference]

A step is one pass of the whole hot path over one decode batch: append the new
rows, then per indexer group indexer scoring + top-K, the fused resolver (with
its host-row copies) and sparse MLA for every layer of the group, then the
one-launch page materialisation when pages complete. The default workload is a
single request at 128K context (64 heads, 4 sparse-MLA layers sharing one
indexer, top-K 2,048, 75 % of pages host-only, hot buffer 4,096 rows).

value: query tokens/s with every step's inputs already in HBM; each step is
timed with CUDA events and L2 is flushed (a 256 MB write) between timed steps.
e2e: the same metric when every step copies its inputs from pinned host memory
and its attention outputs back, inside the timed region.
Under torchrun each rank runs its own independent request (weak scaling) and
rank 0 reports the sum of tokens over the maximum time across ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "HiSparse decode tokens/s (1 GB300) + achieved HBM/host-link GB/s vs roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="ctx128k")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="bound on the oracle's CPU sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-call-timing", action="store_true", help="skip the single-call graph timings")
    ap.add_argument("--extra", default=",".join(EXTRA_WORKLOADS),
                    help="workloads timed after the headline one on a single GPU, reported under 'workloads' "
                         "(empty: none)")
    ap.add_argument("--extra-steps", type=int, default=20, help="timed steps of each extra workload")
    return ap.parse_args()


def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl"
        try:
            import torch
            if not torch.cuda.is_available():
                backend = "gloo"
        except Exception:
            backend = "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def workload_config(name, steps_total, rank):
    from sparse_mla_kv_indexer_gb300 import workload as W
    cfg = W.named_config(name)
    return dataclasses.replace(cfg, steps=max(cfg.steps, steps_total), seed=cfg.seed + rank)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class NvmlSampler:
    """SM clock, its maximum, power and throttle reasons of this process's GPU, read
    through NVML (read-only queries) every few milliseconds on a background thread,
    so that a timed region of tens of milliseconds gets samples."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_slowdown"}

    def __init__(self, cuda_device, period_s=0.005):
        import ctypes
        import threading
        self.samples = []
        self.ok = False
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            rt = None
            for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
                try:
                    rt = ctypes.CDLL(name)
                    break
                except OSError:
                    continue
            bus = ctypes.create_string_buffer(32)
            if rt is None or rt.cudaDeviceGetPCIBusId(bus, 32, ctypes.c_int(cuda_device)) != 0:
                return
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.value, ctypes.byref(h)) != 0:
                return
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self._nv, self._h, self._reasons_fn, self._ct = nv, h, reasons_fn, ctypes
        except Exception:
            return
        self.ok = True
        self._stop = threading.Event()
        self._period = period_s
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def _read(self):
        ct, nv, h = self._ct, self._nv, self._h
        sm, mx, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(sm)) != 0:      # NVML_CLOCK_SM
            return None
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ct.byref(mx))
        nv.nvmlDeviceGetPowerUsage(h, ct.byref(mw))
        self._reasons_fn(h, ct.byref(rs))
        return sm.value, mx.value, mw.value / 1000.0, rs.value

    def _run(self):
        while not self._stop.is_set():
            r = self._read()
            if r:
                self.samples.append(r)
            self._stop.wait(self._period)

    def stop(self):
        if not self.ok:
            return None
        self._stop.set()
        self._t.join(timeout=2)
        if not self.samples:
            return None
        reasons = sorted({name for s in self.samples for bit, name in self.REASONS.items() if s[3] & bit})
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples), "reasons": reasons,
                "power_w": statistics.median(s[2] for s in self.samples),
                "samples": len(self.samples), "source": "nvml"}


class ClockSampler:
    """nvidia-smi clocks line during the timed region; NVML samples (same source,
    every 5 ms) are reported when available, since a short region may see no
    nvidia-smi sample at its 200 ms period."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.gpu = gpu_index
        self.proc = None
        self.nvml = NvmlSampler(gpu_index)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        fast = self.nvml.stop()
        smi = self._stop_smi()
        if fast:
            if smi:
                fast["nvidia_smi_samples"] = smi["samples"]
            return fast
        return smi

    def _stop_smi(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "source": "nvidia-smi"}


# ---------------------------------------------------------------------------
# algorithmic bytes of each hot-path call
# ---------------------------------------------------------------------------
def algorithmic_bytes(cfg, plans, counters_misses_rows):
    """Bytes each call must move at minimum, per call, averaged over the given steps.

    indexer_topk: 128 B per scored key (132 B with FP8 keys: 128 values and a
    scale, vLLM blog Part 2 footnote 3), keys read once per request (shared by its
    query tokens); sparse_mla_decode: per query token 2,048 rows x 660 B plus
    2,176 B of bf16 query and output per head (vLLM blog Part 2, footnote 1);
    resolve_topk: misses x 656 B x layers over the host link; offload_pages:
    64 x 656 B x layers per page over the host link."""
    keys = 0
    for p in plans:
        per_req = {}
        for t in p.tokens:
            per_req[t.req] = max(per_req.get(t.req, 0), t.limit)
        keys += sum(per_req.values())
    keys /= len(plans)
    n_tok = sum(len(p.tokens) for p in plans) / len(plans)
    n_app = n_tok + sum(hi - lo for p in plans for (_, lo, hi) in p.tick.prefill) / len(plans)
    idx = keys * (132 if cfg.idx_fp8 else 128)
    attn = n_tok * (cfg.topk * 660 + cfg.n_heads * 2176)
    offl = sum(len(p.offload) for p in plans) / len(plans) * 64 * 656 * cfg.n_layers
    append = n_app * (cfg.n_layers * 656 + cfg.n_groups * 128) * 2
    return {"indexer_topk": idx, "sparse_mla_decode": attn, "offload_pages": offl, "append": append,
            "resolve_topk": counters_misses_rows * 656 + n_tok * cfg.topk * 8}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Dense bf16 tensor peak: the measured burst figure, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def host_link_probe(torch, H, reps=10):
    """Host-link rates on this machine: single 656-byte rows read from pinned, mapped host
    memory by hs_link_probe (the miss-copy pattern, 16,384 random rows of a 256 MB
    host buffer), and bulk pinned copies H2D / D2H of 64 MB (cudaMemcpyAsync through
    torch). Each the best of `reps` timed repetitions with CUDA events."""
    rows_total = (256 << 20) // 656
    host = torch.empty(rows_total * 656, dtype=torch.uint8, pin_memory=True)
    host.fill_(1)
    n = 16384
    g = torch.Generator().manual_seed(0)
    src = torch.randint(0, rows_total, (n,), generator=g, dtype=torch.int64).cuda()
    dst = torch.empty(n * 656, dtype=torch.uint8, device="cuda")
    bulk_h = torch.empty(64 << 20, dtype=torch.uint8, pin_memory=True)
    bulk_d = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")

    def best(fn, nbytes):
        fn()
        torch.cuda.synchronize()
        t = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            t.append(a.elapsed_time(b) / 1000.0)
        return nbytes / min(t) / 1e9

    single = best(lambda: H.link_probe(host, 656, src, dst), n * 656)
    h2d = best(lambda: bulk_d.copy_(bulk_h, non_blocking=True), bulk_h.numel())
    d2h = best(lambda: bulk_h.copy_(bulk_d, non_blocking=True), bulk_h.numel())
    return {"single_row_gbs": single, "h2d_gbs": h2d, "d2h_gbs": d2h,
            "how": "hs_link_probe: 16,384 random 656-byte rows from a 256 MB pinned mapped buffer; "
                   "bulk: 64 MB pinned copies; best of 10, CUDA events"}


def sources_sha256(files):
    """sha256 over the call's kernel sources and the shared device header, in order."""
    h = hashlib.sha256()
    for f in list(files) + ["hs_internal.cuh"]:
        h.update(open(os.path.join(ROOT, "sparse_mla_kv_indexer_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def ncu_traffic(name, workload):
    """DRAM bytes (read + write) per call of `name` on `workload`: the sum over the call's
    kernels of one single-kernel ncu capture each, committed with the sha256 of the kernel
    sources it was taken on; None when there is no capture or a source has changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d[name + "@" + workload]
        if ent.get("source_sha256") != sources_sha256(ent["sources"]):
            return None
        return ent.get("bytes_per_launch")
    except Exception:
        return None


# ---------------------------------------------------------------------------
# CUDA graphs
# ---------------------------------------------------------------------------
def capture(torch, fn):
    """Capture the hot-path calls issued by fn into a CUDA graph (nothing executes)."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    return g


def time_calls(torch, sess, i, flush, stream, reps=20):
    """Average device time of each hot-path call of step i, each captured alone in a
    graph and replayed `reps` times after an L2 flush. Replaying a call whose inputs
    are unchanged recomputes the same result (the resolver then finds every
    selected token resident or hot)."""
    cfg = sess.run.cfg
    plan, host, d = sess.steps[i]
    pool = sess.run.pool
    g0, l0 = 0, cfg.group_layers(0)[0]
    n = sess.tokens(i)
    ch = sess.run.append_chunk()
    topk, rows, o_l0 = sess.topk[g0][:n], sess.row_ids[g0][:n], sess.out[l0][:n]
    fns = {
        "append": lambda: pool.append_rows(d["app_req"][:ch], d["app_pos"][:ch], d["kv_rows"][:ch], d["idx_keys"][:ch]),
        "indexer_topk": lambda: sess.run.indexer_topk(g0, d["req"], d["limit"], d["q_idx"][g0], d["w_idx"][g0],
                                                      topk),
        "resolve_topk": lambda: pool.resolve_topk(g0, plan.step, d["req"], topk, rows),
        "sparse_mla_decode": lambda: pool.sparse_mla_decode(l0, d["q_attn"][l0], rows,
                                                            sess.run.wl.sm_scale(), o_l0),
    }
    if len(plan.offload):
        fns["offload_pages"] = lambda: pool.offload_pages(d["off_pool"], d["off_host"])
    per_step = {"append": 1, "indexer_topk": cfg.n_groups, "resolve_topk": cfg.n_groups,
                "sparse_mla_decode": cfg.n_layers, "offload_pages": 1}
    out = {}
    for name, fn in fns.items():
        g = capture(torch, fn)
        ev = []
        for r in range(reps):
            flush.fill_(r & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            ev.append((a, b))
        torch.cuda.synchronize()
        out[name] = {"ms": statistics.mean(a.elapsed_time(b) for a, b in ev), "per_step": per_step[name]}
        del g
    return out


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------
class OracleArm:
    """The CPU oracle run over consecutive decode steps of a workload (set up once)."""

    def __init__(self, name, steps, rank=0):
        from oracle.engine import OracleRun
        from sparse_mla_kv_indexer_gb300 import schedule as S
        from sparse_mla_kv_indexer_gb300 import workload as W
        self.cfg = workload_config(name, steps, rank)
        self.sch = S.Schedule(self.cfg)
        self.run = OracleRun(W.Workload(self.cfg), self.sch.setup)
        self.next = 0
        self.cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))

    def step(self):
        """One decode step; returns (query tokens, seconds)."""
        p = self.sch.plan(self.next)
        self.next += 1
        t0 = time.perf_counter()
        self.run.step(p)
        return len(p.tokens), time.perf_counter() - t0


def oracle_sample(name, seconds, rank=0):
    """The oracle over consecutive steps until `seconds` of CPU work (at least one
    step). Returns (tokens/s, sample description, cores)."""
    arm = OracleArm(name, 64, rank)
    toks = 0
    dt = 0.0
    while arm.next < arm.cfg.steps:
        n, t = arm.step()
        toks += n
        dt += t
        if dt >= seconds:
            break
    return toks / dt, f"{arm.next} consecutive decode steps of {name} ({toks} query tokens, {dt:.1f} s)", arm.cores


def config_line(workload, cfg):
    """The `config` object of a bench line (the same for both arms)."""
    return {"workload": workload, "requests_per_gpu": cfg.n_requests, "context": list(cfg.ctx_len)[:4],
            "heads": cfg.n_heads, "topk": cfg.topk, "sparse_layers": cfg.n_layers, "indexer_layers": cfg.n_groups,
            "query_tokens_per_request": cfg.t_q, "l2": "flushed between timed steps (256 MB write)"}


def reference_arm(args, rank, world):
    if rank != 0:
        return 0
    arm = OracleArm(args.workload, args.warmup + args.steps, rank)
    times, toks = [], 0
    for i in range(args.warmup + args.steps):
        n, t = arm.step()
        if i >= args.warmup:
            times.append(t)
            toks += n
    value = toks / sum(times) if times else 0.0
    sample = f"each step is one full decode step of {args.workload} ({toks // max(1, len(times))} query tokens)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * sum(times) / max(1, len(times)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_line(args.workload, arm.cfg),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": arm.cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def measure(args, name, K, Wm, rank, world, local, cpu_baseline):
    """Time `name` on this GPU: K graph-replayed steps after Wm warm-up steps,
    device-resident and end to end; returns the JSON object of the bench line."""
    import torch
    from sparse_mla_kv_indexer_gb300 import schedule as S
    from sparse_mla_kv_indexer_gb300 import workload as W
    from sparse_mla_kv_indexer_gb300.driver import BenchSession, GpuRun

    total = 2 * (Wm + K)
    cfg = workload_config(name, total, rank)
    wl = W.Workload(cfg)
    sch = S.Schedule(cfg)
    plans, occupancy = [], []
    for s in range(total):
        plans.append(sch.plan(s))
        hot = sum(len(v) for v in sch.hot_of.values())
        occupancy.append((int((sch.bt >= 0).sum()), hot, len(sch.free)))
    run = GpuRun(wl, sch.setup)
    dev_sess = BenchSession(run, plans[:Wm + K], mode="device")
    host_sess = BenchSession(run, plans[Wm + K:], mode="host")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    # ---- device-resident timing: one captured CUDA graph per step ----
    for i in range(Wm):
        dev_sess.tick(i)
        dev_sess.step(i)
    run.pool.raise_on_device_error()
    torch.cuda.synchronize()
    graphs = {i: capture(torch, lambda i=i: dev_sess.step(i)) for i in range(Wm, Wm + K)}
    run.pool.counters(reset=True)
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(local) if rank == 0 else None
    step_ev = []
    launches = 0
    t_wall0 = time.perf_counter()
    for i in range(Wm, Wm + K):
        dev_sess.tick(i)
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graphs[i].replay()
        b.record(stream)
        step_ev.append((a, b))
        launches += dev_sess.launches(i)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall0
    clk = clocks.stop() if clocks else None
    barrier(world)
    run.pool.raise_on_device_error()
    counters = run.pool.counters(reset=True)
    del graphs
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    t_total = sum(step_ms) / 1000.0
    t_max = max_over_ranks(t_total, world)
    tokens = sum(dev_sess.tokens(i) for i in range(Wm, Wm + K))
    tokens_all = sum_over_ranks(tokens, world)
    value = tokens_all / t_max

    # ---- each hot-path call alone, replayed from a single-call graph (L2 flushed) ----
    calls = {} if args.no_call_timing else time_calls(torch, dev_sess, Wm + K - 1, flush, stream, reps=20)

    # ---- end-to-end through host buffers: copies in, step, copy out, one graph per step ----
    for i in range(Wm):
        host_sess.tick(i)
        host_sess.step(i)
    torch.cuda.synchronize()
    hgraphs = {i: capture(torch, lambda i=i: host_sess.step(i)) for i in range(Wm, Wm + K)}
    barrier(world)
    e2e_ev = []
    for i in range(Wm, Wm + K):
        host_sess.tick(i)
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        hgraphs[i].replay()
        b.record(stream)
        e2e_ev.append((a, b))
    torch.cuda.synchronize()
    run.pool.raise_on_device_error()
    del hgraphs
    e2e_t = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev) / 1000.0, world)
    e2e_value = sum_over_ranks(sum(host_sess.tokens(i) for i in range(Wm, Wm + K)), world) / e2e_t

    if rank != 0:
        run.close()
        return None

    # ---- roofline of the dominant call ----
    timed_plans = plans[Wm:Wm + K]
    miss_rows = counters.h2d_bytes / 656.0 / K
    alg = algorithmic_bytes(cfg, timed_plans, miss_rows)
    share = {k: v["ms"] * v["per_step"] for k, v in calls.items()} or {"sparse_mla_decode": 0.0}
    dom = max(share, key=share.get)
    avg_ms = calls[dom]["ms"] if calls else 0.0
    peak, peak_kind = measured_peaks()
    # the single-call graph times step Wm + K - 1: its own algorithmic bytes
    dom_bytes = algorithmic_bytes(cfg, [plans[Wm + K - 1]], miss_rows).get(dom, 0.0) if calls else alg.get(dom, 0.0)
    achieved = dom_bytes / (avg_ms / 1000.0) / 1e9 if avg_ms > 0 else 0.0
    tkey = dom + "_fp8" if dom == "indexer_topk" and cfg.idx_fp8 else dom   # key of the committed traffic
    step_bytes = alg["indexer_topk"] * cfg.n_groups + alg["sparse_mla_decode"] * cfg.n_layers
    # step roofline: HBM bytes at the measured copy rate plus miss bytes at the measured
    # single-row host-link rate, or the tensor term (attention 2,176 FLOP per row per head,
    # vLLM blog Part 2 footnote 1; indexer 2 x 128 x H_i per key per query token, run as
    # fp16/fp8 MMAs) when larger
    from sparse_mla_kv_indexer_gb300 import hisparse as HS
    link = host_link_probe(torch, HS)
    miss_bytes = counters.h2d_bytes / K
    n_tok = sum(len(p.tokens) for p in timed_plans) / len(timed_plans)
    keys_scored = alg["indexer_topk"] / (132 if cfg.idx_fp8 else 128)
    flops = (n_tok * cfg.n_layers * cfg.topk * cfg.n_heads * 2176.0 +
             keys_scored * cfg.n_groups * cfg.t_q * 2.0 * 128 * cfg.n_idx_heads)
    tflops, tflops_kind = measured_bf16_tflops()
    t_mem = step_bytes / (peak * 1e9) + miss_bytes / (link["single_row_gbs"] * 1e9)
    t_tensor = flops / (tflops * 1e12)
    roof_step_s = max(t_mem, t_tensor)

    cpu = None
    if cpu_baseline and world == 1:
        v, sample, cores = oracle_sample(name, args.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}
    occ = occupancy[Wm:Wm + K]
    ended = sum(len(p.tick.releases) for p in plans[:Wm + K])
    turn_inputs = sum(len(p.tick.prefill) for p in timed_plans)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": 1000.0 * t_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8->int64 (indexer, exact), fp8-e4m3/bf16->fp32 (attention)",
        "data": "synthetic",
        "config": config_line(name, cfg),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "traffic": ncu_traffic(tkey, name)},
        "step_roofline": {"algorithmic_hbm_bytes": step_bytes, "miss_bytes": miss_bytes,
                          "host_link_gbs": link["single_row_gbs"], "tensor_flops": flops,
                          "tensor_peak_tflops": tflops, "tensor_peak_source": tflops_kind,
                          "bound": "hbm+link" if t_mem >= t_tensor else "tensor",
                          "roofline_ms": roof_step_s * 1e3, "frac": roof_step_s / (t_max / K)},
        "host_link": link,
        "breakdown_ms_per_call": {k: v["ms"] for k, v in calls.items()},
        "calls_per_step": {k: v["per_step"] for k, v in calls.items()},
        "timing": "each timed step is one CUDA graph replay; per-call times from single-call graphs",
        "resolver": {"hits": counters.hits / K, "misses": counters.misses / K, "resident": counters.resident / K,
                     "h2d_bytes_per_step": counters.h2d_bytes / K, "d2h_bytes_per_step": counters.d2h_bytes / K,
                     # the miss bytes of a step at the probe's single-row rate, against the
                     # resolver's whole call time (classification included)
                     "miss_link_us_per_step": miss_bytes / (link["single_row_gbs"] * 1e9) * 1e6,
                     "resolve_us_per_step": (calls["resolve_topk"]["ms"] * calls["resolve_topk"]["per_step"] * 1e3
                                             if "resolve_topk" in calls else None)},
        "pool_pages": {"total": run.setup.num_pages,
                       "block_table_mean": statistics.mean(o[0] for o in occ),
                       "hot_mean": statistics.mean(o[1] for o in occ),
                       "free_min": min(o[2] for o in occ),
                       "requests_ended_by_last_timed_step": ended, "turn_inputs_written_in_timed_steps": turn_inputs},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": statistics.mean(host_sess.h2d_bytes),
                "d2h_bytes_per_step": host_sess.d2h_bytes},
        "gpu_launches": launches,
        "wall_s_timed_loop": wall,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    run.close()
    del run, dev_sess, host_sess, flush
    torch.cuda.empty_cache()
    return line


# workloads timed beside the headline in a default single-GPU run (the second target
# workload of the method, 1M context, and the two batched shapes), each with fewer steps
EXTRA_WORKLOADS = ("ctx1m", "batch32", "multiturn")
EXTRA_KEYS = ("value", "ms_per_step", "steps", "warmup", "roofline", "step_roofline", "resolver", "pool_pages",
              "e2e", "gpu_launches", "clocks", "config", "breakdown_ms_per_call", "calls_per_step")


def main():
    args = parse_args()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        rc = reference_arm(args, rank, world)
        barrier(world)
        return rc
    import torch
    from sparse_mla_kv_indexer_gb300 import build as B
    if rank == 0 or not os.path.exists(B.LIB):
        B.build()
    barrier(world)
    torch.cuda.set_device(local)
    K, Wm = args.steps, max(3, args.warmup)
    line = measure(args, args.workload, K, Wm, rank, world, local, not args.no_cpu_baseline)
    extras = [w for w in (args.extra.split(",") if args.extra else []) if w and w != args.workload]
    if world == 1 and extras:
        line["workloads"] = {}
        for w in extras:
            sub = measure(args, w, min(K, args.extra_steps), Wm, rank, world, local, False)
            line["workloads"][w] = {k: sub[k] for k in EXTRA_KEYS}
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(world)
    return 0


if __name__ == "__main__":
    sys.exit(main())
