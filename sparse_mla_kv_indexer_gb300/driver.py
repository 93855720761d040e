"""Synthetic decode-step driver over the C ABI.

Stands in for the serving engine around the hot path: it owns the caller-side
buffers (KV pool tensors, index caches, pinned host pool), fills them from a
seeded workload, applies the host residency schedule between steps and issues
the hot-path calls of each step:

    append -> per indexer group: indexer_topk -> resolve_topk -> sparse_mla_decode per layer
           -> offload_pages (all layers, one launch)

Every computation runs in libhisparse.so; this module only moves inputs to the
device and results back.
"""
from __future__ import annotations

from typing import Dict, List

import numpy as np

from . import hisparse as H
from .schedule import Setup, StepPlan
from .workload import IDX_DIM, PAGE, ROW_BYTES, Workload

PLAN_FIELDS = 4


def pool_config(wl: Workload, setup: Setup) -> H.PoolConfig:
    cfg = wl.cfg
    max_ctx = -(-setup.n_pages_max * PAGE // 128) * 128
    return H.PoolConfig(
        page_size=PAGE, row_bytes=ROW_BYTES, idx_dim=IDX_DIM, n_idx_heads=cfg.n_idx_heads,
        n_heads=cfg.n_heads, topk=cfg.topk, n_layers=cfg.n_layers,
        layers_per_indexer=cfg.layers_per_indexer, num_pages=setup.num_pages,
        num_idx_pages=setup.num_idx_pages, max_requests=cfg.n_requests, max_ctx=max_ctx,
        max_q_per_req=cfg.t_q, hot_rows=cfg.hot_rows, max_tokens=cfg.n_requests * cfg.t_q,
        idx_format=H.IDX_FP8 if cfg.idx_fp8 else H.IDX_INT8, host_pages=setup.host_pages)


class GpuRun:
    def __init__(self, wl: Workload, setup: Setup, keep_scores: bool = False, device: str = "cuda"):
        import torch
        self.torch = torch
        self.wl = wl
        self.cfg = cfg = wl.cfg
        self.setup = setup
        self.keep_scores = keep_scores
        self.dev = torch.device(device)
        self.pc = pool_config(wl, setup)
        self.max_ctx = self.pc.max_ctx
        R, L, G = cfg.n_requests, cfg.n_layers, cfg.n_groups
        npg, nip = setup.num_pages, setup.num_idx_pages
        # host-side staging of the initial contents
        pool_np = [np.zeros((npg * PAGE, ROW_BYTES), np.uint8) for _ in range(L)]
        fp8 = cfg.idx_fp8
        # key caches: int8 pages [64][128], or FP8 pages [64][128] e4m3 then [64] fp32 scales
        idx_np = [np.zeros((nip, H.IDX_FP8_PAGE_BYTES), np.uint8) if fp8 else np.zeros((nip * PAGE, IDX_DIM), np.int8)
                  for _ in range(G)]
        self.host = torch.zeros(setup.host_pages * L * PAGE * ROW_BYTES, dtype=torch.uint8, pin_memory=True)
        host_np = self.host.numpy().reshape(setup.host_pages, L, PAGE, ROW_BYTES)
        for r in range(R):
            P = setup.prefix_len[r]
            for l in range(L):
                rows = wl.kv_rows(r, l)
                for p in range(-(-P // PAGE)):
                    lo, hi = p * PAGE, min(P, (p + 1) * PAGE)
                    if setup.block_table[r, p] >= 0:
                        b = int(setup.block_table[r, p]) * PAGE
                        pool_np[l][b:b + hi - lo] = rows[lo:hi]
                    if setup.materialised[r, p]:
                        host_np[setup.host_page[r, p], l, :hi - lo] = rows[lo:hi]
            for g in range(G):
                if fp8:
                    codes, scale = wl.idx_keys_fp8(r, g)
                for p in range(-(-P // PAGE)):
                    lo, hi = p * PAGE, min(P, (p + 1) * PAGE)
                    ip = int(setup.idx_page[r, p])
                    if fp8:
                        page = idx_np[g][ip]
                        page[:(hi - lo) * IDX_DIM] = codes[lo:hi].reshape(-1)
                        page[PAGE * IDX_DIM:PAGE * IDX_DIM + 4 * (hi - lo)] = scale[lo:hi].astype("<f4").view(np.uint8)
                    else:
                        idx_np[g][ip * PAGE:ip * PAGE + hi - lo] = wl.idx_keys(r, g)[lo:hi]
        self.kv = [torch.from_numpy(a.reshape(-1)).to(self.dev) for a in pool_np]
        self.idx = [torch.from_numpy(a.reshape(-1)).to(self.dev) for a in idx_np]
        del pool_np, idx_np
        self.pool = H.Pool(self.pc, self.kv, self.idx, self.host)
        for r in range(R):
            self.pool.set_pages(r, 0, block_table=setup.block_table[r].tolist(),
                                idx_pages=setup.idx_page[r].tolist(), host_pages=setup.host_page[r].tolist())
        for (r, g, pages) in setup.leases:
            self.pool.hot_lease(r, g, pages)
        torch.cuda.synchronize()

    # ------------------------------------------------------------------
    def apply_tick(self, tick) -> None:
        for (r, p, pg) in tick.bt_set:
            self.pool.set_pages(r, p, block_table=[pg])
        for r in tick.releases:
            self.pool.hot_release(r)
        for (r, g, pages) in tick.leases:
            self.pool.hot_lease(r, g, pages)

    def step_inputs(self, plan: StepPlan) -> Dict[str, np.ndarray]:
        """Host arrays of one step, in batch order (tokens grouped by request)."""
        cfg, wl, s = self.cfg, self.wl, plan.step
        toks = plan.tokens
        t_q = cfg.t_q
        out = {
            "req": np.array([t.req for t in toks], np.int32),
            "pos": np.array([t.pos for t in toks], np.int32),
            "limit": np.array([t.limit for t in toks], np.int32),
            "kv_rows": np.stack([np.stack([wl.kv_rows(t.req, l)[t.pos] for l in range(cfg.n_layers)]) for t in toks]),
            "idx_keys": np.stack([np.stack([self._key_record(t.req, g, t.pos) for g in range(cfg.n_groups)])
                                  for t in toks]),
            "q_idx": np.stack([np.stack([self._idx_query(t.req, g, s)[0][i % t_q] for i, t in enumerate(toks)])
                               for g in range(cfg.n_groups)]),
            "w_idx": np.stack([np.stack([self._idx_query(t.req, g, s)[1][i % t_q] for i, t in enumerate(toks)])
                               for g in range(cfg.n_groups)]),
            "q_attn": np.stack([np.stack([wl.attn_queries(t.req, l, s)[i % t_q] for i, t in enumerate(toks)])
                                for l in range(cfg.n_layers)]),
            "off_pool": np.array([o[2] for o in plan.offload], np.int32),
            "off_host": np.array([o[3] for o in plan.offload], np.int64),
        }
        return out

    def _key_record(self, r: int, g: int, pos: int) -> np.ndarray:
        """The key written for a new position: 128 int8, or the 132-byte FP8 record."""
        return self.wl.idx_key_records_fp8(r, g)[pos] if self.cfg.idx_fp8 else self.wl.idx_keys(r, g)[pos]

    def _idx_query(self, r: int, g: int, step: int):
        """(index queries [t_q, H_i, 128], head weights [t_q, H_i]) in the pool's key format."""
        if self.cfg.idx_fp8:
            return self.wl.idx_queries_fp8(r, g, step)
        w = self.wl.idx_weights(r, g)
        return self.wl.idx_queries(r, g, step), np.broadcast_to(w, (self.cfg.t_q, w.shape[0]))

    def indexer_topk(self, g, req, limit, q, w, topk, scores=None) -> None:
        """The pool's indexer call for its key format."""
        if self.cfg.idx_fp8:
            self.pool.indexer_topk_fp8(g, req, limit, q, w, topk, scores)
        else:
            self.pool.indexer_topk(g, req, limit, q, w, topk, scores)

    def step(self, plan: StepPlan, collect: bool = True) -> Dict[str, object]:
        torch = self.torch
        cfg, dev = self.cfg, self.dev
        self.apply_tick(plan.tick)
        x = self.step_inputs(plan)
        n = len(plan.tokens)
        K = cfg.topk
        req = torch.from_numpy(x["req"]).to(dev)
        pos = torch.from_numpy(x["pos"]).to(dev)
        limit = torch.from_numpy(x["limit"]).to(dev)
        self.pool.append_rows(req, pos, torch.from_numpy(x["kv_rows"]).to(dev),
                              torch.from_numpy(x["idx_keys"]).to(dev))
        res = {"topk": [], "row_ids": [], "plan": [], "scores": [], "o": [None] * cfg.n_layers,
               "lse": [None] * cfg.n_layers}
        for g in range(cfg.n_groups):
            q = torch.from_numpy(np.ascontiguousarray(x["q_idx"][g])).to(dev)
            w = torch.from_numpy(np.ascontiguousarray(x["w_idx"][g])).to(dev)
            topk = torch.empty((n, K), dtype=torch.int32, device=dev)
            sdt = torch.float32 if cfg.idx_fp8 else torch.int64
            scores = torch.empty((n, self.max_ctx), dtype=sdt, device=dev) if self.keep_scores else None
            self.indexer_topk(g, req, limit, q, w, topk, scores)
            row_ids = torch.empty((n, K), dtype=torch.int32, device=dev)
            plan_t = torch.empty((n, K, PLAN_FIELDS), dtype=torch.int32, device=dev)
            self.pool.resolve_topk(g, plan.step, req, topk, row_ids, plan_t)
            for l in cfg.group_layers(g):
                qa = torch.from_numpy(np.ascontiguousarray(x["q_attn"][l]).view(np.int16)).to(dev)
                o = torch.empty((n, cfg.n_heads, 512), dtype=torch.int16, device=dev)
                lse = torch.empty((n, cfg.n_heads), dtype=torch.float32, device=dev)
                self.pool.sparse_mla_decode(l, qa, row_ids, self.wl.sm_scale(), o, lse)
                if collect:
                    res["o"][l] = o.view(torch.bfloat16).float().cpu().numpy()
                    res["lse"][l] = lse.cpu().numpy()
            if collect:
                res["topk"].append(topk.cpu().numpy())
                res["row_ids"].append(row_ids.cpu().numpy())
                res["plan"].append(plan_t.cpu().numpy())
                res["scores"].append(scores.cpu().numpy() if scores is not None else None)
        if len(plan.offload):
            self.pool.offload_pages(torch.from_numpy(x["off_pool"]).to(dev), torch.from_numpy(x["off_host"]).to(dev))
        res["status"] = self.pool.get_error()
        return res

    def host_pages_view(self) -> np.ndarray:
        L = self.cfg.n_layers
        return self.host.numpy().reshape(self.setup.host_pages, L, PAGE, ROW_BYTES)

    def pool_rows(self, layer: int) -> np.ndarray:
        return self.kv[layer].cpu().numpy().reshape(-1, ROW_BYTES)

    def close(self) -> None:
        self.pool.close()


class BenchSession:
    """Runs decode steps with every step's inputs staged ahead of time.

    device mode: inputs of all steps sit in HBM before timing starts; a step is
    only the hot-path calls.  host mode: each step's inputs sit packed in one pinned
    host buffer (256-byte aligned slices); each step copies it host -> device in one
    copy before its first call, inside the timed region, and the calls read views of
    the device copy. Outputs of up to HOST_WRITE_MAX bytes per step are written by the
    attention straight into pinned host memory (a device -> host transfer by the kernel
    itself: no copy latency after the last layer); larger ones come back in one copy,
    which moves many megabytes faster than the kernels' scattered writes over the link.
    (Splitting the input copy over a side stream to overlap it with the selection, or
    reading every input from host memory, measured slower.)
    """

    HOST_WRITE_MAX = 4 << 20

    def __init__(self, run: GpuRun, plans, mode: str = "device"):
        import torch
        self.torch = torch
        self.run = run
        self.plans = plans
        self.mode = mode
        cfg = run.cfg
        dev = run.dev
        self.steps = []
        for plan in plans:
            x = run.step_inputs(plan)
            arrays = {
                "req": x["req"], "pos": x["pos"], "limit": x["limit"],
                "kv_rows": x["kv_rows"], "idx_keys": x["idx_keys"],
                "q_idx": x["q_idx"], "w_idx": x["w_idx"],
                "q_attn": x["q_attn"].view(np.int16),
                "off_pool": x["off_pool"], "off_host": x["off_host"],
            }
            host = {k: torch.from_numpy(np.ascontiguousarray(v)) for k, v in arrays.items()}
            if mode == "host":
                offs, total = {}, 0
                for k, v in host.items():
                    offs[k] = total
                    total += (v.numel() * v.element_size() + 255) & ~255
                pack = torch.empty(total, dtype=torch.uint8).pin_memory()
                dpack = torch.empty(total, dtype=torch.uint8, device=dev)
                devt = {}
                for k, v in host.items():
                    nb = v.numel() * v.element_size()
                    pack[offs[k]:offs[k] + nb].copy_(torch.from_numpy(np.frombuffer(v.numpy().tobytes(), np.uint8).copy()))
                    devt[k] = dpack[offs[k]:offs[k] + nb].view(v.dtype).view(v.shape)
                host = {"_pack": pack, "_dpack": dpack, "_bytes": sum(v.numel() * v.element_size() for v in host.values())}
            else:
                devt = {k: v.to(dev) for k, v in host.items()}
            self.steps.append((plan, host, devt))
        n = cfg.n_requests * cfg.t_q
        self.n_tokens = n
        K = cfg.topk
        self.topk = [torch.empty((n, K), dtype=torch.int32, device=dev) for _ in range(cfg.n_groups)]
        self.row_ids = [torch.empty((n, K), dtype=torch.int32, device=dev) for _ in range(cfg.n_groups)]
        self.out = torch.empty((cfg.n_layers, n, cfg.n_heads, 512), dtype=torch.int16, device=dev)
        self.out_host = torch.empty_like(self.out, device="cpu").pin_memory() if mode == "host" else None
        self.host_write = mode == "host" and self.out.numel() * self.out.element_size() <= self.HOST_WRITE_MAX
        if self.host_write:
            self.out = self.out_host      # the attention writes its outputs into pinned host memory
        self.h2d_bytes = [h["_bytes"] if mode == "host" else sum(v.numel() * v.element_size() for v in h.values())
                          for _, h, _ in self.steps]
        self.d2h_bytes = self.out.numel() * self.out.element_size() if mode == "host" else 0

    def launches(self, i: int) -> int:
        """Kernels one step launches: append; per indexer group the indexer, the
        select kernel and the resolver (which also copies its misses); one attention
        kernel per layer (the split merge runs inside it); offload when pages complete."""
        cfg = self.run.cfg
        plan = self.steps[i][0]
        return 1 + cfg.n_groups * 3 + cfg.n_layers + (1 if len(plan.offload) else 0)

    def tick(self, i: int) -> None:
        self.run.apply_tick(self.steps[i][0].tick)

    def step(self, i: int, events=None) -> None:
        """Issue step i on the current stream. events: optional dict name -> list of
        (start, end) CUDA event pairs to time each hot-path call."""
        torch = self.torch
        run, cfg = self.run, self.run.cfg
        plan, host, d = self.steps[i]
        pool = run.pool

        def timed(name, fn):
            if events is None:
                fn()
                return
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            events.setdefault(name, []).append((a, b))

        host_mode = self.mode == "host"
        if host_mode:
            host["_dpack"].copy_(host["_pack"], non_blocking=True)   # every input of the step, one copy
        timed("append", lambda: pool.append_rows(d["req"], d["pos"], d["kv_rows"], d["idx_keys"]))
        for g in range(cfg.n_groups):
            timed("indexer_topk", lambda: run.indexer_topk(g, d["req"], d["limit"], d["q_idx"][g], d["w_idx"][g],
                                                           self.topk[g]))
            timed("resolve_topk", lambda: pool.resolve_topk(g, plan.step, d["req"], self.topk[g], self.row_ids[g]))
            for l in cfg.group_layers(g):
                timed("sparse_mla_decode", lambda: pool.sparse_mla_decode(l, d["q_attn"][l], self.row_ids[g],
                                                                          run.wl.sm_scale(), self.out[l]))
        if len(plan.offload):
            timed("offload_pages", lambda: pool.offload_pages(d["off_pool"], d["off_host"]))
        if host_mode and not self.host_write:
            self.out_host.copy_(self.out, non_blocking=True)
