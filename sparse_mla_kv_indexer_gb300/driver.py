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


def _stack(items, shape=None, dtype=None) -> np.ndarray:
    """np.stack, or an empty [0, *shape] array when a step has no query tokens."""
    if items or shape is None:
        return np.stack(items)
    return np.zeros((0,) + tuple(shape), dtype)


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
        # runs of consecutive pages of one request go in one call (a request that ends
        # turns its whole block table into placeholders)
        i, bt = 0, tick.bt_set
        while i < len(bt):
            r, p0, _ = bt[i]
            j = i + 1
            while j < len(bt) and bt[j][0] == r and bt[j][1] == p0 + (j - i):
                j += 1
            self.pool.set_pages(r, p0, block_table=[e[2] for e in bt[i:j]])
            i = j
        for r in tick.releases:
            self.pool.hot_release(r)
        for (r, g, pages) in tick.leases:
            self.pool.hot_lease(r, g, pages)

    def append_chunk(self) -> int:
        """Positions per hs_append_rows call: at most max_tokens, a multiple of 4 so that
        every chunk of 132-byte FP8 key records starts 16-byte aligned."""
        mt = self.pc.max_tokens
        return mt if mt < 4 else mt - mt % 4

    def step_inputs(self, plan: StepPlan) -> Dict[str, np.ndarray]:
        """Host arrays of one step, in batch order (tokens grouped by request)."""
        cfg, wl, s = self.cfg, self.wl, plan.step
        toks = plan.tokens
        t_q = cfg.t_q
        # positions written this step: a beginning turn's input, then the query tokens
        app = [(r, pos) for (r, lo, hi) in plan.tick.prefill for pos in range(lo, hi)] + [(t.req, t.pos) for t in toks]
        assert not plan.tick.prefill or self.append_chunk() % 4 == 0
        out = {
            "req": np.array([t.req for t in toks], np.int32),
            "limit": np.array([t.limit for t in toks], np.int32),
            "app_req": np.array([a[0] for a in app], np.int32),
            "app_pos": np.array([a[1] for a in app], np.int32),
            "kv_rows": np.stack([np.stack([wl.kv_rows(r, l)[pos] for l in range(cfg.n_layers)]) for r, pos in app]),
            "idx_keys": np.stack([np.stack([self._key_record(r, g, pos) for g in range(cfg.n_groups)])
                                  for r, pos in app]),
            "q_idx": _stack([_stack([self._idx_query(t.req, g, s)[0][i % t_q] for i, t in enumerate(toks)],
                                    (cfg.n_idx_heads, IDX_DIM), np.uint8 if cfg.idx_fp8 else np.int8)
                             for g in range(cfg.n_groups)]),
            "w_idx": _stack([_stack([self._idx_query(t.req, g, s)[1][i % t_q] for i, t in enumerate(toks)],
                                    (cfg.n_idx_heads,), np.float32 if cfg.idx_fp8 else np.int8)
                             for g in range(cfg.n_groups)]),
            "q_attn": _stack([_stack([wl.attn_queries(t.req, l, s)[i % t_q] for i, t in enumerate(toks)],
                                     (cfg.n_heads, 576), np.uint16)
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

    def step(self, plan: StepPlan, collect: bool = True, topk_in=None) -> Dict[str, object]:
        """One decode step through the C ABI. topk_in: optional per-group [n, K] host
        arrays that the resolver and attention take instead of the indexer's own
        selection (the indexer still runs; its selection is returned as "topk_own"),
        so that two runs whose selections differ only at a near-tie stay in the same
        residency state."""
        torch = self.torch
        cfg, dev = self.cfg, self.dev
        self.apply_tick(plan.tick)
        x = self.step_inputs(plan)
        n = len(plan.tokens)
        K = cfg.topk
        req = torch.from_numpy(x["req"]).to(dev)
        limit = torch.from_numpy(x["limit"]).to(dev)
        a_req, a_pos = torch.from_numpy(x["app_req"]).to(dev), torch.from_numpy(x["app_pos"]).to(dev)
        a_kv, a_ik = torch.from_numpy(x["kv_rows"]).to(dev), torch.from_numpy(x["idx_keys"]).to(dev)
        ch = self.append_chunk()
        for lo in range(0, a_req.numel(), ch):
            self.pool.append_rows(a_req[lo:lo + ch], a_pos[lo:lo + ch], a_kv[lo:lo + ch], a_ik[lo:lo + ch])
        if n == 0:     # every request has ended
            res = {"topk": [np.zeros((0, K), np.int32)] * cfg.n_groups, "row_ids": [np.zeros((0, K), np.int32)] * cfg.n_groups,
                   "plan": [np.zeros((0, K, PLAN_FIELDS), np.int32)] * cfg.n_groups, "scores": [None] * cfg.n_groups,
                   "o": [np.zeros((0, cfg.n_heads, 512))] * cfg.n_layers, "lse": [np.zeros((0, cfg.n_heads))] * cfg.n_layers}
            if len(plan.offload):
                self.pool.offload_pages(torch.from_numpy(x["off_pool"]).to(dev), torch.from_numpy(x["off_host"]).to(dev))
            res["status"] = self.pool.get_error()
            return res
        res = {"topk": [], "row_ids": [], "plan": [], "scores": [], "o": [None] * cfg.n_layers,
               "lse": [None] * cfg.n_layers}
        for g in range(cfg.n_groups):
            q = torch.from_numpy(np.ascontiguousarray(x["q_idx"][g])).to(dev)
            w = torch.from_numpy(np.ascontiguousarray(x["w_idx"][g])).to(dev)
            topk = torch.empty((n, K), dtype=torch.int32, device=dev)
            sdt = torch.float32 if cfg.idx_fp8 else torch.int64
            scores = torch.empty((n, self.max_ctx), dtype=sdt, device=dev) if self.keep_scores else None
            self.indexer_topk(g, req, limit, q, w, topk, scores)
            if topk_in is not None:
                res.setdefault("topk_own", []).append(topk.cpu().numpy())
                topk = torch.from_numpy(np.ascontiguousarray(topk_in[g], dtype=np.int32)).to(dev)
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
    A step's query tokens are those of the requests still alive; a turn that begins
    writes its input positions in the step's appends.
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
                "req": x["req"], "limit": x["limit"], "app_req": x["app_req"], "app_pos": x["app_pos"],
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
                pack = torch.empty(max(total, 256), dtype=torch.uint8).pin_memory()
                dpack = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
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
        self.n_max = n
        self.n_step = [len(p.tokens) for p in plans]
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
        out_per_tok = cfg.n_layers * cfg.n_heads * 512 * 2
        self.d2h_step = [nt * out_per_tok if mode == "host" else 0 for nt in self.n_step]
        self.d2h_bytes = self.out.numel() * self.out.element_size() if mode == "host" else 0

    def tokens(self, i: int) -> int:
        """Query tokens of step i (the requests alive at that step)."""
        return self.n_step[i]

    def appends(self, i: int) -> int:
        """hs_append_rows calls of step i (turn inputs can need more than one)."""
        n = self.steps[i][2]["app_req"].numel()
        ch = self.run.append_chunk()
        return -(-n // ch)

    def launches(self, i: int) -> int:
        """Kernels one step launches: the appends; per indexer group the indexer, the
        select kernel and the resolver (which also copies its misses); one attention
        kernel per layer (the split merge runs inside it); offload when pages complete."""
        cfg = self.run.cfg
        plan = self.steps[i][0]
        hot = cfg.n_groups * 3 + cfg.n_layers if self.n_step[i] else 0
        return self.appends(i) + hot + (1 if len(plan.offload) else 0)

    def tick(self, i: int) -> None:
        self.run.apply_tick(self.steps[i][0].tick)

    def step(self, i: int, events=None) -> None:
        """Issue step i on the current stream. events: optional dict name -> list of
        (start, end) CUDA event pairs to time each hot-path call."""
        torch = self.torch
        run, cfg = self.run, self.run.cfg
        plan, host, d = self.steps[i]
        pool = run.pool
        n = self.n_step[i]

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
        ch = run.append_chunk()
        for lo in range(0, d["app_req"].numel(), ch):
            timed("append", lambda lo=lo: pool.append_rows(d["app_req"][lo:lo + ch], d["app_pos"][lo:lo + ch],
                                                           d["kv_rows"][lo:lo + ch], d["idx_keys"][lo:lo + ch]))
        if n:
            for g in range(cfg.n_groups):
                topk, rows = self.topk[g][:n], self.row_ids[g][:n]
                timed("indexer_topk", lambda: run.indexer_topk(g, d["req"], d["limit"], d["q_idx"][g], d["w_idx"][g],
                                                               topk))
                timed("resolve_topk", lambda: pool.resolve_topk(g, plan.step, d["req"], topk, rows))
                for l in cfg.group_layers(g):
                    timed("sparse_mla_decode", lambda: pool.sparse_mla_decode(l, d["q_attn"][l], rows,
                                                                              run.wl.sm_scale(), self.out[l][:n]))
        if len(plan.offload):
            timed("offload_pages", lambda: pool.offload_pages(d["off_pool"], d["off_host"]))
        if host_mode and not self.host_write:
            self.out_host.copy_(self.out, non_blocking=True)
