"""Whole decode steps on the CPU, following the per-step procedure of the method.

One step, per "vLLM Part 1" (sections "How it works" and the proactive copy
paragraph) and "vLLM Part 2" (IndexShare, MQA-form sparse MLA):
  0. apply the host tick from the schedule: block-table changes, the hot buffers
     of requests that ended emptied (their pages go back to the pool; "Offload
     only where needed": hot pages are returned when not needed), hot leases;
  1. append the step's new KV rows (every sparse layer) and index keys: the input
     positions of a turn that begins this step, then the step's query tokens;
  2. per indexer group: scores + top-K for every query token, then the
     resolver for every request, then sparse MLA for every layer of the group;
  3. copy the pages this step completed, all layers, to their host pages.
The oracle keeps its own pool, host pool and index cache, filled from the same
workload and schedule the CUDA path uses.
"""
from typing import Dict, List

import numpy as np

from . import indexer, attention, resolver

PAGE = 64


class OracleRun:
    def __init__(self, wl, setup, keep_scores: bool = False):
        self.wl = wl
        cfg = self.cfg = wl.cfg
        self.setup = setup
        self.keep_scores = keep_scores
        R = cfg.n_requests
        self.pool = [np.zeros((setup.num_pages * PAGE, 656), np.uint8) for _ in range(cfg.n_layers)]
        self.host = np.zeros((setup.host_pages, cfg.n_layers, PAGE, 656), np.uint8)
        # key cache rows: 128 int8 values, or the 132-byte FP8 record (codes + fp32 scale)
        self.fp8 = bool(getattr(cfg, "idx_fp8", False))
        self.idx = [np.zeros((setup.num_idx_pages * PAGE, 132 if self.fp8 else 128), np.uint8 if self.fp8 else np.int8)
                    for _ in range(cfg.n_groups)]
        self.bt = setup.block_table.copy()
        self.hp = setup.host_page
        self.ip = setup.idx_page
        self.mat = setup.materialised.copy()
        self.hot = {(r, g): resolver.HotState() for r in range(R) for g in range(cfg.n_groups)}
        for r in range(R):
            P = setup.prefix_len[r]
            for l in range(cfg.n_layers):
                rows = wl.kv_rows(r, l)
                for p in range(-(-P // PAGE)):
                    lo, hi = p * PAGE, min(P, (p + 1) * PAGE)
                    if self.bt[r, p] >= 0:
                        b = int(self.bt[r, p]) * PAGE
                        self.pool[l][b:b + hi - lo] = rows[lo:hi]
                    if self.mat[r, p]:
                        self.host[self.hp[r, p], l, :hi - lo] = rows[lo:hi]
            for g in range(cfg.n_groups):
                keys = self.key_rows(r, g)
                for p in range(-(-P // PAGE)):
                    lo, hi = p * PAGE, min(P, (p + 1) * PAGE)
                    b = int(self.ip[r, p]) * PAGE
                    self.idx[g][b:b + hi - lo] = keys[lo:hi]
        for (r, g, pages) in setup.leases:
            self.hot[(r, g)].lease(pages)

    # ------------------------------------------------------------------
    def apply_tick(self, tick):
        for (r, p, pg) in tick.bt_set:
            self.bt[r, p] = pg
        for r in tick.releases:
            for g in range(self.cfg.n_groups):
                self.hot[(r, g)].release()
        for (r, g, pages) in tick.leases:
            self.hot[(r, g)].lease(pages)

    def append(self, positions):
        """Write the KV row (every layer) and index keys of each (request, position)."""
        for r, pos in positions:
            p, off = pos // PAGE, pos % PAGE
            row = int(self.bt[r, p]) * PAGE + off
            assert self.bt[r, p] >= 0
            for l in range(self.cfg.n_layers):
                self.pool[l][row] = self.wl.kv_rows(r, l)[pos]
            irow = int(self.ip[r, p]) * PAGE + off
            for g in range(self.cfg.n_groups):
                self.idx[g][irow] = self.key_rows(r, g)[pos]

    def key_rows(self, r: int, g: int) -> np.ndarray:
        return self.wl.idx_key_records_fp8(r, g) if self.fp8 else self.wl.idx_keys(r, g)

    def keys_of(self, g: int, r: int, n: int) -> np.ndarray:
        pos = np.arange(n)
        rows = self.ip[r, pos // PAGE].astype(np.int64) * PAGE + pos % PAGE
        return self.idx[g][rows]

    def step(self, plan) -> Dict[str, object]:
        cfg, wl, s = self.cfg, self.wl, plan.step
        self.apply_tick(plan.tick)
        self.append([(r, pos) for (r, lo, hi) in plan.tick.prefill for pos in range(lo, hi)])
        self.append([(t.req, t.pos) for t in plan.tokens])
        toks = plan.tokens
        n = len(toks)
        K = cfg.topk
        out = {"topk": [], "row_ids": [], "kind": [], "slot": [], "evicted": [], "scores": [],
               "misses": [], "o": [None] * cfg.n_layers, "lse": [None] * cfg.n_layers,
               "n_resident": [], "n_hit": []}
        for g in range(cfg.n_groups):
            tk = np.full((n, K), -1, np.int32)
            sc = []
            for i, t in enumerate(toks):
                j = i % cfg.t_q   # tokens come grouped by request, t_q per request
                rows = self.keys_of(g, t.req, t.limit)
                if self.fp8:
                    qc, w = wl.idx_queries_fp8(t.req, g, s)
                    scale = np.ascontiguousarray(rows[:, 128:132]).view("<f4").reshape(-1)
                    sv = indexer.scores_fp8(qc[j], w[j], rows[:, :128], scale)
                    tk[i] = indexer.topk_real(sv, K)
                else:
                    q = wl.idx_queries(t.req, g, s)[j]
                    w = wl.idx_weights(t.req, g)
                    sv = indexer.scores(q, w, rows)
                    tk[i] = indexer.topk(sv, K)
                if self.keep_scores:
                    sc.append(sv)
            row_ids = np.full((n, K), -1, np.int32)
            kind = np.zeros((n, K), np.int32)
            slot = np.full((n, K), -1, np.int32)
            ev = np.full((n, K), -1, np.int32)
            misses = []
            n_res = n_hit = 0
            for r in range(cfg.n_requests):
                idx = [i for i, t in enumerate(toks) if t.req == r]
                if not idx:
                    continue
                res = resolver.resolve(tk[idx], self.bt[r], self.hot[(r, g)], s)
                row_ids[idx], kind[idx], slot[idx], ev[idx] = res.row_ids, res.kind, res.slot, res.evicted
                n_res += res.n_resident
                n_hit += res.n_hit
                for (t, v) in res.misses:
                    p = t // PAGE
                    if not self.mat[r, p]:
                        raise resolver.HostMissingError(f"request {r} token {t}: no host copy")
                    dst = self.hot[(r, g)].slot_row(v)
                    for l in cfg.group_layers(g):
                        self.pool[l][dst] = self.host[self.hp[r, p], l, t % PAGE]
                    misses.append((r, t, v))
            out["topk"].append(tk)
            out["scores"].append(sc)
            out["row_ids"].append(row_ids)
            out["kind"].append(kind)
            out["slot"].append(slot)
            out["evicted"].append(ev)
            out["misses"].append(misses)
            out["n_resident"].append(n_res)
            out["n_hit"].append(n_hit)
            for l in cfg.group_layers(g):
                o = np.zeros((n, cfg.n_heads, 512))
                lse = np.zeros((n, cfg.n_heads))
                for i, t in enumerate(toks):
                    j = i % cfg.t_q
                    qb = wl.attn_queries(t.req, l, s)[j]
                    o[i], lse[i] = attention.sparse_mla_decode(qb, row_ids[i], self.pool[l], wl.sm_scale())
                out["o"][l] = o
                out["lse"][l] = lse
        for (r, p, pg, hpg) in plan.offload:
            for l in range(cfg.n_layers):
                self.host[hpg, l] = self.pool[l][pg * PAGE:(pg + 1) * PAGE]
            self.mat[r, p] = True
        return out
