"""Host-side residency schedule: which pool page holds which KV page, when.

This is the host bookkeeping that runs between decode steps (never inside one):
pool-page allocation for the pages new tokens land in, pressure eviction of
completed, host-materialised pages, hot-buffer leasing, and the list of pages to
materialise on the host after each step. Its decisions depend only on positions
and step counters, never on what the kernels compute, so the whole schedule is
fixed before the run and is an input to both the oracle and the CUDA path. It
holds none of the method's arithmetic.

Readings of "Hybrid HiSparse" (vLLM blog, Part 1, section "How it works") that
this module fixes:
* KV residency is tracked per page; the block table holds real pool pages and
  empty placeholders (-1); the last ``tail_pages`` pages of a request are never
  evicted.
* Under pool pressure a page gives up its pool slot only once it is complete and
  its host copy exists, so the release needs no second copy. Victims are taken
  oldest first: (completion step, request, logical page) ascending; pages
  completed before the run count as step -1.
* Hot-buffer pages are ordinary pool pages leased from the same free list. A
  (request, group) whose block table holds any placeholder is topped up before
  each step to min(cap, leased + T_q * K) rows, in whole pages. Prefix-reuse
  requests start with placeholders for every complete page plus one hot page.
* A page is queued for host materialisation in the step whose committed tokens
  complete it; all sparse layers of the page are copied together.
* Multi-turn histories (the pages' OpenHands-style workload): a turn after the
  first begins with its input positions written into the request's pages before
  that step's decode tokens, like a prefill. When a request's history is done it
  ends: its hot-buffer pages and every pool page of its block table (tail pages
  included) return to the free list, its block-table entries become placeholders
  and its hot buffers are emptied (section "Offload only where needed": hot pages
  are leased on first need and returned when not needed).
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass, field
from typing import Dict, List, Tuple

import numpy as np

from .workload import PAGE, WorkloadConfig


@dataclass
class Token:
    req: int
    pos: int       # position whose KV row this token writes
    limit: int     # causal limit: the token sees positions [0, limit)


@dataclass
class Tick:
    """Host actions applied before a step."""
    bt_set: List[Tuple[int, int, int]] = field(default_factory=list)      # (req, page, pool page or -1)
    leases: List[Tuple[int, int, List[int]]] = field(default_factory=list)  # (req, group, pool pages)
    releases: List[int] = field(default_factory=list)                     # requests that ended
    prefill: List[Tuple[int, int, int]] = field(default_factory=list)     # (req, first pos, end pos) written


@dataclass
class StepPlan:
    step: int
    tick: Tick
    tokens: List[Token]
    offload: List[Tuple[int, int, int, int]]   # (req, page, pool page, host page)


@dataclass
class Setup:
    """State before step 0."""
    num_pages: int
    n_pages_max: int                    # logical pages per request (max over requests)
    block_table: np.ndarray             # [R, n_pages_max] int32, -1 = placeholder / unallocated
    host_page: np.ndarray               # [R, n_pages_max] int64, -1 = none
    materialised: np.ndarray            # [R, n_pages_max] bool: host copy written at setup
    idx_page: np.ndarray                # [R, n_pages_max] int32 index-key cache pages
    num_idx_pages: int
    host_pages: int
    leases: List[Tuple[int, int, List[int]]]   # initial hot pages
    prefix_len: List[int]               # committed tokens per request before step 0


class Schedule:
    def __init__(self, cfg: WorkloadConfig):
        self.cfg = cfg
        R = cfg.n_requests
        self.pressure = cfg.pressure
        self.n_pages_max = max(-(-cfg.final_len(r) // PAGE) for r in range(R))
        self.prefix = [cfg.ctx_len[r] - cfg.t_q for r in range(R)]
        npm = self.n_pages_max
        bt = np.full((R, npm), -1, np.int32)
        hp = np.full((R, npm), -1, np.int64)
        mat = np.zeros((R, npm), bool)
        ip = np.full((R, npm), -1, np.int32)
        host_next = 0
        idx_next = 0
        resident: List[Tuple[int, int]] = []
        for r in range(R):
            n_final = -(-cfg.final_len(r) // PAGE)
            hp[r, :n_final] = np.arange(host_next, host_next + n_final)
            host_next += n_final
            ip[r, :n_final] = np.arange(idx_next, idx_next + n_final)
            idx_next += n_final
            P = self.prefix[r]
            n_prefix = -(-P // PAGE)
            n_complete = P // PAGE
            mat[r, :n_complete] = True
            tail_lo = max(0, n_prefix - cfg.tail_pages)
            if r in cfg.prefix_reuse:
                chosen_res = set(range(n_complete, n_prefix))      # only the partial page
            else:
                cand = np.arange(0, tail_lo)
                rng = np.random.default_rng(np.random.SeedSequence([cfg.request_seed(r), 9]))
                n_host = int(round(cfg.host_only_frac * len(cand)))
                host_only = set(rng.choice(cand, size=n_host, replace=False).tolist()) if n_host else set()
                chosen_res = set(p for p in range(n_prefix) if p not in host_only)
            for p in sorted(chosen_res):
                resident.append((r, p))
        n_res = len(resident)
        init_hot = sum(cfg.n_groups for r in range(R) if r in cfg.prefix_reuse)
        if self.pressure:
            num_pages = n_res + init_hot + cfg.pool_slack_pages
        else:
            if cfg.turns:
                grow = sum(-(-cfg.final_len(r) // PAGE) - self.prefix[r] // PAGE + 1 for r in range(R))
            else:
                grow = sum(-(-(cfg.steps * cfg.accept + cfg.t_q) // PAGE) + 1 for _ in range(R))
            num_pages = n_res + init_hot + R * cfg.n_groups * (cfg.hot_rows // PAGE) + grow + cfg.pool_slack_pages
        for i, (r, p) in enumerate(resident):
            bt[r, p] = i
        free = list(range(n_res, num_pages))
        leases = []
        self.leased = {(r, g): 0 for r in range(R) for g in range(cfg.n_groups)}
        self.hot_of: Dict[Tuple[int, int], List[int]] = {k: [] for k in self.leased}
        for r in cfg.prefix_reuse:
            for g in range(cfg.n_groups):
                pg = free.pop(0)
                leases.append((r, g, [pg]))
                self.leased[(r, g)] = 1
                self.hot_of[(r, g)].append(pg)
        heapq.heapify(free)
        self.free = free
        self.setup = Setup(num_pages, npm, bt.copy(), hp, mat.copy(), ip, idx_next, host_next,
                           leases, list(self.prefix))
        # live state mirrored on the host
        self.bt = bt
        self.mat = mat
        self.hp = hp
        self.completed_step: Dict[Tuple[int, int], int] = {}
        self.evict_heap: List[Tuple[int, int, int]] = []
        for r in range(R):
            for p in range(self.prefix[r] // PAGE):
                if bt[r, p] >= 0:
                    self.evict_heap.append((-1, r, p))
        heapq.heapify(self.evict_heap)
        self.committed = list(self.prefix)
        self.events = [cfg.events(r) for r in range(R)]
        self.alive = [True] * R
        self.evictions = 0

    # ------------------------------------------------------------------
    def _tail_lo(self, r: int, end: int) -> int:
        last = (end - 1) // PAGE
        return max(0, last - self.cfg.tail_pages + 1)

    def _alloc(self, tick: Tick, step_end: List[int]) -> int:
        if not self.free:
            self._evict_one(tick, step_end)
        return heapq.heappop(self.free)

    def _evict_one(self, tick: Tick, step_end: List[int]) -> None:
        while self.evict_heap:
            cs, r, p = heapq.heappop(self.evict_heap)
            if self.bt[r, p] < 0 or not self.mat[r, p]:
                continue
            if p >= self._tail_lo(r, step_end[r]):
                # still in the tail: not eligible now; keep it for later steps
                self._deferred.append((cs, r, p))
                continue
            pg = int(self.bt[r, p])
            self.bt[r, p] = -1
            tick.bt_set.append((r, p, -1))
            heapq.heappush(self.free, pg)
            self.evictions += 1
            return
        raise RuntimeError("pool exhausted: no evictable page (pool too small for the workload)")

    def _needs_hot(self, r: int, end: int) -> bool:
        n = -(-end // PAGE)
        return bool((self.bt[r, :n] < 0).any())

    def _end_request(self, r: int, tick: Tick) -> None:
        """Request end: every pool page of r (block table and hot buffers) to the free list."""
        self.alive[r] = False
        tick.releases.append(r)
        for p in np.nonzero(self.bt[r] >= 0)[0]:
            heapq.heappush(self.free, int(self.bt[r, p]))
            self.bt[r, p] = -1
            tick.bt_set.append((r, int(p), -1))
        for g in range(self.cfg.n_groups):
            for pg in self.hot_of[(r, g)]:
                heapq.heappush(self.free, pg)
            self.hot_of[(r, g)] = []
            self.leased[(r, g)] = 0

    def plan(self, s: int) -> StepPlan:
        cfg = self.cfg
        R = cfg.n_requests
        tick = Tick()
        self._deferred: List[Tuple[int, int, int]] = []
        # 0. requests whose history is done end; a new turn writes its input positions
        live = []
        lo = list(self.committed)
        for r in range(R):
            if not self.alive[r]:
                continue
            if s >= len(self.events[r]):
                self._end_request(r, tick)
                continue
            live.append(r)
            inp = self.events[r][s][0]
            if inp:
                tick.prefill.append((r, self.committed[r], self.committed[r] + inp))
                self.committed[r] += inp
        start = [self.committed[r] for r in range(R)]
        end = [start[r] + cfg.t_q if r in live else start[r] for r in range(R)]
        # 1. pages that this step's positions (turn input and tokens) land in
        for r in live:
            for p in range(lo[r] // PAGE, (end[r] - 1) // PAGE + 1):
                if self.bt[r, p] < 0:
                    pg = self._alloc(tick, end)
                    self.bt[r, p] = pg
                    tick.bt_set.append((r, p, pg))
        # 2. hot leases, repeated until no request newly needs a buffer
        cap_pages = cfg.hot_rows // PAGE
        grow_pages = -(-(cfg.t_q * cfg.topk) // PAGE)
        topped = set()
        changed = True
        while changed:
            changed = False
            for r in live:
                if not self._needs_hot(r, end[r]):
                    continue
                for g in range(cfg.n_groups):
                    if (r, g) in topped:
                        continue
                    topped.add((r, g))
                    cur = self.leased[(r, g)]
                    target = min(cap_pages, cur + grow_pages)
                    if target <= cur:
                        continue
                    pages = [self._alloc(tick, end) for _ in range(target - cur)]
                    changed = True
                    self.leased[(r, g)] = target
                    self.hot_of[(r, g)].extend(pages)
                    tick.leases.append((r, g, pages))
        for item in self._deferred:
            heapq.heappush(self.evict_heap, item)
        # 3. tokens
        tokens = []
        for r in live:
            for j in range(cfg.t_q):
                pos = start[r] + j
                tokens.append(Token(r, pos, pos + 1))
        # 4. commit and offload what this step completes (turn input included)
        offload = []
        for r in live:
            newc = start[r] + cfg.accept
            for p in range(lo[r] // PAGE, newc // PAGE):
                if (p + 1) * PAGE <= newc and not self.mat[r, p]:
                    assert self.bt[r, p] >= 0, "a completing page is always resident"
                    offload.append((r, p, int(self.bt[r, p]), int(self.hp[r, p])))
                    self.mat[r, p] = True
                    self.completed_step[(r, p)] = s
                    heapq.heappush(self.evict_heap, (s, r, p))
            self.committed[r] = newc
        return StepPlan(s, tick, tokens, offload)

    def plans(self) -> List[StepPlan]:
        return [self.plan(s) for s in range(self.cfg.steps)]


def build(cfg: WorkloadConfig) -> Tuple[Setup, List[StepPlan]]:
    """Setup state plus the per-step plans of a run."""
    sch = Schedule(cfg)
    return sch.setup, sch.plans()
