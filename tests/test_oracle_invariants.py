"""Invariants of whole oracle runs over seeded workloads and their schedules.

Pins (from the behaviour the pages state):
* every resolved row id holds exactly the bytes of the requested token, in every
  layer of the group (hot rows and resident rows share one tensor and stride);
* the hot buffer never exceeds its cap ((speculative tokens + 2) x K, or 2 x K);
* the resident tail is never evicted;
* misses = |union| - resident - hits, and only misses move bytes from the host;
* a request with every page resident makes no misses;
* materialised host pages hold the exact bytes of their pool pages.
"""
import numpy as np
import pytest

from oracle.engine import OracleRun
from oracle import resolver
from sparse_mla_kv_indexer_gb300 import schedule as S
from sparse_mla_kv_indexer_gb300 import workload as W

PAGE = 64


def _run(name, **over):
    cfg = W.named_config(name)
    if over:
        cfg = W.WorkloadConfig(**{**cfg.__dict__, **over})
    wl = W.Workload(cfg)
    sch = S.Schedule(cfg)
    setup = sch.setup
    o = OracleRun(wl, setup)
    plans = []
    outs = []
    tails_seen = {}
    for s in range(cfg.steps):
        p = sch.plan(s)
        plans.append(p)
        out = o.step(p)
        outs.append(out)
        # tail pages of every request are resident after the tick
        for r in range(cfg.n_requests):
            end = max(t.pos for t in p.tokens if t.req == r) + 1
            last = (end - 1) // PAGE
            for pg in range(max(0, last - cfg.tail_pages + 1), last + 1):
                if o.bt[r, pg] >= 0:
                    tails_seen.setdefault(r, set()).add(pg)
            for pg in tails_seen.get(r, ()):
                if pg > last - cfg.tail_pages:
                    assert o.bt[r, pg] >= 0, f"tail page {pg} of request {r} evicted at step {s}"
        yield cfg, wl, o, p, out


@pytest.mark.parametrize("name", ["tiny", "small_single", "small_batch", "small_groups",
                                  "small_reuse", "short_ctx"])
def test_run_invariants(name):
    total_miss = 0
    for cfg, wl, o, p, out in _run(name):
        toks = p.tokens
        for g in range(cfg.n_groups):
            rid = out["row_ids"][g]
            tk = out["topk"][g]
            kind = out["kind"][g]
            for i, t in enumerate(toks):
                sel = tk[i]
                valid = sel >= 0
                assert (rid[i][valid] >= 0).all() and (rid[i][~valid] == -1).all()
                assert len(set(sel[valid].tolist())) == int(valid.sum())
                assert (sel[valid] < t.limit).all()
                assert valid.sum() == min(cfg.topk, t.limit)
                for l in cfg.group_layers(g):
                    want = wl.kv_rows(t.req, l)[sel[valid]]
                    got = o.pool[l][rid[i][valid]]
                    assert np.array_equal(got, want), (p.step, g, i, l)
            for r in range(cfg.n_requests):
                hot = o.hot[(r, g)]
                assert len(hot.stamp) <= cfg.hot_rows
                assert len(hot.tok2slot) <= cfg.hot_rows
                idx = [i for i, t in enumerate(toks) if t.req == r]
                union = set(tk[idx][tk[idx] >= 0].tolist())
                nm = sum(1 for (rr, _, _) in out["misses"][g] if rr == r)
                kinds = {}
                for i in idx:
                    for t, k in zip(tk[i], kind[i]):
                        if t >= 0:
                            kinds[int(t)] = int(k)
                assert nm == sum(1 for k in kinds.values() if k == resolver.MISS)
                assert len(union) == len(kinds)
            total_miss += len(out["misses"][g])
        for (r, pg, ppg, hpg) in p.offload:
            for l in range(cfg.n_layers):
                assert np.array_equal(o.host[hpg, l], o.pool[l][ppg * PAGE:(ppg + 1) * PAGE])
                assert np.array_equal(o.host[hpg, l], wl.kv_rows(r, l)[pg * PAGE:(pg + 1) * PAGE])
    assert total_miss > 0


def test_fully_resident_request_has_no_misses():
    for cfg, wl, o, p, out in _run("small_single", host_only_frac=0.0):
        for g in range(cfg.n_groups):
            assert out["misses"][g] == []
            assert out["n_hit"][g] == 0
            assert all(len(h.stamp) == 0 for h in o.hot.values())


def test_hot_cap_rule_matches_pages():
    for name in ["tiny", "ctx128k", "ctx1m"]:
        cfg = W.named_config(name)
        assert cfg.hot_rows == 2 * cfg.topk
    for name in ["batch32", "multiturn"]:
        cfg = W.named_config(name)
        assert cfg.hot_rows == (cfg.t_q - 1 + 2) * cfg.topk


def test_schedule_pool_pages_never_shared():
    cfg = W.named_config("small_batch")
    sch = S.Schedule(cfg)
    owner = {}
    for r in range(cfg.n_requests):
        for pg in sch.setup.block_table[r]:
            if pg >= 0:
                assert pg not in owner
                owner[int(pg)] = "kv"
    for (r, g, pages) in sch.setup.leases:
        for pg in pages:
            assert pg not in owner
            owner[pg] = "hot"
    hot_pages = set(pg for pg, k in owner.items() if k == "hot")
    for s in range(cfg.steps):
        p = sch.plan(s)
        for (r, g, pages) in p.tick.leases:
            hot_pages.update(pages)
        live = [int(x) for x in sch.bt.ravel() if x >= 0]
        assert len(live) == len(set(live))
        assert not (set(live) & hot_pages)
        assert not (set(sch.free) & (set(live) | hot_pages))
        assert len(set(live)) + len(hot_pages) + len(sch.free) == sch.setup.num_pages
    assert sch.evictions > 0
