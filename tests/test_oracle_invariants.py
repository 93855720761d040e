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
        # tail pages of every live request are resident after the tick
        for r in sorted(set(t.req for t in p.tokens)):
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
                                  "small_reuse", "short_ctx", "small_multiturn"])
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


@pytest.mark.parametrize("name", ["small_batch", "small_multiturn"])
def test_schedule_pool_pages_never_shared(name):
    """Every pool page has exactly one owner (a block-table entry, a hot buffer or the
    free list) after every step, across evictions, request ends and re-leases."""
    cfg = W.named_config(name)
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
    hot = {(r, g): list(pages) for (r, g, pages) in sch.setup.leases}
    released_pages = set()
    reused = 0
    for s in range(cfg.steps):
        p = sch.plan(s)
        for r in p.tick.releases:            # the schedule's own record of a request end
            for g in range(cfg.n_groups):
                released_pages.update(hot.pop((r, g), []))
        for (r, g, pages) in p.tick.leases:
            reused += len(released_pages & set(pages))
            hot.setdefault((r, g), []).extend(pages)
        hot_pages = [pg for v in hot.values() for pg in v]
        assert sorted(hot_pages) == sorted(pg for v in sch.hot_of.values() for pg in v)
        live = [int(x) for x in sch.bt.ravel() if x >= 0]
        reused += len(released_pages & set(live))
        assert len(live) == len(set(live)) and len(hot_pages) == len(set(hot_pages))
        assert not (set(live) & set(hot_pages))
        assert not (set(sch.free) & (set(live) | set(hot_pages)))
        assert len(set(live)) + len(hot_pages) + len(sch.free) == sch.setup.num_pages
        for r in p.tick.releases:
            assert (sch.bt[r] < 0).all() and all(not sch.hot_of[(r, g)] for g in range(cfg.n_groups))
    assert sch.evictions > 0
    if cfg.turns:
        assert released_pages and reused > 0, "pages of ended requests are leased again"


def test_multiturn_schedule_crosses_turns_and_ends_requests():
    """small_multiturn: turn inputs are written at the turn boundaries of each request's
    history, and requests whose history is done end (release, no more tokens)."""
    cfg = W.named_config("small_multiturn")
    sch = S.Schedule(cfg)
    prefills, ends, toks = [], [], []
    for s in range(cfg.steps):
        p = sch.plan(s)
        prefills += [(s, r, hi - lo) for (r, lo, hi) in p.tick.prefill]
        ends += [(s, r) for r in p.tick.releases]
        toks.append(sorted(set(t.req for t in p.tokens)))
        for (r, lo, hi) in p.tick.prefill:      # the turn's input lands right before its tokens
            assert min(t.pos for t in p.tokens if t.req == r) == hi
    assert all(n == cfg.turn_input for (_, _, n) in prefills)
    # history steps (0, 4, 7, 2) with 3 steps per turn and 3 turns
    assert sorted((s, r) for (s, r, _) in prefills) == [(1, 3), (2, 1), (3, 0), (4, 3), (6, 0)]
    assert ends == [(2, 2), (5, 1), (7, 3)]
    for (s, r) in ends:
        assert all(r not in toks[t] for t in range(s, cfg.steps))


def test_multiturn_config_matches_the_pages_shape():
    """The full multi-turn shape: 64 requests, 13 turns (74,160 first-turn tokens, +753
    input and 220 output tokens per turn at 3 per step), contexts 74K..86K, 25 %
    prefix-reuse requests."""
    cfg = W.named_config("multiturn")
    assert cfg.n_requests == 64 and cfg.turns == 13 and cfg.turn_input == 753
    assert cfg.turn_steps * cfg.accept >= 220 > (cfg.turn_steps - 1) * cfg.accept
    assert len(cfg.prefix_reuse) == 16
    assert 74160 <= min(cfg.ctx_len) - cfg.t_q and max(cfg.ctx_len) <= 74160 + 12 * 753 + 13 * 222 + cfg.t_q
    assert all(h < cfg.turns * cfg.turn_steps for h in cfg.history_step)
