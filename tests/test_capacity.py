"""Capacity report (host side): plain residency against Hybrid HiSparse on one KV budget."""
import json
import os

import pytest

from sparse_mla_kv_indexer_gb300 import capacity as C
from sparse_mla_kv_indexer_gb300 import schedule as S
from sparse_mla_kv_indexer_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _pages_model():
    """The pages' model: 78 MLA layers x 656 B, 21 indexer layers x 132 B, 788 B MTP
    (vLLM blog Part 2, footnote 3), top-K 2,048, one indexer per 4 sparse layers."""
    return C.KVLayout(78, 21, row_bytes=656, key_bytes=132, extra_bytes_per_token=788), C.HiSparsePolicy()


def test_layout_reproduces_the_pages_bytes_per_token_and_per_million():
    g = json.load(open(GOLDEN))
    layout, _ = _pages_model()
    assert layout.plain_bytes_per_token() == g["kv_bytes_per_token"]["value"]
    gib = C.plain_bytes_per_request(g["kv_gib_per_1m_tokens"]["tokens"], layout) / (1 << 30)
    assert abs(gib - g["kv_gib_per_1m_tokens"]["value"]) <= g["kv_gib_per_1m_tokens"]["abs_tol"]


def test_plain_concurrency_equals_page_by_page_allocation():
    layout = C.KVLayout(4, 1)
    per_page = C.PAGE * layout.plain_bytes_per_token()
    for L in (1, 63, 64, 65, 4097, 131072):
        budget_pages = 5000
        budget = budget_pages * per_page + 123
        free, n = budget_pages, 0
        while free >= C.pages(L):           # admit whole requests until the next one does not fit
            free -= C.pages(L)
            n += 1
        assert C.report(budget, [L], layout, C.HiSparsePolicy())[0].plain == n


def test_crossover_matches_the_pages_qualitative_shape():
    layout, policy = _pages_model()
    budget = 100 << 30
    Lx = C.crossover_context(layout, policy)
    assert 1000 < Lx < 1 << 20
    short, long_ = C.report(budget, [int(Lx / 4), int(Lx * 4)], layout, policy)
    assert short.plain > short.hisparse          # the fixed hot-buffer cost dominates short contexts
    assert long_.hisparse > long_.plain          # bounded sparse-MLA residency wins long ones
    r = C.report(budget, [1 << 20], layout, policy)[0]
    assert r.host_pool_bytes == r.hisparse * C.host_bytes_per_request(1 << 20, layout)


def test_mtp_hot_factor_and_pool_pages_match_the_schedule():
    # the 1M shape: 8 sparse layers, 2 indexers, hot cap 4,096 rows per group, 16 tail
    # pages resident; the schedule reserves exactly the tail and the hot buffers
    # (plus its growth pages and slack) for the request
    cfg = W.named_config("ctx1m")
    sch = S.Schedule(cfg)
    layout = C.KVLayout(cfg.n_layers, cfg.n_groups)
    policy = C.HiSparsePolicy(cfg.topk, cfg.hot_rows // cfg.topk, cfg.layers_per_indexer, cfg.tail_pages)
    grow = -(-(cfg.steps * cfg.accept + cfg.t_q) // C.PAGE) + 1
    assert C.hisparse_pool_pages_per_request(layout, policy, max(cfg.ctx_len)) == \
        sch.setup.num_pages - grow - cfg.pool_slack_pages
    assert C.HiSparsePolicy.mtp_hot_factor(3) == 5      # (num_speculative_tokens + 2) x top-K


def test_cli_prints_a_table(capsys):
    C.main(["--kv-gib", "50", "--contexts", "8192,1048576"])
    out = capsys.readouterr().out
    assert "crossover" in out and "1048576" in out


@pytest.mark.parametrize("name", ["batch32", "multiturn"])
def test_capacity_matches_measured_pool_occupancy(name):
    """The capacity model against the pool pages the residency schedule actually holds
    for the 32-request and the multi-turn shapes, step by step (host side: the
    schedule is what the bench and the tests drive; no kernel runs here).

    Once a hot buffer has had the steps it needs to fill, every request that reads
    from the host holds exactly the model's HiSparse floor, its resident tail plus
    its hot buffers; the rest of the pool is the surplus residency that pressure
    eviction lets go of page by page. Pool pages are conserved, and the model's
    HiSparse concurrency on the measured pool covers the requests the run carries."""
    import dataclasses
    cfg = dataclasses.replace(W.named_config(name), steps=8)
    sch = S.Schedule(cfg)
    layout = C.KVLayout(cfg.n_layers, cfg.n_groups)
    policy = C.HiSparsePolicy(cfg.topk, cfg.hot_rows // cfg.topk, cfg.layers_per_indexer, cfg.tail_pages)
    grow = -(-cfg.t_q * cfg.topk // C.PAGE)
    fill = -(-policy.hot_pages() // grow)        # steps a hot buffer needs to reach its cap
    checked = 0
    for s in range(cfg.steps):
        p = sch.plan(s)
        used = int((sch.bt >= 0).sum()) + sum(len(v) for v in sch.hot_of.values())
        assert used + len(sch.free) == sch.setup.num_pages
        live = sorted(set(t.req for t in p.tokens))
        for r in live:
            end = max(t.pos for t in p.tokens if t.req == r) + 1
            hot = sum(len(sch.hot_of[(r, g)]) for g in range(cfg.n_groups))
            assert hot <= C.n_groups(layout, policy) * policy.hot_pages()
            last = (end - 1) // C.PAGE
            tail = [pg for pg in range(max(0, last - cfg.tail_pages + 1), last + 1)]
            if r in cfg.prefix_reuse or s < fill or not (sch.bt[r, :last + 1] < 0).any():
                continue
            assert all(sch.bt[r, pg] >= 0 for pg in tail)
            assert len(tail) + hot == C.hisparse_pool_pages_per_request(layout, policy, end), (s, r)
            checked += 1
        floor = max(C.hisparse_pool_pages_per_request(layout, policy, max(t.limit for t in p.tokens if t.req == r))
                    for r in live)
        assert sch.setup.num_pages // floor >= len(live)
    assert checked > 0
