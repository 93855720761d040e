"""Parity of the CUDA path (through the C ABI) with the CPU oracle, step by step.

Bit-exact: indexer scores, top-K sets, resolver plans (kind, slot, row id,
evicted token), pool bytes behind every row id, page copies to host.
Attention: max |err| <= 1e-2 and relative L2 <= 5e-3 against the fp64 oracle
on the dequantised FP8 inputs; lse within 5e-3.
"""
import numpy as np
import pytest

from oracle.engine import OracleRun
from sparse_mla_kv_indexer_gb300 import schedule as S
from sparse_mla_kv_indexer_gb300 import workload as W

pytestmark = pytest.mark.gpu

ATOL = 1e-2
REL_L2 = 5e-3
LSE_TOL = 5e-3


def _setup(name, **over):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_indexer_gb300.driver import GpuRun
    cfg = W.named_config(name)
    if over:
        cfg = W.WorkloadConfig(**{**cfg.__dict__, **over})
    wl = W.Workload(cfg)
    sch = S.Schedule(cfg)
    plans = [sch.plan(s) for s in range(cfg.steps)]
    oracle = OracleRun(wl, sch.setup, keep_scores=True)
    gpu = GpuRun(wl, sch.setup, keep_scores=True)
    return cfg, wl, plans, oracle, gpu


def check_step(cfg, wl, plan, o, g, gpu, oracle, exact_scores=True):
    assert g["status"] == 0, f"device status {g['status']}"
    toks = plan.tokens
    for grp in range(cfg.n_groups):
        for i, t in enumerate(toks):
            if exact_scores:
                assert np.array_equal(g["scores"][grp][i, :t.limit], o["scores"][grp][i]), (plan.step, grp, i)
        assert np.array_equal(g["topk"][grp], o["topk"][grp]), (plan.step, grp)
        pg = g["plan"][grp]
        assert np.array_equal(g["row_ids"][grp], o["row_ids"][grp]), (plan.step, grp)
        assert np.array_equal(pg[..., 0], o["kind"][grp])
        assert np.array_equal(pg[..., 1], o["slot"][grp])
        assert np.array_equal(pg[..., 2], o["row_ids"][grp])
        assert np.array_equal(pg[..., 3], o["evicted"][grp])
        # every row id holds exactly the bytes of its token, in every layer of the group
        for l in cfg.group_layers(grp):
            rows = gpu.pool_rows(l)
            for i, t in enumerate(toks):
                sel = o["topk"][grp][i]
                v = sel >= 0
                assert np.array_equal(rows[g["row_ids"][grp][i][v]], wl.kv_rows(t.req, l)[sel[v]])
    for l in range(cfg.n_layers):
        go, oo = g["o"][l], o["o"][l]
        err = np.abs(go - oo).max()
        rel = np.linalg.norm(go - oo) / np.linalg.norm(oo)
        assert err <= ATOL and rel <= REL_L2, (plan.step, l, err, rel)
        assert np.abs(g["lse"][l] - o["lse"][l]).max() <= LSE_TOL, (plan.step, l)
    host = gpu.host_pages_view()
    for (r, p, ppg, hpg) in plan.offload:
        assert np.array_equal(host[hpg], oracle.host[hpg]), (plan.step, r, p)


@pytest.mark.parametrize("name", ["tiny", "short_ctx", "small_single", "small_batch", "small_groups",
                                  "small_reuse", "small_mtp"])
def test_parity_small_configs(name):
    cfg, wl, plans, oracle, gpu = _setup(name)
    try:
        total_miss = total_h2d = 0
        for plan in plans:
            o = oracle.step(plan)
            g = gpu.step(plan)
            check_step(cfg, wl, plan, o, g, gpu, oracle)
            for grp in range(cfg.n_groups):
                total_miss += len(o["misses"][grp])
                total_h2d += len(o["misses"][grp]) * len(cfg.group_layers(grp)) * W.ROW_BYTES
        c = gpu.pool.counters()
        assert c.misses == total_miss and total_miss > 0
        assert c.h2d_bytes == total_h2d
    finally:
        gpu.close()


def test_parity_multiturn_turn_inputs_and_request_end():
    """Multi-turn histories: turn inputs written between decode steps (hs_append_rows),
    requests that end (hs_hot_release and their block tables cleared) and their pages
    leased again by the others. Every step matches the oracle as above, and the whole
    KV pool and index caches equal the oracle's byte for byte after every step."""
    cfg, wl, plans, oracle, gpu = _setup("small_multiturn")
    try:
        ends = prefills = 0
        for plan in plans:
            o = oracle.step(plan)
            g = gpu.step(plan)
            check_step(cfg, wl, plan, o, g, gpu, oracle)
            for l in range(cfg.n_layers):
                assert np.array_equal(gpu.pool_rows(l), oracle.pool[l]), (plan.step, l)
            for grp in range(cfg.n_groups):
                got = gpu.idx[grp].cpu().numpy().reshape(oracle.idx[grp].shape)
                assert np.array_equal(got, oracle.idx[grp].view(got.dtype)), (plan.step, grp)
            ends += len(plan.tick.releases)
            prefills += len(plan.tick.prefill)
        assert ends == 3 and prefills == 5
        c = gpu.pool.counters()
        assert c.misses > 0 and c.d2h_bytes > 0
    finally:
        gpu.close()


@pytest.mark.parametrize("name,over", [
    # 16 query tokens x 9 row splits: 64 heads per CTA, merge through L2, odd split count
    ("small_batch", dict(topk=1152, hot_rows=5 * 1152, pressure=False)),
    # 1 query token x 9 row splits: 16 heads per CTA, merge through distributed shared memory
    ("small_single", dict(topk=1152, hot_rows=2 * 1152)),
    # top-K 128: a single row split, no cluster and no merge (16 and 64 heads per CTA)
    ("small_single", dict(topk=128, hot_rows=2 * 128)),
    ("small_batch", dict(topk=128, hot_rows=5 * 128, pressure=False)),
])
def test_parity_odd_split_count(name, over):
    cfg, wl, plans, oracle, gpu = _setup(name, **over)
    try:
        for plan in plans:
            o = oracle.step(plan)
            g = gpu.step(plan)
            check_step(cfg, wl, plan, o, g, gpu, oracle)
    finally:
        gpu.close()


@pytest.mark.parametrize("name,over", [
    # 32 query heads (two head groups of 16 per token) and 48 index heads (N = 48 MMAs)
    ("small_single", dict(n_heads=32, n_idx_heads=48)),
    # 32 query heads and 32 index heads with 4 MTP tokens per request
    ("small_batch", dict(n_heads=32, n_idx_heads=32)),
])
def test_parity_other_head_counts(name, over):
    cfg, wl, plans, oracle, gpu = _setup(name, **over)
    try:
        for plan in plans:
            o = oracle.step(plan)
            g = gpu.step(plan)
            check_step(cfg, wl, plan, o, g, gpu, oracle)
    finally:
        gpu.close()


def test_parity_tiny_all_pages_resident_no_misses():
    cfg, wl, plans, oracle, gpu = _setup("tiny", host_only_frac=0.0)
    try:
        for plan in plans:
            o = oracle.step(plan)
            g = gpu.step(plan)
            check_step(cfg, wl, plan, o, g, gpu, oracle)
        assert gpu.pool.counters().misses == 0
    finally:
        gpu.close()


def test_replay_reproduces_the_resolved_rows_and_changes_no_state():
    # multi-request MTP batch with misses, eviction and pool pressure; the oracle
    # never replays, so any state a replay changed would show in the next step
    cfg, wl, plans, oracle, gpu = _setup("small_batch")
    import torch
    try:
        for plan in plans:
            o = oracle.step(plan)
            g = gpu.step(plan)
            check_step(cfg, wl, plan, o, g, gpu, oracle)
            req = torch.tensor([t.req for t in plan.tokens], dtype=torch.int32, device="cuda")
            c0 = gpu.pool.counters()
            for grp in range(cfg.n_groups):
                topk = torch.from_numpy(np.ascontiguousarray(g["topk"][grp])).cuda()
                rows = torch.full_like(topk, -7)
                gpu.pool.replay_topk(grp, req, topk, rows)
                assert np.array_equal(rows.cpu().numpy(), g["row_ids"][grp]), (plan.step, grp)
            c1 = gpu.pool.counters()
            assert (c0.resident, c0.hits, c0.misses, c0.h2d_bytes) == (c1.resident, c1.hits, c1.misses, c1.h2d_bytes)
            assert gpu.pool.get_error() == 0
    finally:
        gpu.close()


def test_replay_of_an_unresolved_token_reports_not_resolved():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=16, n_heads=16, topk=256,
                      n_layers=1, layers_per_indexer=1, num_pages=4, num_idx_pages=4, max_requests=1,
                      max_ctx=256, max_q_per_req=1, hot_rows=512, max_tokens=1, idx_format=0, host_pages=4)
    kv = [torch.zeros(4 * 64 * 656, dtype=torch.uint8, device="cuda")]
    ix = [torch.zeros(4 * 64 * 128, dtype=torch.int8, device="cuda")]
    host = torch.zeros(4 * 64 * 656, dtype=torch.uint8, pin_memory=True)
    pool = H.Pool(pc, kv, ix, host)
    try:
        # page 0 resident at pool page 2, page 1 host-only and never resolved
        pool.set_pages(0, 0, block_table=[2, -1], idx_pages=[0, 1], host_pages=[0, 1])
        req = torch.zeros(1, dtype=torch.int32, device="cuda")
        topk = torch.full((1, 256), -1, dtype=torch.int32, device="cuda")
        topk[0, :3] = torch.tensor([5, 70, 63], dtype=torch.int32)
        rows = torch.empty_like(topk)
        pool.replay_topk(0, req, topk, rows)
        assert pool.get_error() == 10   # HS_ERR_NOT_RESOLVED
        assert rows[0, :4].cpu().tolist() == [2 * 64 + 5, -1, 2 * 64 + 63, -1]
    finally:
        pool.close()
