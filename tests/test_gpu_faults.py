"""Failure detection on the device and the host, without faulting or hanging the GPU.

Device-detected errors go to the pool's status word (read and cleared by
hs_get_error); each case is provoked with valid memory accesses only:
  * a bounded wait that runs out (hs_wait_selftest) -> HS_ERR_TIMEOUT, and the
    context then runs a full decode step;
  * more misses than the hot buffer has slots -> HS_ERR_CAPACITY;
  * a selected token whose page is a placeholder without a host copy -> HS_ERR_HOST_MISSING;
  * a row id beyond the pool -> HS_ERR_BAD_ID (the row is skipped).
Host-side argument checks return HS_ERR_INVALID and launch nothing: a misaligned
query, page ids outside the pool, a hot lease beyond the cap."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

TIMEOUT, CAPACITY, HOST_MISSING, BAD_ID, INVALID = 5, 3, 6, 7, 1


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _pool(torch, H, hot_rows=64, num_pages=8, host_pages=64):
    pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=16, n_heads=16, topk=128,
                      n_layers=1, layers_per_indexer=1, num_pages=num_pages, num_idx_pages=64, max_requests=1,
                      max_ctx=4096, max_q_per_req=1, hot_rows=hot_rows, max_tokens=1, idx_format=0,
                      host_pages=host_pages)
    kv = [torch.zeros(num_pages * 64 * 656, dtype=torch.uint8, device="cuda")]
    ix = [torch.zeros(64 * 64 * 128, dtype=torch.int8, device="cuda")]
    host = torch.zeros(host_pages * 64 * 656, dtype=torch.uint8, pin_memory=True)
    return H.Pool(pc, kv, ix, host)


def _resolve(torch, pool, tokens, step):
    req = torch.zeros(1, dtype=torch.int32, device="cuda")
    topk = torch.tensor([tokens], dtype=torch.int32, device="cuda")
    rows = torch.empty_like(topk)
    pool.resolve_topk(0, step, req, topk, rows)
    torch.cuda.synchronize()
    return rows.cpu().numpy()[0]


def test_wait_timeout_is_reported_and_the_context_stays_usable():
    torch = _torch()
    from oracle.engine import OracleRun
    from sparse_mla_kv_indexer_gb300 import schedule as S
    from sparse_mla_kv_indexer_gb300 import workload as W
    from sparse_mla_kv_indexer_gb300.driver import GpuRun
    cfg = W.named_config("tiny")
    wl = W.Workload(cfg)
    sch = S.Schedule(cfg)
    gpu = GpuRun(wl, sch.setup)
    gpu.pool.wait_selftest()
    assert gpu.pool.get_error() == TIMEOUT
    assert gpu.pool.get_error() == 0           # read and cleared
    plan = sch.plan(0)                         # a full step afterwards, checked against the oracle
    g = gpu.step(plan)
    o = OracleRun(wl, sch.setup).step(plan)
    assert g["status"] == 0
    assert np.array_equal(g["topk"][0], o["topk"][0]) and np.array_equal(g["row_ids"][0], o["row_ids"][0])


def test_more_misses_than_hot_slots_is_capacity():
    torch = _torch()
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    pool = _pool(torch, H, hot_rows=64)
    try:
        pool.set_pages(0, 0, block_table=[-1] * 64, host_pages=list(range(64)))   # nothing resident
        pool.hot_lease(0, 0, [0])                                                  # 64 slots
        _resolve(torch, pool, list(range(128)), 1)                                 # 128 misses
        assert pool.get_error() == CAPACITY
    finally:
        pool.close()


def test_placeholder_without_host_copy_is_host_missing():
    torch = _torch()
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    pool = _pool(torch, H, hot_rows=256)
    try:
        pool.set_pages(0, 0, block_table=[-1] * 64, host_pages=[-1, -1] + list(range(2, 64)))
        pool.hot_lease(0, 0, [0, 1])
        _resolve(torch, pool, list(range(64, 192)), 1)   # pages 1-2: page 1 has no host copy
        assert pool.get_error() == HOST_MISSING
        _resolve(torch, pool, list(range(128, 256)), 2)  # pages 2-3, both materialised: no error
        assert pool.get_error() == 0
    finally:
        pool.close()


def test_row_id_beyond_the_pool_is_bad_id_and_skipped():
    torch = _torch()
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    pool = _pool(torch, H)
    try:
        q = torch.randn(1, 16, 576, device="cuda").to(torch.bfloat16).view(torch.int16)
        out = torch.zeros(1, 16, 512, dtype=torch.int16, device="cuda")
        rows = torch.full((1, 128), -1, dtype=torch.int32, device="cuda")
        rows[0, 0] = 8 * 64          # one past the last row of the 8-page pool
        rows[0, 1] = 5
        pool.sparse_mla_decode(0, q, rows, 0.05, out)
        torch.cuda.synchronize()
        assert pool.get_error() == BAD_ID
        assert bool(torch.isfinite(out.view(torch.bfloat16).float()).all())
    finally:
        pool.close()


def test_host_side_checks_launch_nothing():
    torch = _torch()
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    pool = _pool(torch, H)
    try:
        q = torch.zeros(1 * 16 * 576 + 8, dtype=torch.int16, device="cuda")[1:1 + 16 * 576].view(1, 16, 576)
        out = torch.zeros(1, 16, 512, dtype=torch.int16, device="cuda")
        rows = torch.full((1, 128), -1, dtype=torch.int32, device="cuda")
        with pytest.raises(H.HisparseError) as e:       # q 2 bytes off a 16-byte boundary
            pool.sparse_mla_decode(0, q, rows, 0.05, out)
        assert e.value.status == INVALID
        with pytest.raises(H.HisparseError) as e:       # a page id outside the pool
            pool.set_pages(0, 0, block_table=[8])
        assert e.value.status == INVALID
        with pytest.raises(H.HisparseError) as e:       # a lease beyond the hot cap (1 page)
            pool.hot_lease(0, 0, [0, 1])
        assert e.value.status == INVALID
        assert pool.get_error() == 0                    # nothing reached the device
    finally:
        pool.close()


def test_selection_wait_timeout_then_recovery_on_the_same_pool():
    """The grid-wide top-K selection when one of its CTAs never arrives at a wait
    (hs_select_selftest: as when another stream holds an SM): the others give up
    after a second with HS_ERR_TIMEOUT and leave the token's scratch half used. The
    next call on the same pool, before the error is read, still selects exactly what
    the oracle selects (the scratch-free path); hs_get_error reports the timeout and
    clears the scratch; the call after that takes the grid-wide path again and the
    whole step (resolver, attention, page copies) matches the oracle. The local
    selection mode (hs_set_select_mode) selects the same tokens."""
    torch = _torch()
    from oracle.engine import OracleRun
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    from sparse_mla_kv_indexer_gb300 import schedule as S
    from sparse_mla_kv_indexer_gb300 import workload as W
    from sparse_mla_kv_indexer_gb300.driver import GpuRun
    from test_gpu_parity import check_step
    cfg = W.named_config("small_single")
    wl = W.Workload(cfg)
    sch = S.Schedule(cfg)
    plans = [sch.plan(s) for s in range(2)]
    oracle = OracleRun(wl, sch.setup)
    gpu = GpuRun(wl, sch.setup)
    try:
        check_step(cfg, wl, plans[0], oracle.step(plans[0]), gpu.step(plans[0]), gpu, oracle, exact_scores=False)
        o1 = oracle.step(plans[1])
        gpu.apply_tick(plans[1].tick)
        x = gpu.step_inputs(plans[1])
        dev = gpu.dev
        t = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in x.items() if k != "q_attn"}
        gpu.pool.append_rows(t["app_req"], t["app_pos"], t["kv_rows"], t["idx_keys"])
        n, K = len(plans[1].tokens), cfg.topk

        def select():
            out = torch.full((n, K), -7, dtype=torch.int32, device=dev)
            gpu.pool.indexer_topk(0, t["req"], t["limit"], t["q_idx"][0], t["w_idx"][0], out)
            torch.cuda.synchronize()
            return out.cpu().numpy()

        want = o1["topk"][0]
        assert np.array_equal(select(), want)                  # grid-wide path, scores left in the pool
        junk = torch.empty((n, K), dtype=torch.int32, device=dev)
        gpu.pool.select_selftest(t["limit"], junk)              # one CTA per token withholds its arrivals
        torch.cuda.synchronize()
        assert np.array_equal(select(), want)                  # half-used scratch: routed around
        assert gpu.pool.get_error() == TIMEOUT                 # reported once, scratch cleared
        assert np.array_equal(select(), want)                  # grid-wide path again
        assert gpu.pool.get_error() == 0
        gpu.pool.set_select_mode(H.SELECT_LOCAL)
        assert np.array_equal(select(), want)                  # no grid-wide waits at all
        gpu.pool.set_select_mode(H.SELECT_AUTO)
        with pytest.raises(H.HisparseError):
            gpu.pool.set_select_mode(7)
        # the rest of step 1 on the same pool, from its own selection
        topk = torch.from_numpy(select()).to(dev)
        rows = torch.empty_like(topk)
        plan_t = torch.empty((n, K, 4), dtype=torch.int32, device=dev)
        gpu.pool.resolve_topk(0, plans[1].step, t["req"], topk, rows, plan_t)
        qa = torch.from_numpy(np.ascontiguousarray(x["q_attn"][0]).view(np.int16)).to(dev)
        o = torch.empty((n, cfg.n_heads, 512), dtype=torch.int16, device=dev)
        gpu.pool.sparse_mla_decode(0, qa, rows, wl.sm_scale(), o)
        assert gpu.pool.get_error() == 0
        assert np.array_equal(rows.cpu().numpy(), o1["row_ids"][0])
        assert np.array_equal(plan_t.cpu().numpy()[..., 0], o1["kind"][0])
        go = o.view(torch.bfloat16).float().cpu().numpy()
        d = go - o1["o"][0]
        assert np.abs(d).max() <= 1e-2 and np.linalg.norm(d) / np.linalg.norm(o1["o"][0]) <= 5e-3
    finally:
        gpu.close()
