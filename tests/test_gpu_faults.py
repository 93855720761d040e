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
