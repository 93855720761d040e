"""The residency calls (hs_request_set_pages, hs_hot_lease) take the caller's host
arrays by value: the caller may overwrite them as soon as the call returns, even
when they are page-locked and the stream is still busy with earlier work, so that
the stream-ordered copies run long after the return. The device tables are read
back through the hot path: hs_replay_topk gives page * 64 + offset for a resident
token, and hs_resolve_topk places a missed token in a slot of the leased page."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _pool(torch, H):
    pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=16, n_heads=16, topk=128,
                      n_layers=1, layers_per_indexer=1, num_pages=8, num_idx_pages=64, max_requests=1,
                      max_ctx=4096, max_q_per_req=1, hot_rows=64, max_tokens=1, idx_format=0, host_pages=64)
    kv = [torch.zeros(8 * 64 * 656, dtype=torch.uint8, device="cuda")]
    ix = [torch.zeros(64 * 64 * 128, dtype=torch.int8, device="cuda")]
    host = torch.zeros(64 * 64 * 656, dtype=torch.uint8, pin_memory=True)
    return H.Pool(pc, kv, ix, host)


def _busy(torch):
    torch.cuda._sleep(200_000_000)   # ~0.1 s of device work ahead of the copies


def test_page_locked_arrays_may_be_reused_at_return():
    torch = _torch()
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    pool = _pool(torch, H)
    try:
        st = torch.cuda.current_stream().cuda_stream
        req = torch.zeros(1, dtype=torch.int32, device="cuda")
        topk = torch.arange(128, dtype=torch.int32, device="cuda").view(1, 128)   # tokens of pages 0 and 1
        rows = torch.empty_like(topk)

        # block table: pages 0 and 1 resident in pool pages 3 and 5
        bt = torch.full((64,), -1, dtype=torch.int32).pin_memory()
        bt[0], bt[1] = 3, 5
        _busy(torch)
        assert H.lib.hs_request_set_pages(pool.handle, 0, 0, 64, bt.data_ptr(), None, None, st) == 0
        bt.fill_(7)                    # overwritten while the copy is still queued
        pool.replay_topk(0, req, topk, rows)
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        want = np.concatenate([3 * 64 + np.arange(64), 5 * 64 + np.arange(64)])
        assert np.array_equal(rows.cpu().numpy()[0], want)

        # hot lease: page 2 of the request goes host-only, its misses land in leased pool page 6
        pool.set_pages(0, 2, block_table=[-1], host_pages=[0])
        lease = torch.tensor([6], dtype=torch.int32).pin_memory()
        _busy(torch)
        assert H.lib.hs_hot_lease(pool.handle, 0, 0, 1, lease.data_ptr(), st) == 0
        lease.fill_(4)
        topk2 = torch.full((1, 128), -1, dtype=torch.int32, device="cuda")
        topk2[0, :64] = torch.arange(128, 192, dtype=torch.int32, device="cuda")
        rows2 = torch.empty_like(topk2)
        pool.resolve_topk(0, 1, req, topk2, rows2)
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        got = rows2.cpu().numpy()[0]
        assert np.all(got[:64] // 64 == 6) and len(set(got[:64].tolist())) == 64
        assert np.all(got[64:] == -1)
    finally:
        pool.close()
