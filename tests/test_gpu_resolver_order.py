"""hs_resolve_topk with several query tokens per request: the union of the rows is
formed by merging the ascending top-K rows by rank, and rows in any other order
(entries shuffled, pads in the middle) are sorted whole instead. Two identical
pools resolve the same selections, one as hs_indexer_topk writes them (ascending,
pads at the end) and one with every row shuffled; the row ids and plan entries of
each (token, entry) and the hot-buffer decisions must agree, over steps with
resident rows, hits, misses and evictions, and the ascending pool must match the
oracle's resolver entry by entry."""
import numpy as np
import pytest

from oracle import resolver as OR

pytestmark = pytest.mark.gpu

K, T, CTX, RESIDENT, HOT_PAGES = 128, 4, 4096, 4, 10


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _pool(torch, H):
    n_pages = RESIDENT + HOT_PAGES
    pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=16, n_heads=16, topk=K,
                      n_layers=1, layers_per_indexer=1, num_pages=n_pages, num_idx_pages=64, max_requests=1,
                      max_ctx=CTX, max_q_per_req=T, hot_rows=HOT_PAGES * 64, max_tokens=T, idx_format=0,
                      host_pages=64)
    kv = [torch.zeros(n_pages * 64 * 656, dtype=torch.uint8, device="cuda")]
    ix = [torch.zeros(64 * 64 * 128, dtype=torch.int8, device="cuda")]
    host = torch.zeros(64 * 64 * 656, dtype=torch.uint8, pin_memory=True)
    pool = H.Pool(pc, kv, ix, host)
    pool.set_pages(0, 0, block_table=list(range(RESIDENT)) + [-1] * (CTX // 64 - RESIDENT),
                   host_pages=list(range(CTX // 64)))
    pool.hot_lease(0, 0, list(range(RESIDENT, RESIDENT + HOT_PAGES)))
    return pool


def _rows(rng, centre):
    """T ascending top-K rows around a shared centre (overlapping), some short."""
    rows = np.full((T, K), -1, np.int32)
    for j in range(T):
        n = K if j % 2 == 0 else K - 1 - 17 * j
        lo = max(0, centre - 300)
        rows[j, :n] = np.sort(rng.choice(np.arange(lo, min(CTX, lo + 600)), size=n, replace=False))
    return rows


def test_shuffled_rows_resolve_like_ascending_rows():
    torch = _torch()
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    rng = np.random.default_rng(5)
    pa, pb = _pool(torch, H), _pool(torch, H)
    bt = np.array(list(range(RESIDENT)) + [-1] * (CTX // 64 - RESIDENT))
    hot = OR.HotState()
    hot.lease(range(RESIDENT, RESIDENT + HOT_PAGES))
    try:
        req = torch.zeros(T, dtype=torch.int32, device="cuda")
        for step, centre in enumerate([400, 700, 2500, 720, 3600], start=1):
            rows = _rows(rng, centre)
            perm = np.stack([rng.permutation(K) for _ in range(T)])
            shuffled = np.take_along_axis(rows, perm, axis=1)
            out = []
            for pool, sel in ((pa, rows), (pb, shuffled)):
                topk = torch.from_numpy(np.ascontiguousarray(sel)).to("cuda")
                row_ids = torch.empty_like(topk)
                plan = torch.empty((T, K, 4), dtype=torch.int32, device="cuda")
                pool.resolve_topk(0, step, req, topk, row_ids, plan)
                torch.cuda.synchronize()
                assert pool.get_error() == 0, step
                out.append((row_ids.cpu().numpy(), plan.cpu().numpy()))
            (ra, pla), (rb, plb) = out
            o = OR.resolve(rows, bt, hot, step)
            assert np.array_equal(pla, np.stack([o.kind, o.slot, o.row_ids, o.evicted], axis=-1)), step
            assert np.array_equal(np.take_along_axis(ra, perm, axis=1), rb), step
            assert np.array_equal(np.take_along_axis(pla, perm[:, :, None], axis=1), plb), step
            kinds = set(pla[..., 0].ravel().tolist())
            if step == 1:
                assert {1, 3} <= kinds        # resident rows and misses
            if step == 4:
                assert 2 in kinds             # hits on rows copied at step 2
        ca, cb = pa.counters(), pb.counters()
        assert (ca.resident, ca.hits, ca.misses) == (cb.resident, cb.hits, cb.misses)
        assert ca.misses > HOT_PAGES * 64    # the hot buffer filled and slots were reused
    finally:
        pa.close()
        pb.close()
