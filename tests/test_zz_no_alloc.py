"""The no-allocation indexer entry point against the regular one.

hs_indexer_topk_noalloc serves callers that cannot allocate device memory (an
engine that has handed all free HBM to its KV pool, or code running during
stream capture): its score scratch is a fixed array inside the library instead
of pool-owned memory. This file is collected last so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

from sparse_mla_kv_indexer_gb300 import schedule as S
from sparse_mla_kv_indexer_gb300 import workload as W

pytestmark = pytest.mark.gpu


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def test_noalloc_matches_regular_on_two_calls_in_a_row():
    torch = _torch()
    from sparse_mla_kv_indexer_gb300.driver import GpuRun
    cfg = W.named_config("small_batch")          # 4 requests x 4 query tokens, K = 512
    wl = W.Workload(cfg)
    sch = S.Schedule(cfg)
    gpu = GpuRun(wl, sch.setup)
    try:
        dev = gpu.dev
        for s in range(2):                          # two calls in a row, different steps
            plan = sch.plan(s)
            gpu.apply_tick(plan.tick)
            x = gpu.step_inputs(plan)
            n, K = len(plan.tokens), cfg.topk
            req = torch.from_numpy(x["req"]).to(dev)
            limit = torch.from_numpy(x["limit"]).to(dev)
            gpu.pool.append_rows(torch.from_numpy(x["app_req"]).to(dev), torch.from_numpy(x["app_pos"]).to(dev),
                                 torch.from_numpy(x["kv_rows"]).to(dev), torch.from_numpy(x["idx_keys"]).to(dev))
            for g in range(cfg.n_groups):
                q = torch.from_numpy(np.ascontiguousarray(x["q_idx"][g])).to(dev)
                w = torch.from_numpy(np.ascontiguousarray(x["w_idx"][g])).to(dev)
                ref = torch.full((n, K), -7, dtype=torch.int32, device=dev)
                got = torch.full((n, K), -7, dtype=torch.int32, device=dev)
                gpu.pool.indexer_topk(g, req, limit, q, w, ref)
                gpu.pool.indexer_topk_noalloc(g, req, limit, q, w, got)
                assert gpu.pool.get_error() == 0
                # top-K is integer work: the two entry points agree exactly
                assert torch.equal(got, ref), (s, g)
                assert int((ref >= 0).sum()) == sum(min(K, t.limit) for t in plan.tokens)
    finally:
        gpu.close()


def test_noalloc_rejects_requests_beyond_its_scratch():
    torch = _torch()
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    max_ctx = 1 << 20                               # 4 tokens x 1M positions > 2^21 scores
    pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=16, n_heads=16, topk=256,
                      n_layers=1, layers_per_indexer=1, num_pages=4, num_idx_pages=4, max_requests=1,
                      max_ctx=max_ctx, max_q_per_req=4, hot_rows=512, max_tokens=4, idx_format=0, host_pages=1)
    kv = [torch.zeros(4 * 64 * 656, dtype=torch.uint8, device="cuda")]
    ix = [torch.zeros(4 * 64 * 128, dtype=torch.int8, device="cuda")]
    host = torch.zeros(64 * 656, dtype=torch.uint8, pin_memory=True)
    pool = H.Pool(pc, kv, ix, host)
    try:
        pool.set_pages(0, 0, idx_pages=[0, 1])
        req = torch.zeros(4, dtype=torch.int32, device="cuda")
        limit = torch.full((4,), 100, dtype=torch.int32, device="cuda")
        q = torch.zeros((4, 16, 128), dtype=torch.int8, device="cuda")
        w = torch.ones((4, 16), dtype=torch.int8, device="cuda")
        out = torch.empty((4, 256), dtype=torch.int32, device="cuda")
        with pytest.raises(H.HisparseError) as e:
            pool.indexer_topk_noalloc(0, req, limit, q, w, out)
        assert e.value.status == 9
        H.lib.hs_status_string.restype = ctypes.c_char_p
        assert b"scratch" in H.lib.hs_status_string(9)
        # within the limit (1 token x 1M positions = 2^20 scores) the call is accepted
        pool.indexer_topk_noalloc(0, req[:1], limit[:1], q[:1], w[:1], out[:1])
        assert pool.get_error() == 0
        assert out[0, :100].cpu().tolist() == list(range(100))
    finally:
        pool.close()
