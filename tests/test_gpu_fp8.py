"""FP8 index keys (the pages' key record: 128 e4m3 values and an fp32 scale,
"Serving GLM-5.3 with PCP, DCP and Hybrid HiSparse", footnote 3) through
hs_indexer_topk_fp8, against the fp64 oracle.

Scores: the GPU contracts e4m3 keys and queries on the tensor cores (exact
products, fp32 sums of 128) and sums 64 weighted heads in fp32; its error is a
small multiple of 2^-24 of the key's L1 magnitude
    B_t = scale_t * sum_h |w_h| * sum_d |q_hd| |k_td|,
so every score must lie within TOL * B_t of the oracle's. Top-K: the sets must
be equal except for tokens whose oracle score is within 2 * TOL * B_t of the
oracle's K-th score (a near-tie the fp32 rounding may order either way). The
resolver and attention then take the oracle's selection (uploaded to the GPU), so
both sides stay in the same residency state through every step, and the rest of
the step is compared as for int8 keys.
"""
import dataclasses

import numpy as np
import pytest

from oracle import formats
from test_gpu_parity import _setup, check_step

pytestmark = pytest.mark.gpu

TOL = 2.0 ** -14


def _l1_bound(qc, w, rows):
    q = np.abs(formats.e4m3_to_f64(qc))
    k = np.abs(formats.e4m3_to_f64(rows[:, :128]))
    scale = np.ascontiguousarray(rows[:, 128:132]).view("<f4").reshape(-1).astype(np.float64)
    return scale * ((k @ q.T) @ np.abs(np.asarray(w, np.float64)))


def run_fp8_parity(cfg, wl, plans, oracle, gpu):
    """Every step: scores within the bound, the GPU's own top-K equal to the oracle's
    except at near-ties, and (from the oracle's selection) plans, rows, attention and
    page copies as for int8 keys. Returns the number of selections that differed."""
    K = cfg.topk
    differing = 0
    for plan in plans:
        o = oracle.step(plan)
        g = gpu.step(plan, topk_in=o["topk"])
        assert g["status"] == 0, g["status"]
        for grp in range(cfg.n_groups):
            for i, t in enumerate(plan.tokens):
                qc, w = wl.idx_queries_fp8(t.req, grp, plan.step)
                j = i % cfg.t_q
                b = _l1_bound(qc[j], w[j], oracle.keys_of(grp, t.req, t.limit))
                so = o["scores"][grp][i]
                sg = g["scores"][grp][i, :t.limit].astype(np.float64)
                assert np.all(np.abs(sg - so) <= TOL * b + 1e-30), (plan.step, grp, i)
                ot, gt = o["topk"][grp][i], g["topk_own"][grp][i]
                assert np.all(np.diff(gt[gt >= 0]) > 0) and (gt >= 0).sum() == min(K, t.limit)
                if not np.array_equal(ot, gt):
                    differing += 1
                    kth = np.sort(so)[::-1][min(K, t.limit) - 1]
                    for tok in set(ot[ot >= 0].tolist()) ^ set(gt[gt >= 0].tolist()):
                        assert abs(so[tok] - kth) <= 2 * TOL * b[tok], (plan.step, grp, i, tok)
        check_step(cfg, wl, plan, o, g, gpu, oracle, exact_scores=False)
    return differing


@pytest.mark.parametrize("name", ["tiny_fp8", "small_batch_fp8", "small_groups_fp8"])
def test_fp8_indexer_parity(name):
    cfg, wl, plans, oracle, gpu = _setup(name)
    try:
        run_fp8_parity(cfg, wl, plans, oracle, gpu)
    finally:
        gpu.close()


def test_fp8_indexer_parity_full_size_128k():
    """The 128K shape with FP8 keys, two steps, in the launch configuration the bench times."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from oracle.engine import OracleRun
    from sparse_mla_kv_indexer_gb300 import schedule as S
    from sparse_mla_kv_indexer_gb300 import workload as W
    from sparse_mla_kv_indexer_gb300.driver import GpuRun
    cfg = dataclasses.replace(W.named_config("ctx128k_fp8"), steps=2)
    wl = W.Workload(cfg)
    sch = S.Schedule(cfg)
    plans = [sch.plan(s) for s in range(cfg.steps)]
    oracle = OracleRun(wl, sch.setup, keep_scores=True)
    gpu = GpuRun(wl, sch.setup, keep_scores=True)
    try:
        run_fp8_parity(cfg, wl, plans, oracle, gpu)
    finally:
        gpu.close()


def test_each_indexer_entry_rejects_the_other_key_format():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    for fmt in (H.IDX_INT8, H.IDX_FP8):
        pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=16, n_heads=16, topk=256,
                          n_layers=1, layers_per_indexer=1, num_pages=4, num_idx_pages=4, max_requests=1,
                          max_ctx=256, max_q_per_req=1, hot_rows=512, max_tokens=1, idx_format=fmt, host_pages=1)
        kv = [torch.zeros(4 * 64 * 656, dtype=torch.uint8, device="cuda")]
        ix = [torch.zeros(4 * H.IDX_FP8_PAGE_BYTES, dtype=torch.uint8, device="cuda")]
        host = torch.zeros(64 * 656, dtype=torch.uint8, pin_memory=True)
        pool = H.Pool(pc, kv, ix, host)
        try:
            req = torch.zeros(1, dtype=torch.int32, device="cuda")
            lim = torch.full((1,), 10, dtype=torch.int32, device="cuda")
            q = torch.zeros((1, 16, 128), dtype=torch.int8, device="cuda")
            topk = torch.empty((1, 256), dtype=torch.int32, device="cuda")
            with pytest.raises(H.HisparseError) as e:
                if fmt == H.IDX_INT8:
                    pool.indexer_topk_fp8(0, req, lim, q.view(torch.uint8), torch.ones((1, 16), device="cuda"), topk)
                else:
                    pool.indexer_topk(0, req, lim, q, torch.ones((1, 16), dtype=torch.int8, device="cuda"), topk)
            assert e.value.status == 1
        finally:
            pool.close()
