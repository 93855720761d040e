"""Top-K selection edge cases through hs_indexer_topk, against the oracle's full sort.

Key caches are built so that the scores are crowded: every key equal (all scores
tie, the K lowest token ids win), all scores zero, three distinct scores over
262,144 tokens, and plain random keys. Each runs with 1 and 2 query tokens (the
wide selection, one group of CTAs per token over the whole GPU; with one token the
scoring kernel fills the selection's first histogram), with 8 query tokens (the
cluster selection) and through hs_indexer_topk_noalloc (the cluster selection, no
pool scratch); ragged limits and limits below K are included, and a one-token call
with every token selected is followed by a full one (its sums must have been cleared).
The oracle's top-K (vLLM blog Part 1, "Sparsity when you need it"; ties to the
lower token index) is a full sort of the exact int64 scores.
"""
import numpy as np
import pytest

from oracle import indexer as OI
from sparse_mla_kv_indexer_gb300 import workload as W

pytestmark = pytest.mark.gpu

CTX = 262144
K = 2048
HI = 16


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _keys(kind, rng):
    if kind == "equal":
        k = rng.integers(1, 40, size=128, dtype=np.int64)
        return np.broadcast_to(k, (CTX, 128)).astype(np.int8)
    if kind == "three":
        base = rng.integers(-60, 60, size=(3, 128), dtype=np.int64)
        return base[rng.integers(0, 3, size=CTX)].astype(np.int8)
    return np.clip(np.rint(rng.normal(0, 32, size=(CTX, 128))), -127, 127).astype(np.int8)


def _queries(kind, n_tok, rng):
    if kind == "zero":
        q = np.zeros((n_tok, HI, 128), np.int8)
    else:
        q = np.clip(np.rint(rng.normal(0, 32, size=(n_tok, HI, 128))), -127, 127).astype(np.int8)
        if kind == "equal":
            q = np.abs(q)           # positive dot products with the all-positive key
    w = rng.integers(1, 17, size=(n_tok, HI)).astype(np.int8)
    return q, w


# (request of each token, limit of each token), run in this order
BATCHES = [
    ([0], [CTX]),
    ([0], [1500]),
    ([0], [CTX - 77]),
    ([0, 1], [CTX - 1000, 131073]),
    ([0, 0, 0, 0, 1, 1, 1, 1], [200001, 200002, 200003, 200004, 1000, 1001, K + 1, CTX]),
]


@pytest.mark.parametrize("kind", ["equal", "zero", "three", "random"])
def test_selection_matches_full_sort(kind):
    torch = _torch()
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    rng = np.random.default_rng({"equal": 1, "zero": 2, "three": 3, "random": 4}[kind])
    keys = _keys("equal" if kind == "zero" else kind, rng)
    pages = CTX // 64
    pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=HI, n_heads=16, topk=K,
                      n_layers=1, layers_per_indexer=1, num_pages=4, num_idx_pages=pages, max_requests=2,
                      max_ctx=CTX, max_q_per_req=4, hot_rows=4096, max_tokens=8, idx_format=H.IDX_INT8,
                      host_pages=1)
    kv = [torch.zeros(4 * 64 * 656, dtype=torch.uint8, device="cuda")]
    ix = [torch.from_numpy(np.ascontiguousarray(keys).reshape(-1)).to("cuda")]
    host = torch.zeros(64 * 656, dtype=torch.uint8, pin_memory=True)
    pool = H.Pool(pc, kv, ix, host)
    try:
        for r in range(2):
            pool.set_pages(r, 0, idx_pages=list(range(pages)))
        for reqs, limits in BATCHES:
            n_tok = len(reqs)
            q, w = _queries(kind, n_tok, rng)
            want = np.stack([OI.topk(OI.scores(q[i], w[i], keys[:limits[i]]), K) for i in range(n_tok)])
            d_req = torch.tensor(reqs, dtype=torch.int32, device="cuda")
            d_lim = torch.tensor(limits, dtype=torch.int32, device="cuda")
            d_q = torch.from_numpy(q.reshape(n_tok, -1)).to("cuda")
            d_w = torch.from_numpy(w).to("cuda")
            for entry in ("regular", "noalloc"):
                out = torch.full((n_tok, K), -7, dtype=torch.int32, device="cuda")
                for _ in range(2):   # the wide selection clears its scratch for the next call
                    if entry == "regular":
                        pool.indexer_topk(0, d_req, d_lim, d_q, d_w, out)
                    else:
                        pool.indexer_topk_noalloc(0, d_req, d_lim, d_q, d_w, out)
                    torch.cuda.synchronize()
                    assert pool.get_error() == 0, (kind, n_tok, entry)
                    got = out.cpu().numpy()
                    for i in range(n_tok):
                        assert np.array_equal(got[i], want[i]), (kind, n_tok, entry, i)
            if kind == "equal":
                for i in range(n_tok):   # all scores tie: the K lowest token ids
                    m = min(K, limits[i])
                    assert np.array_equal(want[i][:m], np.arange(m)), i
    finally:
        pool.close()


# ---- FP8 keys (128 e4m3 values and an fp32 scale per key) ------------------------
#
# Every key value, query value and head weight is a small integer (e4m3 holds the
# integers up to 16 exactly) and every scale a power of two, so each score
# (|sum_d q k| <= 128 * 64 per head, 16 heads, |w| <= 16, below 2^24) is exact in
# fp32 whatever the order of the sums: the scores and the top-K must equal the fp64
# oracle's exactly, ties included. All queries zero makes every head product a
# signed zero (-0 where a key value is negative); the score of such a token is 0
# and ties with the +0 scores.

def _fp8_keys(kind, rng):
    if kind == "equal":
        k = np.broadcast_to(rng.integers(1, 9, size=128).astype(np.float32), (CTX, 128))
        scale = np.ones(CTX, np.float32)
    elif kind == "three":
        base = rng.integers(-8, 9, size=(3, 128)).astype(np.float32)
        k = base[rng.integers(0, 3, size=CTX)]
        scale = np.ones(CTX, np.float32)
    else:   # "zero" and "random": mixed signs, scales 1/2, 1 or 2
        k = rng.integers(-8, 9, size=(CTX, 128)).astype(np.float32)
        scale = np.float32(2.0) ** rng.integers(-1, 2, size=CTX).astype(np.float32)
    return W.encode_e4m3(np.ascontiguousarray(k)), scale.astype(np.float32)


def _fp8_queries(kind, n_tok, rng):
    if kind == "zero":
        q = np.zeros((n_tok, HI, 128), np.float32)
    else:
        q = rng.integers(-8, 9, size=(n_tok, HI, 128)).astype(np.float32)
        if kind == "equal":
            q = np.abs(q)
    w = rng.integers(1, 17, size=(n_tok, HI)).astype(np.float32)
    if kind == "random":
        w *= np.where(rng.random((n_tok, HI)) < 0.25, -1.0, 1.0).astype(np.float32)   # negative scores too
    return W.encode_e4m3(q), w


def _fp8_pages(codes, scale):
    n = codes.shape[0] // 64
    page = np.empty((n, 64 * 128 + 64 * 4), np.uint8)
    page[:, :64 * 128] = codes.reshape(n, 64 * 128)
    page[:, 64 * 128:] = scale.astype("<f4").view(np.uint8).reshape(n, 64 * 4)
    return page.reshape(-1)


@pytest.mark.parametrize("kind", ["equal", "zero", "three", "random"])
def test_fp8_selection_matches_full_sort(kind):
    torch = _torch()
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    rng = np.random.default_rng({"equal": 11, "zero": 12, "three": 13, "random": 14}[kind])
    codes, scale = _fp8_keys(kind, rng)
    pages = CTX // 64
    pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=HI, n_heads=16, topk=K,
                      n_layers=1, layers_per_indexer=1, num_pages=4, num_idx_pages=pages, max_requests=2,
                      max_ctx=CTX, max_q_per_req=4, hot_rows=4096, max_tokens=8, idx_format=H.IDX_FP8,
                      host_pages=1)
    kv = [torch.zeros(4 * 64 * 656, dtype=torch.uint8, device="cuda")]
    ix = [torch.from_numpy(_fp8_pages(codes, scale)).to("cuda")]
    host = torch.zeros(64 * 656, dtype=torch.uint8, pin_memory=True)
    pool = H.Pool(pc, kv, ix, host)
    try:
        for r in range(2):
            pool.set_pages(r, 0, idx_pages=list(range(pages)))
        for reqs, limits in BATCHES:
            n_tok = len(reqs)
            qc, w = _fp8_queries(kind, n_tok, rng)
            so = [OI.scores_fp8(qc[i], w[i], codes[:limits[i]], scale[:limits[i]]) for i in range(n_tok)]
            want = np.stack([OI.topk_real(s, K) for s in so])
            d_req = torch.tensor(reqs, dtype=torch.int32, device="cuda")
            d_lim = torch.tensor(limits, dtype=torch.int32, device="cuda")
            d_q = torch.from_numpy(qc.reshape(n_tok, -1)).to("cuda")
            d_w = torch.from_numpy(w).to("cuda")
            out = torch.full((n_tok, K), -7, dtype=torch.int32, device="cuda")
            sc = torch.full((n_tok, CTX), float("nan"), dtype=torch.float32, device="cuda")
            for _ in range(2):   # the wide selection clears its scratch for the next call
                pool.indexer_topk_fp8(0, d_req, d_lim, d_q, d_w, out, sc)
                torch.cuda.synchronize()
                assert pool.get_error() == 0, (kind, n_tok)
                got, gs = out.cpu().numpy(), sc.cpu().numpy()
                for i in range(n_tok):
                    assert np.array_equal(gs[i, :limits[i]].astype(np.float64), so[i]), (kind, n_tok, i)
                    assert np.array_equal(got[i], want[i]), (kind, n_tok, i)
            if kind in ("equal", "zero"):
                for i in range(n_tok):   # all scores tie: the K lowest token ids
                    m = min(K, limits[i])
                    assert np.array_equal(want[i][:m], np.arange(m)), i
    finally:
        pool.close()
