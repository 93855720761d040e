"""Top-K selection for many query tokens (the chunked selection: every token's keys in
8,192-key chunks spread over the GPU), through hs_indexer_topk, against the oracle's
full sort (vLLM blog Part 1, "Sparsity when you need it": the top-K of the exact
int64 scores, ties to the lower token index, ascending token order).

36 query tokens (9 requests x 4) with ragged limits: below K, exactly K, K + 1, one
and two keys past a chunk boundary, a full chunk, and long ones. The key caches make
the threshold bucket small (random keys: the chunks emit at their offsets), crowded
(three distinct scores: the bucket overflows the 4,096-key list and the token is
selected in full) and fully tied (every score equal, or every score zero). Each call
runs twice, so the second one starts from the sums the first one cleared, and is
checked, for the first 16 tokens, against the no-allocation entry point (the cluster
selection) too.
"""
import numpy as np
import pytest

from oracle import indexer as OI

pytestmark = pytest.mark.gpu

CTX = 131072
K = 2048
HI = 16
N_REQ, T_Q = 9, 4
NOALLOC_TOKENS = (1 << 21) // CTX
LIMITS = [CTX, 1500, K, K + 1, 8193, 8194, 8192, 16385, CTX - 77, 100000, 65536, 3,
          CTX, CTX - 1, 40000, 2 * K, 24577, 9000, 120000, 70001, 1, 50000, 8191, 33333,
          CTX, 90000, 12345, K - 1, 131000, 60000, 16384, 77777, 100, 110000, 20000, CTX]


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _keys(kind, rng):
    if kind in ("equal", "zero"):
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
            q = np.abs(q)
    w = rng.integers(1, 17, size=(n_tok, HI)).astype(np.int8)
    return q, w


@pytest.mark.parametrize("kind", ["random", "three", "equal", "zero"])
def test_many_token_selection_matches_full_sort(kind):
    torch = _torch()
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    rng = np.random.default_rng({"random": 21, "three": 22, "equal": 23, "zero": 24}[kind])
    keys = _keys(kind, rng)
    n_tok = N_REQ * T_Q
    assert len(LIMITS) == n_tok
    pages = CTX // 64
    pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=HI, n_heads=16, topk=K,
                      n_layers=1, layers_per_indexer=1, num_pages=4, num_idx_pages=pages, max_requests=N_REQ,
                      max_ctx=CTX, max_q_per_req=T_Q, hot_rows=4096, max_tokens=n_tok, idx_format=H.IDX_INT8,
                      host_pages=1)
    kv = [torch.zeros(4 * 64 * 656, dtype=torch.uint8, device="cuda")]
    ix = [torch.from_numpy(np.ascontiguousarray(keys).reshape(-1)).to("cuda")]
    host = torch.zeros(64 * 656, dtype=torch.uint8, pin_memory=True)
    pool = H.Pool(pc, kv, ix, host)
    try:
        for r in range(N_REQ):
            pool.set_pages(r, 0, idx_pages=list(range(pages)))
        reqs = [i // T_Q for i in range(n_tok)]
        q, w = _queries(kind, n_tok, rng)
        want = np.stack([OI.topk(OI.scores(q[i], w[i], keys[:LIMITS[i]]), K) for i in range(n_tok)])
        d_req = torch.tensor(reqs, dtype=torch.int32, device="cuda")
        d_lim = torch.tensor(LIMITS, dtype=torch.int32, device="cuda")
        d_q = torch.from_numpy(q.reshape(n_tok, -1)).to("cuda")
        d_w = torch.from_numpy(w).to("cuda")
        for entry in ("regular", "noalloc"):
            # the no-allocation entry's fixed scratch holds 2^21 scores: 16 tokens at this context
            m = n_tok if entry == "regular" else NOALLOC_TOKENS
            for rep in range(2):
                out = torch.full((m, K), -7, dtype=torch.int32, device="cuda")
                if entry == "regular":
                    pool.indexer_topk(0, d_req, d_lim, d_q, d_w, out)
                else:
                    pool.indexer_topk_noalloc(0, d_req[:m], d_lim[:m], d_q[:m], d_w[:m], out)
                torch.cuda.synchronize()
                assert pool.get_error() == 0, (kind, entry, rep)
                got = out.cpu().numpy()
                for i in range(m):
                    assert np.array_equal(got[i], want[i]), (kind, entry, rep, i, LIMITS[i])
        if kind in ("equal", "zero"):
            for i in range(n_tok):   # all scores tie: the K lowest token ids
                m = min(K, LIMITS[i])
                assert np.array_equal(want[i][:m], np.arange(m)), i
    finally:
        pool.close()


# ---- FP8 keys: the same chunked selection over order-preserving keys of fp32 scores ----
# Small integer key and query values and power-of-two scales keep every score exact in
# fp32 (see test_gpu_select.py), so the top-K must equal the fp64 oracle's, ties included.

@pytest.mark.parametrize("kind", ["random", "three"])
def test_many_token_fp8_selection_matches_full_sort(kind):
    torch = _torch()
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    from test_gpu_select import _fp8_keys, _fp8_pages, _fp8_queries
    rng = np.random.default_rng({"random": 31, "three": 32}[kind])
    codes, scale = _fp8_keys(kind, rng)
    codes, scale = np.ascontiguousarray(codes[:CTX]), np.ascontiguousarray(scale[:CTX])
    n_tok = N_REQ * T_Q
    pages = CTX // 64
    pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=HI, n_heads=16, topk=K,
                      n_layers=1, layers_per_indexer=1, num_pages=4, num_idx_pages=pages, max_requests=N_REQ,
                      max_ctx=CTX, max_q_per_req=T_Q, hot_rows=4096, max_tokens=n_tok, idx_format=H.IDX_FP8,
                      host_pages=1)
    kv = [torch.zeros(4 * 64 * 656, dtype=torch.uint8, device="cuda")]
    ix = [torch.from_numpy(_fp8_pages(codes, scale)).to("cuda")]
    host = torch.zeros(64 * 656, dtype=torch.uint8, pin_memory=True)
    pool = H.Pool(pc, kv, ix, host)
    try:
        for r in range(N_REQ):
            pool.set_pages(r, 0, idx_pages=list(range(pages)))
        reqs = [i // T_Q for i in range(n_tok)]
        qc, w = _fp8_queries(kind, n_tok, rng)
        so = [OI.scores_fp8(qc[i], w[i], codes[:LIMITS[i]], scale[:LIMITS[i]]) for i in range(n_tok)]
        want = np.stack([OI.topk_real(s, K) for s in so])
        d_req = torch.tensor(reqs, dtype=torch.int32, device="cuda")
        d_lim = torch.tensor(LIMITS, dtype=torch.int32, device="cuda")
        d_q = torch.from_numpy(qc.reshape(n_tok, -1)).to("cuda")
        d_w = torch.from_numpy(w).to("cuda")
        sc = torch.full((n_tok, CTX), float("nan"), dtype=torch.float32, device="cuda")
        for rep in range(2):
            out = torch.full((n_tok, K), -7, dtype=torch.int32, device="cuda")
            pool.indexer_topk_fp8(0, d_req, d_lim, d_q, d_w, out, sc)
            torch.cuda.synchronize()
            assert pool.get_error() == 0, (kind, rep)
            got = out.cpu().numpy()
            for i in range(n_tok):
                assert np.array_equal(got[i], want[i]), (kind, rep, i, LIMITS[i])
    finally:
        pool.close()
