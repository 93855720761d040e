"""Pool limits enforced by hs_pool_init on a GPU: the longest context (HS_MAX_CTX)
is accepted, one page more is rejected."""
import pytest

pytestmark = pytest.mark.gpu


def _pool(torch, H, max_ctx):
    pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=16, n_heads=16, topk=256,
                      n_layers=1, layers_per_indexer=1, num_pages=4, num_idx_pages=4, max_requests=1,
                      max_ctx=max_ctx, max_q_per_req=1, hot_rows=512, max_tokens=1, idx_format=0, host_pages=1)
    kv = [torch.zeros(4 * 64 * 656, dtype=torch.uint8, device="cuda")]
    ix = [torch.zeros(4 * 64 * 128, dtype=torch.int8, device="cuda")]
    host = torch.zeros(64 * 656, dtype=torch.uint8, pin_memory=True)
    return H.Pool(pc, kv, ix, host)


def test_longest_context_accepted_and_one_page_more_rejected():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    pool = _pool(torch, H, H.MAX_CTX)
    pool.close()
    with pytest.raises(H.HisparseError) as e:
        _pool(torch, H, H.MAX_CTX + 128)
    assert e.value.status == 1   # HS_ERR_INVALID
