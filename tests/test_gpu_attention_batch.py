"""Sparse MLA decode with many query tokens (the one-CTA-per-token kernel), through
the C ABI, against the fp64 oracle ("Serving GLM-5.3 with PCP, DCP and Hybrid
HiSparse", footnote 1: 576-dim QK, 512-dim PV, every row serving all 64 heads).

The rows are built so that the kernel's online softmax must move its reference
maximum: for some tokens a row far above the others (a large multiple of one
head's query) sits in a late block of 128 rows, after the maximum of the early
blocks was taken. Other tokens have pads (-1) at the end, -1 scattered inside, or
no valid row at all (output zero, lse -inf).
Tolerance as for every attention test: max |err| <= 1e-2, relative L2 <= 5e-3.
"""
import numpy as np
import pytest

from oracle import attention
from sparse_mla_kv_indexer_gb300 import workload as W

pytestmark = pytest.mark.gpu

ATOL = 1e-2
REL_L2 = 5e-3


def _bf16(x):
    return W.round_to_bf16_bits(np.asarray(x, np.float32))


def test_many_token_attention_with_late_maximum_pads_and_empty_tokens():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    rng = np.random.default_rng(7)
    n, K, H_ = 24, 2048, 64
    n_rows = 64 * 64
    x = W.bf16_bits_to_f32(_bf16(rng.standard_normal((n_rows, 576), dtype=np.float32)))
    q_bits = _bf16(rng.standard_normal((n, H_, 576), dtype=np.float32))
    q = W.bf16_bits_to_f32(q_bits)
    row_ids = np.stack([rng.permutation(n_rows)[:K] for _ in range(n)]).astype(np.int32)
    # dominant rows: token i's row at position pos_i is its head (i % 64) query scaled
    # to a largest magnitude of 2.5, so that head's score for the row is about 17 above
    # the others (25 in log2 units, past the kernel's 2^8 lazy-rescale bound) while
    # the row's values stay where a bf16 output rounds them within the tolerance
    planted = {}
    for i, pos in [(0, K - 1), (1, 1900), (2, 0), (3, 777), (4, 1500), (5, 2047)]:
        r = int(row_ids[i, pos])
        qh = q[i, i % H_]
        x[r] = qh * (2.5 / np.abs(qh).max())
        planted[i] = r
    row_ids[6, 1000:] = -1                 # pads at the end
    row_ids[7, ::3] = -1                   # scattered -1
    row_ids[8, :] = -1                     # no valid row
    row_ids[9, :128] = -1                  # an empty first block
    rows = W.quantise_rows(W.bf16_bits_to_f32(_bf16(x)))
    pc = H.PoolConfig(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=64, n_heads=H_, topk=K, n_layers=1,
                      layers_per_indexer=1, num_pages=64, num_idx_pages=1, max_requests=1, max_ctx=4096,
                      max_q_per_req=1, hot_rows=4096, max_tokens=n, idx_format=H.IDX_INT8, host_pages=1)
    kv = [torch.from_numpy(rows.reshape(-1).copy()).cuda()]
    ix = [torch.zeros(64 * 128, dtype=torch.int8, device="cuda")]
    host = torch.zeros(64 * 656, dtype=torch.uint8, pin_memory=True)
    pool = H.Pool(pc, kv, ix, host)
    try:
        dq = torch.from_numpy(q_bits.view(np.int16).copy()).cuda()
        dr = torch.from_numpy(row_ids).cuda()
        out = torch.full((n, H_, 512), 0x7FC0, dtype=torch.int16, device="cuda")
        lse = torch.full((n, H_), 123.0, dtype=torch.float32, device="cuda")
        scale = 1.0 / np.sqrt(576.0)
        pool.sparse_mla_decode(0, dq, dr, scale, out, lse)
        assert pool.get_error() == 0
        o = out.view(torch.bfloat16).float().cpu().numpy()
        l = lse.cpu().numpy()
    finally:
        pool.close()
    for i in range(n):
        oo, ol = attention.sparse_mla_decode(q_bits[i], row_ids[i], rows, scale)
        if i == 8:
            assert np.all(o[i] == 0) and np.all(np.isneginf(l[i]))
            continue
        d = o[i] - oo
        err, rel = np.abs(d).max(), np.linalg.norm(d) / np.linalg.norm(oo)
        assert err <= ATOL and rel <= REL_L2, (i, err, rel)
        assert np.abs(l[i] - ol).max() <= 5e-3, (i, np.abs(l[i] - ol).max())
    for i, r in planted.items():   # the dominant row decides its head's output
        h = i % H_
        v = attention.dequant_rows(rows[r:r + 1])[0, :512]
        assert np.abs(o[i, h] - v).max() <= 2e-2 * max(1.0, np.abs(v).max()), i
