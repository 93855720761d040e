"""hs_link_probe, the host-link measurement aid: it must copy exactly the requested
single rows from pinned host memory (the miss-copy pattern whose rate the step
roofline charges miss bytes against) and reject bad sizes."""
import pytest

pytestmark = pytest.mark.gpu


def test_link_probe_copies_the_requested_rows():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    rows, rb = 1000, 656
    g = torch.Generator().manual_seed(3)
    host = torch.randint(0, 256, (rows * rb,), generator=g, dtype=torch.uint8).pin_memory()
    want = [5, 999, 0, 5, -1, 1000, 17]
    src = torch.tensor(want, dtype=torch.int64, device="cuda")
    dst = torch.full((len(want) * rb,), 7, dtype=torch.uint8, device="cuda")
    H.link_probe(host, rb, src, dst)
    torch.cuda.synchronize()
    d = dst.cpu().view(len(want), rb)
    h = host.view(rows, rb)
    for i, r in enumerate(want):
        if 0 <= r < rows:
            assert torch.equal(d[i], h[r]), i
        else:   # an index outside the host rows leaves its destination unchanged
            assert bool((d[i] == 7).all()), i
    with pytest.raises(H.HisparseError):
        H.link_probe(host, 650, src, dst)     # row size not a multiple of 16
