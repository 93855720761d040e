"""The seeded input generator: encodings match library conversions, seeds are stable."""
import numpy as np
import pytest

from sparse_mla_kv_indexer_gb300 import workload as W


def test_e4m3_encoder_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-460, 460, 20000), rng.uniform(-0.02, 0.02, 20000),
                        np.array([0.0, -0.0, 448.0, -448.0, 2 ** -9, 2 ** -10, 3 * 2 ** -11])]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(W.encode_e4m3(x), ref)


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    y = np.random.default_rng(1).standard_normal(100000).astype(np.float32) * 7
    ref = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.round_to_bf16_bits(y), ref)


def test_inputs_are_deterministic_and_shaped():
    cfg = W.named_config("tiny")
    a, b = W.Workload(cfg), W.Workload(cfg)
    assert np.array_equal(a.kv_rows(0, 0), b.kv_rows(0, 0))
    assert a.kv_rows(0, 0).shape == (cfg.final_len(0), 656)
    assert a.idx_keys(0, 0).dtype == np.int8 and np.abs(a.idx_keys(0, 0).astype(int)).max() <= 127
    w = a.idx_weights(0, 0)
    assert w.min() >= 1 and w.max() <= 16
    q = a.idx_queries(0, 0, 3)
    assert q.shape == (1, 16, 128)
    assert a.attn_queries(0, 0, 2).shape == (1, 16, 576)


def test_clusters_planted_and_targeted():
    cfg = W.named_config("small_single")
    wl = W.Workload(cfg)
    cl = wl.clusters(0)
    assert len(cl.starts) == cfg.n_clusters
    ends = cl.starts + cfg.cluster_len
    assert (cl.starts[1:] >= ends[:-1]).all()
    k = wl.idx_keys(0, 0).astype(np.int64)
    s = int(cl.starts[0])
    inside = (k[s:s + cfg.cluster_len] * cl.dirs[0]).mean()
    outside = (k[:s] * cl.dirs[0]).mean() if s else 0.0
    assert inside > 60 and abs(outside) < 10
