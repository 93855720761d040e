"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every test here checks the oracle against something other than itself: numbers
printed by the pages, hand-worked cases, brute force on tiny inputs, library
routines for special cases, closed forms and invariants.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import attention, closed_forms, formats, indexer, resolver
from sparse_mla_kv_indexer_gb300 import workload as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# element formats
# ----------------------------------------------------------------------------
def test_e4m3_known_codes():
    # OCP OFP8 E4M3: bias 7, max finite 448, min normal 2^-6, min subnormal 2^-9
    codes = np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x40, 0x7E, 0xB8, 0xFE, 0x80], np.uint8)
    want = [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 2.0, 448.0, -1.0, -448.0, -0.0]
    got = formats.e4m3_to_f64(codes)
    assert np.array_equal(got, np.array(want))
    assert np.isnan(formats.e4m3_to_f64(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_matches_torch_all_codes():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = formats.e4m3_to_f64(codes)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])
    assert (np.isnan(ref) == np.isnan(got)).all()


def test_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=5000).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]          # finite values only
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(formats.bf16_to_f64(bits), ref)


def test_row_decode_hand_built():
    row = np.zeros((1, 656), np.uint8)
    row[0, 0] = 0x38          # 1.0 in group 0
    row[0, 200] = 0xC0        # -2.0 in group 1
    row[0, 511] = 0x01        # 2^-9 in group 3
    row[0, 512:528] = np.array([2.0, 0.5, 1.0, 8.0], "<f4").view(np.uint8)
    row[0, 528:530] = np.array([0x3F80], "<u2").view(np.uint8)   # rope[0] = 1.0
    row[0, 654:656] = np.array([0xC040], "<u2").view(np.uint8)   # rope[63] = -3.0
    x = formats.dequant_rows(row)[0]
    assert x[0] == 2.0 and x[200] == -1.0 and x[511] == 8.0 * 2.0 ** -9
    assert x[512] == 1.0 and x[575] == -3.0
    assert np.count_nonzero(x) == 5


def test_quantise_then_decode_within_e4m3_bound():
    # round-to-nearest e4m3 has relative error <= 2^-4 on normals and absolute
    # error <= 2^-10 * scale on subnormals; rope bf16 is carried exactly.
    rng = np.random.default_rng(2)
    x = W.bf16_bits_to_f32(W.round_to_bf16_bits(rng.standard_normal((64, 576), dtype=np.float32)))
    rows = W.quantise_rows(x)
    y = formats.dequant_rows(rows)
    scale = np.ascontiguousarray(rows[:, 512:528]).view("<f4").astype(np.float64)
    s = np.repeat(scale, 128, axis=1)
    err = np.abs(y[:, :512] - x[:, :512])
    bound = np.maximum(np.abs(x[:, :512]) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-6)
    assert (err <= bound).all()
    # the group maximum maps to exactly 448 * scale
    g = np.abs(x[:, :512]).reshape(64, 4, 128).max(axis=2)
    assert np.allclose(g, 448 * scale, rtol=1e-6)
    assert np.array_equal(y[:, 512:], x[:, 512:].astype(np.float64))


# ----------------------------------------------------------------------------
# indexer scores
# ----------------------------------------------------------------------------
def _dense(spec):
    v = np.zeros(128, np.int64)
    if spec == "all127":
        v[:] = 127
    else:
        for d, x in spec.items():
            v[int(d)] = x
    return v


def test_scores_hand_worked():
    g = _load("indexer_hand.json")
    q = np.stack([_dense(s) for s in g["q"]]).astype(np.int8)
    keys = np.stack([_dense(s) for s in g["keys"]]).astype(np.int8)
    w = np.array(g["w"], np.int8)
    assert indexer.scores(q, w, keys).tolist() == g["scores"]


def test_scores_max_case():
    g = _load("indexer_hand.json")
    q = np.full((64, 128), 127, np.int8)
    w = np.full(64, 16, np.int8)
    k = np.full((1, 128), 127, np.int8)
    assert int(indexer.scores(q, w, k)[0]) == g["max_case_score"]


def test_scores_brute_force_loops():
    rng = np.random.default_rng(3)
    h, n = 5, 17
    q = rng.integers(-128, 128, size=(h, 128)).astype(np.int8)
    w = rng.integers(-128, 128, size=h).astype(np.int8)
    keys = rng.integers(-128, 128, size=(n, 128)).astype(np.int8)
    want = []
    for t in range(n):
        tot = 0
        for hh in range(h):
            dot = 0
            for d in range(128):
                dot += int(q[hh, d]) * int(keys[t, d])
            tot += int(w[hh]) * max(0, dot)
        want.append(tot)
    assert indexer.scores(q, w, keys).tolist() == want


def test_scores_all_positive_dots_collapse():
    # when every q_h . k is positive, sum_h w_h relu(q_h . k) = (sum_h w_h q_h) . k
    rng = np.random.default_rng(4)
    q = rng.integers(1, 128, size=(6, 128)).astype(np.int8)
    k = rng.integers(1, 128, size=(9, 128)).astype(np.int8)
    w = rng.integers(1, 17, size=6).astype(np.int8)
    collapsed = k.astype(np.int64) @ (w.astype(np.int64) @ q.astype(np.int64))
    assert np.array_equal(indexer.scores(q, w, k), collapsed)


def test_scores_single_head_unit_weight_is_relu_dot():
    q = np.zeros((1, 128), np.int8); q[0, :3] = [1, -2, 3]
    k = np.zeros((3, 128), np.int8)
    k[0, :3] = [1, 1, 1]      # 1 - 2 + 3 = 2
    k[1, :3] = [0, 5, 0]      # -10 -> 0
    k[2, :3] = [4, 0, 4]      # 16
    assert indexer.scores(q, np.ones(1, np.int8), k).tolist() == [2, 0, 16]


# ----------------------------------------------------------------------------
# top-K
# ----------------------------------------------------------------------------
def _brute_topk(s, k):
    s = list(int(x) for x in s)
    chosen = []
    alive = set(range(len(s)))
    for _ in range(min(k, len(s))):
        best = None
        for t in sorted(alive):
            if best is None or s[t] > s[best]:
                best = t
        chosen.append(best)
        alive.remove(best)
    return sorted(chosen) + [-1] * (k - len(chosen))


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 80))
    s = rng.integers(0, 6, size=n).astype(np.int64)      # heavy ties
    k = int(rng.integers(1, 40))
    assert indexer.topk(s, k).tolist() == _brute_topk(s, k)


def test_topk_all_zero_takes_lowest_tokens():
    assert indexer.topk(np.zeros(100, np.int64), 16).tolist() == list(range(16))


def test_topk_short_context_pads():
    out = indexer.topk(np.array([5, 1, 9], np.int64), 6)
    assert out.tolist() == [0, 1, 2, -1, -1, -1]


def test_topk_threshold_property():
    rng = np.random.default_rng(7)
    s = rng.integers(0, 1 << 40, size=3000).astype(np.int64)
    sel = indexer.topk(s, 100)
    mask = np.zeros(3000, bool); mask[sel] = True
    assert s[mask].min() > s[~mask].max()


# ----------------------------------------------------------------------------
# resolver
# ----------------------------------------------------------------------------
def _sel(ranges):
    out = []
    for lo, hi in ranges:
        out.extend(range(lo, hi))
    return np.array([out], np.int32)


def test_resolver_hand_worked_sequence():
    g = _load("resolver_hand.json")
    bt = np.array(g["block_table"], np.int32)
    hot = resolver.HotState()
    hot.lease(g["hot_pages"])
    for step, st in enumerate(g["steps"]):
        sel = _sel(st["select"])
        res = resolver.resolve(sel, bt, hot, step)
        pos = {int(t): i for i, t in enumerate(sel[0])}
        for tok, (kind, slot, row, ev) in st["expect"].items():
            i = pos[int(tok)]
            got = [int(res.kind[0, i]), int(res.slot[0, i]), int(res.row_ids[0, i]), int(res.evicted[0, i])]
            assert got == [kind, slot, row, ev], (step, tok, got)
        assert len(res.misses) == st["n_miss"]
        assert res.n_hit == st["n_hit"] and res.n_resident == st["n_resident"]


def test_resolver_release_then_lease_again():
    """Request end empties the hot buffer; a later lease starts from empty slots
    (hand-worked fixture, tests/golden/resolver_release_hand.json)."""
    g = _load("resolver_release_hand.json")
    bt = np.array(g["block_table"], np.int32)
    hot = resolver.HotState()
    for act in g["actions"]:
        if "lease" in act:
            hot.lease(act["lease"])
        elif act.get("release"):
            hot.release()
            assert hot.pages == [] and hot.tok2slot == {}
        else:
            sel = _sel(act["select"])
            res = resolver.resolve(sel, bt, hot, act["step"])
            pos = {int(t): i for i, t in enumerate(sel[0])}
            for tok, (kind, slot, row, ev) in act["expect"].items():
                i = pos[int(tok)]
                got = [int(res.kind[0, i]), int(res.slot[0, i]), int(res.row_ids[0, i]), int(res.evicted[0, i])]
                assert got == [kind, slot, row, ev], (act["step"], tok, got)
            assert len(res.misses) == act["n_miss"]
            assert res.n_hit == act["n_hit"] and res.n_resident == act["n_resident"]
        if "slots" in act:
            assert len(hot.stamp) == len(hot.slot_token) == act["slots"]
        # no token holds a slot twice and every map entry points back at its token
        assert all(hot.slot_token[v] == t for t, v in hot.tok2slot.items())


def test_resolver_capacity_error():
    bt = np.array([-1, -1], np.int32)
    hot = resolver.HotState()
    hot.lease([3])
    with pytest.raises(resolver.CapacityError):
        resolver.resolve(np.arange(65, dtype=np.int32)[None], bt, hot, 0)


def test_resolver_fully_resident_changes_nothing():
    bt = np.arange(8, dtype=np.int32) + 100
    hot = resolver.HotState()
    hot.lease([1])
    sel = np.array([[0, 5, 77, 300, 511, -1]], np.int32)
    res = resolver.resolve(sel, bt, hot, 0)
    assert res.misses == [] and res.n_hit == 0 and res.n_resident == 5
    assert res.row_ids[0].tolist() == [6400, 6405, 101 * 64 + 13, 104 * 64 + 44, 107 * 64 + 63, -1]
    assert hot.stamp == [-1] * 64 and hot.tok2slot == {}


def test_resolver_mtp_union_resolves_once():
    bt = np.array([-1, -1], np.int32)
    hot = resolver.HotState()
    hot.lease([9, 4])
    sel = np.array([[3, 10, 70], [10, 70, 71]], np.int32)
    res = resolver.resolve(sel, bt, hot, 0)
    # union {3, 10, 70, 71} misses once each, in ascending token order, slots 0..3
    assert [t for t, _ in res.misses] == [3, 10, 70, 71]
    assert res.slot.tolist() == [[0, 1, 2], [1, 2, 3]]
    assert res.row_ids.tolist() == [[576, 577, 578], [577, 578, 579]]


def test_replay_follows_the_hand_worked_sequence_and_changes_nothing():
    import copy
    g = _load("resolver_hand.json")
    bt = np.array(g["block_table"], np.int32)
    hot = resolver.HotState()
    hot.lease(g["hot_pages"])
    for step, st in enumerate(g["steps"]):
        sel = _sel(st["select"])
        resolver.resolve(sel, bt, hot, step)
        before = copy.deepcopy(hot)
        rows = resolver.replay(sel, bt, hot)
        pos = {int(t): i for i, t in enumerate(sel[0])}
        for tok, (_, _, row, _) in st["expect"].items():
            assert int(rows[0, pos[int(tok)]]) == row, (step, tok)
        assert hot == before     # no stamp refreshed, no slot reassigned


def test_replay_of_an_unresolved_or_evicted_token_is_an_error():
    g = _load("resolver_hand.json")
    bt = np.array(g["block_table"], np.int32)
    hot = resolver.HotState()
    hot.lease(g["hot_pages"])
    with pytest.raises(resolver.NotResolvedError):      # nothing resolved yet
        resolver.replay(np.array([[70]], np.int32), bt, hot)
    assert resolver.replay(np.array([[0, 200, -1]], np.int32), bt, hot).tolist() == [[640, 712, -1]]
    for step in range(2):                                # step 1 evicts token 96 (fixture)
        resolver.resolve(_sel(g["steps"][step]["select"]), bt, hot, step)
    with pytest.raises(resolver.NotResolvedError):
        resolver.replay(np.array([[96]], np.int32), bt, hot)


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------
def _rand_rows(rng, n):
    x = W.bf16_bits_to_f32(W.round_to_bf16_bits(rng.standard_normal((n, 576), dtype=np.float32)))
    return W.quantise_rows(x)


def _dense_loop_attention(qf, kv, mask, sm_scale):
    """Dense masked attention over ALL rows, masked-out rows weighted 0 (plain loops)."""
    H, n = qf.shape[0], kv.shape[0]
    o = np.zeros((H, 512))
    lse = np.zeros(H)
    for h in range(H):
        z = [sm_scale * float(np.dot(qf[h], kv[t])) if mask[t] else -math.inf for t in range(n)]
        m = max(z)
        e = [math.exp(v - m) if v != -math.inf else 0.0 for v in z]
        tot = sum(e)
        for t in range(n):
            if e[t]:
                o[h] += (e[t] / tot) * kv[t, :512]
        lse[h] = m + math.log(tot)
    return o, lse


def test_sparse_equals_dense_masked():
    rng = np.random.default_rng(5)
    n, H = 40, 3
    pool = _rand_rows(rng, n)
    q = W.round_to_bf16_bits(rng.standard_normal((H, 576), dtype=np.float32))
    sel = np.sort(rng.choice(n, size=13, replace=False))
    ids = np.concatenate([sel, [-1, -1]]).astype(np.int32)
    o, lse = attention.sparse_mla_decode(q, ids, pool, 1 / 24)
    mask = np.zeros(n, bool); mask[sel] = True
    o2, lse2 = _dense_loop_attention(formats.bf16_to_f64(q), formats.dequant_rows(pool), mask, 1 / 24)
    assert np.allclose(o, o2, rtol=1e-12, atol=1e-13) and np.allclose(lse, lse2, rtol=1e-13)


def test_topk_covering_context_equals_full_dense_attention():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(6)
    n, H = 30, 4
    pool = _rand_rows(rng, n)
    q = W.round_to_bf16_bits(rng.standard_normal((H, 576), dtype=np.float32))
    ids = indexer.topk(np.zeros(n, np.int64), 64)   # K >= L selects every token
    o, lse = attention.sparse_mla_decode(q, ids, pool, 0.05)
    kv = formats.dequant_rows(pool)
    z = 0.05 * formats.bf16_to_f64(q) @ kv.T
    p = scipy_special.softmax(z, axis=1)
    assert np.allclose(o, p @ kv[:, :512], rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, scipy_special.logsumexp(z, axis=1), rtol=1e-13)


def test_uniform_rows_give_that_row():
    rng = np.random.default_rng(8)
    row = _rand_rows(rng, 1)
    pool = np.repeat(row, 10, axis=0)
    q = W.round_to_bf16_bits(rng.standard_normal((2, 576), dtype=np.float32))
    o, lse = attention.sparse_mla_decode(q, np.arange(10, dtype=np.int32), pool, 0.1)
    v = formats.dequant_rows(row)[0, :512]
    assert np.allclose(o, np.broadcast_to(v, o.shape), rtol=1e-12, atol=1e-14)
    z = 0.1 * formats.bf16_to_f64(q) @ formats.dequant_rows(row)[0]
    assert np.allclose(lse, z + math.log(10), rtol=1e-12)


def test_one_hot_dominance():
    rng = np.random.default_rng(9)
    pool = _rand_rows(rng, 12)
    kv = formats.dequant_rows(pool)
    target = 7
    qf = kv[target] * 50.0                       # q . k_target dwarfs the rest
    q = W.round_to_bf16_bits(qf[None].astype(np.float32))
    o, _ = attention.sparse_mla_decode(q, np.arange(12, dtype=np.int32), pool, 1.0)
    assert np.allclose(o[0], kv[target, :512], atol=1e-9)


def test_single_row():
    rng = np.random.default_rng(10)
    pool = _rand_rows(rng, 3)
    q = W.round_to_bf16_bits(rng.standard_normal((1, 576), dtype=np.float32))
    o, lse = attention.sparse_mla_decode(q, np.array([-1, 2, -1], np.int32), pool, 0.3)
    kv = formats.dequant_rows(pool[2:3])[0]
    assert np.array_equal(o[0], kv[:512])
    assert np.isclose(lse[0], 0.3 * float(formats.bf16_to_f64(q)[0] @ kv), rtol=1e-13)


# ----------------------------------------------------------------------------
# closed forms printed by the pages
# ----------------------------------------------------------------------------
def _close(got, ent):
    v = ent["value"]
    if "rel_tol" in ent:
        return abs(got - v) <= ent["rel_tol"] * abs(v)
    if "abs_tol" in ent:
        return abs(got - v) <= ent["abs_tol"]
    return got == v


def test_closed_forms_match_pages():
    g = _load("closed_forms.json")
    cf = closed_forms
    assert _close(cf.row_bytes(), g["fp8_ds_mla_row_bytes"])
    assert _close(cf.bytes_per_selected_row(), g["selected_row_bytes"])
    assert _close(2048 * cf.bytes_per_selected_row(), g["query_bytes_rows_2048"])
    assert _close(cf.q_o_bytes_per_head(), g["q_o_bytes_per_head"])
    assert _close(cf.flops_per_row_per_head(), g["flops_per_row_per_head"])
    assert _close(cf.query_flops(8) / 1e6, g["heads8_mflops"])
    assert _close(cf.query_bytes(8) / 1e6, g["heads8_mbytes"])
    assert _close(cf.flops_per_byte(8), g["heads8_flops_per_byte"])
    assert _close(cf.query_flops(64) / 1e6, g["heads64_mflops"])
    assert _close(cf.query_bytes(64) / 1e6, g["heads64_mbytes"])
    assert _close(cf.flops_per_byte(64), g["heads64_flops_per_byte"])
    e = g["h200_ridge_flops_per_byte"]
    assert _close(cf.ridge_flops_per_byte(e["tflops"], e["tbps"]), e)
    assert _close(cf.kv_bytes_per_token(), g["kv_bytes_per_token"])
    e = g["kv_gib_per_1m_tokens"]
    assert _close(cf.kv_bytes_per_token() * e["tokens"] / 2 ** 30, e)
    assert _close(cf.kv_bytes_per_token() * 2 ** 20 / 2 ** 30 / 8, g["dcp8_gib_per_gpu"])
    assert _close(128 + 4, g["indexer_key_bytes"])


def test_workload_rows_have_the_page_row_size():
    cfg = W.named_config("ctx1m")
    # 1M tokens x 656 B per sparse layer is about 0.69 GB
    assert abs(1048576 * W.ROW_BYTES / 1e9 - 0.69) < 0.005
    assert W.ROW_BYTES == closed_forms.row_bytes()
    assert cfg.hot_rows == 2 * cfg.topk
    assert W.named_config("batch32").hot_rows == (3 + 2) * 2048


# ----------------------------------------------------------------------------
# FP8 indexer keys
# ----------------------------------------------------------------------------
def test_fp8_scores_equal_the_exact_integer_scores_on_small_integers():
    # integers of magnitude <= 16 are exact in e4m3; with unit scales the FP8 score
    # must be the exact int64 score of the integer path (pinned above)
    rng = np.random.default_rng(11)
    q = rng.integers(-16, 17, size=(8, 128))
    k = rng.integers(-16, 17, size=(300, 128))
    w = rng.integers(1, 17, size=8)
    ref = indexer.scores(q.astype(np.int8), w.astype(np.int8), k.astype(np.int8))
    got = indexer.scores_fp8(W.encode_e4m3(q.astype(np.float32)), w.astype(np.float32),
                             W.encode_e4m3(k.astype(np.float32)), np.ones(300, np.float32))
    assert np.array_equal(got, ref.astype(np.float64))


def test_fp8_scores_scale_with_the_key_scale_and_ignore_negative_dots():
    rng = np.random.default_rng(12)
    qc = W.encode_e4m3(rng.standard_normal((4, 128)).astype(np.float32))
    kc = W.encode_e4m3(rng.standard_normal((50, 128)).astype(np.float32))
    w = rng.standard_normal(4).astype(np.float32)
    s1 = indexer.scores_fp8(qc, w, kc, np.ones(50, np.float32))
    s3 = indexer.scores_fp8(qc, w, kc, np.full(50, 0.375, np.float32))
    assert np.allclose(s3, 0.375 * s1, rtol=0, atol=1e-12)
    # a key opposite to every query row scores 0 whatever the weights
    qpos = np.full((4, 128), 0x38, np.uint8)    # e4m3 +1.0
    neg = np.full((1, 128), 0xB8, np.uint8)     # e4m3 -1.0
    assert np.all(indexer.scores_fp8(qpos, w, neg, np.ones(1, np.float32)) == 0.0)


def test_topk_real_breaks_ties_toward_the_lower_token():
    s = np.array([0.5, 2.0, 2.0, -1.0, 2.0, 0.5])
    assert indexer.topk_real(s, 4).tolist() == [0, 1, 2, 4]
    assert indexer.topk_real(s, 8).tolist() == [0, 1, 2, 3, 4, 5, -1, -1]
