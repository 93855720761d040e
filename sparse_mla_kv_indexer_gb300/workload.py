"""Seeded synthetic inputs for the sparse-MLA decode step.

This module draws random numbers and lays out bytes. It holds none of the
method's arithmetic: no indexer scoring, no top-K, no residency resolution, no
FP8 decoding, no attention and no page copies. Both the CPU oracle and the CUDA
path consume exactly the arrays produced here, so every comparison between the
two runs on identical inputs.

Row layout of one sparse-MLA KV row (656 bytes, the ``fp8_ds_mla`` size given in
the footnotes of "vLLM Part 2: PCP/DCP and P/D deployment with HiSparse"):

    bytes [0, 512)    512 x FP8 e4m3 latent values
    bytes [512, 528)  4 x fp32 scale, one per 128 latent values (little endian)
    bytes [528, 656)  64 x bf16 rope values (little endian)

The pages give only the 656-byte total; this split is the one reading in which
512 FP8 latent dims with per-128 fp32 scales and 64 bf16 rope dims add up to
exactly 656 bytes.

Quantisation of the synthetic KV (an input-synthesis step, done once here):
scale = amax(group) / 448 (1 when the group is all zero), value / scale rounded
to the nearest e4m3 code with ties to even, saturated at +-448.

Index keys and index queries are int8 drawn from round(N(0, 32^2)) clamped to
[-127, 127]; head weights are integers U[1, 16]; attention queries are bf16
N(0, 1). Planted clusters (config shapes for 128K, batch and 1M runs): spans of
512 tokens carry a +-96 bias along a random sign direction, and each quarter of
the index heads is biased toward one target cluster, so top-K sets overlap from
step to step. Query drift: q_t = clamp(q_{t-1} + round(N(0, 4^2))).
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Dict, List, Tuple

import numpy as np

PAGE = 64
ROW_BYTES = 656
LATENT = 512
ROPE = 64
QK_DIM = LATENT + ROPE
IDX_DIM = 128
GROUP = 128
SCALE_OFF = LATENT
ROPE_OFF = LATENT + 16
KV_CHUNK = 1 << 15


# --------------------------------------------------------------------------
# Configurations
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class WorkloadConfig:
    """Shapes and structure of one synthetic decode workload."""

    name: str
    config_id: int
    n_requests: int
    ctx_len: Tuple[int, ...]          # context L per request at step 0 (includes the step-0 tokens)
    n_heads: int = 64                 # attention query heads H
    n_idx_heads: int = 64             # index heads H_i
    topk: int = 2048                  # K
    n_layers: int = 4                 # sparse-MLA layers
    layers_per_indexer: int = 4       # IndexShare group size
    steps: int = 8
    t_q: int = 1                      # query tokens per request per step
    accept: int = 1                   # positions committed per step
    tail_pages: int = 8               # last pages that are never evicted
    host_only_frac: float = 0.75      # fraction of non-tail prefix pages that start host-only
    hot_rows: int = 4096              # hot-buffer capacity per (request, group)
    n_clusters: int = 0
    cluster_len: int = 512
    cluster_bias: int = 96
    drift_sigma: float = 4.0
    jump_prob: float = 0.0
    pool_slack_pages: int = 16        # free pool pages beyond what setup occupies
    prefix_reuse: Tuple[int, ...] = ()  # requests starting with placeholders + 1 hot page
    pressure: bool = False            # pool holds only the setup residency + slack: growth evicts
    idx_fp8: bool = False             # index keys as 128 e4m3 values + an fp32 scale (132-byte record)
    seed: int = 0
    # Multi-turn histories (0 turns: one open-ended decode). A request's history is
    # `turns` turns of `turn_steps` decode steps each; every turn after the first
    # starts by writing `turn_input` new input positions (written like a prefill, not
    # decoded). `history_step[r]` is where request r stands in its history at step 0;
    # a request whose history is done ends and leaves the batch.
    turns: int = 0
    turn_input: int = 0
    turn_steps: int = 0
    history_step: Tuple[int, ...] = ()

    @property
    def n_groups(self) -> int:
        return -(-self.n_layers // self.layers_per_indexer)

    def group_layers(self, g: int) -> List[int]:
        lo = g * self.layers_per_indexer
        return list(range(lo, min(self.n_layers, lo + self.layers_per_indexer)))

    def events(self, r: int) -> List[Tuple[int, int]]:
        """(turn-input positions written, decode positions committed) of request r at
        each step of the run, while it lives: a request that ends stops early."""
        if self.turns == 0:
            return [(0, self.accept)] * self.steps
        out = []
        for s in range(self.steps):
            h = self.history_step[r] + s
            if h >= self.turns * self.turn_steps:
                break
            boundary = s > 0 and h % self.turn_steps == 0
            out.append((self.turn_input if boundary else 0, self.accept))
        return out

    def final_len(self, r: int) -> int:
        """Highest position written by the run, plus one."""
        committed = self.ctx_len[r] - self.t_q
        end = committed
        for inp, acc in self.events(r):
            committed += inp
            end = committed + self.t_q
            committed += acc
        return end

    def max_ctx(self) -> int:
        m = max(self.final_len(r) for r in range(self.n_requests))
        return -(-m // PAGE) * PAGE

    def request_seed(self, r: int) -> int:
        return 1000 * self.config_id + r + 1_000_003 * self.seed


def _loguniform_lengths(n: int, lo: int, hi: int, seed: int) -> Tuple[int, ...]:
    rng = np.random.default_rng(np.random.SeedSequence([seed, 77]))
    v = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
    return tuple(int(x) for x in np.round(v))


def _history_context(first: int, turn_input: int, turn_steps: int, accept: int, h: int) -> int:
    """Committed positions of a multi-turn request after h decode steps of its history:
    the first turn's input, the input of every later turn begun, accept per step."""
    return first + (h // turn_steps) * turn_input + h * accept


def named_config(name: str) -> WorkloadConfig:
    """The workloads of the method's decode path, by name.

    tiny        1 request, L = 4,096, 16 heads, 1 indexer + 1 layer, K = 256
    ctx128k     1 request, L = 131,072, 64 heads, 4 layers / 1 indexer, K = 2,048
    batch32     32 requests, L log-uniform in [8K, 256K], MTP3 (4 query tokens, 3 accepted)
    ctx1m       1 request, L = 1,048,576, 8 layers / 2 indexers, only the last 16 pages resident
    multiturn   64 requests with 13-turn histories (74,160 first-turn tokens, +753 input and
                220 output tokens per turn), MTP3, 40 % pool, 25 % prefix-reuse requests;
                requests end when their histories do
    The small_* variants keep every structural feature at sizes the oracle finishes in seconds.
    """
    if name == "tiny":
        return WorkloadConfig(name, 1, 1, (4096,), n_heads=16, n_idx_heads=16, topk=256,
                              n_layers=1, layers_per_indexer=1, steps=8, tail_pages=4,
                              host_only_frac=0.5, hot_rows=512, pool_slack_pages=4)
    if name == "ctx128k":
        return WorkloadConfig(name, 2, 1, (131072,), steps=64, tail_pages=8,
                              host_only_frac=0.75, hot_rows=4096, n_clusters=32)
    if name == "batch32":
        return WorkloadConfig(name, 3, 32, _loguniform_lengths(32, 8192, 262144, 3), steps=32,
                              t_q=4, accept=3, tail_pages=8, host_only_frac=0.5,
                              hot_rows=(3 + 2) * 2048, n_clusters=32, pressure=True)
    if name == "ctx1m":
        return WorkloadConfig(name, 4, 1, (1048576,), n_layers=8, layers_per_indexer=4,
                              steps=128, tail_pages=16, host_only_frac=1.0, hot_rows=4096,
                              n_clusters=32, drift_sigma=1.0, jump_prob=0.1)
    if name == "multiturn":
        # 13-turn histories: a 74,160-token first turn, then +753 input tokens per turn;
        # 220 output tokens per turn decoded at MTP3 (74 steps of 3 accepted tokens).
        # The 48 ongoing requests stand at spread points of their histories, the 16
        # prefix-reuse requests early in their first turn.
        turn_steps, turns, first, inp = 74, 13, 74160, 753
        hist = tuple((r * 131 + 17) % (turns * turn_steps) if r < 48 else (r * 7) % turn_steps for r in range(64))
        ctx = tuple(_history_context(first, inp, turn_steps, 3, h) + 4 for h in hist)
        return WorkloadConfig(name, 5, 64, ctx, steps=74, t_q=4, accept=3,
                              tail_pages=8, host_only_frac=0.6, hot_rows=(3 + 2) * 2048,
                              n_clusters=32, prefix_reuse=tuple(range(48, 64)), pressure=True,
                              turns=turns, turn_input=inp, turn_steps=turn_steps, history_step=hist)
    # Reduced variants used by parity tests: same structure, fewer tokens.
    if name == "small_single":
        return WorkloadConfig(name, 12, 1, (16384,), steps=6, tail_pages=8,
                              host_only_frac=0.75, hot_rows=4096, n_clusters=16)
    if name == "small_batch":
        return WorkloadConfig(name, 13, 4, (5000, 9000, 3000, 12001), topk=512, steps=6, t_q=4,
                              accept=3, tail_pages=4, host_only_frac=0.5, hot_rows=(3 + 2) * 512,
                              n_clusters=8, pool_slack_pages=8, pressure=True)
    if name == "small_groups":
        return WorkloadConfig(name, 14, 1, (20000,), n_layers=8, layers_per_indexer=4, steps=6,
                              tail_pages=16, host_only_frac=1.0, hot_rows=4096, n_clusters=16,
                              drift_sigma=1.0, jump_prob=0.5)
    if name == "small_reuse":
        return WorkloadConfig(name, 15, 3, (6000, 7000, 6500), topk=512, steps=5, t_q=4, accept=3,
                              tail_pages=4, host_only_frac=0.4, hot_rows=(3 + 2) * 512,
                              n_clusters=8, prefix_reuse=(2,), pressure=True)
    if name == "small_multiturn":
        # 3-turn histories of 3 steps per turn and +100 input tokens per turn, so that
        # 8 steps cross five turn boundaries and end three requests (their pages go back
        # to the pool and are leased again by the others)
        turn_steps, turns, inp = 3, 3, 100
        hist = (0, 4, 7, 2)
        first = (5000, 6000, 3000, 4000)
        ctx = tuple(_history_context(first[r], inp, turn_steps, 3, hist[r]) + 4 for r in range(4))
        return WorkloadConfig(name, 17, 4, ctx, topk=512, steps=8, t_q=4, accept=3, tail_pages=4,
                              host_only_frac=0.5, hot_rows=(3 + 2) * 512, n_clusters=8, pool_slack_pages=64,
                              prefix_reuse=(3,), pressure=True, turns=turns, turn_input=inp,
                              turn_steps=turn_steps, history_step=hist)
    if name == "small_mtp":
        # 6 requests x 4 MTP tokens at top-K 2,048: enough query tokens for the
        # one-CTA-per-token attention; the shortest context is below K (pads)
        return WorkloadConfig(name, 18, 6, (1500, 2600, 4000, 5200, 7000, 9100), steps=4, t_q=4, accept=3,
                              tail_pages=4, host_only_frac=0.5, hot_rows=(3 + 2) * 2048, n_clusters=8)
    if name.endswith("_fp8"):   # the same shape with FP8 index keys
        return dataclasses.replace(named_config(name[:-4]), name=name, idx_fp8=True)
    if name == "short_ctx":
        # context shorter than K: every earlier token is selected, pads are -1
        return WorkloadConfig(name, 16, 2, (1500, 700), n_heads=16, n_idx_heads=16, topk=2048,
                              n_layers=1, layers_per_indexer=1, steps=3, t_q=2, accept=2,
                              tail_pages=2, host_only_frac=0.5, hot_rows=3 * 2048)
    raise KeyError(name)


CONFIG_NAMES = ("tiny", "ctx128k", "batch32", "ctx1m", "multiturn")


# --------------------------------------------------------------------------
# Element encodings used to synthesise inputs
# --------------------------------------------------------------------------
def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (a widening; used only to build inputs)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def encode_e4m3(v: np.ndarray) -> np.ndarray:
    """float32 -> FP8 e4m3 byte, round to nearest even, saturate to +-448.

    e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
    subnormal (m * 2^-9); the all-ones code 0x7F / 0xFF is NaN, so the largest
    finite magnitude is 1.75 * 2^8 = 448. Normal values are rounded on the
    binary32 bit pattern (keep 3 of 23 mantissa bits, ties to even, rebias the
    exponent from 127 to 7); magnitudes below 2^-6 are multiples of 2^-9.
    """
    v = np.ascontiguousarray(v, dtype=np.float32)
    b = v.view(np.uint32)
    sign = ((b >> np.uint32(31)).astype(np.uint8)) << np.uint8(7)
    a = b & np.uint32(0x7FFFFFFF)
    r = (a + np.uint32(0x7FFFF) + ((a >> np.uint32(20)) & np.uint32(1))) >> np.uint32(20)
    code_n = np.minimum(r.astype(np.int64) - (120 << 3), 0x7E)
    sub = a < np.uint32(0x3C800000)                     # |v| < 2^-6
    code_s = np.rint(np.abs(v).astype(np.float64) * 512.0).astype(np.int64)
    code = np.where(sub, code_s, code_n).astype(np.uint8)
    return code | sign


def quantise_rows(x: np.ndarray) -> np.ndarray:
    """[n, 576] float32 (bf16-exact) -> [n, 656] uint8 rows in the layout above."""
    n = x.shape[0]
    out = np.empty((n, ROW_BYTES), dtype=np.uint8)
    lat = x[:, :LATENT].reshape(n, LATENT // GROUP, GROUP)
    amax = np.abs(lat).max(axis=2)
    scale = np.where(amax > 0, amax.astype(np.float32) / np.float32(448.0), np.float32(1.0))
    scale = scale.astype(np.float32)
    q = lat / scale[:, :, None]
    out[:, :LATENT] = encode_e4m3(q.reshape(n, LATENT))
    out[:, SCALE_OFF:SCALE_OFF + 16] = scale.astype("<f4").view(np.uint8).reshape(n, 16)
    rope = round_to_bf16_bits(x[:, LATENT:])
    out[:, ROPE_OFF:] = rope.astype("<u2").view(np.uint8).reshape(n, 2 * ROPE)
    return out


# --------------------------------------------------------------------------
# The workload: static cache content and per-step queries
# --------------------------------------------------------------------------
def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(k) & 0xFFFFFFFF for k in key]))


@dataclass
class _Clusters:
    starts: np.ndarray      # [C] first token of each planted span
    dirs: np.ndarray        # [C, 128] +-1 directions


class Workload:
    """All inputs of a run: cache contents (KV rows and index keys by position),
    index queries and weights, attention queries, for every request and step."""

    def __init__(self, cfg: WorkloadConfig):
        self.cfg = cfg
        self._kv: Dict[Tuple[int, int], np.ndarray] = {}
        self._ik: Dict[Tuple[int, int], np.ndarray] = {}
        self._iq: Dict[Tuple[int, int], np.ndarray] = {}
        self._clusters: Dict[int, _Clusters] = {}

    # -- planted clusters (per request, shared by its indexer layers) --------
    def clusters(self, r: int) -> _Clusters:
        if r not in self._clusters:
            cfg = self.cfg
            rng = _rng(cfg.request_seed(r), 1)
            c = cfg.n_clusters
            prefix = cfg.ctx_len[r] - cfg.t_q
            if c == 0 or prefix < c * cfg.cluster_len:
                self._clusters[r] = _Clusters(np.zeros(0, np.int64), np.zeros((0, IDX_DIM), np.int64))
            else:
                seg = prefix // c
                slack = seg - cfg.cluster_len
                starts = np.arange(c, dtype=np.int64) * seg + rng.integers(0, slack + 1, size=c)
                dirs = rng.integers(0, 2, size=(c, IDX_DIM)).astype(np.int64) * 2 - 1
                self._clusters[r] = _Clusters(starts, dirs)
        return self._clusters[r]

    # -- KV rows --------------------------------------------------------------
    def kv_rows(self, r: int, layer: int) -> np.ndarray:
        """[final_len, 656] uint8: the KV row of every position of request r, layer.

        Rows are drawn in chunks of 32,768 positions, each chunk from its own
        seed, so chunks are generated in parallel and are independent of how
        long the run is."""
        key = (r, layer)
        if key not in self._kv:
            n = self.cfg.final_len(r)
            out = np.empty((n, ROW_BYTES), dtype=np.uint8)
            seed = self.cfg.request_seed(r)

            def fill(ci: int) -> None:
                lo = ci * KV_CHUNK
                hi = min(n, lo + KV_CHUNK)
                rng = _rng(seed, 2, layer, ci)
                x = rng.standard_normal((KV_CHUNK, QK_DIM), dtype=np.float32)[:hi - lo]
                x = bf16_bits_to_f32(round_to_bf16_bits(x))
                out[lo:hi] = quantise_rows(x)

            chunks = range(-(-n // KV_CHUNK))
            if len(chunks) > 1:
                with ThreadPoolExecutor(max_workers=min(len(chunks), os.cpu_count() or 1)) as ex:
                    list(ex.map(fill, chunks))
            else:
                for ci in chunks:
                    fill(ci)
            self._kv[key] = out
        return self._kv[key]

    # -- index keys -------------------------------------------------------------
    def idx_keys(self, r: int, il: int) -> np.ndarray:
        """[final_len, 128] int8 index key of every position."""
        key = (r, il)
        if key not in self._ik:
            cfg = self.cfg
            n = cfg.final_len(r)
            rng = _rng(cfg.request_seed(r), 3, il)
            k = np.rint(rng.standard_normal((n, IDX_DIM), dtype=np.float32) * 32.0).astype(np.int64)
            cl = self.clusters(r)
            for c in range(len(cl.starts)):
                s = int(cl.starts[c])
                k[s:s + cfg.cluster_len] += cfg.cluster_bias * cl.dirs[c]
            self._ik[key] = np.clip(k, -127, 127).astype(np.int8)
        return self._ik[key]

    def idx_keys_fp8(self, r: int, il: int):
        """FP8 form of the same keys: ([final_len, 128] e4m3 codes, [final_len] fp32
        scales), scale = amax / 448 per key (1 for an all-zero key)."""
        key = ("fp8", r, il)
        if key not in self._ik:
            k = self.idx_keys(r, il).astype(np.float32)
            amax = np.abs(k).max(axis=1)
            scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
            self._ik[key] = (encode_e4m3(k / scale[:, None]), scale)
        return self._ik[key]

    def idx_key_records_fp8(self, r: int, il: int) -> np.ndarray:
        """[final_len, 132] bytes: the e4m3 codes, then the scale (little-endian fp32)."""
        codes, scale = self.idx_keys_fp8(r, il)
        rec = np.empty((codes.shape[0], IDX_DIM + 4), np.uint8)
        rec[:, :IDX_DIM] = codes
        rec[:, IDX_DIM:] = scale.astype("<f4").view(np.uint8).reshape(-1, 4)
        return rec

    def idx_queries_fp8(self, r: int, il: int, step: int):
        """FP8 form of a step's index queries: ([t_q, H_i, 128] e4m3 codes, [t_q, H_i]
        fp32 weights); each head's scale amax / 448 is folded into its weight."""
        q = self.idx_queries(r, il, step).astype(np.float32)
        amax = np.abs(q).max(axis=2)
        qs = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
        w = (self.idx_weights(r, il).astype(np.float32)[None, :] * qs).astype(np.float32)
        return encode_e4m3(q / qs[:, :, None]), w

    def idx_weights(self, r: int, il: int) -> np.ndarray:
        """[H_i] int8 head weights, integers U[1, 16], fixed across steps."""
        rng = _rng(self.cfg.request_seed(r), 4, il)
        return rng.integers(1, 17, size=self.cfg.n_idx_heads).astype(np.int8)

    def _idx_query_chain(self, r: int, il: int) -> np.ndarray:
        """[steps * t_q, H_i, 128] int8: one index query per (step, query token)."""
        key = (r, il)
        if key not in self._iq:
            cfg = self.cfg
            rng = _rng(cfg.request_seed(r), 5, il)
            hi_ = cfg.n_idx_heads
            q = np.rint(rng.standard_normal((hi_, IDX_DIM)) * 32.0).astype(np.int64)
            cl = self.clusters(r)
            nq = len(cl.starts)
            targets = None
            quarter = np.arange(hi_) * 4 // hi_
            if nq >= 4:
                targets = rng.choice(nq, size=4, replace=False)
                q += cfg.cluster_bias * cl.dirs[targets[quarter]]
            q = np.clip(q, -127, 127)
            chain = []
            n = cfg.steps * cfg.t_q
            for i in range(n):
                if i > 0:
                    q = np.clip(q + np.rint(rng.standard_normal(q.shape) * cfg.drift_sigma).astype(np.int64),
                                -127, 127)
                    if targets is not None and i % cfg.t_q == 0 and cfg.jump_prob > 0:
                        if rng.random() < cfg.jump_prob:
                            a = int(rng.integers(0, 4))
                            new = int(rng.integers(0, nq))
                            sel = quarter == a
                            q[sel] = np.clip(q[sel] + cfg.cluster_bias * (cl.dirs[new] - cl.dirs[targets[a]]),
                                             -127, 127)
                            targets[a] = new
                chain.append(q.copy())
            self._iq[key] = np.stack(chain).astype(np.int8)
        return self._iq[key]

    def idx_queries(self, r: int, il: int, step: int) -> np.ndarray:
        """[t_q, H_i, 128] int8 index queries of request r at a step."""
        t = self.cfg.t_q
        return self._idx_query_chain(r, il)[step * t:(step + 1) * t]

    def attn_queries(self, r: int, layer: int, step: int) -> np.ndarray:
        """[t_q, H, 576] bf16 bit patterns (uint16), N(0, 1), fresh every step."""
        rng = _rng(self.cfg.request_seed(r), 6, layer, step)
        x = rng.standard_normal((self.cfg.t_q, self.cfg.n_heads, QK_DIM), dtype=np.float32)
        return round_to_bf16_bits(x)

    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(QK_DIM)
