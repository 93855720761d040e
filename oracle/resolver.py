"""Residency resolution of a top-K selection (the fused resolver).

"vLLM Part 1", section "How it works", hybrid residency: a fused kernel resolves
the top-K; resident tokens are read in place, hot tokens are read and have their
LRU entry refreshed, and a miss copies a single row from pinned host memory into
an LRU slot. Hot-buffer pages are ordinary KV blocks leased from the same pool,
and the resolver hands the attention HMA row ids (pool page * 64 + offset) for
resident and hot rows alike. With MTP the verification tokens of a request are
resolved together ("the hot buffer must hold all verification tokens at once").

Readings where the pages are silent (one hot buffer per request and indexer
group; deterministic LRU):
  U = ascending union of the selected tokens of the request's query tokens.
  For t in U, page p = t // 64:
    block_table[p] >= 0          -> RESIDENT, row = block_table[p] * 64 + t % 64
    t has a hot slot             -> HIT, stamp[slot] = step
    otherwise                    -> MISS
  Victims: leased slots whose stamp is not this step, ordered by (stamp, slot)
  ascending (empty slots carry stamp -1, so free slots go first). Misses, in
  ascending token order, take victims in that order; the victim's old token
  loses its slot; the slot gets the token and stamp = step, and host row t of
  every layer of the group is copied into the slot's pool row.
  More misses than victims is a capacity error.
"""
from dataclasses import dataclass, field
from typing import Dict, List

import numpy as np

PAGE = 64
PAD, RESIDENT, HIT, MISS = 0, 1, 2, 3


class CapacityError(RuntimeError):
    pass


class HostMissingError(RuntimeError):
    pass


@dataclass
class HotState:
    pages: List[int] = field(default_factory=list)
    slot_token: List[int] = field(default_factory=list)
    stamp: List[int] = field(default_factory=list)
    tok2slot: Dict[int, int] = field(default_factory=dict)

    def lease(self, pages):
        for pg in pages:
            self.pages.append(int(pg))
            self.slot_token.extend([-1] * PAGE)
            self.stamp.extend([-1] * PAGE)

    def release(self):
        self.pages.clear()
        self.slot_token.clear()
        self.stamp.clear()
        self.tok2slot.clear()

    def slot_row(self, slot: int) -> int:
        return self.pages[slot // PAGE] * PAGE + slot % PAGE


@dataclass
class Resolution:
    row_ids: np.ndarray        # [T, K] int32
    kind: np.ndarray           # [T, K] int32
    slot: np.ndarray           # [T, K] int32 (-1 unless HIT / MISS)
    evicted: np.ndarray        # [T, K] int32 (old token of a MISS victim slot, else -1)
    misses: List[tuple]        # (token, slot) in assignment order
    n_resident: int
    n_hit: int


def resolve(topk_rows: np.ndarray, block_table: np.ndarray, hot: HotState, step: int) -> Resolution:
    topk_rows = np.asarray(topk_rows)
    U = sorted(set(int(t) for t in topk_rows.ravel() if t >= 0))
    info = {}
    misses = []
    n_res = n_hit = 0
    for t in U:
        p = t // PAGE
        if block_table[p] >= 0:
            info[t] = (RESIDENT, -1, int(block_table[p]) * PAGE + t % PAGE, -1)
            n_res += 1
        elif t in hot.tok2slot:
            s = hot.tok2slot[t]
            hot.stamp[s] = step
            info[t] = (HIT, s, hot.slot_row(s), -1)
            n_hit += 1
        else:
            misses.append(t)
    if misses:
        victims = sorted((s for s in range(len(hot.stamp)) if hot.stamp[s] != step),
                         key=lambda s: (hot.stamp[s], s))
        if len(misses) > len(victims):
            raise CapacityError(f"{len(misses)} misses, {len(victims)} victim slots")
    assigned = []
    for i, t in enumerate(misses):
        v = victims[i]
        old = hot.slot_token[v]
        if old >= 0:
            del hot.tok2slot[old]
        hot.slot_token[v] = t
        hot.stamp[v] = step
        hot.tok2slot[t] = v
        info[t] = (MISS, v, hot.slot_row(v), old)
        assigned.append((t, v))
    shape = topk_rows.shape
    row_ids = np.full(shape, -1, np.int32)
    kind = np.zeros(shape, np.int32)
    slot = np.full(shape, -1, np.int32)
    evicted = np.full(shape, -1, np.int32)
    for idx in np.ndindex(*shape):
        t = int(topk_rows[idx])
        if t < 0:
            continue
        k, s, row, old = info[t]
        row_ids[idx], kind[idx], slot[idx], evicted[idx] = row, k, s, old
    return Resolution(row_ids, kind, slot, evicted, assigned, n_res, n_hit)


class NotResolvedError(RuntimeError):
    pass


def replay(topk_rows: np.ndarray, block_table: np.ndarray, hot: HotState) -> np.ndarray:
    """Replay of a resolver plan ("vLLM Part 1", section "Composing with the rest of
    vLLM": speculative decoding works through per-step replayable resolver plans
    that share the request's hot state).

    Reading: a replay maps each selected token to the row the last resolve gave it,
    from the residency maps as they stand, and changes nothing: no stamp is
    refreshed, no victim is taken. A resident page gives its row in place, a token
    holding a hot slot gives that slot's row; a token that is neither was not
    resolved and is an error. Pads (-1) stay -1."""
    topk_rows = np.asarray(topk_rows)
    row_ids = np.full(topk_rows.shape, -1, np.int32)
    for idx in np.ndindex(*topk_rows.shape):
        t = int(topk_rows[idx])
        if t < 0:
            continue
        p = t // PAGE
        if block_table[p] >= 0:
            row_ids[idx] = int(block_table[p]) * PAGE + t % PAGE
        elif t in hot.tok2slot:
            row_ids[idx] = hot.slot_row(hot.tok2slot[t])
        else:
            raise NotResolvedError(f"token {t} is neither resident nor in the hot buffer")
    return row_ids
