"""Capacity report: how many requests of a given context fit in a KV budget, all
resident versus with Hybrid HiSparse, and the host pool HiSparse then needs.

"vLLM introduces Hybrid HiSparse hybrid sparse offloading for GLM 5.3" (vLLM blog
Part 1), section "Estimate what your configuration gains": a calculator compares
plain GPU-resident KV with hybrid sparse offload on the same HBM, and reports the
smallest HiSparse host pool that keeps host memory from limiting the concurrency
the GPU-side indexer and hot buffers allow. Its qualitative shape is on the page.
Each hot buffer is a fixed GPU cost per request, so plain residency fits more
requests at short contexts, and HiSparse more at long ones. The note under the
calculator sizes a hot buffer with MTP at (num_speculative_tokens + 2) x top-K.

The page prints no formula; this module restates the comparison from the byte
layout of this pool (one page index across every sparse layer's KV tensor):
  plain     per request: pages(L) x 64 x (row x sparse layers + key x indexer layers + extra)
  HiSparse  per request: pages(L) x 64 x (key x indexer layers + extra)       index keys stay resident
                         + tail pages x 64 x row x sparse layers              the tail is never evicted
                         + groups x hot pages x 64 x row x sparse layers      hot pages are pool pages
  host pool for n requests: n x pages(L) x 64 x row x sparse layers           every page materialised
with pages(L) = ceil(L / 64). `extra` is per-token KV that stays resident in both
(the pages' MTP layer, 788 B). Planning estimates, like the page's: runtime
workspace, length skew and scheduling lower what is reached.
"""
from __future__ import annotations

import argparse
from dataclasses import dataclass
from typing import List

PAGE = 64


@dataclass(frozen=True)
class KVLayout:
    n_sparse_layers: int
    n_indexer_layers: int
    row_bytes: int = 656          # FP8 latent + 4 fp32 scales + bf16 rope
    key_bytes: int = 128          # int8 index key (132 with the pages' FP8 + scale)
    extra_bytes_per_token: int = 0

    def plain_bytes_per_token(self) -> int:
        return self.row_bytes * self.n_sparse_layers + self.key_bytes * self.n_indexer_layers + self.extra_bytes_per_token

    def resident_bytes_per_token(self) -> int:
        """Bytes per token HiSparse keeps on the GPU for the whole context."""
        return self.key_bytes * self.n_indexer_layers + self.extra_bytes_per_token


@dataclass(frozen=True)
class HiSparsePolicy:
    topk: int = 2048
    hot_factor: int = 2           # hot rows per (request, indexer group) = hot_factor x topk
    layers_per_indexer: int = 4
    tail_pages: int = 8

    def hot_pages(self) -> int:
        return -(-self.hot_factor * self.topk // PAGE)

    @staticmethod
    def mtp_hot_factor(num_speculative_tokens: int) -> int:
        return num_speculative_tokens + 2


def pages(context: int) -> int:
    return -(-context // PAGE)


def n_groups(layout: KVLayout, policy: HiSparsePolicy) -> int:
    return -(-layout.n_sparse_layers // policy.layers_per_indexer)


def plain_bytes_per_request(context: int, layout: KVLayout) -> int:
    return pages(context) * PAGE * layout.plain_bytes_per_token()


def hisparse_pool_pages_per_request(layout: KVLayout, policy: HiSparsePolicy, context: int) -> int:
    """Sparse-MLA pool pages a request holds under HiSparse: its tail and its hot buffers."""
    return min(pages(context), policy.tail_pages) + n_groups(layout, policy) * policy.hot_pages()


def hisparse_bytes_per_request(context: int, layout: KVLayout, policy: HiSparsePolicy) -> int:
    keys = pages(context) * PAGE * layout.resident_bytes_per_token()
    pool = hisparse_pool_pages_per_request(layout, policy, context) * PAGE * layout.row_bytes * layout.n_sparse_layers
    return keys + pool


def host_bytes_per_request(context: int, layout: KVLayout) -> int:
    return pages(context) * PAGE * layout.row_bytes * layout.n_sparse_layers


def crossover_context(layout: KVLayout, policy: HiSparsePolicy) -> float:
    """Context above which HiSparse fits more requests than plain residency, with
    per-request costs taken as continuous in L (page rounding ignored)."""
    fixed = (policy.tail_pages + n_groups(layout, policy) * policy.hot_pages()) * PAGE * layout.row_bytes \
        * layout.n_sparse_layers
    slope = layout.plain_bytes_per_token() - layout.resident_bytes_per_token()
    return fixed / slope


@dataclass
class CapacityRow:
    context: int
    plain: int                    # concurrent requests, all KV resident
    hisparse: int                 # concurrent requests with HiSparse, host pool unlimited
    gain: float
    host_pool_bytes: int          # smallest host pool for `hisparse` requests


def report(kv_budget_bytes: int, contexts: List[int], layout: KVLayout, policy: HiSparsePolicy) -> List[CapacityRow]:
    rows = []
    for L in contexts:
        plain = kv_budget_bytes // plain_bytes_per_request(L, layout)
        hs = kv_budget_bytes // hisparse_bytes_per_request(L, layout, policy)
        rows.append(CapacityRow(L, int(plain), int(hs), (hs / plain) if plain else float("inf"),
                                int(hs) * host_bytes_per_request(L, layout)))
    return rows


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description="HiSparse capacity report from the pool's byte layout")
    ap.add_argument("--kv-gib", type=float, default=100.0, help="HBM given to KV, GiB")
    ap.add_argument("--sparse-layers", type=int, default=78)
    ap.add_argument("--indexer-layers", type=int, default=21)
    ap.add_argument("--key-bytes", type=int, default=132)
    ap.add_argument("--extra-bytes", type=int, default=788, help="resident KV per token outside the sparse layers")
    ap.add_argument("--topk", type=int, default=2048)
    ap.add_argument("--layers-per-indexer", type=int, default=4)
    ap.add_argument("--num-speculative-tokens", type=int, default=0)
    ap.add_argument("--tail-pages", type=int, default=8)
    ap.add_argument("--contexts", default="8192,32768,131072,262144,1048576")
    a = ap.parse_args(argv)
    layout = KVLayout(a.sparse_layers, a.indexer_layers, key_bytes=a.key_bytes, extra_bytes_per_token=a.extra_bytes)
    hot = HiSparsePolicy.mtp_hot_factor(a.num_speculative_tokens) if a.num_speculative_tokens else 2
    policy = HiSparsePolicy(a.topk, hot, a.layers_per_indexer, a.tail_pages)
    budget = int(a.kv_gib * (1 << 30))
    print(f"KV budget {a.kv_gib} GiB; plain {layout.plain_bytes_per_token()} B/token; HiSparse resident "
          f"{layout.resident_bytes_per_token()} B/token + {hisparse_pool_pages_per_request(layout, policy, 1 << 30)} "
          f"pool pages per request; crossover ~{crossover_context(layout, policy):.0f} tokens")
    print(f"{'context':>10} {'plain':>8} {'HiSparse':>9} {'gain':>7} {'host pool GiB':>14}")
    for r in report(budget, [int(x) for x in a.contexts.split(",")], layout, policy):
        print(f"{r.context:>10} {r.plain:>8} {r.hisparse:>9} {r.gain:>7.2f} {r.host_pool_bytes / (1 << 30):>14.1f}")


if __name__ == "__main__":
    main()
